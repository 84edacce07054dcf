// RMSNorm backward with the pre-norm residual add fused in front: dx = dh +
// the norm's gradient at the stored h (the kernels are in rmsnorm_bwd.cuh).
#include "rmsnorm_bwd.cuh"

namespace ftk {

cudaError_t launch_rmsnorm_add_bwd(DType dt, bool vec, bool wide, const RmsNormBwdArgs &a,
                                   const DeviceInfo &dev, cudaStream_t s) {
  return launch_bwd_form<true>(dt, vec, wide, a, dev, s);
}

}  // namespace ftk
