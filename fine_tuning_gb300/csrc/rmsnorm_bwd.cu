// RMSNorm backward, plain form (the kernels are in rmsnorm_bwd.cuh); the
// residual-add form is instantiated in rmsnorm_add_bwd.cu.
#include "rmsnorm_bwd.cuh"

namespace ftk {

int64_t rmsnorm_bwd_partial_rows(int64_t T, const DeviceInfo &dev) {
  const int64_t cap = (int64_t)dev.sms * kMaxBlocksPerSm;
  return T < cap ? T : cap;
}

cudaError_t launch_rmsnorm_bwd(DType dt, bool vec, bool wide, const RmsNormBwdArgs &a,
                               const DeviceInfo &dev, cudaStream_t s) {
  if (a.dh) return launch_rmsnorm_add_bwd(dt, vec, wide, a, dev, s);
  return launch_bwd_form<false>(dt, vec, wide, a, dev, s);
}

}  // namespace ftk
