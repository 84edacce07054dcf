// Host-side interface between the C ABI (ftk_api.cu) and the kernel
// translation units.  Arguments arrive here already validated; each launcher
// picks the kernel instance (storage type, index width, packet width, row
// plan) and launches it on the caller's stream.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace ftk {

enum class DType : int { F32 = 0, BF16 = 1 };

inline int dtype_bytes(DType t) { return t == DType::F32 ? 4 : 2; }

struct DeviceInfo {
  int device = 0;
  int sms = 0;            // streaming multiprocessors
  int max_smem_optin = 0;  // dynamic shared memory a CTA may opt into
};

// Cached per device; the only state the library keeps.
cudaError_t current_device_info(DeviceInfo *out);

// How one RMSNorm row is spread over threads: W warps per row, V packets of
// `pack` elements per thread, R rows per CTA.  `generic` = the row does not
// fit in registers and the CTA-per-row two-pass kernels are used instead.
struct RowPlan {
  int pack = 1;
  int W = 1, V = 1, R = 1;
  bool generic = false;
  int threads() const { return generic ? 256 : 32 * W * R; }
};
RowPlan plan_rmsnorm_row(int64_t H, int pack);

struct RmsNormFwdArgs {
  const void *x;
  int64_t ldx;
  const void *w;
  void *y;
  int64_t ldy;
  float *rstd;  // nullable
  int64_t T, H;
  float eps;
};
cudaError_t launch_rmsnorm_fwd(DType dt, bool vec, bool wide, const RmsNormFwdArgs &a,
                               const DeviceInfo &dev, cudaStream_t s);

struct RmsNormBwdArgs {
  const void *dy;
  int64_t lddy;
  const void *x;
  int64_t ldx;
  const void *w;
  const float *rstd;  // nullable: recompute
  void *dx;
  int64_t lddx;
  float *dw;
  float *ws;          // [ws_rows, H] fp32 partials
  int64_t ws_rows;
  int64_t T, H;
  float eps;
};
// Upper bound on the partial rows the backward kernel writes (any plan).
int64_t rmsnorm_bwd_partial_rows(int64_t T, const DeviceInfo &dev);
cudaError_t launch_rmsnorm_bwd(DType dt, bool vec, bool wide, const RmsNormBwdArgs &a,
                               const DeviceInfo &dev, cudaStream_t s);

struct SwigluFwdArgs {
  const void *g, *u;
  int64_t ld_gu;
  void *h;
  int64_t ld_h;
  int64_t T, I;
};
cudaError_t launch_swiglu_fwd(DType dt, bool vec, bool wide, const SwigluFwdArgs &a,
                              const DeviceInfo &dev, cudaStream_t s);

struct SwigluBwdArgs {
  const void *dh;
  int64_t ld_dh;
  const void *g, *u;
  int64_t ld_gu;
  void *dg, *du;
  int64_t ld_dgu;
  int64_t T, I;
};
cudaError_t launch_swiglu_bwd(DType dt, bool vec, bool wide, const SwigluBwdArgs &a,
                              const DeviceInfo &dev, cudaStream_t s);

constexpr int kRopeMaxHalf = 256;  // D <= 512

struct RopeArgs {
  void *q;
  int64_t ld_q;
  void *k;
  int64_t ld_k;
  const int32_t *cu;
  int32_t B;
  int64_t T;
  int32_t Hq, Hkv, D;
  double theta;
  bool backward;
};
cudaError_t launch_qk_rope(DType dt, bool vec, bool wide, const RopeArgs &a,
                           const DeviceInfo &dev, cudaStream_t s);

}  // namespace ftk
