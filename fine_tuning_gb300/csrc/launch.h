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

// Cached per device; with the status word below, the only state the
// library keeps.
cudaError_t current_device_info(DeviceInfo *out);

// Device address of the status word (bit kStatusWaitTimeout: a bounded
// wait in some kernel ran out); cached per device.
cudaError_t device_status_ptr(const DeviceInfo &dev, unsigned **out);
cudaError_t read_device_status(unsigned *flags, bool clear);
cudaError_t launch_wait_timeout_selftest(const DeviceInfo &dev, long long limit_cycles,
                                         cudaStream_t s);

// Launches `kernel` on `s` as a programmatic dependent of the previous
// kernel in the stream (see pdl_wait in common.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// SM clock cycles a pipeline wait may take before it gives up (~1 s).
constexpr long long kWaitLimitCycles = 2000000000LL;

// How one RMSNorm row is spread over threads: W warps per row, V packets of
// `pack` elements per thread, R rows per CTA.  `generic` = the row does not
// fit in registers and the CTA-per-row two-pass kernels are used instead.
struct RowPlan {
  int pack = 1;
  int W = 1, V = 1, R = 1;
  bool generic = false;
  int threads() const { return generic ? 256 : 32 * W * R; }
};
// W = ceil(packets / (32 * vmax)) warps per row (at most 8), then V packets
// per thread rounded up to 1, 2, 3, 4, 6 or 8.
RowPlan plan_rmsnorm_row(int64_t H, int pack, int vmax);

// The bulk-copy pipeline on top of a row plan: every row group owns a ring
// of S shared-memory stages, each holding `nbuf` rows (x, or x and dy).
// Shared memory layout: [R*S mbarriers][R*W float2 reduction slots]
// [R*S stages of stage_bytes], stages 128-byte aligned.  S = 0 means the
// pipeline does not fit and the register kernels are used.
struct StagedPlan {
  int S = 0;
  uint32_t row_bytes = 0, stage_bytes = 0;
  size_t off_red = 0, off_stage = 0, smem = 0;
};
StagedPlan plan_rmsnorm_staged(const RowPlan &p, int64_t H, int elem_bytes, int nbuf,
                               const DeviceInfo &dev);

// Resident CTAs per SM of `kernel` at this shape, capped at `cap` (cached).
// Also lifts the kernel's dynamic shared memory limit to the device maximum
// the first time it sees the kernel on a device.
int blocks_per_sm(const void *kernel, int threads, size_t smem, const DeviceInfo &dev, int cap);

struct RmsNormFwdArgs {
  const void *x;
  int64_t ldx;
  const void *w;
  void *y;
  int64_t ldy;
  float *rstd;  // nullable
  int64_t T, H;
  float eps;
  // residual add fused in front (h = x + res stored, norm of h); res null: plain norm
  const void *res = nullptr;
  int64_t ldr = 0;
  void *h = nullptr;
  int64_t ldh = 0;
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
  // residual add fused in front: x is the stored h, and dx = dh + norm backward;
  // dh null: plain norm
  const void *dh = nullptr;
  int64_t lddh = 0;
};
// Upper bound on the partial rows the backward kernel writes (any plan).
int64_t rmsnorm_bwd_partial_rows(int64_t T, const DeviceInfo &dev);
cudaError_t launch_rmsnorm_bwd(DType dt, bool vec, bool wide, const RmsNormBwdArgs &a,
                               const DeviceInfo &dev, cudaStream_t s);
// the dh != nullptr form (called by launch_rmsnorm_bwd)
cudaError_t launch_rmsnorm_add_bwd(DType dt, bool vec, bool wide, const RmsNormBwdArgs &a,
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
  void *h = nullptr;  // nullable: re-emit the forward's h
  int64_t ld_h = 0;
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
  const double *inv_freq = nullptr;  // HOST [D/2]: replaces theta^(-2i/D) when set
  const uint32_t *skip = nullptr;    // DEVICE word: non-zero leaves q, k untouched
};
cudaError_t launch_qk_rope(DType dt, bool vec, bool wide, const RopeArgs &a,
                           const DeviceInfo &dev, cudaStream_t s);

// The sequence-boundary check (seqlens_check.cu): status = the
// FTK_SEQLENS_* bits found in cu[0..B] against T, written by one CTA.
cudaError_t launch_check_seqlens(const int32_t *cu, int32_t B, int64_t T, uint32_t *status,
                                 cudaStream_t s);

// Per-head QK-RMSNorm fused with RoPE (qk_norm_rope.cu).  Forward: q, k in,
// oq, ok out (may be q, k), rq/rk written when set.  Backward: gq, gk (the
// output gradients) and the pre-norm q, k in; oq, ok receive the pre-norm
// gradients (may be gq, gk); rq/rk read when set (else recomputed); the
// partial rows go to ws and dwq/dwk (nullable) receive the weight gradients.
struct QkNormRopeArgs {
  const void *q;
  int64_t ld_q;
  const void *k;
  int64_t ld_k;
  const void *gq;
  int64_t ld_gq;
  const void *gk;
  int64_t ld_gk;
  void *oq;
  int64_t ld_oq;
  void *ok;
  int64_t ld_ok;
  const void *wq, *wk;
  float *rq, *rk;
  float *dwq, *dwk;
  float *ws;  // [ws_rows][2D]
  int64_t ws_rows;
  const int32_t *cu;
  int32_t B;
  int64_t T;
  int32_t Hq, Hkv, D;
  double theta;
  const double *inv_freq;  // HOST [D/2], nullable
  float eps;
  bool backward;
  const uint32_t *skip = nullptr;  // DEVICE word: non-zero leaves every output untouched
};
// Upper bound on the partial rows the backward writes.
int64_t qk_norm_rope_partial_rows(int64_t T, const DeviceInfo &dev);
cudaError_t launch_qk_norm_rope(DType dt, bool vec, bool wide, const QkNormRopeArgs &a,
                                const DeviceInfo &dev, cudaStream_t s);

// Cross-entropy of the LM head (cce.cu).  bf16 h [T, ldh], W [V, ldw];
// y int32 [T] (valid when 0 <= y < V).  Forward: loss (1 float) and lse [T].
// Backward: dloss (1 float, device) in, dh bf16 [T, lddh] and dW fp32
// [V, lddw] out.  ws: the workspace of the matching *_workspace_bytes.
struct CceArgs {
  const void *h;
  int64_t ldh;
  const void *w;
  int64_t ldw;
  const int32_t *y;
  int64_t T, H, V;
  float *loss, *lse;
  const float *dloss;
  void *dh;
  int64_t lddh;
  float *dw;
  int64_t lddw;
  void *ws;
};
size_t cce_fwd_workspace_bytes(int64_t T, int64_t V);
size_t cce_bwd_workspace_bytes(int64_t T, int64_t H, int64_t V);
int64_t cce_bwd_chunk(int64_t T, int64_t H, int64_t V, int sms);
cudaError_t launch_cce_fwd(const CceArgs &a, const DeviceInfo &dev, cudaStream_t s);
cudaError_t launch_cce_bwd(const CceArgs &a, const DeviceInfo &dev, cudaStream_t s);
// C fp32 [M, ldc] = A B^T on the tensor cores (bf16, tc_gemm.cuh): A stored
// [M, lda] (K-major) or, with a_mn, [K, lda] (MN-major); B stored [N, ldb]
// or, with b_mn, [K, ldb].
cudaError_t launch_gemm_bf16(const void *a, int64_t lda, bool a_mn, const void *b, int64_t ldb,
                             bool b_mn, float *c, int64_t ldc, int64_t M, int64_t N, int64_t K,
                             const DeviceInfo &dev, cudaStream_t s);

}  // namespace ftk
