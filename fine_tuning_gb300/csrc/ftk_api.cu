// The C ABI declared in include/ftk.h: argument validation, choice of index
// width and packet width, and dispatch to the kernel launchers.  Nothing here
// touches device memory or synchronises; every error is found on the host
// before a launch.
#include <stdint.h>

#include <cmath>
#include <cstring>
#include <mutex>
#include <string>

#include "ftk.h"
#include "launch.h"

namespace {

using ftk::DType;

thread_local std::string g_last_cuda_error;

ftk_status cuda_fail(cudaError_t e) {
  g_last_cuda_error = std::string(cudaGetErrorName(e)) + ": " + cudaGetErrorString(e);
  return FTK_ERR_CUDA;
}

ftk_status finish(cudaError_t e) { return e == cudaSuccess ? FTK_OK : cuda_fail(e); }

bool valid_dtype(ftk_dtype d) { return d == FTK_F32 || d == FTK_BF16; }

// 32-bit offsets are used only while every offset a kernel can form, plus
// the overshoot of its last loop step, stays below 2^31.
constexpr int64_t kNarrowLimit = (int64_t(1) << 31) - (int64_t(1) << 24);

// A [rows, len] view with row stride ld (elements of es bytes).
struct View {
  uintptr_t base;
  int64_t rows, ld, len, es;
  uintptr_t end() const { return base + (uintptr_t)(((rows - 1) * ld + len) * es); }
  int64_t max_offset() const { return (rows - 1) * ld + len; }
};

View view(const void *p, int64_t rows, int64_t ld, int64_t len, int64_t es) {
  return View{(uintptr_t)p, rows, ld, len, es};
}

bool same_view(const View &a, const View &b) {
  return a.base == b.base && a.ld == b.ld && a.len == b.len && a.es == b.es;
}

// Conservative: false only when the two element sets are provably disjoint
// (disjoint byte ranges, or equal strides with interleaved row slices as in a
// fused QKV or gate_up buffer).
bool may_overlap(const View &a, const View &b) {
  if (a.rows <= 0 || b.rows <= 0 || a.len <= 0 || b.len <= 0) return false;
  if (a.end() <= b.base || b.end() <= a.base) return false;
  if (a.ld == b.ld && a.es == b.es) {
    const int64_t period = a.ld * a.es;
    const int64_t la = a.len * a.es, lb = b.len * b.es;
    int64_t d = (int64_t)(b.base - a.base) % period;
    if (d < 0) d += period;
    if (d >= la && d + lb <= period) return false;
  }
  return true;
}

bool aligned(const void *p, size_t n) { return ((uintptr_t)p % n) == 0; }

std::mutex g_dev_mutex;
ftk::DeviceInfo g_dev_cache[64];
bool g_dev_known[64];

cudaError_t device_info(ftk::DeviceInfo *out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) {
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (g_dev_known[dev]) {
      *out = g_dev_cache[dev];
      return cudaSuccess;
    }
  }
  ftk::DeviceInfo d;
  d.device = dev;
  e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64) {
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    g_dev_cache[dev] = d;
    g_dev_known[dev] = true;
  }
  *out = d;
  return cudaSuccess;
}

}  // namespace

namespace ftk {
cudaError_t current_device_info(DeviceInfo *out) { return device_info(out); }
}  // namespace ftk

extern "C" {

FTK_API const char *ftk_version(void) { return "0.1.0"; }

FTK_API const char *ftk_status_str(ftk_status s) {
  switch (s) {
    case FTK_OK: return "ok";
    case FTK_ERR_NULL: return "a required pointer is NULL";
    case FTK_ERR_SHAPE: return "invalid size or stride";
    case FTK_ERR_ALIGN: return "pointer not aligned to its element size";
    case FTK_ERR_DTYPE: return "unknown dtype";
    case FTK_ERR_WORKSPACE: return "workspace missing or too small";
    case FTK_ERR_CUDA: return "CUDA error";
    case FTK_ERR_ALIAS: return "buffers overlap where that is not allowed";
  }
  return "unknown status";
}

FTK_API const char *ftk_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

FTK_API ftk_status ftk_device_status(uint32_t *flags, int clear) {
  if (!flags) return FTK_ERR_NULL;
  unsigned v = 0;
  cudaError_t e = ftk::read_device_status(&v, clear != 0);
  if (e != cudaSuccess) return cuda_fail(e);
  *flags = v;
  return FTK_OK;
}

FTK_API ftk_status ftk_selftest_wait_timeout(int64_t limit_cycles, ftk_stream_t stream) {
  if (limit_cycles < 0) return FTK_ERR_SHAPE;
  ftk::DeviceInfo dev;
  cudaError_t e = device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  return finish(ftk::launch_wait_timeout_selftest(dev, limit_cycles, (cudaStream_t)stream));
}

// ------------------------------------------------------------------ RMSNorm

}  // extern "C"

namespace {

// Shared by the plain and the residual-add forward; res == nullptr is the
// plain norm (h unused).
ftk_status rmsnorm_fwd_checked(const void *x, int64_t ldx, const void *res, int64_t ldr,
                               const void *w, void *h, int64_t ldh, void *y, int64_t ldy,
                               float *rstd, int64_t T, int64_t H, float eps, ftk_dtype dtype,
                               ftk_stream_t stream) {
  const bool add = res != nullptr;
  if (!valid_dtype(dtype)) return FTK_ERR_DTYPE;
  if (T < 0 || H < 1 || ldx < H || ldy < H || T >= (int64_t(1) << 31)) return FTK_ERR_SHAPE;
  if (add && (ldr < H || ldh < H)) return FTK_ERR_SHAPE;
  if (T == 0) return FTK_OK;
  if (!x || !w || !y || (add && !h)) return FTK_ERR_NULL;
  const DType dt = (DType)dtype;
  const int64_t es = ftk::dtype_bytes(dt);
  if (!aligned(x, es) || !aligned(w, es) || !aligned(y, es) || !aligned(rstd, 4) ||
      !aligned(res, es) || !aligned(h, es))
    return FTK_ERR_ALIGN;
  const View vx = view(x, T, ldx, H, es), vy = view(y, T, ldy, H, es);
  const View vw = view(w, 1, H, H, es), vr = view(rstd, 1, T, T, 4);
  const View vres = view(res, add ? T : 0, ldr, H, es), vh = view(h, add ? T : 0, ldh, H, es);
  if (!add) {
    if (!same_view(vx, vy) && may_overlap(vx, vy)) return FTK_ERR_ALIAS;
  } else {
    // h may replace x or res in place; y overlaps nothing
    if (!same_view(vh, vx) && may_overlap(vh, vx)) return FTK_ERR_ALIAS;
    if (!same_view(vh, vres) && may_overlap(vh, vres)) return FTK_ERR_ALIAS;
    if (may_overlap(vh, vw) || may_overlap(vh, vy)) return FTK_ERR_ALIAS;
    if (may_overlap(vy, vx) || may_overlap(vy, vres)) return FTK_ERR_ALIAS;
    if (rstd && (may_overlap(vr, vres) || may_overlap(vr, vh))) return FTK_ERR_ALIAS;
  }
  if (may_overlap(vy, vw)) return FTK_ERR_ALIAS;
  if (rstd && (may_overlap(vr, vx) || may_overlap(vr, vy) || may_overlap(vr, vw)))
    return FTK_ERR_ALIAS;

  const int n = dt == DType::F32 ? 4 : 8;
  bool vec = aligned(x, 16) && aligned(y, 16) && aligned(w, 16) && H % n == 0 && ldx % n == 0 &&
             ldy % n == 0;
  if (add) vec = vec && aligned(res, 16) && aligned(h, 16) && ldr % n == 0 && ldh % n == 0;
  bool wide = vx.max_offset() > kNarrowLimit || vy.max_offset() > kNarrowLimit;
  if (add) wide = wide || vres.max_offset() > kNarrowLimit || vh.max_offset() > kNarrowLimit;
  ftk::DeviceInfo dev;
  cudaError_t e = device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  ftk::RmsNormFwdArgs a{x, ldx, w, y, ldy, rstd, T, H, eps};
  if (add) {
    a.res = res;
    a.ldr = ldr;
    a.h = h;
    a.ldh = ldh;
  }
  return finish(ftk::launch_rmsnorm_fwd(dt, vec, wide, a, dev, (cudaStream_t)stream));
}

// Shared by the plain and the residual-add backward; dh == nullptr is the
// plain norm.  x is the norm's input (the stored h of the add form).
ftk_status rmsnorm_bwd_checked(const void *dy, int64_t lddy, const void *dh, int64_t lddh,
                               const void *x, int64_t ldx, const void *w, const float *rstd,
                               void *dx, int64_t lddx, float *dw, void *workspace,
                               size_t workspace_bytes, int64_t T, int64_t H, float eps,
                               ftk_dtype dtype, ftk_stream_t stream) {
  const bool add = dh != nullptr;
  if (!valid_dtype(dtype)) return FTK_ERR_DTYPE;
  if (T < 0 || H < 1 || lddy < H || ldx < H || lddx < H || T >= (int64_t(1) << 31))
    return FTK_ERR_SHAPE;
  if (add && lddh < H) return FTK_ERR_SHAPE;
  if (T == 0) return FTK_OK;
  if (!dy || !x || !w || !dx || !dw) return FTK_ERR_NULL;
  if (!workspace) return FTK_ERR_WORKSPACE;
  const DType dt = (DType)dtype;
  const int64_t es = ftk::dtype_bytes(dt);
  if (!aligned(dy, es) || !aligned(x, es) || !aligned(w, es) || !aligned(dx, es) ||
      !aligned(dh, es) || !aligned(rstd, 4) || !aligned(dw, 4) || !aligned(workspace, 16))
    return FTK_ERR_ALIGN;
  const int64_t ws_rows = (int64_t)(workspace_bytes / ((size_t)H * sizeof(float)));
  if (ws_rows < 1) return FTK_ERR_WORKSPACE;

  const View vdy = view(dy, T, lddy, H, es), vx = view(x, T, ldx, H, es);
  const View vdh = view(dh, add ? T : 0, lddh, H, es);
  const View vdx = view(dx, T, lddx, H, es), vw = view(w, 1, H, H, es);
  const View vr = view(rstd, 1, T, T, 4), vdw = view(dw, 1, H, H, 4);
  const View vws = view(workspace, 1, ws_rows * H, ws_rows * H, 4);
  if (!same_view(vdx, vdy) && may_overlap(vdx, vdy)) return FTK_ERR_ALIAS;
  if (!same_view(vdx, vdh) && may_overlap(vdx, vdh)) return FTK_ERR_ALIAS;
  const View outs[3] = {vdx, vdw, vws};
  for (int i = 0; i < 3; ++i) {
    if (i != 0 && (may_overlap(outs[i], vdy) || may_overlap(outs[i], vdh))) return FTK_ERR_ALIAS;
    if (may_overlap(outs[i], vx) || may_overlap(outs[i], vw)) return FTK_ERR_ALIAS;
    if (rstd && may_overlap(outs[i], vr)) return FTK_ERR_ALIAS;
    for (int k = i + 1; k < 3; ++k)
      if (may_overlap(outs[i], outs[k])) return FTK_ERR_ALIAS;
  }

  const int n = dt == DType::F32 ? 4 : 8;
  bool vec = aligned(dy, 16) && aligned(x, 16) && aligned(w, 16) && aligned(dx, 16) &&
             H % n == 0 && lddy % n == 0 && ldx % n == 0 && lddx % n == 0;
  if (add) vec = vec && aligned(dh, 16) && lddh % n == 0;
  const bool wide = vdy.max_offset() > kNarrowLimit || vx.max_offset() > kNarrowLimit ||
                    vdx.max_offset() > kNarrowLimit ||
                    (add && vdh.max_offset() > kNarrowLimit);
  ftk::DeviceInfo dev;
  cudaError_t e = device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  ftk::RmsNormBwdArgs a{dy, lddy, x, ldx, w, rstd, dx, lddx, dw, (float *)workspace, ws_rows,
                        T, H, eps};
  if (add) {
    a.dh = dh;
    a.lddh = lddh;
  }
  return finish(ftk::launch_rmsnorm_bwd(dt, vec, wide, a, dev, (cudaStream_t)stream));
}

}  // namespace

extern "C" {

FTK_API ftk_status ftk_rmsnorm_fwd(const void *x, int64_t ldx, const void *w, void *y,
                                   int64_t ldy, float *rstd, int64_t T, int64_t H, float eps,
                                   ftk_dtype dtype, ftk_stream_t stream) {
  return rmsnorm_fwd_checked(x, ldx, nullptr, 0, w, nullptr, 0, y, ldy, rstd, T, H, eps, dtype,
                             stream);
}

FTK_API ftk_status ftk_rmsnorm_add_fwd(const void *x, int64_t ldx, const void *res,
                                       int64_t ldr, const void *w, void *h, int64_t ldh,
                                       void *y, int64_t ldy, float *rstd, int64_t T,
                                       int64_t H, float eps, ftk_dtype dtype,
                                       ftk_stream_t stream) {
  if (!res && T > 0) return FTK_ERR_NULL;
  return rmsnorm_fwd_checked(x, ldx, res, ldr, w, h, ldh, y, ldy, rstd, T, H, eps, dtype,
                             stream);
}

FTK_API size_t ftk_rmsnorm_bwd_workspace_bytes(int64_t T, int64_t H, ftk_dtype dtype) {
  if (!valid_dtype(dtype) || T <= 0 || H <= 0) return 0;
  ftk::DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return 0;
  return (size_t)ftk::rmsnorm_bwd_partial_rows(T, dev) * (size_t)H * sizeof(float);
}

FTK_API ftk_status ftk_rmsnorm_bwd(const void *dy, int64_t lddy, const void *x, int64_t ldx,
                                   const void *w, const float *rstd, void *dx, int64_t lddx,
                                   float *dw, void *workspace, size_t workspace_bytes, int64_t T,
                                   int64_t H, float eps, ftk_dtype dtype, ftk_stream_t stream) {
  return rmsnorm_bwd_checked(dy, lddy, nullptr, 0, x, ldx, w, rstd, dx, lddx, dw, workspace,
                             workspace_bytes, T, H, eps, dtype, stream);
}

FTK_API ftk_status ftk_rmsnorm_add_bwd(const void *dy, int64_t lddy, const void *dh,
                                       int64_t lddh, const void *h, int64_t ldh,
                                       const void *w, const float *rstd, void *dx,
                                       int64_t lddx, float *dw, void *workspace,
                                       size_t workspace_bytes, int64_t T, int64_t H,
                                       float eps, ftk_dtype dtype, ftk_stream_t stream) {
  if (!dh && T > 0) return FTK_ERR_NULL;
  return rmsnorm_bwd_checked(dy, lddy, dh, lddh, h, ldh, w, rstd, dx, lddx, dw, workspace,
                             workspace_bytes, T, H, eps, dtype, stream);
}

// ------------------------------------------------------------------- SwiGLU

FTK_API ftk_status ftk_swiglu_fwd(const void *g, const void *u, int64_t ld_gu, void *h,
                                  int64_t ld_h, int64_t T, int64_t I, ftk_dtype dtype,
                                  ftk_stream_t stream) {
  if (!valid_dtype(dtype)) return FTK_ERR_DTYPE;
  if (T < 0 || I < 0 || ld_gu < I || ld_h < I) return FTK_ERR_SHAPE;
  if (T == 0 || I == 0) return FTK_OK;
  if (!g || !u || !h) return FTK_ERR_NULL;
  const DType dt = (DType)dtype;
  const int64_t es = ftk::dtype_bytes(dt);
  if (!aligned(g, es) || !aligned(u, es) || !aligned(h, es)) return FTK_ERR_ALIGN;
  const View vg = view(g, T, ld_gu, I, es), vu = view(u, T, ld_gu, I, es);
  const View vh = view(h, T, ld_h, I, es);
  if (!same_view(vh, vg) && may_overlap(vh, vg)) return FTK_ERR_ALIAS;
  if (!same_view(vh, vu) && may_overlap(vh, vu)) return FTK_ERR_ALIAS;

  const int n = dt == DType::F32 ? 4 : 8;
  const bool vec = aligned(g, 16) && aligned(u, 16) && aligned(h, 16) && I % n == 0 &&
                   ld_gu % n == 0 && ld_h % n == 0;
  const bool wide = vg.max_offset() > kNarrowLimit || vu.max_offset() > kNarrowLimit ||
                    vh.max_offset() > kNarrowLimit || T * I > kNarrowLimit;
  ftk::DeviceInfo dev;
  cudaError_t e = device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  ftk::SwigluFwdArgs a{g, u, ld_gu, h, ld_h, T, I};
  return finish(ftk::launch_swiglu_fwd(dt, vec, wide, a, dev, (cudaStream_t)stream));
}

}  // extern "C"

namespace {

// Shared by ftk_swiglu_bwd and ftk_swiglu_bwd_h; h == nullptr: no re-emitted h.
ftk_status swiglu_bwd_checked(const void *dh, int64_t ld_dh, const void *g, const void *u,
                              int64_t ld_gu, void *dg, void *du, int64_t ld_dgu, void *h,
                              int64_t ld_h, int64_t T, int64_t I, ftk_dtype dtype,
                              ftk_stream_t stream) {
  const bool emit = h != nullptr;
  if (!valid_dtype(dtype)) return FTK_ERR_DTYPE;
  if (T < 0 || I < 0 || ld_dh < I || ld_gu < I || ld_dgu < I || (emit && ld_h < I))
    return FTK_ERR_SHAPE;
  if (T == 0 || I == 0) return FTK_OK;
  if (!dh || !g || !u || !dg || !du) return FTK_ERR_NULL;
  const DType dt = (DType)dtype;
  const int64_t es = ftk::dtype_bytes(dt);
  if (!aligned(dh, es) || !aligned(g, es) || !aligned(u, es) || !aligned(dg, es) ||
      !aligned(du, es) || !aligned(h, es))
    return FTK_ERR_ALIGN;
  const View vdh = view(dh, T, ld_dh, I, es), vg = view(g, T, ld_gu, I, es);
  const View vu = view(u, T, ld_gu, I, es), vdg = view(dg, T, ld_dgu, I, es);
  const View vdu = view(du, T, ld_dgu, I, es), vh = view(h, emit ? T : 0, ld_h, I, es);
  // every thread reads all its inputs before it writes, so an output may
  // replace an input exactly; outputs never overlap one another
  if (may_overlap(vdg, vdu) || may_overlap(vh, vdg) || may_overlap(vh, vdu))
    return FTK_ERR_ALIAS;
  const View ins[3] = {vdh, vg, vu};
  for (const View &o : {vdg, vdu, vh})
    for (const View &i : ins)
      if (!same_view(o, i) && may_overlap(o, i)) return FTK_ERR_ALIAS;

  const int n = dt == DType::F32 ? 4 : 8;
  bool vec = aligned(dh, 16) && aligned(g, 16) && aligned(u, 16) && aligned(dg, 16) &&
             aligned(du, 16) && I % n == 0 && ld_dh % n == 0 && ld_gu % n == 0 &&
             ld_dgu % n == 0;
  if (emit) vec = vec && aligned(h, 16) && ld_h % n == 0;
  const bool wide = vdh.max_offset() > kNarrowLimit || vg.max_offset() > kNarrowLimit ||
                    vu.max_offset() > kNarrowLimit || vdg.max_offset() > kNarrowLimit ||
                    vdu.max_offset() > kNarrowLimit || (emit && vh.max_offset() > kNarrowLimit) ||
                    T * I > kNarrowLimit;
  ftk::DeviceInfo dev;
  cudaError_t e = device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  ftk::SwigluBwdArgs a{dh, ld_dh, g, u, ld_gu, dg, du, ld_dgu, T, I};
  a.h = h;
  a.ld_h = ld_h;
  return finish(ftk::launch_swiglu_bwd(dt, vec, wide, a, dev, (cudaStream_t)stream));
}

}  // namespace

extern "C" {

FTK_API ftk_status ftk_swiglu_bwd(const void *dh, int64_t ld_dh, const void *g, const void *u,
                                  int64_t ld_gu, void *dg, void *du, int64_t ld_dgu, int64_t T,
                                  int64_t I, ftk_dtype dtype, ftk_stream_t stream) {
  return swiglu_bwd_checked(dh, ld_dh, g, u, ld_gu, dg, du, ld_dgu, nullptr, 0, T, I, dtype,
                            stream);
}

FTK_API ftk_status ftk_swiglu_bwd_h(const void *dh, int64_t ld_dh, const void *g, const void *u,
                                    int64_t ld_gu, void *dg, void *du, int64_t ld_dgu, void *h,
                                    int64_t ld_h, int64_t T, int64_t I, ftk_dtype dtype,
                                    ftk_stream_t stream) {
  if (!h && T > 0 && I > 0) return FTK_ERR_NULL;
  return swiglu_bwd_checked(dh, ld_dh, g, u, ld_gu, dg, du, ld_dgu, h, ld_h, T, I, dtype,
                            stream);
}

// ------------------------------------------------------------------ QK-RoPE

// inv_freq (HOST, nullable) replaces theta's table when given; skip (DEVICE,
// nullable) is the word of the boundary check that guards the rotation.
static ftk_status qk_rope(void *q, int64_t ld_q, void *k, int64_t ld_k, const int32_t *cu,
                          int32_t B, int64_t T, int32_t Hq, int32_t Hkv, int32_t D, double theta,
                          const double *inv_freq, ftk_dtype dtype, ftk_stream_t stream,
                          bool backward, const uint32_t *skip = nullptr) {
  if (!valid_dtype(dtype)) return FTK_ERR_DTYPE;
  if (T < 0 || B < 0 || Hq < 0 || Hkv < 0 || Hq + Hkv < 1 || D < 2 || D % 2 != 0 ||
      D / 2 > ftk::kRopeMaxHalf || T >= (int64_t(1) << 31))
    return FTK_ERR_SHAPE;
  if (inv_freq) {
    for (int32_t i = 0; i < D / 2; ++i)
      if (!(inv_freq[i] >= 0.0 && inv_freq[i] <= 1.0)) return FTK_ERR_SHAPE;  // NaN fails too
  } else if (!(theta > 0.0)) {
    return FTK_ERR_SHAPE;
  }
  if ((Hq > 0 && ld_q < (int64_t)Hq * D) || (Hkv > 0 && ld_k < (int64_t)Hkv * D))
    return FTK_ERR_SHAPE;
  if (T == 0) return FTK_OK;
  if (B < 1) return FTK_ERR_SHAPE;
  if (!cu || (Hq > 0 && !q) || (Hkv > 0 && !k)) return FTK_ERR_NULL;
  const DType dt = (DType)dtype;
  const int64_t es = ftk::dtype_bytes(dt);
  if ((Hq > 0 && !aligned(q, es)) || (Hkv > 0 && !aligned(k, es)) || !aligned(cu, 4))
    return FTK_ERR_ALIGN;
  const View vq = view(q, Hq > 0 ? T : 0, ld_q, (int64_t)Hq * D, es);
  const View vk = view(k, Hkv > 0 ? T : 0, ld_k, (int64_t)Hkv * D, es);
  const View vc = view(cu, 1, (int64_t)B + 1, (int64_t)B + 1, 4);
  if (may_overlap(vq, vk) || may_overlap(vc, vq) || may_overlap(vc, vk)) return FTK_ERR_ALIAS;
  if (skip) {
    if (!aligned(skip, 4)) return FTK_ERR_ALIGN;
    const View vs = view(skip, 1, 1, 1, 4);
    if (may_overlap(vs, vq) || may_overlap(vs, vk)) return FTK_ERR_ALIAS;
  }

  const int n = dt == DType::F32 ? 4 : 8;
  const bool vec = (D / 2) % n == 0 && (Hq == 0 || (aligned(q, 16) && ld_q % n == 0)) &&
                   (Hkv == 0 || (aligned(k, 16) && ld_k % n == 0));
  const bool wide = (Hq > 0 && vq.max_offset() > kNarrowLimit) ||
                    (Hkv > 0 && vk.max_offset() > kNarrowLimit);
  ftk::DeviceInfo dev;
  cudaError_t e = device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  ftk::RopeArgs a{q, ld_q, k, ld_k, cu, B, T, Hq, Hkv, D, theta, backward};
  a.inv_freq = inv_freq;
  a.skip = skip;
  return finish(ftk::launch_qk_rope(dt, vec, wide, a, dev, (cudaStream_t)stream));
}

FTK_API ftk_status ftk_check_seqlens(const int32_t *cu_seqlens, int32_t B, int64_t T,
                                     uint32_t *status, ftk_stream_t stream) {
  if (B < 0 || T < 0) return FTK_ERR_SHAPE;
  if (!cu_seqlens || !status) return FTK_ERR_NULL;
  if (!aligned(cu_seqlens, 4) || !aligned(status, 4)) return FTK_ERR_ALIGN;
  if (may_overlap(view(cu_seqlens, 1, (int64_t)B + 1, (int64_t)B + 1, 4), view(status, 1, 1, 1, 4)))
    return FTK_ERR_ALIAS;
  return finish(ftk::launch_check_seqlens(cu_seqlens, B, T, status, (cudaStream_t)stream));
}

FTK_API ftk_status ftk_qk_rope_fwd_checked(void *q, int64_t ld_q, void *k, int64_t ld_k,
                                           const int32_t *cu_seqlens, int32_t B, int64_t T,
                                           int32_t Hq, int32_t Hkv, int32_t D, double theta,
                                           const double *inv_freq,
                                           const uint32_t *seqlens_status, ftk_dtype dtype,
                                           ftk_stream_t stream) {
  if (!seqlens_status && T > 0) return FTK_ERR_NULL;
  return qk_rope(q, ld_q, k, ld_k, cu_seqlens, B, T, Hq, Hkv, D, theta, inv_freq, dtype, stream,
                 false, seqlens_status);
}

FTK_API ftk_status ftk_qk_rope_bwd_checked(void *dq, int64_t ld_q, void *dk, int64_t ld_k,
                                           const int32_t *cu_seqlens, int32_t B, int64_t T,
                                           int32_t Hq, int32_t Hkv, int32_t D, double theta,
                                           const double *inv_freq,
                                           const uint32_t *seqlens_status, ftk_dtype dtype,
                                           ftk_stream_t stream) {
  if (!seqlens_status && T > 0) return FTK_ERR_NULL;
  return qk_rope(dq, ld_q, dk, ld_k, cu_seqlens, B, T, Hq, Hkv, D, theta, inv_freq, dtype,
                 stream, true, seqlens_status);
}

FTK_API ftk_status ftk_qk_rope_fwd(void *q, int64_t ld_q, void *k, int64_t ld_k,
                                   const int32_t *cu_seqlens, int32_t B, int64_t T, int32_t Hq,
                                   int32_t Hkv, int32_t D, double theta, ftk_dtype dtype,
                                   ftk_stream_t stream) {
  return qk_rope(q, ld_q, k, ld_k, cu_seqlens, B, T, Hq, Hkv, D, theta, nullptr, dtype, stream,
                 false);
}

FTK_API ftk_status ftk_qk_rope_bwd(void *dq, int64_t ld_q, void *dk, int64_t ld_k,
                                   const int32_t *cu_seqlens, int32_t B, int64_t T, int32_t Hq,
                                   int32_t Hkv, int32_t D, double theta, ftk_dtype dtype,
                                   ftk_stream_t stream) {
  return qk_rope(dq, ld_q, dk, ld_k, cu_seqlens, B, T, Hq, Hkv, D, theta, nullptr, dtype, stream,
                 true);
}

FTK_API ftk_status ftk_qk_rope_freq_fwd(void *q, int64_t ld_q, void *k, int64_t ld_k,
                                        const int32_t *cu_seqlens, int32_t B, int64_t T,
                                        int32_t Hq, int32_t Hkv, int32_t D,
                                        const double *inv_freq, ftk_dtype dtype,
                                        ftk_stream_t stream) {
  if (!inv_freq) return FTK_ERR_NULL;
  return qk_rope(q, ld_q, k, ld_k, cu_seqlens, B, T, Hq, Hkv, D, 0.0, inv_freq, dtype, stream,
                 false);
}

FTK_API ftk_status ftk_qk_rope_freq_bwd(void *dq, int64_t ld_q, void *dk, int64_t ld_k,
                                        const int32_t *cu_seqlens, int32_t B, int64_t T,
                                        int32_t Hq, int32_t Hkv, int32_t D,
                                        const double *inv_freq, ftk_dtype dtype,
                                        ftk_stream_t stream) {
  if (!inv_freq) return FTK_ERR_NULL;
  return qk_rope(dq, ld_q, dk, ld_k, cu_seqlens, B, T, Hq, Hkv, D, 0.0, inv_freq, dtype, stream,
                 true);
}

// -------------------------------------------------- QK-RMSNorm fused with RoPE

}  // extern "C"

namespace {

struct NormRopeShape {
  int64_t T;
  int32_t B, Hq, Hkv, D;
};

// Shape, frequency and eps checks shared by the fused forward and backward.
ftk_status norm_rope_shape(const NormRopeShape &sh, double theta, const double *inv_freq,
                           float eps) {
  if (sh.T < 0 || sh.B < 0 || sh.Hq < 0 || sh.Hkv < 0 || sh.Hq + sh.Hkv < 1 || sh.D < 2 ||
      sh.D % 2 != 0 || sh.D / 2 > ftk::kRopeMaxHalf || sh.T >= (int64_t(1) << 31))
    return FTK_ERR_SHAPE;
  if (!(eps >= 0.0f) || !std::isfinite(eps)) return FTK_ERR_SHAPE;
  if (inv_freq) {
    for (int32_t i = 0; i < sh.D / 2; ++i)
      if (!(inv_freq[i] >= 0.0 && inv_freq[i] <= 1.0)) return FTK_ERR_SHAPE;
  } else if (!(theta > 0.0)) {
    return FTK_ERR_SHAPE;
  }
  return FTK_OK;
}

}  // namespace

// skip (DEVICE, nullable): the boundary check's word; non-zero leaves every
// output untouched.
static ftk_status qk_norm_rope_fwd(const void *q, int64_t ld_q, const void *k, int64_t ld_k,
                                   const void *wq, const void *wk, void *q_out, int64_t ld_qo,
                                   void *k_out, int64_t ld_ko, float *rstd_q, float *rstd_k,
                                   const int32_t *cu_seqlens, int32_t B, int64_t T, int32_t Hq,
                                   int32_t Hkv, int32_t D, double theta, const double *inv_freq,
                                   float eps, ftk_dtype dtype, ftk_stream_t stream,
                                   const uint32_t *skip) {
  if (!valid_dtype(dtype)) return FTK_ERR_DTYPE;
  const NormRopeShape sh{T, B, Hq, Hkv, D};
  ftk_status st = norm_rope_shape(sh, theta, inv_freq, eps);
  if (st != FTK_OK) return st;
  const int64_t wq_ = (int64_t)Hq * D, wk_ = (int64_t)Hkv * D;
  if ((Hq > 0 && (ld_q < wq_ || ld_qo < wq_)) || (Hkv > 0 && (ld_k < wk_ || ld_ko < wk_)))
    return FTK_ERR_SHAPE;
  if (T == 0) return FTK_OK;
  if (B < 1) return FTK_ERR_SHAPE;
  if (!cu_seqlens || (Hq > 0 && (!q || !wq || !q_out)) || (Hkv > 0 && (!k || !wk || !k_out)))
    return FTK_ERR_NULL;
  const DType dt = (DType)dtype;
  const int64_t es = ftk::dtype_bytes(dt);
  if (!aligned(q, es) || !aligned(k, es) || !aligned(wq, es) || !aligned(wk, es) ||
      !aligned(q_out, es) || !aligned(k_out, es) || !aligned(rstd_q, 4) ||
      !aligned(rstd_k, 4) || !aligned(cu_seqlens, 4))
    return FTK_ERR_ALIGN;
  const int64_t rq_n = Hq > 0 ? T : 0, rk_n = Hkv > 0 ? T : 0;
  const View vq = view(q, rq_n, ld_q, wq_, es), vk = view(k, rk_n, ld_k, wk_, es);
  const View voq = view(q_out, rq_n, ld_qo, wq_, es), vok = view(k_out, rk_n, ld_ko, wk_, es);
  const View vwq = view(wq, Hq > 0 ? 1 : 0, D, D, es), vwk = view(wk, Hkv > 0 ? 1 : 0, D, D, es);
  const View vrq = view(rstd_q, rstd_q && Hq > 0 ? 1 : 0, T * Hq, T * Hq, 4);
  const View vrk = view(rstd_k, rstd_k && Hkv > 0 ? 1 : 0, T * Hkv, T * Hkv, 4);
  const View vc = view(cu_seqlens, 1, (int64_t)B + 1, (int64_t)B + 1, 4);
  // an output may replace its own input exactly; nothing else overlaps an output
  if (!same_view(voq, vq) && may_overlap(voq, vq)) return FTK_ERR_ALIAS;
  if (!same_view(vok, vk) && may_overlap(vok, vk)) return FTK_ERR_ALIAS;
  const View outs[4] = {voq, vok, vrq, vrk};
  const View ins[5] = {vq, vk, vwq, vwk, vc};
  for (int i = 0; i < 4; ++i) {
    for (int m = 0; m < 5; ++m) {
      if ((i == 0 && m == 0) || (i == 1 && m == 1)) continue;  // handled above
      if (may_overlap(outs[i], ins[m])) return FTK_ERR_ALIAS;
    }
    for (int m = i + 1; m < 4; ++m)
      if (may_overlap(outs[i], outs[m])) return FTK_ERR_ALIAS;
  }
  if (skip) {
    if (!aligned(skip, 4)) return FTK_ERR_ALIGN;
    const View vs = view(skip, 1, 1, 1, 4);
    for (int i = 0; i < 4; ++i)
      if (may_overlap(vs, outs[i])) return FTK_ERR_ALIAS;
  }
  const int n = dt == DType::F32 ? 4 : 8;
  const bool vec = (D / 2) % n == 0 &&
                   (Hq == 0 || (aligned(q, 16) && aligned(q_out, 16) && aligned(wq, 16) &&
                                ld_q % n == 0 && ld_qo % n == 0)) &&
                   (Hkv == 0 || (aligned(k, 16) && aligned(k_out, 16) && aligned(wk, 16) &&
                                 ld_k % n == 0 && ld_ko % n == 0));
  const int64_t hmax = Hq > Hkv ? Hq : Hkv;
  const bool wide = vq.max_offset() > kNarrowLimit || vk.max_offset() > kNarrowLimit ||
                    voq.max_offset() > kNarrowLimit || vok.max_offset() > kNarrowLimit ||
                    T * hmax > kNarrowLimit;
  ftk::DeviceInfo dev;
  cudaError_t e = device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  ftk::QkNormRopeArgs a{q,     ld_q,   k,      ld_k,      nullptr, 0,     nullptr, 0,
                        q_out, ld_qo,  k_out,  ld_ko,     wq,      wk,    rstd_q,  rstd_k,
                        nullptr, nullptr, nullptr, 0,     cu_seqlens, B,  T,       Hq,
                        Hkv,   D,      theta,  inv_freq,  eps,     false};
  a.skip = skip;
  return finish(ftk::launch_qk_norm_rope(dt, vec, wide, a, dev, (cudaStream_t)stream));
}

extern "C" {

FTK_API ftk_status ftk_qk_norm_rope_fwd(const void *q, int64_t ld_q, const void *k, int64_t ld_k,
                                        const void *wq, const void *wk, void *q_out,
                                        int64_t ld_qo, void *k_out, int64_t ld_ko,
                                        float *rstd_q, float *rstd_k,
                                        const int32_t *cu_seqlens, int32_t B, int64_t T,
                                        int32_t Hq, int32_t Hkv, int32_t D, double theta,
                                        const double *inv_freq, float eps, ftk_dtype dtype,
                                        ftk_stream_t stream) {
  return qk_norm_rope_fwd(q, ld_q, k, ld_k, wq, wk, q_out, ld_qo, k_out, ld_ko, rstd_q, rstd_k,
                          cu_seqlens, B, T, Hq, Hkv, D, theta, inv_freq, eps, dtype, stream,
                          nullptr);
}

FTK_API ftk_status ftk_qk_norm_rope_fwd_checked(
    const void *q, int64_t ld_q, const void *k, int64_t ld_k, const void *wq, const void *wk,
    void *q_out, int64_t ld_qo, void *k_out, int64_t ld_ko, float *rstd_q, float *rstd_k,
    const int32_t *cu_seqlens, int32_t B, int64_t T, int32_t Hq, int32_t Hkv, int32_t D,
    double theta, const double *inv_freq, float eps, const uint32_t *seqlens_status,
    ftk_dtype dtype, ftk_stream_t stream) {
  if (!seqlens_status && T > 0) return FTK_ERR_NULL;
  return qk_norm_rope_fwd(q, ld_q, k, ld_k, wq, wk, q_out, ld_qo, k_out, ld_ko, rstd_q, rstd_k,
                          cu_seqlens, B, T, Hq, Hkv, D, theta, inv_freq, eps, dtype, stream,
                          seqlens_status);
}

FTK_API size_t ftk_qk_norm_rope_bwd_workspace_bytes(int64_t T, int32_t D, ftk_dtype dtype) {
  if (!valid_dtype(dtype) || T <= 0 || D < 2 || D % 2 != 0) return 0;
  ftk::DeviceInfo dev;
  if (device_info(&dev) != cudaSuccess) return 0;
  return (size_t)ftk::qk_norm_rope_partial_rows(T, dev) * 2 * (size_t)D * sizeof(float);
}

}  // extern "C"

static ftk_status qk_norm_rope_bwd(const void *dq_out, int64_t ld_gq, const void *dk_out,
                                   int64_t ld_gk, const void *q, int64_t ld_q, const void *k,
                                   int64_t ld_k, const void *wq, const void *wk,
                                   const float *rstd_q, const float *rstd_k, void *dq,
                                   int64_t ld_dq, void *dk, int64_t ld_dk, float *dwq, float *dwk,
                                   void *workspace, size_t workspace_bytes,
                                   const int32_t *cu_seqlens, int32_t B, int64_t T, int32_t Hq,
                                   int32_t Hkv, int32_t D, double theta, const double *inv_freq,
                                   float eps, ftk_dtype dtype, ftk_stream_t stream,
                                   const uint32_t *skip) {
  if (!valid_dtype(dtype)) return FTK_ERR_DTYPE;
  const NormRopeShape sh{T, B, Hq, Hkv, D};
  ftk_status st = norm_rope_shape(sh, theta, inv_freq, eps);
  if (st != FTK_OK) return st;
  const int64_t wq_ = (int64_t)Hq * D, wk_ = (int64_t)Hkv * D;
  if ((Hq > 0 && (ld_q < wq_ || ld_gq < wq_ || ld_dq < wq_)) ||
      (Hkv > 0 && (ld_k < wk_ || ld_gk < wk_ || ld_dk < wk_)))
    return FTK_ERR_SHAPE;
  if (T == 0) return FTK_OK;
  if (B < 1) return FTK_ERR_SHAPE;
  if (!cu_seqlens || (Hq > 0 && (!q || !wq || !dq_out || !dq || !dwq)) ||
      (Hkv > 0 && (!k || !wk || !dk_out || !dk || !dwk)))
    return FTK_ERR_NULL;
  // rstd: every needed one, or none (recompute)
  const bool have_r = (Hq > 0 && rstd_q) || (Hkv > 0 && rstd_k);
  if (have_r && ((Hq > 0 && !rstd_q) || (Hkv > 0 && !rstd_k))) return FTK_ERR_NULL;
  if (!workspace) return FTK_ERR_WORKSPACE;
  const DType dt = (DType)dtype;
  const int64_t es = ftk::dtype_bytes(dt);
  if (!aligned(q, es) || !aligned(k, es) || !aligned(wq, es) || !aligned(wk, es) ||
      !aligned(dq_out, es) || !aligned(dk_out, es) || !aligned(dq, es) || !aligned(dk, es) ||
      !aligned(rstd_q, 4) || !aligned(rstd_k, 4) || !aligned(dwq, 4) || !aligned(dwk, 4) ||
      !aligned(workspace, 16) || !aligned(cu_seqlens, 4))
    return FTK_ERR_ALIGN;
  const int64_t ws_rows = (int64_t)(workspace_bytes / (2 * (size_t)D * sizeof(float)));
  if (ws_rows < 1) return FTK_ERR_WORKSPACE;
  const int64_t rq_n = Hq > 0 ? T : 0, rk_n = Hkv > 0 ? T : 0;
  const View vq = view(q, rq_n, ld_q, wq_, es), vk = view(k, rk_n, ld_k, wk_, es);
  const View vgq = view(dq_out, rq_n, ld_gq, wq_, es), vgk = view(dk_out, rk_n, ld_gk, wk_, es);
  const View vdq = view(dq, rq_n, ld_dq, wq_, es), vdk = view(dk, rk_n, ld_dk, wk_, es);
  const View vwq = view(wq, Hq > 0 ? 1 : 0, D, D, es), vwk = view(wk, Hkv > 0 ? 1 : 0, D, D, es);
  const View vrq = view(rstd_q, rstd_q && Hq > 0 ? 1 : 0, T * Hq, T * Hq, 4);
  const View vrk = view(rstd_k, rstd_k && Hkv > 0 ? 1 : 0, T * Hkv, T * Hkv, 4);
  const View vdwq = view(dwq, Hq > 0 ? 1 : 0, D, D, 4), vdwk = view(dwk, Hkv > 0 ? 1 : 0, D, D, 4);
  const View vws = view(workspace, 1, ws_rows * 2 * D, ws_rows * 2 * D, 4);
  const View vc = view(cu_seqlens, 1, (int64_t)B + 1, (int64_t)B + 1, 4);
  // dq / dk may replace the output gradients exactly; nothing else overlaps an output
  if (!same_view(vdq, vgq) && may_overlap(vdq, vgq)) return FTK_ERR_ALIAS;
  if (!same_view(vdk, vgk) && may_overlap(vdk, vgk)) return FTK_ERR_ALIAS;
  const View outs[5] = {vdq, vdk, vdwq, vdwk, vws};
  const View ins[9] = {vgq, vgk, vq, vk, vwq, vwk, vrq, vrk, vc};
  for (int i = 0; i < 5; ++i) {
    for (int m = 0; m < 9; ++m) {
      if ((i == 0 && m == 0) || (i == 1 && m == 1)) continue;  // handled above
      if (may_overlap(outs[i], ins[m])) return FTK_ERR_ALIAS;
    }
    for (int m = i + 1; m < 5; ++m)
      if (may_overlap(outs[i], outs[m])) return FTK_ERR_ALIAS;
  }
  if (skip) {
    if (!aligned(skip, 4)) return FTK_ERR_ALIGN;
    const View vs = view(skip, 1, 1, 1, 4);
    for (int i = 0; i < 5; ++i)
      if (may_overlap(vs, outs[i])) return FTK_ERR_ALIAS;
  }
  const int n = dt == DType::F32 ? 4 : 8;
  const bool vec =
      (D / 2) % n == 0 &&
      (Hq == 0 || (aligned(q, 16) && aligned(dq_out, 16) && aligned(dq, 16) && aligned(wq, 16) &&
                   ld_q % n == 0 && ld_gq % n == 0 && ld_dq % n == 0)) &&
      (Hkv == 0 || (aligned(k, 16) && aligned(dk_out, 16) && aligned(dk, 16) &&
                    aligned(wk, 16) && ld_k % n == 0 && ld_gk % n == 0 && ld_dk % n == 0));
  const int64_t hmax = Hq > Hkv ? Hq : Hkv;
  const bool wide = vq.max_offset() > kNarrowLimit || vk.max_offset() > kNarrowLimit ||
                    vgq.max_offset() > kNarrowLimit || vgk.max_offset() > kNarrowLimit ||
                    vdq.max_offset() > kNarrowLimit || vdk.max_offset() > kNarrowLimit ||
                    T * hmax > kNarrowLimit;
  ftk::DeviceInfo dev;
  cudaError_t e = device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  ftk::QkNormRopeArgs a{q,      ld_q,   k,      ld_k,   dq_out,   ld_gq,  dk_out,
                        ld_gk,  dq,     ld_dq,  dk,     ld_dk,    wq,     wk,
                        have_r ? (float *)rstd_q : nullptr,
                        have_r ? (float *)rstd_k : nullptr,
                        Hq > 0 ? dwq : nullptr, Hkv > 0 ? dwk : nullptr,
                        (float *)workspace, ws_rows, cu_seqlens, B, T, Hq, Hkv, D,
                        theta,  inv_freq, eps,  true};
  a.skip = skip;
  return finish(ftk::launch_qk_norm_rope(dt, vec, wide, a, dev, (cudaStream_t)stream));
}

extern "C" {

FTK_API ftk_status ftk_qk_norm_rope_bwd(const void *dq_out, int64_t ld_gq, const void *dk_out,
                                        int64_t ld_gk, const void *q, int64_t ld_q,
                                        const void *k, int64_t ld_k, const void *wq,
                                        const void *wk, const float *rstd_q,
                                        const float *rstd_k, void *dq, int64_t ld_dq, void *dk,
                                        int64_t ld_dk, float *dwq, float *dwk, void *workspace,
                                        size_t workspace_bytes, const int32_t *cu_seqlens,
                                        int32_t B, int64_t T, int32_t Hq, int32_t Hkv, int32_t D,
                                        double theta, const double *inv_freq, float eps,
                                        ftk_dtype dtype, ftk_stream_t stream) {
  return qk_norm_rope_bwd(dq_out, ld_gq, dk_out, ld_gk, q, ld_q, k, ld_k, wq, wk, rstd_q, rstd_k,
                          dq, ld_dq, dk, ld_dk, dwq, dwk, workspace, workspace_bytes, cu_seqlens,
                          B, T, Hq, Hkv, D, theta, inv_freq, eps, dtype, stream, nullptr);
}

FTK_API ftk_status ftk_qk_norm_rope_bwd_checked(
    const void *dq_out, int64_t ld_gq, const void *dk_out, int64_t ld_gk, const void *q,
    int64_t ld_q, const void *k, int64_t ld_k, const void *wq, const void *wk,
    const float *rstd_q, const float *rstd_k, void *dq, int64_t ld_dq, void *dk, int64_t ld_dk,
    float *dwq, float *dwk, void *workspace, size_t workspace_bytes, const int32_t *cu_seqlens,
    int32_t B, int64_t T, int32_t Hq, int32_t Hkv, int32_t D, double theta,
    const double *inv_freq, float eps, const uint32_t *seqlens_status, ftk_dtype dtype,
    ftk_stream_t stream) {
  if (!seqlens_status && T > 0) return FTK_ERR_NULL;
  return qk_norm_rope_bwd(dq_out, ld_gq, dk_out, ld_gk, q, ld_q, k, ld_k, wq, wk, rstd_q, rstd_k,
                          dq, ld_dq, dk, ld_dk, dwq, dwk, workspace, workspace_bytes, cu_seqlens,
                          B, T, Hq, Hkv, D, theta, inv_freq, eps, dtype, stream, seqlens_status);
}

// ------------------------------------------------------ tensor-core GEMM

FTK_API ftk_status ftk_gemm_bf16_ex(const void *a, int64_t lda, int a_mn, const void *b,
                                    int64_t ldb, int b_mn, float *c, int64_t ldc, int64_t M,
                                    int64_t N, int64_t K, ftk_stream_t stream) {
  if (M < 0 || N < 0 || K < 0 || lda < (a_mn ? M : K) || ldb < (b_mn ? N : K) || ldc < N ||
      M >= (int64_t(1) << 31) || N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31))
    return FTK_ERR_SHAPE;
  if (M == 0 || N == 0) return FTK_OK;
  if (!a || !b || !c) return FTK_ERR_NULL;
  if (K > 0 && (!aligned(a, 16) || !aligned(b, 16) || lda % 8 != 0 || ldb % 8 != 0))
    return FTK_ERR_ALIGN;
  if (!aligned(c, 4)) return FTK_ERR_ALIGN;
  if (K == 0) return FTK_ERR_SHAPE;  // an empty contraction has nothing to run on
  const View va = a_mn ? view(a, K, lda, M, 2) : view(a, M, lda, K, 2);
  const View vb = b_mn ? view(b, K, ldb, N, 2) : view(b, N, ldb, K, 2);
  const View vc = view(c, M, ldc, N, 4);
  if (may_overlap(vc, va) || may_overlap(vc, vb)) return FTK_ERR_ALIAS;
  ftk::DeviceInfo dev;
  cudaError_t e = device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  return finish(ftk::launch_gemm_bf16(a, lda, a_mn != 0, b, ldb, b_mn != 0, c, ldc, M, N, K, dev,
                                      (cudaStream_t)stream));
}

FTK_API ftk_status ftk_gemm_bf16(const void *a, int64_t lda, const void *b, int64_t ldb,
                                 float *c, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                 ftk_stream_t stream) {
  return ftk_gemm_bf16_ex(a, lda, 0, b, ldb, 0, c, ldc, M, N, K, stream);
}

// ------------------------------------------------------ Cut Cross-Entropy

FTK_API size_t ftk_cce_fwd_workspace_bytes(int64_t T, int64_t V) {
  if (T <= 0 || V <= 0) return 0;
  return ftk::cce_fwd_workspace_bytes(T, V);
}

FTK_API size_t ftk_cce_bwd_workspace_bytes(int64_t T, int64_t H, int64_t V) {
  if (T <= 0 || H <= 0 || V <= 0) return 0;
  return ftk::cce_bwd_workspace_bytes(T, H, V);
}

FTK_API int64_t ftk_cce_bwd_chunk(int64_t T, int64_t H, int64_t V, int32_t sms) {
  if (T <= 0 || H <= 0 || V <= 0 || sms <= 0) return 0;
  return ftk::cce_bwd_chunk(T, H, V, sms);
}

}  // extern "C"

namespace {

// Checks shared by the CCE forward and backward: shapes, the TMA rules on
// h and W (16-byte aligned bases, row strides a multiple of 8 elements), y.
ftk_status cce_common(const void *h, int64_t ldh, const void *w, int64_t ldw, const int32_t *y,
                      int64_t T, int64_t H, int64_t V, ftk_dtype dtype) {
  if (!valid_dtype(dtype)) return FTK_ERR_DTYPE;
  if (dtype != FTK_BF16) return FTK_ERR_DTYPE;  // the tensor-core path is bf16
  if (T < 0 || H < 1 || V < 1 || ldh < H || ldw < H || T >= (int64_t(1) << 31) ||
      V >= (int64_t(1) << 31) || H >= (int64_t(1) << 31))
    return FTK_ERR_SHAPE;
  if (T == 0) return FTK_OK;
  if (!h || !w || !y) return FTK_ERR_NULL;
  if (!aligned(h, 16) || !aligned(w, 16) || ldh % 8 != 0 || ldw % 8 != 0 || !aligned(y, 4))
    return FTK_ERR_ALIGN;
  return FTK_OK;
}

}  // namespace

extern "C" {

FTK_API ftk_status ftk_cce_fwd(const void *h, int64_t ldh, const void *w, int64_t ldw,
                               const int32_t *y, int64_t T, int64_t H, int64_t V, float *loss,
                               float *lse, void *workspace, size_t workspace_bytes,
                               ftk_dtype dtype, ftk_stream_t stream) {
  ftk_status st = cce_common(h, ldh, w, ldw, y, T, H, V, dtype);
  if (st != FTK_OK || T == 0) return st;
  if (!loss || !lse) return FTK_ERR_NULL;
  if (!workspace || workspace_bytes < ftk::cce_fwd_workspace_bytes(T, V))
    return FTK_ERR_WORKSPACE;
  if (!aligned(loss, 4) || !aligned(lse, 4) || !aligned(workspace, 256)) return FTK_ERR_ALIGN;
  const View vh = view(h, T, ldh, H, 2), vw = view(w, V, ldw, H, 2), vy = view(y, 1, T, T, 4);
  const View vl = view(loss, 1, 1, 1, 4), vs = view(lse, 1, T, T, 4);
  const View vws = view(workspace, 1, (int64_t)workspace_bytes, (int64_t)workspace_bytes, 1);
  const View outs[3] = {vl, vs, vws}, ins[3] = {vh, vw, vy};
  for (int i = 0; i < 3; ++i) {
    for (int m = 0; m < 3; ++m)
      if (may_overlap(outs[i], ins[m])) return FTK_ERR_ALIAS;
    for (int m = i + 1; m < 3; ++m)
      if (may_overlap(outs[i], outs[m])) return FTK_ERR_ALIAS;
  }
  ftk::DeviceInfo dev;
  cudaError_t e = device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  ftk::CceArgs a{h, ldh, w, ldw, y, T, H, V, loss, lse, nullptr, nullptr, 0, nullptr, 0,
                 workspace};
  return finish(ftk::launch_cce_fwd(a, dev, (cudaStream_t)stream));
}

FTK_API ftk_status ftk_cce_bwd(const void *h, int64_t ldh, const void *w, int64_t ldw,
                               const int32_t *y, const float *lse, const float *dloss,
                               int64_t T, int64_t H, int64_t V, void *dh, int64_t lddh,
                               float *dw, int64_t lddw, void *workspace,
                               size_t workspace_bytes, ftk_dtype dtype, ftk_stream_t stream) {
  ftk_status st = cce_common(h, ldh, w, ldw, y, T, H, V, dtype);
  if (st != FTK_OK) return st;
  if (lddh < H || lddw < H) return FTK_ERR_SHAPE;
  if (T == 0) return FTK_OK;
  if (!lse || !dloss || !dh || !dw) return FTK_ERR_NULL;
  if (!workspace || workspace_bytes < ftk::cce_bwd_workspace_bytes(T, H, V))
    return FTK_ERR_WORKSPACE;
  if (!aligned(lse, 4) || !aligned(dloss, 4) || !aligned(dh, 2) || !aligned(dw, 4) ||
      !aligned(workspace, 256))
    return FTK_ERR_ALIGN;
  const View vh = view(h, T, ldh, H, 2), vw = view(w, V, ldw, H, 2), vy = view(y, 1, T, T, 4);
  const View vs = view(lse, 1, T, T, 4), vg = view(dloss, 1, 1, 1, 4);
  const View vdh = view(dh, T, lddh, H, 2), vdw = view(dw, V, lddw, H, 4);
  const View vws = view(workspace, 1, (int64_t)workspace_bytes, (int64_t)workspace_bytes, 1);
  const View outs[3] = {vdh, vdw, vws}, ins[5] = {vh, vw, vy, vs, vg};
  for (int i = 0; i < 3; ++i) {
    for (int m = 0; m < 5; ++m)
      if (may_overlap(outs[i], ins[m])) return FTK_ERR_ALIAS;
    for (int m = i + 1; m < 3; ++m)
      if (may_overlap(outs[i], outs[m])) return FTK_ERR_ALIAS;
  }
  ftk::DeviceInfo dev;
  cudaError_t e = device_info(&dev);
  if (e != cudaSuccess) return cuda_fail(e);
  ftk::CceArgs a{h, ldh, w, ldw, y, T, H, V, nullptr, (float *)lse, dloss, dh, lddh, dw, lddw,
                 workspace};
  return finish(ftk::launch_cce_bwd(a, dev, (cudaStream_t)stream));
}

}  // extern "C"
