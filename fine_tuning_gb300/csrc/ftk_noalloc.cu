// ftk_rmsnorm_bwd_noalloc: the RMSNorm backward for callers that cannot
// allocate device memory.
//
// ftk_rmsnorm_bwd needs a caller-provided workspace for its per-CTA dw
// partial sums.  Some callers cannot provide one: code running where
// cudaMalloc is not allowed or not wanted (inside a pre-sized memory pool
// whose budget is fixed, a runtime that forbids allocation after start-up,
// or a plugin handed only input and output pointers by its host framework).
// This entry point uses instead a scratch array that lives in the library
// itself: a file-scope __device__ array of fixed size, created when the
// library is loaded on a device and held by that device until the process
// exits.  It allocates nothing per call.
//
// Set-up: the first call on each device looks up the array's device address
// with cudaGetSymbolAddress (the symbol's name in host code is only a
// host-side stand-in, never a device address) and caches it for that
// device.  Make that first call before any stream capture.
//
// The array is shared by every call on a device and keeps the last call's
// contents.  Nothing in it needs to start at zero: each call writes every
// partial row it later sums.  Calls whose executions overlap on the GPU
// (different streams, or a graph replayed concurrently) race on the array
// and must be serialised by the caller.
#include <mutex>

#include "ftk.h"
#include "launch.h"

namespace {

// 4 MiB of fp32 dw partial sums: P rows of H values.  One row must fit, so
// H <= 1,048,576; a larger H leaves fewer rows and thus fewer CTAs.
constexpr size_t kScratchFloats = size_t(1) << 20;

static __device__ __align__(256) float g_dw_scratch[kScratchFloats];

std::mutex g_scratch_mutex;
float *g_scratch_ptr[64];

// Device address of g_dw_scratch on the current device (set-up on first use).
cudaError_t scratch_on_current_device(float **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_dw_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<float *>(p);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

FTK_API ftk_status ftk_rmsnorm_bwd_noalloc(const void *dy, int64_t lddy, const void *x,
                                           int64_t ldx, const void *w, const float *rstd,
                                           void *dx, int64_t lddx, float *dw, int64_t T,
                                           int64_t H, float eps, ftk_dtype dtype,
                                           ftk_stream_t stream) {
  if (H > (int64_t)kScratchFloats) return FTK_ERR_WORKSPACE;  // one partial row must fit
  if (T <= 0 || H < 1)  // empty or invalid: no set-up, same answer as ftk_rmsnorm_bwd
    return ftk_rmsnorm_bwd(dy, lddy, x, ldx, w, rstd, dx, lddx, dw, nullptr, 0, T, H, eps,
                           dtype, stream);
  float *scratch = nullptr;
  cudaError_t e = scratch_on_current_device(&scratch);
  if (e != cudaSuccess) return FTK_ERR_CUDA;
  return ftk_rmsnorm_bwd(dy, lddy, x, ldx, w, rstd, dx, lddx, dw, scratch,
                         kScratchFloats * sizeof(float), T, H, eps, dtype, stream);
}

}  // extern "C"
