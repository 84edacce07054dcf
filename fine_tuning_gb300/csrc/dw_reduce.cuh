// Second pass of the deterministic weight gradients (RMSNorm's dw, the
// per-head QK-norm's dwq and dwk): out[j] = sum_{p < P} ws[p, j] over the
// fp32 partial rows the first pass wrote, one per CTA, in a fixed order.
#pragma once

#include "common.cuh"
#include "launch.h"

namespace ftk {

namespace {

// out[j] = sum_{p < P} ws[p * ld + j] for the columns j < H: a CTA owns 32
// columns; its 32 warps take the rows p = warp, warp + 32, ... and their sums
// are added in warp order.  Column j goes to out0[j] when j < split, else to
// out1[j - split] (two weights whose partial rows sit side by side); a null
// output is skipped.  Each thread loads its rows kReduceBatch at a time, all
// loads of a batch issued before the first add (up to 512 partial rows, one
// L2 round trip), and adds them in row order.
constexpr int kReduceWarps = 32;
constexpr int kReduceBatch = 16;

__global__ void __launch_bounds__(32 * kReduceWarps)
dw_reduce(const float *__restrict__ ws, int P, int H, int ld, float *__restrict__ out0, int split,
          float *__restrict__ out1, const uint32_t *__restrict__ skip) {
  __shared__ float part[kReduceWarps][33];
  pdl_wait();
  pdl_trigger();
  if (skip != nullptr && *skip != 0u) return;  // the first pass was skipped: outputs untouched
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int col = blockIdx.x * 32 + lane;
  float s = 0.f;
  if (col < H) {
    for (int p0 = warp; p0 < P; p0 += kReduceWarps * kReduceBatch) {
      float v[kReduceBatch];
#pragma unroll
      for (int i = 0; i < kReduceBatch; ++i) {
        const int p = p0 + i * kReduceWarps;
        v[i] = p < P ? __ldcg(ws + (size_t)p * ld + col) : 0.f;
      }
#pragma unroll
      for (int i = 0; i < kReduceBatch; ++i) s += v[i];  // + 0 past P leaves s unchanged
    }
  }
  part[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && col < H) {
    float t = 0.f;
#pragma unroll
    for (int i = 0; i < kReduceWarps; ++i) t += part[i][lane];
    float *const out = col < split ? out0 : out1;
    if (out) out[col < split ? col : col - split] = t;
  }
}

// Launches dw_reduce on the P partial rows (row stride ld) of H columns
// (PDL, like the first pass); columns [0, split) go to out0, the rest to
// out1; a non-zero word at `skip` (DEVICE, nullable) leaves both untouched.
// Also reports an error left by the first pass's launch.
inline cudaError_t launch_dw_reduce(const float *ws, int64_t P, int64_t H, int64_t ld,
                                    float *out0, int64_t split, float *out1, cudaStream_t s,
                                    const uint32_t *skip = nullptr) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = launch_pdl(dw_reduce, dim3((unsigned)ceil_div(H, (int64_t)32)), dim3(32 * kReduceWarps), 0,
                 s, ws, (int)P, (int)H, (int)ld, out0, (int)split, out1, skip);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// The single-output form: out[j] for all H columns.
inline cudaError_t launch_dw_reduce(const float *ws, int64_t P, int64_t H, int64_t ld, float *out,
                                    cudaStream_t s) {
  return launch_dw_reduce(ws, P, H, ld, out, H, nullptr, s);
}

}  // namespace

}  // namespace ftk
