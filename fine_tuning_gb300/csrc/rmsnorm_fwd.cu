// RMSNorm forward:  y[t,j] = x[t,j] * r[t] * w[j],
//                   r[t]   = 1 / sqrt(mean_j x[t,j]^2 + eps)
// (Chronicals, arXiv 2601.02609, abstract, optimisation (1): fused RMSNorm.)
//
// One row is read from HBM once and written once.  A group of W warps owns a
// row: each thread holds V packets of the row in registers, the sum of
// squares is reduced with warp shuffles (and, for W > 1, through shared
// memory in a fixed order), then every thread scales its own packets.  R row
// groups share a CTA so that CTAs stay at 128-256 threads for any H.
// Rows too long for registers take a CTA-per-row two-pass kernel.
#include "common.cuh"
#include "launch.h"

namespace ftk {

RowPlan plan_rmsnorm_row(int64_t H, int pack) {
  RowPlan p;
  p.pack = pack;
  const int64_t hp = H / pack;  // packets per row
  int64_t W = ceil_div(hp, (int64_t)128);
  if (W > 8) W = 8;
  int64_t V = ceil_div(hp, 32 * W);
  static const int kV[] = {1, 2, 3, 4, 6, 8};
  int v = 0;
  for (int c : kV)
    if (c >= V) { v = c; break; }
  if (v == 0) {
    p.generic = true;
    return p;
  }
  p.W = (int)W;
  p.V = v;
  p.R = (int)(8 / W) > 0 ? (int)(8 / W) : 1;
  return p;
}

template <typename T, typename Idx, int N, int V>
__global__ void __launch_bounds__(256)
rmsnorm_fwd_rows(const T *x, Idx ldx, const T *__restrict__ w, T *y, Idx ldy,
                 float *__restrict__ rstd, Idx rows, int hp, float inv_h, float eps,
                 int W, int R) {
  extern __shared__ float red[];  // [R][W] warp partial sums
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / W, wig = warp - grp * W;
  const int gi = wig * 32 + lane, G = W * 32;
  const Idx row = (Idx)blockIdx.x * R + grp;
  const bool active = row < rows;

  Packet<T, N> xv[V];
  float ss = 0.f;
  if (active) {
    const T *xr = x + row * ldx;
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const int c = gi + k * G;
      if (c < hp) xv[k] = load_packet_stream<T, N>(xr + (Idx)c * N);
    }
#pragma unroll
    for (int k = 0; k < V; ++k) {
      if (gi + k * G < hp) {
#pragma unroll
        for (int e = 0; e < N; ++e) {
          const float f = xv[k].get(e);
          ss = fmaf(f, f, ss);
        }
      }
    }
  }
  ss = warp_sum(ss);
  if (W > 1) {
    if (lane == 0) red[grp * W + wig] = ss;
    __syncthreads();
    ss = 0.f;
    for (int i = 0; i < W; ++i) ss += red[grp * W + i];
  }
  if (!active) return;

  const float r = rsqrtf(fmaf(ss, inv_h, eps));
  if (rstd != nullptr && gi == 0) rstd[row] = r;
  T *yr = y + row * ldy;
#pragma unroll
  for (int k = 0; k < V; ++k) {
    const int c = gi + k * G;
    if (c < hp) {
      const Packet<T, N> wv = load_packet<T, N>(w + (Idx)c * N);
      Packet<T, N> o;
#pragma unroll
      for (int e = 0; e < N; ++e) o.set(e, (xv[k].get(e) * r) * wv.get(e));
      store_packet<T, N>(yr + (Idx)c * N, o);
    }
  }
}

// Rows longer than the register plan: one CTA per row (grid-stride over
// rows), sum of squares first, then a second pass that re-reads x (from L2).
template <typename T, typename Idx>
__global__ void __launch_bounds__(256)
rmsnorm_fwd_generic(const T *x, Idx ldx, const T *__restrict__ w, T *y, Idx ldy,
                    float *__restrict__ rstd, Idx rows, Idx H, float inv_h, float eps) {
  __shared__ float red[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (Idx row = blockIdx.x; row < rows; row += gridDim.x) {
    const T *xr = x + row * ldx;
    float ss = 0.f;
    for (Idx j = threadIdx.x; j < H; j += blockDim.x) {
      const float f = to_float(xr[j]);
      ss = fmaf(f, f, ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();
    ss = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) ss += red[i];
    __syncthreads();  // red is reused by the next row
    const float r = rsqrtf(fmaf(ss, inv_h, eps));
    if (rstd != nullptr && threadIdx.x == 0) rstd[row] = r;
    T *yr = y + row * ldy;
    for (Idx j = threadIdx.x; j < H; j += blockDim.x)
      yr[j] = from_float<T>((to_float(xr[j]) * r) * to_float(w[j]));
  }
}

template <typename T, typename Idx, int N>
static cudaError_t fwd_rows(const RowPlan &p, const RmsNormFwdArgs &a, cudaStream_t s) {
  const Idx rows = (Idx)a.T;
  const dim3 grid((unsigned)ceil_div(a.T, (int64_t)p.R));
  const size_t smem = sizeof(float) * p.R * p.W;
  const int hp = (int)(a.H / N);
  const float inv_h = (float)(1.0 / (double)a.H);
#define FTK_FWD_CASE(VV)                                                          \
  case VV:                                                                        \
    rmsnorm_fwd_rows<T, Idx, N, VV><<<grid, p.threads(), smem, s>>>(               \
        (const T *)a.x, (Idx)a.ldx, (const T *)a.w, (T *)a.y, (Idx)a.ldy, a.rstd, \
        rows, hp, inv_h, a.eps, p.W, p.R);                                        \
    break;
  switch (p.V) {
    FTK_FWD_CASE(1)
    FTK_FWD_CASE(2)
    FTK_FWD_CASE(3)
    FTK_FWD_CASE(4)
    FTK_FWD_CASE(6)
    FTK_FWD_CASE(8)
    default:
      return cudaErrorInvalidConfiguration;
  }
#undef FTK_FWD_CASE
  return cudaGetLastError();
}

template <typename T, typename Idx>
static cudaError_t fwd_typed(bool vec, const RmsNormFwdArgs &a, const DeviceInfo &dev,
                             cudaStream_t s) {
  constexpr int NV = VecWidth<T>::value;
  const RowPlan p = plan_rmsnorm_row(a.H, vec ? NV : 1);
  if (p.generic) {
    int64_t grid = a.T < (int64_t)dev.sms * 16 ? a.T : (int64_t)dev.sms * 16;
    rmsnorm_fwd_generic<T, Idx><<<(unsigned)grid, 256, 0, s>>>(
        (const T *)a.x, (Idx)a.ldx, (const T *)a.w, (T *)a.y, (Idx)a.ldy, a.rstd,
        (Idx)a.T, (Idx)a.H, (float)(1.0 / (double)a.H), a.eps);
    return cudaGetLastError();
  }
  return vec ? fwd_rows<T, Idx, NV>(p, a, s) : fwd_rows<T, Idx, 1>(p, a, s);
}

cudaError_t launch_rmsnorm_fwd(DType dt, bool vec, bool wide, const RmsNormFwdArgs &a,
                               const DeviceInfo &dev, cudaStream_t s) {
  if (dt == DType::F32)
    return wide ? fwd_typed<float, int64_t>(vec, a, dev, s)
                : fwd_typed<float, int32_t>(vec, a, dev, s);
  return wide ? fwd_typed<bf16, int64_t>(vec, a, dev, s)
              : fwd_typed<bf16, int32_t>(vec, a, dev, s);
}

}  // namespace ftk
