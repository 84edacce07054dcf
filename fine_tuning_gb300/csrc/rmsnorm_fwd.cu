// RMSNorm forward:  y[t,j] = x[t,j] * r[t] * w[j],
//                   r[t]   = 1 / sqrt(mean_j x[t,j]^2 + eps)
// (Chronicals, arXiv 2601.02609, abstract, optimisation (1): fused RMSNorm.)
//
// One row is read from HBM once and written once.  A group of W warps owns a
// row; the sum of squares is reduced with warp shuffles (and, for W > 1,
// through shared memory in a fixed order), then every thread scales its own
// packets.  R row groups share a CTA so that CTAs stay at 128-256 threads.
//
// 16-byte aligned rows take rmsnorm_fwd_staged: a persistent grid in which
// one elected thread per row group streams the group's next S rows into a
// ring of shared-memory stages with bulk copies (cp.async.bulk, the TMA
// engine's 1-D mode) completing on mbarriers; the warps compute from shared
// memory.  Bytes in flight then cost no registers, and a row's copy starts
// S rows before it is needed.  Other rows hold their packets in registers
// (rmsnorm_fwd_rows); rows too long for either take a CTA-per-row kernel.
#include "common.cuh"
#include "launch.h"

namespace ftk {

RowPlan plan_rmsnorm_row(int64_t H, int pack, int vmax) {
  RowPlan p;
  p.pack = pack;
  const int64_t hp = H / pack;  // packets per row
  int64_t W = ceil_div(hp, (int64_t)32 * vmax);
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

StagedPlan plan_rmsnorm_staged(const RowPlan &p, int64_t H, int elem_bytes, int nbuf,
                               const DeviceInfo &dev) {
  StagedPlan sp;
  if (p.generic || p.pack == 1) return sp;
  sp.row_bytes = (uint32_t)(H * elem_bytes);
  sp.stage_bytes = sp.row_bytes * (uint32_t)nbuf;
  // Aim for ~6 row groups computing per SM (at least 2 CTAs) and ~200 KiB of
  // stages per SM in all; each group gets 2..8 stages.
  const int ctas = p.R >= 3 ? 2 : (6 + p.R - 1) / p.R;
  int S = (int)((204800 / ctas) / ((size_t)p.R * sp.stage_bytes));
  S = S < 2 ? 2 : (S > 8 ? 8 : S);
  for (; S >= 2; --S) {
    sp.off_red = ((size_t)p.R * S * 8 + 15) / 16 * 16;
    sp.off_stage = (sp.off_red + (size_t)p.R * p.W * 8 + 127) / 128 * 128;
    sp.smem = sp.off_stage + (size_t)p.R * S * sp.stage_bytes;
    if (sp.smem <= (size_t)dev.max_smem_optin) {
      sp.S = S;
      return sp;
    }
  }
  sp.S = 0;
  return sp;
}

template <typename T, typename Idx, int N, int V>
__global__ void __launch_bounds__(256)
rmsnorm_fwd_staged(const T *x, Idx ldx, const T *__restrict__ w, T *y, Idx ldy,
                   float *__restrict__ rstd, Idx rows, int hp, float inv_h, float eps, int W,
                   int R, int S, uint32_t off_red, uint32_t off_stage, uint32_t row_bytes,
                   unsigned *status, long long wait_limit) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem);  // [R][S]
  float *red = reinterpret_cast<float *>(smem + off_red);  // [R][W]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / W, wig = warp - grp * W;
  const int gi = wig * 32 + lane, G = W * 32;
  const bool leader = gi == 0;

  for (int i = threadIdx.x; i < R * S; i += blockDim.x) mbar_init(&bars[i], 1);
  if (threadIdx.x == 0) fence_mbar_init();
  __syncthreads();
  pdl_wait();
  pdl_trigger();

  uint64_t *gb = bars + grp * S;
  unsigned char *ring = smem + off_stage + (size_t)grp * S * row_bytes;
  const Idx stride = (Idx)gridDim.x * R;
  const Idx first = (Idx)blockIdx.x * R + grp;

  int issued = 0;  // copies issued by the leader
  if (leader) {
    for (int s = 0; s < S; ++s) {
      const Idx row = first + (Idx)s * stride;
      if (row >= rows) break;
      mbar_arrive_expect_tx(&gb[s], row_bytes);
      bulk_copy_g2s(ring + (size_t)s * row_bytes, x + row * ldx, row_bytes, &gb[s]);
      ++issued;
    }
  }
  Packet<T, N> wv[V];
#pragma unroll
  for (int k = 0; k < V; ++k) {
    const int c = gi + k * G;
    if (c < hp) wv[k] = load_packet<T, N>(w + (Idx)c * N);
  }

  bool live = true;  // false once one of this thread's waits has run out
  int it = 0;
  for (Idx row = first; row < rows; row += stride, ++it) {
    const int s = it % S;
    if (live) live = mbar_wait_bounded(&gb[s], (uint32_t)((it / S) & 1), wait_limit, status);
    const T *xs = reinterpret_cast<const T *>(ring + (size_t)s * row_bytes);
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const int c = gi + k * G;
      if (c < hp) {
        const Packet<T, N> v = *reinterpret_cast<const Packet<T, N> *>(xs + c * N);
#pragma unroll
        for (int e = 0; e < N; ++e) {
          const float f = v.get(e);
          ss = fmaf(f, f, ss);
        }
      }
    }
    ss = warp_sum(ss);
    if (W > 1) {
      if (lane == 0) red[grp * W + wig] = ss;
      named_barrier(1 + grp, G);
      ss = 0.f;
      for (int i = 0; i < W; ++i) ss += red[grp * W + i];
    }
    const float r = rsqrtf(fmaf(ss, inv_h, eps));
    if (rstd != nullptr && leader) rstd[row] = r;
    T *yr = y + row * ldy;
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const int c = gi + k * G;
      if (c < hp) {
        const Packet<T, N> v = *reinterpret_cast<const Packet<T, N> *>(xs + c * N);
        Packet<T, N> o;
#pragma unroll
        for (int e = 0; e < N; ++e) o.set(e, (v.get(e) * r) * wv[k].get(e));
        store_packet<T, N>(yr + (Idx)c * N, o);
      }
    }
    // the whole group has read stage s (and the reduction slots): refill it
    if (W > 1)
      named_barrier(1 + grp, G);
    else
      __syncwarp();
    if (leader) {
      const Idx next = row + (Idx)S * stride;
      if (next < rows) {
        fence_proxy_async_smem();
        mbar_arrive_expect_tx(&gb[s], row_bytes);
        bulk_copy_g2s(ring + (size_t)s * row_bytes, x + next * ldx, row_bytes, &gb[s]);
        ++issued;
      }
    }
  }
  // after a wait ran out, let the copies still in flight land (bounded)
  // before the CTA's shared memory is released
  if (leader && !live)
    for (int i = it; i < issued; ++i)
      mbar_wait_bounded(&gb[i % S], (uint32_t)((i / S) & 1), wait_limit, status);
}

template <typename T, typename Idx, int N, int V>
__global__ void __launch_bounds__(256)
rmsnorm_fwd_rows(const T *x, Idx ldx, const T *__restrict__ w, T *y, Idx ldy,
                 float *__restrict__ rstd, Idx rows, int hp, float inv_h, float eps,
                 int W, int R) {
  extern __shared__ float red[];  // [R][W] warp partial sums
  pdl_wait();
  pdl_trigger();
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
  pdl_wait();
  pdl_trigger();
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
    {                                                                             \
      cudaError_t le_ = launch_pdl(rmsnorm_fwd_rows<T, Idx, N, VV>, dim3(grid), dim3(p.threads()), smem, s, \
                                    (const T *)a.x, (Idx)a.ldx, (const T *)a.w, (T *)a.y, (Idx)a.ldy, a.rstd, rows, hp, inv_h, a.eps, p.W, p.R); \
      if (le_ != cudaSuccess) return le_;                                          \
    }                                        \
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

template <typename T, typename Idx, int N, int V>
static cudaError_t fwd_staged_v(const RowPlan &p, const StagedPlan &sp, const RmsNormFwdArgs &a,
                                const DeviceInfo &dev, cudaStream_t s) {
  auto kern = rmsnorm_fwd_staged<T, Idx, N, V>;
  const int threads = p.threads();
  const int occ = blocks_per_sm((const void *)kern, threads, sp.smem, dev, 8);
  int64_t P = ceil_div(a.T, (int64_t)p.R);
  if (P > (int64_t)dev.sms * occ) P = (int64_t)dev.sms * occ;
  unsigned *status = nullptr;
  cudaError_t e = device_status_ptr(dev, &status);
  if (e != cudaSuccess) return e;
  {
    cudaError_t le_ = launch_pdl(kern, dim3((unsigned)P), dim3(threads), sp.smem, s,
                                 (const T *)a.x, (Idx)a.ldx, (const T *)a.w, (T *)a.y, (Idx)a.ldy, a.rstd, (Idx)a.T,
      (int)(a.H / N), (float)(1.0 / (double)a.H), a.eps, p.W, p.R, sp.S, (uint32_t)sp.off_red,
      (uint32_t)sp.off_stage, sp.row_bytes, status, kWaitLimitCycles);
    if (le_ != cudaSuccess) return le_;
  }
  return cudaGetLastError();
}

template <typename T, typename Idx, int N>
static cudaError_t fwd_staged(const RowPlan &p, const StagedPlan &sp, const RmsNormFwdArgs &a,
                              const DeviceInfo &dev, cudaStream_t s) {
  switch (p.V) {
    case 1: return fwd_staged_v<T, Idx, N, 1>(p, sp, a, dev, s);
    case 2: return fwd_staged_v<T, Idx, N, 2>(p, sp, a, dev, s);
    case 3: return fwd_staged_v<T, Idx, N, 3>(p, sp, a, dev, s);
    case 4: return fwd_staged_v<T, Idx, N, 4>(p, sp, a, dev, s);
    case 6: return fwd_staged_v<T, Idx, N, 6>(p, sp, a, dev, s);
    case 8: return fwd_staged_v<T, Idx, N, 8>(p, sp, a, dev, s);
    default: return cudaErrorInvalidConfiguration;
  }
}

template <typename T, typename Idx>
static cudaError_t fwd_typed(bool vec, const RmsNormFwdArgs &a, const DeviceInfo &dev,
                             cudaStream_t s) {
  constexpr int NV = VecWidth<T>::value;
  const RowPlan p = plan_rmsnorm_row(a.H, vec ? NV : 1, 4);
  // The staged pipeline pays off once every row group streams a dozen rows
  // or more; smaller batches finish sooner with one row per group and the
  // hardware scheduler refilling SMs (rmsnorm_fwd_rows).
  if (vec && !p.generic && a.T >= (int64_t)12 * p.R * 2 * dev.sms) {
    const StagedPlan sp = plan_rmsnorm_staged(p, a.H, (int)sizeof(T), 1, dev);
    if (sp.S > 0) return fwd_staged<T, Idx, NV>(p, sp, a, dev, s);
  }
  if (p.generic) {
    int64_t grid = a.T < (int64_t)dev.sms * 16 ? a.T : (int64_t)dev.sms * 16;
    {
      cudaError_t le_ = launch_pdl(rmsnorm_fwd_generic<T, Idx>, dim3((unsigned)grid), dim3(256), 0, s,
                                   (const T *)a.x, (Idx)a.ldx, (const T *)a.w, (T *)a.y, (Idx)a.ldy, a.rstd,
        (Idx)a.T, (Idx)a.H, (float)(1.0 / (double)a.H), a.eps);
      if (le_ != cudaSuccess) return le_;
    }
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
