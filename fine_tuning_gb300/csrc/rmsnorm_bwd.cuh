// RMSNorm backward (gradient of sum(dy * y), y = x * r * w):
//   c[t]    = sum_j dy[t,j] w[j] x[t,j]
//   dx[t,j] = r[t] w[j] dy[t,j] - r[t]^3 x[t,j] c[t] / H
//   dw[j]   = sum_t dy[t,j] x[t,j] r[t]
// (Chronicals, arXiv 2601.02609, abstract, optimisation (1): fused RMSNorm;
// the page gives no formula, this is the standard gradient.)
// With ADD (the pre-norm residual step h = x + res in front of the norm) the
// norm's input x is the stored h, and the gradient the residual stream
// carries into h, dh, is added: dx = dh + the expression above.  That one
// tensor is the gradient of both addends.
//
// Pass 1: a persistent grid of P CTAs walks the rows with a fixed stride.
// Each thread keeps its slice of w in registers for the whole kernel and
// accumulates dy*x*r for its columns in fp32 registers over the rows its
// group visits.  At the end the R row groups of a CTA are summed in shared
// memory in a fixed order and the CTA writes one fp32 row of partials to the
// workspace.  16-byte aligned rows of one warp (without dh) take
// rmsnorm_bwd_pipe, each lane streaming its packets of the next rows through
// a per-warp cp.async ring.  Other 16-byte aligned rows (rmsnorm_bwd_staged)
// have one elected thread per row group stream the next S rows of x and dy
// (and dh) into a ring of shared-memory stages with bulk copies
// (cp.async.bulk, completing on mbarriers) while the warps compute from
// shared memory; the rest hold their packets in registers
// (rmsnorm_bwd_rows).
// Pass 2 (dw_reduce): dw[j] = sum_p ws[p, j], rows in a fixed order.
// The row -> CTA map and every summation order are fixed, so dw is bitwise
// reproducible; no CTA ever waits on another.
//
// The kernels are templates on ADD; rmsnorm_bwd.cu instantiates the plain
// norm and rmsnorm_add_bwd.cu the residual form, so the two compile apart.
#pragma once

#include "common.cuh"
#include "dw_reduce.cuh"
#include "launch.h"
#include "pair_math.cuh"

namespace ftk {

namespace {

constexpr int kMaxBlocksPerSm = 8;

template <typename T, typename Idx> struct BwdParams {
  const T *dy;
  Idx lddy;
  const T *x;  // the norm's input (the stored h when ADD)
  Idx ldx;
  const T *dh;  // ADD only
  Idx lddh;
  const T *w;
  const float *rstd;  // nullable: recompute
  T *dx;
  Idx lddx;
  float *ws;
  Idx rows;
  int hp, H;  // packets per row, columns
  float inv_h, eps;
  int W, R;
};

// One output value: the norm's gradient, plus dh when ADD.
template <bool ADD>
__device__ __forceinline__ float dx_value(float a, float xf, float r, float wf, float gf,
                                          float dhf) {
  const float v = fmaf(-a, xf, r * wf * gf);
  return ADD ? dhf + v : v;
}

// Rows of one or two warps' plan (W <= 2): persistent, one row per group of
// W warps at a time, rows row, row + (8 / W) P, ...; each lane copies its
// packets of x and dy (and dh, and r when saved) of the group's next rows
// (bwd_pipe_bufs - 1 of them) into its warp's shared-memory ring with
// cp.async while it works on the current one.  Lane l of warp w in the
// group owns packets w 32 + l + k 32W (the row plan's columns and summation
// order); with W = 2 the two warps' sums meet in shared memory (slots
// double-buffered by row parity) behind a named barrier of the pair and are
// added in the plan's order.  The CTA's row groups combine their dw sums in
// a fixed order at the end, in the ring's memory, into the CTA's partial
// row.
// Ring depth in rows: 3 for rows of one warp (few rows per warp, so the
// loads of two rows ahead cover the ramp), 2 for two-warp rows (measured
// faster there).
template <int W> constexpr int bwd_pipe_bufs() { return W == 1 ? 3 : 2; }
template <int V, bool ADD> constexpr int bwd_pipe_slots() { return (ADD ? 3 : 2) * V + 1; }
template <int V, int W, bool ADD> constexpr size_t bwd_pipe_smem() {
  return sizeof(uint4) * 8 * bwd_pipe_bufs<W>() * bwd_pipe_slots<V, ADD>() * 32;  // 8 warps
}

template <typename T, typename Idx, int N, int V, int W, bool HAS_RSTD, bool ADD>
__global__ void __launch_bounds__(256) rmsnorm_bwd_pipe(const BwdParams<T, Idx> a) {
  constexpr int kSl = bwd_pipe_slots<V, ADD>();  // x[V], dy[V] (, dh[V]), r
  constexpr int kBufs = bwd_pipe_bufs<W>();
  constexpr int R = 8 / W;                       // row groups per CTA
  extern __shared__ uint4 ring[];                // [warps][kBufs][kSl][32]
  __shared__ float2 red[2][R][W];                // the groups' warp sums, by row parity
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / W, wig = warp - grp * W;
  const int hp = a.hp;
  uint4 *my = ring + warp * (kBufs * kSl * 32);
  auto col = [&](int k) { return wig * 32 + lane + k * 32 * W; };
  pdl_wait();
  pdl_trigger();

  Packet<T, N> wv[V];
#pragma unroll
  for (int k = 0; k < V; ++k)
    if (col(k) < hp) wv[k] = load_packet<T, N>(a.w + (Idx)col(k) * N);
  float acc[V][N];
#pragma unroll
  for (int k = 0; k < V; ++k)
#pragma unroll
    for (int e = 0; e < N; ++e) acc[k][e] = 0.f;

  const Idx step = (Idx)gridDim.x * R;
  auto stage = [&](Idx r, int b) {
    if (r < a.rows) {
      uint4 *d = my + b * kSl * 32 + lane;
#pragma unroll
      for (int k = 0; k < V; ++k) {
        const int c = col(k);
        if (c < hp) {
          cp_async16(d + k * 32, a.x + r * a.ldx + (Idx)c * N);
          cp_async16(d + (V + k) * 32, a.dy + r * a.lddy + (Idx)c * N);
          if (ADD) cp_async16(d + (2 * V + k) * 32, a.dh + r * a.lddh + (Idx)c * N);
        }
      }
      if (HAS_RSTD) cp_async4(d + (kSl - 1) * 32, a.rstd + r);
    }
    cp_async_commit();  // one group per row on every lane, empty or not
  };
  Idx row = (Idx)blockIdx.x * R + grp;
#pragma unroll
  for (int i = 0; i < kBufs - 1; ++i) stage(row + i * step, i);
  int b = 0, parity = 0;
  while (row < a.rows) {  // uniform across the group's warps
    // the loads of the next kBufs - 1 rows fly meanwhile
    stage(row + (kBufs - 1) * step, b == 0 ? kBufs - 1 : b - 1);
    cp_async_wait<kBufs - 1>();  // this lane's copies of `row` have landed
    const uint4 *d = my + b * kSl * 32 + lane;
    Packet<T, N> xv[V], gv[V];
    float2 cs = make_float2(0.f, 0.f);  // (sum dy*w*x, sum x*x)
    float2 s2 = make_float2(0.f, 0.f);  // sum x*x in the forward's order
#pragma unroll
    for (int k = 0; k < V; ++k) {
      if (col(k) < hp) {
        *reinterpret_cast<uint4 *>(&xv[k]) = d[k * 32];
        *reinterpret_cast<uint4 *>(&gv[k]) = d[(V + k) * 32];
#pragma unroll
        for (int e = 0; e < N; ++e) cs.x = fmaf(gv[k].get(e) * wv[k].get(e), xv[k].get(e), cs.x);
        if (!HAS_RSTD) sumsq_packet<T, N>(s2, xv[k]);
      }
    }
    if (!HAS_RSTD) cs.y = sumsq_total<T, N>(s2);
    if (HAS_RSTD)
      cs.x = warp_sum(cs.x);
    else
      cs = warp_sum2(cs);
    if (W > 1) {
      float2 *slot = red[parity][grp];
      if (lane == 0) slot[wig] = cs;
      group_barrier(grp, 32 * W);
      cs = make_float2(0.f, 0.f);
#pragma unroll
      for (int i = 0; i < W; ++i) {
        cs.x += slot[i].x;
        cs.y += slot[i].y;
      }
      parity ^= 1;
    }
    const float r = HAS_RSTD ? *reinterpret_cast<const float *>(d + (kSl - 1) * 32)
                             : rsqrtf(fmaf(cs.y, a.inv_h, a.eps));
    const float am = r * r * r * cs.x * a.inv_h;
    T *dr = a.dx + row * a.lddx;
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const int c = col(k);
      if (c < hp) {
        Packet<T, N> hv, o;
        if (ADD) *reinterpret_cast<uint4 *>(&hv) = d[(2 * V + k) * 32];
#pragma unroll
        for (int e = 0; e < N; ++e) {
          const float xf = xv[k].get(e), gf = gv[k].get(e);
          o.set(e, dx_value<ADD>(am, xf, r, wv[k].get(e), gf, ADD ? hv.get(e) : 0.f));
          acc[k][e] = fmaf(gf * xf, r, acc[k][e]);
        }
        store_packet<T, N>(dr + (Idx)c * N, o);
      }
    }
    row += step;
    b = b == kBufs - 1 ? 0 : b + 1;
  }
  cp_async_wait<0>();
  __syncthreads();  // every warp is done with its ring: it becomes [R][H] partials
  float *part = reinterpret_cast<float *>(ring);
  float *mine = part + grp * a.H;
#pragma unroll
  for (int k = 0; k < V; ++k) {
    const int c = col(k);
    if (c < hp)
#pragma unroll
      for (int e = 0; e < N; ++e) mine[c * N + e] = acc[k][e];
  }
  __syncthreads();
  float *dst = a.ws + (size_t)blockIdx.x * a.H;
  for (int j = threadIdx.x; j < a.H; j += blockDim.x) {
    float sum = 0.f;
    for (int g = 0; g < R; ++g) sum += part[g * a.H + j];
    dst[j] = sum;
  }
}

// bf16 rows of one warp (the backward of rmsnorm_fwd_lean):
// rmsnorm_bwd_pipe's persistent grid and per-warp cp.async ring (x, dy, with
// ADD dh, and r of the next rows, kLeanBwdBufs rows deep) with the lean pair
// arithmetic.  A row takes two sweeps over the lane's packets,
// held packed in registers: the first forms c = sum dy w x (and, without a
// saved r, sum x^2 in the forward's lean order), the second dx and the dw
// pair sums, which stay in registers across all the rows a warp visits.
// Both sweeps read the packets from the ring (the second re-reads them
// rather than keep 2V unpacked packets live across the row's reduction,
// which would spill).  Lane l owns packets l + 32 k (k < V).
constexpr int kLeanBwdBufs = 3;

template <int V, bool ADD> constexpr size_t bwd_lean_smem() {
  return sizeof(uint4) * 8 * kLeanBwdBufs * ((ADD ? 3 : 2) * V + 1) * 32;  // 8 warps
}

template <typename Idx, int V, bool HAS_RSTD, bool ADD>
__global__ void __launch_bounds__(256, 2) rmsnorm_bwd_lean(const BwdParams<bf16, Idx> a) {
  constexpr int kSl = (ADD ? 3 : 2) * V + 1;  // x[V], dy[V] (, dh[V]), r
  constexpr int kR = kSl - 1;                 // r's slot
  extern __shared__ uint4 ring[];  // [warps][kLeanBwdBufs][kSl][32]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint4 *const my = ring + warp * (kLeanBwdBufs * kSl * 32) + lane;
  pdl_wait();
  pdl_trigger();
  bool on[V];
  float2 wf[V][4], acc[V][4];
#pragma unroll
  for (int k = 0; k < V; ++k) {
    on[k] = lane + 32 * k < a.hp;
    uint4 u = make_uint4(0u, 0u, 0u, 0u);
    if (on[k]) u = *reinterpret_cast<const uint4 *>(a.w + (lane + 32 * k) * 8);
    unpack8(u, wf[k]);
#pragma unroll
    for (int p = 0; p < 4; ++p) acc[k][p] = make_float2(0.f, 0.f);
  }
  const Idx step = (Idx)gridDim.x * 8;
  Idx row = (Idx)blockIdx.x * 8 + warp;
  Idx srow = row;
  const bf16 *sx = a.x + row * a.ldx + lane * 8;
  const bf16 *sg = a.dy + row * a.lddy + lane * 8;
  const bf16 *sh = ADD ? a.dh + row * a.lddh + lane * 8 : nullptr;
  const Idx sx_step = step * a.ldx, sg_step = step * a.lddy, sh_step = ADD ? step * a.lddh : 0;
  int sslot = 0;
  auto stage = [&]() {
    if (srow < a.rows) {
      uint4 *d = my + sslot * (kSl * 32);
#pragma unroll
      for (int k = 0; k < V; ++k) {
        if (on[k]) {
          cp_async16(d + k * 32, sx + k * 256);
          cp_async16(d + (V + k) * 32, sg + k * 256);
          if (ADD) cp_async16(d + (2 * V + k) * 32, sh + k * 256);
        }
      }
      if (HAS_RSTD) cp_async4(d + kR * 32, a.rstd + srow);
    }
    cp_async_commit();  // one group per row on every lane, empty or not
    srow += step;
    sx += sx_step;
    sg += sg_step;
    if (ADD) sh += sh_step;
    sslot = sslot + 1 == kLeanBwdBufs ? 0 : sslot + 1;
  };
#pragma unroll
  for (int i = 0; i < kLeanBwdBufs - 1; ++i) stage();
  bf16 *dst = a.dx + row * a.lddx + lane * 8;
  const Idx dst_step = step * a.lddx;
  int slot = 0;
  while (row < a.rows) {  // warp-uniform
    stage();
    cp_async_wait<kLeanBwdBufs - 1>();  // this lane's copies of `row` have landed
    const uint4 *d = my + slot * (kSl * 32);
    float2 c2 = make_float2(0.f, 0.f), s2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < V; ++k) {
      float2 xf[4], gf[4];
      unpack8(on[k] ? d[k * 32] : make_uint4(0u, 0u, 0u, 0u), xf);
      unpack8(on[k] ? d[(V + k) * 32] : make_uint4(0u, 0u, 0u, 0u), gf);
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        c2 = __ffma2_rn(__fmul2_rn(gf[p], wf[k][p]), xf[p], c2);
        if (!HAS_RSTD) lean_sumsq_step(s2, xf[p]);
      }
    }
    float c, r;
    if (HAS_RSTD) {
      c = warp_sum(lean_lane_total(c2));
      r = *reinterpret_cast<const float *>(d + kR * 32);
    } else {
      const float2 cs = warp_sum2(make_float2(lean_lane_total(c2), lean_lane_total(s2)));
      c = cs.x;
      r = rsqrtf(fmaf(cs.y, a.inv_h, a.eps));
    }
    const float am = r * r * r * c * a.inv_h;
    const float2 r2 = make_float2(r, r), nam2 = make_float2(-am, -am);
    asm volatile("" ::: "memory");  // re-read the ring below instead of keeping the packets
#pragma unroll
    for (int k = 0; k < V; ++k) {
      if (on[k]) {
        float2 xf[4], gf[4], o[4];
        unpack8(d[k * 32], xf);
        unpack8(d[(V + k) * 32], gf);
#pragma unroll
        float2 hf[4];
        if (ADD) unpack8(d[(2 * V + k) * 32], hf);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          // dx = (dh +) r w dy - r^3 x c / H;  dw += dy x r
          o[p] = __ffma2_rn(nam2, xf[p], __fmul2_rn(r2, __fmul2_rn(gf[p], wf[k][p])));
          if (ADD) o[p] = __fadd2_rn(hf[p], o[p]);
          acc[k][p] = __ffma2_rn(__fmul2_rn(gf[p], xf[p]), r2, acc[k][p]);
        }
        *reinterpret_cast<uint4 *>(dst + k * 256) = pack8(o);
      }
    }
    row += step;
    dst += dst_step;
    slot = slot + 1 == kLeanBwdBufs ? 0 : slot + 1;
  }
  cp_async_wait<0>();
  __syncthreads();  // every warp is done with its ring: it becomes [8][H] partials
  float *part = reinterpret_cast<float *>(ring);
  float2 *mine = reinterpret_cast<float2 *>(part + warp * a.H);
#pragma unroll
  for (int k = 0; k < V; ++k)
    if (on[k])
#pragma unroll
      for (int p = 0; p < 4; ++p) mine[(lane + 32 * k) * 4 + p] = acc[k][p];
  __syncthreads();
  float *dstw = a.ws + (size_t)blockIdx.x * a.H;
  for (int j = threadIdx.x; j < a.H; j += blockDim.x) {
    float sum = 0.f;
#pragma unroll
    for (int g = 0; g < 8; ++g) sum += part[g * a.H + j];
    dstw[j] = sum;
  }
}

template <typename T, typename Idx, int N, int V, bool HAS_RSTD, bool ADD>
__global__ void __launch_bounds__(256) rmsnorm_bwd_rows(const BwdParams<T, Idx> a) {
  // [2][R][W] float2 reduction slots (double-buffered by row parity), then,
  // when R > 1, [R][H] fp32 dw partials for the final combine.
  extern __shared__ float smem[];
  const int W = a.W, R = a.R, hp = a.hp;
  float2 *red = reinterpret_cast<float2 *>(smem);
  float *part = smem + 4 * R * W;
  pdl_wait();
  pdl_trigger();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / W, wig = warp - grp * W;
  const int gi = wig * 32 + lane, G = W * 32;

  Packet<T, N> wv[V];
#pragma unroll
  for (int k = 0; k < V; ++k) {
    const int c = gi + k * G;
    if (c < hp) wv[k] = load_packet<T, N>(a.w + (Idx)c * N);
  }
  float acc[V][N];
#pragma unroll
  for (int k = 0; k < V; ++k)
#pragma unroll
    for (int e = 0; e < N; ++e) acc[k][e] = 0.f;

  int parity = 0;
  const Idx step = (Idx)gridDim.x * R;
  for (Idx base = (Idx)blockIdx.x * R; base < a.rows; base += step, parity ^= 1) {
    const Idx row = base + grp;
    const bool active = row < a.rows;
    Packet<T, N> xv[V], gv[V], hv[ADD ? V : 1];
    float r = 0.f;
    float2 cs = make_float2(0.f, 0.f);  // (sum dy*w*x, sum x*x)
    if (active) {
      const T *xr = a.x + row * a.ldx;
      const T *gr = a.dy + row * a.lddy;
#pragma unroll
      for (int k = 0; k < V; ++k) {
        const int c = gi + k * G;
        if (c < hp) {
          xv[k] = load_packet_stream<T, N>(xr + (Idx)c * N);
          gv[k] = load_packet_stream<T, N>(gr + (Idx)c * N);
          if (ADD) hv[ADD ? k : 0] = load_packet_stream<T, N>(a.dh + row * a.lddh + (Idx)c * N);
        }
      }
      if (HAS_RSTD) r = a.rstd[row];
      float2 s2 = make_float2(0.f, 0.f);  // sum x*x in the forward's order
#pragma unroll
      for (int k = 0; k < V; ++k) {
        if (gi + k * G < hp) {
#pragma unroll
          for (int e = 0; e < N; ++e) cs.x = fmaf(gv[k].get(e) * wv[k].get(e), xv[k].get(e), cs.x);
          if (!HAS_RSTD) sumsq_packet<T, N>(s2, xv[k]);
        }
      }
      if (!HAS_RSTD) cs.y = sumsq_total<T, N>(s2);
    }
    if (HAS_RSTD) {
      cs.x = warp_sum(cs.x);
    } else {
      cs = warp_sum2(cs);
    }
    if (W > 1) {
      float2 *slot = red + (parity * R + grp) * W;
      if (lane == 0) slot[wig] = cs;
      __syncthreads();
      cs = make_float2(0.f, 0.f);
      for (int i = 0; i < W; ++i) {
        cs.x += slot[i].x;
        cs.y += slot[i].y;
      }
    }
    if (active) {
      if (!HAS_RSTD) r = rsqrtf(fmaf(cs.y, a.inv_h, a.eps));
      const float am = r * r * r * cs.x * a.inv_h;
      T *dr = a.dx + row * a.lddx;
#pragma unroll
      for (int k = 0; k < V; ++k) {
        const int c = gi + k * G;
        if (c < hp) {
          Packet<T, N> o;
#pragma unroll
          for (int e = 0; e < N; ++e) {
            const float xf = xv[k].get(e), gf = gv[k].get(e);
            o.set(e, dx_value<ADD>(am, xf, r, wv[k].get(e), gf,
                                   ADD ? hv[ADD ? k : 0].get(e) : 0.f));
            acc[k][e] = fmaf(gf * xf, r, acc[k][e]);
          }
          store_packet<T, N>(dr + (Idx)c * N, o);
        }
      }
    }
  }

  float *dst = a.ws + (size_t)blockIdx.x * a.H;
  if (R == 1) {
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const int c = gi + k * G;
      if (c < hp)
#pragma unroll
        for (int e = 0; e < N; ++e) dst[c * N + e] = acc[k][e];
    }
    return;
  }
  float *mine = part + grp * a.H;
#pragma unroll
  for (int k = 0; k < V; ++k) {
    const int c = gi + k * G;
    if (c < hp)
#pragma unroll
      for (int e = 0; e < N; ++e) mine[c * N + e] = acc[k][e];
  }
  __syncthreads();
  for (int j = threadIdx.x; j < a.H; j += blockDim.x) {
    float sum = 0.f;
    for (int g = 0; g < R; ++g) sum += part[g * a.H + j];
    dst[j] = sum;
  }
}

// The staged backward's group barrier.  Its occupancy is set by registers
// (2-3 CTAs per SM), not by named barriers, yet the barrier's form still
// measured: at H = 5,120 the plain backward ran 1.4% faster with a run-time
// barrier id (2,333 against 2,366 us) and the residual form 1.7% faster with
// constant ids (3,028 against 3,080 us).
template <bool ADD> __device__ __forceinline__ void staged_bwd_barrier(int grp, int threads) {
  if constexpr (ADD)
    group_barrier(grp, threads);
  else
    named_barrier(1 + grp, threads);
}

template <typename T, typename Idx, int N, int V, bool HAS_RSTD, bool ADD>
__global__ void __launch_bounds__(256)
rmsnorm_bwd_staged(const BwdParams<T, Idx> a, int S, uint32_t off_red, uint32_t off_stage,
                   uint32_t row_bytes, unsigned *status, long long wait_limit) {
  extern __shared__ __align__(128) unsigned char sbuf[];
  const int W = a.W, R = a.R, hp = a.hp;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sbuf);  // [R][S]
  float2 *red = reinterpret_cast<float2 *>(sbuf + off_red);  // [R][W]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / W, wig = warp - grp * W;
  const int gi = wig * 32 + lane, G = W * 32;
  const bool leader = gi == 0;
  const uint32_t stage_bytes = (ADD ? 3 : 2) * row_bytes;  // x row, dy row (, dh row)

  for (int i = threadIdx.x; i < R * S; i += blockDim.x) mbar_init(&bars[i], 1);
  if (threadIdx.x == 0) fence_mbar_init();
  __syncthreads();
  pdl_wait();
  pdl_trigger();

  uint64_t *gb = bars + grp * S;
  unsigned char *ring = sbuf + off_stage + (size_t)grp * S * stage_bytes;
  const Idx stride = (Idx)gridDim.x * R;
  const Idx first = (Idx)blockIdx.x * R + grp;

  auto issue = [&](int s, Idx row) {
    unsigned char *st = ring + (size_t)s * stage_bytes;
    mbar_arrive_expect_tx(&gb[s], stage_bytes);
    bulk_copy_g2s(st, a.x + row * a.ldx, row_bytes, &gb[s]);
    bulk_copy_g2s(st + row_bytes, a.dy + row * a.lddy, row_bytes, &gb[s]);
    if (ADD) bulk_copy_g2s(st + 2 * row_bytes, a.dh + row * a.lddh, row_bytes, &gb[s]);
  };
  int issued = 0;
  if (leader) {
    for (int s = 0; s < S; ++s) {
      const Idx row = first + (Idx)s * stride;
      if (row >= a.rows) break;
      issue(s, row);
      ++issued;
    }
  }
  Packet<T, N> wv[V];
#pragma unroll
  for (int k = 0; k < V; ++k) {
    const int c = gi + k * G;
    if (c < hp) wv[k] = load_packet<T, N>(a.w + (Idx)c * N);
  }
  float acc[V][N];
#pragma unroll
  for (int k = 0; k < V; ++k)
#pragma unroll
    for (int e = 0; e < N; ++e) acc[k][e] = 0.f;

  bool live = true;
  int it = 0;
  // the saved r of each row is loaded one iteration ahead: the rows arrive
  // through the stages long before they are needed, so a load issued at the
  // row's own iteration would put a DRAM round trip on every row's path
  float r_next = (HAS_RSTD && first < a.rows) ? a.rstd[first] : 0.f;
  for (Idx row = first; row < a.rows; row += stride, ++it) {
    const int s = it % S;
    float r = r_next;
    if (HAS_RSTD && row + stride < a.rows) r_next = a.rstd[row + stride];
    if (live) live = mbar_wait_bounded(&gb[s], (uint32_t)((it / S) & 1), wait_limit, status);
    const unsigned char *st = ring + (size_t)s * stage_bytes;
    const T *xs = reinterpret_cast<const T *>(st);
    const T *gs = reinterpret_cast<const T *>(st + row_bytes);
    const T *hs = reinterpret_cast<const T *>(st + (ADD ? 2 : 1) * row_bytes);
    float2 cs = make_float2(0.f, 0.f);  // (sum dy*w*x, sum x*x)
    float2 s2 = make_float2(0.f, 0.f);  // sum x*x in the forward's order
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const int c = gi + k * G;
      if (c < hp) {
        const Packet<T, N> xv = *reinterpret_cast<const Packet<T, N> *>(xs + c * N);
        const Packet<T, N> gv = *reinterpret_cast<const Packet<T, N> *>(gs + c * N);
#pragma unroll
        for (int e = 0; e < N; ++e) cs.x = fmaf(gv.get(e) * wv[k].get(e), xv.get(e), cs.x);
        if (!HAS_RSTD) sumsq_packet<T, N>(s2, xv);
      }
    }
    if (!HAS_RSTD) cs.y = sumsq_total<T, N>(s2);
    if (HAS_RSTD)
      cs.x = warp_sum(cs.x);
    else
      cs = warp_sum2(cs);
    if (W > 1) {
      if (lane == 0) red[grp * W + wig] = cs;
      staged_bwd_barrier<ADD>(grp, G);
      cs = make_float2(0.f, 0.f);
      for (int i = 0; i < W; ++i) {
        cs.x += red[grp * W + i].x;
        cs.y += red[grp * W + i].y;
      }
    }
    if (!HAS_RSTD) r = rsqrtf(fmaf(cs.y, a.inv_h, a.eps));
    const float am = r * r * r * cs.x * a.inv_h;
    T *dr = a.dx + row * a.lddx;
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const int c = gi + k * G;
      if (c < hp) {
        const Packet<T, N> xv = *reinterpret_cast<const Packet<T, N> *>(xs + c * N);
        const Packet<T, N> gv = *reinterpret_cast<const Packet<T, N> *>(gs + c * N);
        Packet<T, N> hv;
        if (ADD) hv = *reinterpret_cast<const Packet<T, N> *>(hs + c * N);
        Packet<T, N> o;
#pragma unroll
        for (int e = 0; e < N; ++e) {
          const float xf = xv.get(e), gf = gv.get(e);
          o.set(e, dx_value<ADD>(am, xf, r, wv[k].get(e), gf, ADD ? hv.get(e) : 0.f));
          acc[k][e] = fmaf(gf * xf, r, acc[k][e]);
        }
        store_packet<T, N>(dr + (Idx)c * N, o);
      }
    }
    if (W > 1)
      staged_bwd_barrier<ADD>(grp, G);
    else
      __syncwarp();
    if (leader) {
      const Idx next = row + (Idx)S * stride;
      if (next < a.rows) {
        fence_proxy_async_smem();
        issue(s, next);
        ++issued;
      }
    }
  }
  if (leader && !live)
    for (int i = it; i < issued; ++i)
      mbar_wait_bounded(&gb[i % S], (uint32_t)((i / S) & 1), wait_limit, status);

  float *dst = a.ws + (size_t)blockIdx.x * a.H;
  if (R == 1) {
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const int c = gi + k * G;
      if (c < hp)
#pragma unroll
        for (int e = 0; e < N; ++e) dst[c * N + e] = acc[k][e];
    }
    return;
  }
  // the stages are free now: combine the R groups there in a fixed order
  __syncthreads();
  float *part = reinterpret_cast<float *>(sbuf + off_stage);
  float *mine = part + grp * a.H;
#pragma unroll
  for (int k = 0; k < V; ++k) {
    const int c = gi + k * G;
    if (c < hp)
#pragma unroll
      for (int e = 0; e < N; ++e) mine[c * N + e] = acc[k][e];
  }
  __syncthreads();
  for (int j = threadIdx.x; j < a.H; j += blockDim.x) {
    float sum = 0.f;
    for (int g = 0; g < R; ++g) sum += part[g * a.H + j];
    dst[j] = sum;
  }
}

// Rows too long for registers: one CTA per row at a time, persistent grid,
// two passes over the row; the CTA's dw partial row lives in the workspace
// and is updated in place (each CTA owns its row, so no atomics).
template <typename T, typename Idx, bool HAS_RSTD, bool ADD>
__global__ void __launch_bounds__(256) rmsnorm_bwd_generic(const BwdParams<T, Idx> a, Idx H) {
  __shared__ float2 red[8];
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float *mine = a.ws + (size_t)blockIdx.x * H;
  for (Idx j = threadIdx.x; j < H; j += blockDim.x) mine[j] = 0.f;
  for (Idx row = blockIdx.x; row < a.rows; row += gridDim.x) {
    const T *xr = a.x + row * a.ldx;
    const T *gr = a.dy + row * a.lddy;
    float2 cs = make_float2(0.f, 0.f);
    for (Idx j = threadIdx.x; j < H; j += blockDim.x) {
      const float xf = to_float(xr[j]);
      cs.x = fmaf(to_float(gr[j]) * to_float(a.w[j]), xf, cs.x);
      cs.y = fmaf(xf, xf, cs.y);
    }
    cs = warp_sum2(cs);
    if (lane == 0) red[warp] = cs;
    __syncthreads();
    cs = make_float2(0.f, 0.f);
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) {
      cs.x += red[i].x;
      cs.y += red[i].y;
    }
    __syncthreads();
    const float r = HAS_RSTD ? a.rstd[row] : rsqrtf(fmaf(cs.y, a.inv_h, a.eps));
    const float am = r * r * r * cs.x * a.inv_h;
    T *dr = a.dx + row * a.lddx;
    const T *hr = ADD ? a.dh + row * a.lddh : nullptr;
    for (Idx j = threadIdx.x; j < H; j += blockDim.x) {
      const float xf = to_float(xr[j]), gf = to_float(gr[j]);
      dr[j] = from_float<T>(
          dx_value<ADD>(am, xf, r, to_float(a.w[j]), gf, ADD ? to_float(hr[j]) : 0.f));
      mine[j] = fmaf(gf * xf, r, mine[j]);
    }
  }
}

cudaError_t launch_dw_reduce(const RmsNormBwdArgs &a, int64_t P, cudaStream_t s) {
  return launch_dw_reduce(a.ws, P, a.H, a.H, a.dw, s);
}

// Resident CTAs per SM of the saved-rstd and recomputing forms of a
// backward kernel, the smaller of the two.  The CTA count, and with it the
// row -> CTA map and the order in which dw is summed, is then the same in
// both modes, so dw does not depend on whether rstd was saved.
inline int min_blocks_per_sm(const void *with_rstd, const void *without, int threads, size_t smem,
                             const DeviceInfo &dev) {
  const int a = blocks_per_sm(with_rstd, threads, smem, dev, kMaxBlocksPerSm);
  const int b = blocks_per_sm(without, threads, smem, dev, kMaxBlocksPerSm);
  return a < b ? a : b;
}

template <typename T, typename Idx, int N, int V, bool HAS_RSTD, bool ADD>
cudaError_t bwd_rows_v(const RowPlan &p, const BwdParams<T, Idx> &k, const RmsNormBwdArgs &a,
                       const DeviceInfo &dev, cudaStream_t s) {
  auto kern = rmsnorm_bwd_rows<T, Idx, N, V, HAS_RSTD, ADD>;
  const int threads = p.threads();
  const size_t smem = sizeof(float) * (4 * p.R * p.W + (p.R > 1 ? (size_t)p.R * a.H : 0));
  if (smem > (size_t)dev.max_smem_optin) return cudaErrorInvalidConfiguration;
  // the grid must not depend on whether rstd is saved (dw's summation order)
  const int occ = min_blocks_per_sm((const void *)rmsnorm_bwd_rows<T, Idx, N, V, true, ADD>,
                                    (const void *)rmsnorm_bwd_rows<T, Idx, N, V, false, ADD>,
                                    threads, smem, dev);
  int64_t P = ceil_div(a.T, (int64_t)p.R);
  if (P > (int64_t)dev.sms * occ) P = (int64_t)dev.sms * occ;
  if (P > a.ws_rows) P = a.ws_rows;
  cudaError_t e = launch_pdl(kern, dim3((unsigned)P), dim3(threads), smem, s, k);
  if (e != cudaSuccess) return e;
  return launch_dw_reduce(a, P, s);
}

template <typename T, typename Idx, int N, int V, bool HAS_RSTD, bool ADD>
cudaError_t bwd_staged_v(const RowPlan &p, const StagedPlan &sp, const BwdParams<T, Idx> &k,
                         const RmsNormBwdArgs &a, const DeviceInfo &dev, cudaStream_t s) {
  auto kern = rmsnorm_bwd_staged<T, Idx, N, V, HAS_RSTD, ADD>;
  const int threads = p.threads();
  // the grid must not depend on whether rstd is saved (dw's summation order)
  const int occ = min_blocks_per_sm((const void *)rmsnorm_bwd_staged<T, Idx, N, V, true, ADD>,
                                    (const void *)rmsnorm_bwd_staged<T, Idx, N, V, false, ADD>,
                                    threads, sp.smem, dev);
  int64_t P = ceil_div(a.T, (int64_t)p.R);
  if (P > (int64_t)dev.sms * occ) P = (int64_t)dev.sms * occ;
  if (P > a.ws_rows) P = a.ws_rows;
  unsigned *status = nullptr;
  cudaError_t e = device_status_ptr(dev, &status);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kern, dim3((unsigned)P), dim3(threads), sp.smem, s, k, sp.S,
                 (uint32_t)sp.off_red, (uint32_t)sp.off_stage, sp.row_bytes, status,
                 kWaitLimitCycles);
  if (e != cudaSuccess) return e;
  return launch_dw_reduce(a, P, s);
}

template <typename T, typename Idx, int N, int V, int W, bool HAS_RSTD, bool ADD>
cudaError_t bwd_pipe_v(const BwdParams<T, Idx> &k, const RmsNormBwdArgs &a, const DeviceInfo &dev,
                       cudaStream_t s) {
  auto kern = rmsnorm_bwd_pipe<T, Idx, N, V, W, HAS_RSTD, ADD>;
  constexpr size_t smem = bwd_pipe_smem<V, W, ADD>();
  static_assert(smem >= sizeof(float) * (8 / W) * 32 * W * V * N,
                "the ring holds the [R][H] partials");
  // the grid must not depend on whether rstd is saved (dw's summation order)
  const int occ = min_blocks_per_sm((const void *)rmsnorm_bwd_pipe<T, Idx, N, V, W, true, ADD>,
                                    (const void *)rmsnorm_bwd_pipe<T, Idx, N, V, W, false, ADD>,
                                    256, smem, dev);
  int64_t P = ceil_div(a.T, (int64_t)(8 / W));
  if (P > (int64_t)dev.sms * occ) P = (int64_t)dev.sms * occ;
  if (P > a.ws_rows) P = a.ws_rows;
  cudaError_t e = launch_pdl(kern, dim3((unsigned)P), dim3(256), smem, s, k);
  if (e != cudaSuccess) return e;
  return launch_dw_reduce(a, P, s);
}

template <typename Idx, int V, bool HAS_RSTD, bool ADD>
cudaError_t bwd_lean_v(const BwdParams<bf16, Idx> &k, const RmsNormBwdArgs &a,
                       const DeviceInfo &dev, cudaStream_t s) {
  auto kern = rmsnorm_bwd_lean<Idx, V, HAS_RSTD, ADD>;
  constexpr size_t smem = bwd_lean_smem<V, ADD>();
  static_assert(smem >= sizeof(float) * 8 * 32 * V * 8, "the ring holds the [8][H] partials");
  // the grid must not depend on whether rstd is saved (dw's summation order)
  const int occ = min_blocks_per_sm((const void *)rmsnorm_bwd_lean<Idx, V, true, ADD>,
                                    (const void *)rmsnorm_bwd_lean<Idx, V, false, ADD>, 256,
                                    smem, dev);
  int64_t P = ceil_div(a.T, (int64_t)8);
  if (P > (int64_t)dev.sms * occ) P = (int64_t)dev.sms * occ;
  if (P > a.ws_rows) P = a.ws_rows;
  cudaError_t e = launch_pdl(kern, dim3((unsigned)P), dim3(256), smem, s, k);
  if (e != cudaSuccess) return e;
  return launch_dw_reduce(a, P, s);
}

template <typename T, typename Idx, int N, bool HAS_RSTD, bool ADD>
cudaError_t bwd_planned(const RowPlan &p, const StagedPlan *sp, const BwdParams<T, Idx> &k,
                        const RmsNormBwdArgs &a, const DeviceInfo &dev, cudaStream_t s) {
#define FTK_BWD_V(VV)                                                              \
  case VV:                                                                         \
    return sp ? bwd_staged_v<T, Idx, N, VV, HAS_RSTD, ADD>(p, *sp, k, a, dev, s)   \
              : bwd_rows_v<T, Idx, N, VV, HAS_RSTD, ADD>(p, k, a, dev, s);
  switch (p.V) {
    FTK_BWD_V(1)
    FTK_BWD_V(2)
    FTK_BWD_V(3)
    FTK_BWD_V(4)
    FTK_BWD_V(6)
    FTK_BWD_V(8)
    default:
      return cudaErrorInvalidConfiguration;
  }
#undef FTK_BWD_V
}

template <typename T, typename Idx, bool HAS_RSTD, bool ADD>
cudaError_t bwd_typed(bool vec, const RmsNormBwdArgs &a, const DeviceInfo &dev,
                      cudaStream_t s) {
  constexpr int NV = VecWidth<T>::value;
  // the forward's plan: the same per-thread columns and summation order, so
  // an rstd recomputed here equals the one the forward saved bit for bit
  const RowPlan p = plan_rmsnorm_row(a.H, vec ? NV : 1, 4);
  const BwdParams<T, Idx> k{(const T *)a.dy, (Idx)a.lddy, (const T *)a.x, (Idx)a.ldx,
                            (const T *)a.dh, (Idx)a.lddh, (const T *)a.w, a.rstd,
                            (T *)a.dx,       (Idx)a.lddx, a.ws,           (Idx)a.T,
                            (int)(a.H / (vec ? NV : 1)),  (int)a.H,
                            (float)(1.0 / (double)a.H),   a.eps,
                            p.W,             p.R};
  if (p.generic) {
    int64_t P = a.T < (int64_t)dev.sms * 4 ? a.T : (int64_t)dev.sms * 4;
    if (P > a.ws_rows) P = a.ws_rows;
    cudaError_t e = launch_pdl(rmsnorm_bwd_generic<T, Idx, HAS_RSTD, ADD>, dim3((unsigned)P),
                               dim3(256), 0, s, k, (Idx)a.H);
    if (e != cudaSuccess) return e;
    return launch_dw_reduce(a, P, s);
  }
  // rows of one or two warps' plan: the per-warp cp.async pipeline (not
  // with the residual gradient: its third input costs the registers of a
  // second CTA per SM, and the staged ring measured faster there)
  if constexpr (sizeof(T) == 2) {  // bf16 rows of one warp: the lean form (the forward's order)
    if (vec && p.W == 1) {
      switch (p.V) {
        case 1: return bwd_lean_v<Idx, 1, HAS_RSTD, ADD>(k, a, dev, s);
        case 2: return bwd_lean_v<Idx, 2, HAS_RSTD, ADD>(k, a, dev, s);
        case 3: return bwd_lean_v<Idx, 3, HAS_RSTD, ADD>(k, a, dev, s);
        case 4: return bwd_lean_v<Idx, 4, HAS_RSTD, ADD>(k, a, dev, s);
        default: break;
      }
    }
  }
  if constexpr (!ADD) {
    if (vec && p.W == 1) {
      switch (p.V) {
        case 1: return bwd_pipe_v<T, Idx, NV, 1, 1, HAS_RSTD, ADD>(k, a, dev, s);
        case 2: return bwd_pipe_v<T, Idx, NV, 2, 1, HAS_RSTD, ADD>(k, a, dev, s);
        case 3: return bwd_pipe_v<T, Idx, NV, 3, 1, HAS_RSTD, ADD>(k, a, dev, s);
        case 4: return bwd_pipe_v<T, Idx, NV, 4, 1, HAS_RSTD, ADD>(k, a, dev, s);
        default: break;
      }
    }
    if (vec && p.W == 2 && p.V == 4) return bwd_pipe_v<T, Idx, NV, 4, 2, HAS_RSTD, ADD>(k, a, dev, s);
  }
  if (vec) {
    const StagedPlan sp = plan_rmsnorm_staged(p, a.H, (int)sizeof(T), ADD ? 3 : 2, dev);
    if (sp.S > 0) return bwd_planned<T, Idx, NV, HAS_RSTD, ADD>(p, &sp, k, a, dev, s);
    return bwd_planned<T, Idx, NV, HAS_RSTD, ADD>(p, nullptr, k, a, dev, s);
  }
  return bwd_planned<T, Idx, 1, HAS_RSTD, ADD>(p, nullptr, k, a, dev, s);
}

template <typename T, typename Idx, bool ADD>
cudaError_t bwd_rstd_or_not(bool vec, const RmsNormBwdArgs &a, const DeviceInfo &dev,
                            cudaStream_t s) {
  return a.rstd ? bwd_typed<T, Idx, true, ADD>(vec, a, dev, s)
                : bwd_typed<T, Idx, false, ADD>(vec, a, dev, s);
}

template <bool ADD>
cudaError_t launch_bwd_form(DType dt, bool vec, bool wide, const RmsNormBwdArgs &a,
                            const DeviceInfo &dev, cudaStream_t s) {
  if (dt == DType::F32)
    return wide ? bwd_rstd_or_not<float, int64_t, ADD>(vec, a, dev, s)
                : bwd_rstd_or_not<float, int32_t, ADD>(vec, a, dev, s);
  return wide ? bwd_rstd_or_not<bf16, int64_t, ADD>(vec, a, dev, s)
              : bwd_rstd_or_not<bf16, int32_t, ADD>(vec, a, dev, s);
}

}  // namespace

}  // namespace ftk
