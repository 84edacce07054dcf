// RMSNorm forward:  y[t,j] = x[t,j] * r[t] * w[j],
//                   r[t]   = 1 / sqrt(mean_j x[t,j]^2 + eps)
// (Chronicals, arXiv 2601.02609, abstract, optimisation (1): fused RMSNorm.)
// With ADD, the pre-norm residual step fused in front of it: h = x + res is
// added in fp32, rounded to the storage type and stored, and the norm runs
// on that stored h (exactly what a separate add followed by the norm gives).
//
// One row is read from HBM once and written once.  A group of W warps owns a
// row; the sum of squares is reduced with warp shuffles (and, for W > 1,
// through shared memory in a fixed order), then every thread scales its own
// packets.  R row groups share a CTA so that CTAs stay at 128-256 threads.
//
// 16-byte aligned rows of one or two warps' plan take rmsnorm_fwd_pipe: a
// persistent grid of single warps, each lane streaming its packets of the
// rows ahead through a per-warp cp.async ring.  Longer aligned rows take
// rmsnorm_fwd_staged once the batch is large: a persistent grid in which one
// elected thread per row group streams the group's next S rows into a ring
// of shared-memory stages with bulk copies (cp.async.bulk, the TMA engine's
// 1-D mode) completing on mbarriers; the warps compute from shared memory.
// Bytes in flight then cost no registers, and a row's copy starts S rows
// before it is needed.  Other rows hold their packets in registers
// (rmsnorm_fwd_rows); rows too long for either take a CTA-per-row kernel.
#include "common.cuh"
#include "launch.h"
#include "pair_math.cuh"

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

namespace {

template <typename T, typename Idx> struct FwdParams {
  const T *x;
  Idx ldx;
  const T *res;  // ADD only
  Idx ldr;
  const T *w;
  T *y;
  Idx ldy;
  T *h;  // ADD only
  Idx ldh;
  float *rstd;  // nullable
  Idx rows;
  int hp;  // packets per row
  float inv_h, eps;
  int W, R;
};

// The row's value as the norm sees it: x, or (ADD) x + res rounded to T.
template <typename T, int N, bool ADD>
__device__ __forceinline__ Packet<T, N> norm_input(const Packet<T, N> &xv,
                                                   const Packet<T, N> &rv) {
  if constexpr (!ADD) {
    return xv;
  } else {
    Packet<T, N> h;
#pragma unroll
    for (int e = 0; e < N; ++e) h.set(e, xv.get(e) + rv.get(e));
    return h;
  }
}

// Packet c of a staged row as the norm sees it; the res row (read only with
// ADD) follows the x row in the stage.
template <typename T, int N, bool ADD>
__device__ __forceinline__ Packet<T, N> staged_input(const T *xs, const T *rs, int c) {
  const Packet<T, N> xv = *reinterpret_cast<const Packet<T, N> *>(xs + c * N);
  if constexpr (!ADD) {
    return xv;
  } else {
    return norm_input<T, N, true>(xv, *reinterpret_cast<const Packet<T, N> *>(rs + c * N));
  }
}

template <typename T, typename Idx, int N, int V, bool ADD>
__global__ void __launch_bounds__(256)
rmsnorm_fwd_staged(const FwdParams<T, Idx> a, int S, uint32_t off_red, uint32_t off_stage,
                   uint32_t row_bytes, unsigned *status, long long wait_limit) {
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem);  // [R][S]
  float *red = reinterpret_cast<float *>(smem + off_red);  // [2][R][W], by row parity
  const int W = a.W, R = a.R;
  // Multi-warp groups with three or more stages refill a row's stage at the
  // next row's reduction barrier (by then the whole group is past the row),
  // which saves a barrier per row; with two stages that would leave the
  // next row half a row of lead, so they refill behind a second barrier at
  // the end of the row.  (With the residual, whose stages are twice as
  // large, the early refill measured slower: it keeps the second barrier.)
  const bool early = !ADD && W > 1 && S > 2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / W, wig = warp - grp * W;
  const int gi = wig * 32 + lane, G = W * 32;
  const bool leader = gi == 0;
  const uint32_t stage_bytes = (ADD ? 2 : 1) * row_bytes;  // x row (then res row)

  for (int i = threadIdx.x; i < R * S; i += blockDim.x) mbar_init(&bars[i], 1);
  if (threadIdx.x == 0) fence_mbar_init();
  __syncthreads();
  pdl_wait();
  pdl_trigger();

  uint64_t *gb = bars + grp * S;
  unsigned char *ring = smem + off_stage + (size_t)grp * S * stage_bytes;
  const Idx stride = (Idx)gridDim.x * R;
  const Idx first = (Idx)blockIdx.x * R + grp;

  auto issue = [&](int s, Idx row) {
    unsigned char *st = ring + (size_t)s * stage_bytes;
    mbar_arrive_expect_tx(&gb[s], stage_bytes);
    bulk_copy_g2s(st, a.x + row * a.ldx, row_bytes, &gb[s]);
    if (ADD) bulk_copy_g2s(st + row_bytes, a.res + row * a.ldr, row_bytes, &gb[s]);
  };
  int issued = 0;  // copies issued by the leader
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
    if (c < a.hp) wv[k] = load_packet<T, N>(a.w + (Idx)c * N);
  }

  bool live = true;  // false once one of this thread's waits has run out
  int it = 0;
  for (Idx row = first; row < a.rows; row += stride, ++it) {
    const int s = it % S;
    if (live) live = mbar_wait_bounded(&gb[s], (uint32_t)((it / S) & 1), wait_limit, status);
    const T *xs = reinterpret_cast<const T *>(ring + (size_t)s * stage_bytes);
    const T *rs = reinterpret_cast<const T *>(ring + (size_t)s * stage_bytes + row_bytes);
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const int c = gi + k * G;
      if (c < a.hp) {
        const Packet<T, N> v = staged_input<T, N, ADD>(xs, rs, c);
        sumsq_packet<T, N>(acc, v);
      }
    }
    float ss = warp_sum(sumsq_total<T, N>(acc));
    if (W > 1) {
      // with the early refill the slots alternate by row parity: a warp one
      // row ahead writes the other half, and none gets two rows ahead
      // without passing this barrier again (otherwise the end-of-row
      // barrier keeps the slots)
      float *slot = red + ((early ? (it & 1) * R : 0) + grp) * W;
      if (lane == 0) slot[wig] = ss;
      group_barrier(grp, G);
      ss = 0.f;
      for (int i = 0; i < W; ++i) ss += slot[i];
      if (early && leader && it > 0) {  // the previous row's stage is free
        const Idx next = row + (Idx)(S - 1) * stride;
        if (next < a.rows) {
          fence_proxy_async_smem();
          issue((it - 1) % S, next);
          ++issued;
        }
      }
    }
    const float r = rsqrtf(fmaf(ss, a.inv_h, a.eps));
    if (a.rstd != nullptr && leader) a.rstd[row] = r;
    T *yr = a.y + row * a.ldy;
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const int c = gi + k * G;
      if (c < a.hp) {
        const Packet<T, N> v = staged_input<T, N, ADD>(xs, rs, c);
        if (ADD) store_packet<T, N>(a.h + row * a.ldh + (Idx)c * N, v);
        store_packet<T, N>(yr + (Idx)c * N, scale_packet<T, N, !ADD>(v, r, wv[k]));
      }
    }
    if (!early) {
      // the whole group has read stage s: refill it
      if (W > 1)
        group_barrier(grp, G);
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
  }
  // after a wait ran out, let the copies still in flight land (bounded)
  // before the CTA's shared memory is released
  if (leader && !live)
    for (int i = it; i < issued; ++i)
      mbar_wait_bounded(&gb[i % S], (uint32_t)((i / S) & 1), wait_limit, status);
}

template <typename T, typename Idx, int N, int V, bool ADD>
__global__ void __launch_bounds__(256) rmsnorm_fwd_rows(const FwdParams<T, Idx> a) {
  extern __shared__ float red[];  // [R][W] warp partial sums
  pdl_wait();
  pdl_trigger();
  const int W = a.W, R = a.R;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / W, wig = warp - grp * W;
  const int gi = wig * 32 + lane, G = W * 32;
  const Idx row = (Idx)blockIdx.x * R + grp;
  const bool active = row < a.rows;

  Packet<T, N> xv[V];
  float2 acc = make_float2(0.f, 0.f);
  if (active) {
    const T *xr = a.x + row * a.ldx;
    const T *rr = ADD ? a.res + row * a.ldr : nullptr;
    Packet<T, N> rv[ADD ? V : 1];
#pragma unroll
    for (int k = 0; k < V; ++k) {
      const int c = gi + k * G;
      if (c < a.hp) {
        xv[k] = load_packet_stream<T, N>(xr + (Idx)c * N);
        if (ADD) rv[ADD ? k : 0] = load_packet_stream<T, N>(rr + (Idx)c * N);
      }
    }
#pragma unroll
    for (int k = 0; k < V; ++k) {
      if (gi + k * G < a.hp) {
        if (ADD) xv[k] = norm_input<T, N, ADD>(xv[k], rv[ADD ? k : 0]);
        sumsq_packet<T, N>(acc, xv[k]);
      }
    }
  }
  float ss = warp_sum(sumsq_total<T, N>(acc));
  if (W > 1) {
    if (lane == 0) red[grp * W + wig] = ss;
    __syncthreads();
    ss = 0.f;
    for (int i = 0; i < W; ++i) ss += red[grp * W + i];
  }
  if (!active) return;

  const float r = rsqrtf(fmaf(ss, a.inv_h, a.eps));
  if (a.rstd != nullptr && gi == 0) a.rstd[row] = r;
  T *yr = a.y + row * a.ldy;
#pragma unroll
  for (int k = 0; k < V; ++k) {
    const int c = gi + k * G;
    if (c < a.hp) {
      if (ADD) store_packet<T, N>(a.h + row * a.ldh + (Idx)c * N, xv[k]);
      const Packet<T, N> wv = load_packet<T, N>(a.w + (Idx)c * N);
      store_packet<T, N>(yr + (Idx)c * N, scale_packet<T, N, !ADD>(xv[k], r, wv));
    }
  }
}

// Rows of one or two warps' plan (W <= 2): persistent, one row per warp at
// a time, rows row, row + 8P, ...  Each lane copies its packets of the rows
// kBufs - 1 ahead into a per-warp shared-memory ring with cp.async while it
// normalises the current row, so the loads of later rows overlap the
// arithmetic and the stores of this one.  The warp plays the plan's W warps
// in turn: lane l owns packets w 32 + l + k 32W (w < W, k < V), sums the
// squares of each w separately in the plan's order, and adds the W warp
// sums in order, so the row sum is the plan's bit for bit and an rstd the
// backward recomputes is identical.
template <int W, int V, bool ADD> struct FwdPipe {
  static constexpr int kBufs = (ADD || W * V > 4) ? 2 : 4;  // rows in the ring per warp
  static constexpr int kSl = (ADD ? 2 : 1) * W * V;         // 16-byte slots per lane per row
};

template <typename T, typename Idx, int N, int V, int W, bool ADD>
__global__ void __launch_bounds__(256) rmsnorm_fwd_pipe(const FwdParams<T, Idx> a) {
  constexpr int kBufs = FwdPipe<W, V, ADD>::kBufs;
  constexpr int kSl = FwdPipe<W, V, ADD>::kSl;  // x (, res), W V packets each
  constexpr int kP = W * V;                     // packets per lane
  extern __shared__ uint4 ring[];               // [warps][kBufs][kSl][32]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint4 *my = ring + warp * (kBufs * kSl * 32);
  // packet i = w V + k of this lane: column w 32 + lane + k 32W
  auto col = [&](int i) { return (i / V) * 32 + lane + (i % V) * 32 * W; };
  pdl_wait();
  pdl_trigger();
  Packet<T, N> wv[kP];
#pragma unroll
  for (int i = 0; i < kP; ++i)
    if (col(i) < a.hp) wv[i] = load_packet<T, N>(a.w + (Idx)col(i) * N);
  const Idx step = (Idx)gridDim.x * (blockDim.x >> 5);
  auto stage = [&](Idx r, int b) {
    if (r < a.rows) {
      const T *xr = a.x + r * a.ldx;
#pragma unroll
      for (int i = 0; i < kP; ++i) {
        const int c = col(i);
        if (c < a.hp) {
          cp_async16(my + (b * kSl + i) * 32 + lane, xr + (Idx)c * N);
          if (ADD) cp_async16(my + (b * kSl + kP + i) * 32 + lane, a.res + r * a.ldr + (Idx)c * N);
        }
      }
    }
    cp_async_commit();  // one group per row on every lane, empty or not
  };
  Idx row = (Idx)blockIdx.x * (blockDim.x >> 5) + warp, r2 = row;
  stage(r2, 0);
  for (int i = 1; i < kBufs - 1; ++i) {
    r2 += step;
    stage(r2, i);
  }
  int b = 0;
  while (row < a.rows) {  // warp-uniform
    r2 += step;
    stage(r2, b == 0 ? kBufs - 1 : b - 1);  // the next rows' loads fly meanwhile
    cp_async_wait<kBufs - 1>();              // this lane's copies of `row` have landed
    Packet<T, N> xv[kP];
    float2 part[W];
#pragma unroll
    for (int w = 0; w < W; ++w) part[w] = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < kP; ++i) {
      if (col(i) < a.hp) {
        *reinterpret_cast<uint4 *>(&xv[i]) = my[(b * kSl + i) * 32 + lane];
        if (ADD) {
          Packet<T, N> rv;
          *reinterpret_cast<uint4 *>(&rv) = my[(b * kSl + kP + i) * 32 + lane];
          xv[i] = norm_input<T, N, ADD>(xv[i], rv);
        }
        sumsq_packet<T, N>(part[i / V], xv[i]);
      }
    }
    float ss = 0.f;
    if (W == 1) {
      ss = warp_sum(sumsq_total<T, N>(part[0]));
    } else {
#pragma unroll
      for (int w = 0; w < W; ++w) ss += warp_sum(sumsq_total<T, N>(part[w]));  // the plan's order
    }
    const float r = rsqrtf(fmaf(ss, a.inv_h, a.eps));
    if (a.rstd != nullptr && lane == 0) a.rstd[row] = r;
    T *yr = a.y + row * a.ldy;
#pragma unroll
    for (int i = 0; i < kP; ++i) {
      const int c = col(i);
      if (c < a.hp) {
        if (ADD) store_packet<T, N>(a.h + row * a.ldh + (Idx)c * N, xv[i]);
        store_packet<T, N>(yr + (Idx)c * N, scale_packet<T, N, !ADD>(xv[i], r, wv[i]));
      }
    }
    row += step;
    b = b + 1 == kBufs ? 0 : b + 1;
  }
  cp_async_wait<0>();
}

// bf16 rows of one warp (H <= 1,024, 16-byte aligned): rmsnorm_fwd_pipe's
// persistent grid and per-warp cp.async ring, with the lean arithmetic of
// pair_math.cuh: the weights are unpacked to fp32 pairs once per warp,
// each packet once per row, every product is a pair instruction, and the
// ring and row addresses advance as running pointers.  With ADD the ring
// holds the x and res rows; h = x + res is added in fp32 pairs, rounded,
// stored, and the norm runs on the stored h, so y and r equal the plain
// lean norm of that h bit for bit.  Lane l owns packets l + 32 k (k < V).
template <bool ADD> constexpr int lean_fwd_bufs() { return ADD ? 3 : 4; }

// Three CTAs per SM; two with ADD, whose rows carry twice the bytes and
// whose packets would not fit three CTAs' registers.
template <typename Idx, int V, bool ADD>
__global__ void __launch_bounds__(256, ADD ? 2 : 3) rmsnorm_fwd_lean(const FwdParams<bf16, Idx> a) {
  constexpr int kBufs = lean_fwd_bufs<ADD>();
  constexpr int kSl = (ADD ? 2 : 1) * V;  // x (, res) packets per lane per row
  extern __shared__ uint4 ring[];        // [warps][kBufs][kSl][32]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint4 *const my = ring + warp * (kBufs * kSl * 32) + lane;
  pdl_wait();
  pdl_trigger();
  bool on[V];
  float2 wf[V][4];
#pragma unroll
  for (int k = 0; k < V; ++k) {
    on[k] = lane + 32 * k < a.hp;
    uint4 u = make_uint4(0u, 0u, 0u, 0u);
    if (on[k]) u = *reinterpret_cast<const uint4 *>(a.w + (lane + 32 * k) * 8);
    unpack8(u, wf[k]);
  }
  const Idx step = (Idx)gridDim.x * 8;
  Idx row = (Idx)blockIdx.x * 8 + warp;
  // the next row to stage, its source addresses and its ring slot
  Idx srow = row;
  const bf16 *src = a.x + row * a.ldx + lane * 8;
  const bf16 *srs = ADD ? a.res + row * a.ldr + lane * 8 : nullptr;
  const Idx src_step = step * a.ldx, srs_step = ADD ? step * a.ldr : 0;
  int sslot = 0;
  auto stage = [&]() {
    if (srow < a.rows) {
      uint4 *d = my + sslot * (kSl * 32);
#pragma unroll
      for (int k = 0; k < V; ++k) {
        if (on[k]) {
          cp_async16(d + k * 32, src + k * 256);
          if (ADD) cp_async16(d + (V + k) * 32, srs + k * 256);
        }
      }
    }
    cp_async_commit();  // one group per row on every lane, empty or not
    srow += step;
    src += src_step;
    if (ADD) srs += srs_step;
    sslot = sslot + 1 == kBufs ? 0 : sslot + 1;
  };
#pragma unroll
  for (int i = 0; i < kBufs - 1; ++i) stage();
  bf16 *dst = a.y + row * a.ldy + lane * 8;
  bf16 *dsth = ADD ? a.h + row * a.ldh + lane * 8 : nullptr;
  const Idx dst_step = step * a.ldy, dsth_step = ADD ? step * a.ldh : 0;
  int slot = 0;
  while (row < a.rows) {  // warp-uniform
    stage();                    // the next rows' loads fly meanwhile
    cp_async_wait<kBufs - 1>();  // this lane's copies of `row` have landed
    const uint4 *d = my + slot * (kSl * 32);
    float2 xf[V][4];
    float2 acc = make_float2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < V; ++k) {
      uint4 u = make_uint4(0u, 0u, 0u, 0u);
      if (on[k]) u = d[k * 32];
      if (ADD) {
        // h = x + res in fp32, rounded once; the norm sees the stored h
        float2 rf[4];
        unpack8(on[k] ? d[(V + k) * 32] : make_uint4(0u, 0u, 0u, 0u), rf);
        unpack8(u, xf[k]);
#pragma unroll
        for (int p = 0; p < 4; ++p) xf[k][p] = __fadd2_rn(xf[k][p], rf[p]);
        u = pack8(xf[k]);
        if (on[k]) *reinterpret_cast<uint4 *>(dsth + k * 256) = u;
      }
      unpack8(u, xf[k]);
#pragma unroll
      for (int p = 0; p < 4; ++p) lean_sumsq_step(acc, xf[k][p]);
    }
    const float ss = warp_sum(lean_lane_total(acc));
    const float r = rsqrtf(fmaf(ss, a.inv_h, a.eps));
    if (a.rstd != nullptr && lane == 0) a.rstd[row] = r;
    const float2 r2 = make_float2(r, r);
#pragma unroll
    for (int k = 0; k < V; ++k) {
      if (on[k]) {
        float2 o[4];
#pragma unroll
        for (int p = 0; p < 4; ++p) o[p] = __fmul2_rn(__fmul2_rn(xf[k][p], r2), wf[k][p]);
        *reinterpret_cast<uint4 *>(dst + k * 256) = pack8(o);
      }
    }
    row += step;
    dst += dst_step;
    if (ADD) dsth += dsth_step;
    slot = slot + 1 == kBufs ? 0 : slot + 1;
  }
  cp_async_wait<0>();
}

// Rows longer than the register plan: one CTA per row (grid-stride over
// rows), sum of squares first (writing h when ADD), then a second pass that
// re-reads the row (from L2).
template <typename T, typename Idx, bool ADD>
__global__ void __launch_bounds__(256) rmsnorm_fwd_generic(const FwdParams<T, Idx> a, Idx H) {
  __shared__ float red[8];
  pdl_wait();
  pdl_trigger();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (Idx row = blockIdx.x; row < a.rows; row += gridDim.x) {
    const T *xr = a.x + row * a.ldx;
    const T *rr = ADD ? a.res + row * a.ldr : nullptr;
    T *hr = ADD ? a.h + row * a.ldh : nullptr;
    float ss = 0.f;
    for (Idx j = threadIdx.x; j < H; j += blockDim.x) {
      T v = xr[j];
      if (ADD) {
        v = from_float<T>(to_float(v) + to_float(rr[j]));
        hr[j] = v;
      }
      const float f = to_float(v);
      ss = fmaf(f, f, ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) red[warp] = ss;
    __syncthreads();  // also orders this CTA's h writes before the re-reads
    ss = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) ss += red[i];
    __syncthreads();  // red is reused by the next row
    const float r = rsqrtf(fmaf(ss, a.inv_h, a.eps));
    if (a.rstd != nullptr && threadIdx.x == 0) a.rstd[row] = r;
    T *yr = a.y + row * a.ldy;
    const T *src = ADD ? hr : xr;
    for (Idx j = threadIdx.x; j < H; j += blockDim.x)
      yr[j] = from_float<T>((to_float(src[j]) * r) * to_float(a.w[j]));
  }
}

template <typename T, typename Idx, int N, int V, bool ADD>
cudaError_t fwd_rows_v(const RowPlan &p, const FwdParams<T, Idx> &k, cudaStream_t s) {
  const dim3 grid((unsigned)ceil_div((int64_t)k.rows, (int64_t)p.R));
  const size_t smem = sizeof(float) * p.R * p.W;
  cudaError_t le = launch_pdl(rmsnorm_fwd_rows<T, Idx, N, V, ADD>, grid, dim3(p.threads()), smem,
                              s, k);
  if (le != cudaSuccess) return le;
  return cudaGetLastError();
}

template <typename T, typename Idx, int N, int V, int W, bool ADD>
cudaError_t fwd_pipe_v(const FwdParams<T, Idx> &k, const DeviceInfo &dev, cudaStream_t s) {
  auto kern = rmsnorm_fwd_pipe<T, Idx, N, V, W, ADD>;
  const size_t smem =
      sizeof(uint4) * 8 * FwdPipe<W, V, ADD>::kBufs * FwdPipe<W, V, ADD>::kSl * 32;  // 8 warps
  const int occ = blocks_per_sm((const void *)kern, 256, smem, dev, 8);
  int64_t P = ceil_div((int64_t)k.rows, (int64_t)8);
  if (P > (int64_t)dev.sms * occ) P = (int64_t)dev.sms * occ;
  cudaError_t le = launch_pdl(kern, dim3((unsigned)P), dim3(256), smem, s, k);
  if (le != cudaSuccess) return le;
  return cudaGetLastError();
}

template <typename Idx, int V, bool ADD>
cudaError_t fwd_lean_v(const FwdParams<bf16, Idx> &k, const DeviceInfo &dev, cudaStream_t s) {
  auto kern = rmsnorm_fwd_lean<Idx, V, ADD>;
  const size_t smem =
      sizeof(uint4) * 8 * lean_fwd_bufs<ADD>() * (ADD ? 2 : 1) * V * 32;  // 8 warps
  const int occ = blocks_per_sm((const void *)kern, 256, smem, dev, 8);
  int64_t P = ceil_div((int64_t)k.rows, (int64_t)8);
  if (P > (int64_t)dev.sms * occ) P = (int64_t)dev.sms * occ;
  cudaError_t le = launch_pdl(kern, dim3((unsigned)P), dim3(256), smem, s, k);
  if (le != cudaSuccess) return le;
  return cudaGetLastError();
}

// Resident CTAs per SM of the staged forward, at most.  Fewer row groups
// streaming at once measured faster at H = 5,120 (groups of 5 warps, 524,288
// rows): the plain norm 1,641 us with 3 CTAs per SM, 1,653 us with 4 and
// 1,850 us with 6; with the residual (two rows per stage) 3,205 us with 4
// and 3,311 us with 3.
template <bool ADD> constexpr int fwd_staged_blocks() { return ADD ? 4 : 3; }

template <typename T, typename Idx, int N, int V, bool ADD>
cudaError_t fwd_staged_v(const RowPlan &p, const StagedPlan &sp, const FwdParams<T, Idx> &k,
                         const DeviceInfo &dev, cudaStream_t s) {
  auto kern = rmsnorm_fwd_staged<T, Idx, N, V, ADD>;
  const int threads = p.threads();
  const int occ = blocks_per_sm((const void *)kern, threads, sp.smem, dev, fwd_staged_blocks<ADD>());
  int64_t P = ceil_div((int64_t)k.rows, (int64_t)p.R);
  if (P > (int64_t)dev.sms * occ) P = (int64_t)dev.sms * occ;
  unsigned *status = nullptr;
  cudaError_t e = device_status_ptr(dev, &status);
  if (e != cudaSuccess) return e;
  cudaError_t le = launch_pdl(kern, dim3((unsigned)P), dim3(threads), sp.smem, s, k, sp.S,
                              (uint32_t)sp.off_red, (uint32_t)sp.off_stage, sp.row_bytes, status,
                              kWaitLimitCycles);
  if (le != cudaSuccess) return le;
  return cudaGetLastError();
}

template <typename T, typename Idx, int N, bool ADD>
cudaError_t fwd_planned(const RowPlan &p, const StagedPlan *sp, const FwdParams<T, Idx> &k,
                        const DeviceInfo &dev, cudaStream_t s) {
#define FTK_FWD_V(VV)                                                   \
  case VV:                                                              \
    return sp ? fwd_staged_v<T, Idx, N, VV, ADD>(p, *sp, k, dev, s)     \
              : fwd_rows_v<T, Idx, N, VV, ADD>(p, k, s);
  switch (p.V) {
    FTK_FWD_V(1)
    FTK_FWD_V(2)
    FTK_FWD_V(3)
    FTK_FWD_V(4)
    FTK_FWD_V(6)
    FTK_FWD_V(8)
    default:
      return cudaErrorInvalidConfiguration;
  }
#undef FTK_FWD_V
}

template <typename T, typename Idx, bool ADD>
cudaError_t fwd_typed(bool vec, const RmsNormFwdArgs &a, const DeviceInfo &dev, cudaStream_t s) {
  constexpr int NV = VecWidth<T>::value;
  const RowPlan p = plan_rmsnorm_row(a.H, vec ? NV : 1, 4);
  FwdParams<T, Idx> k{(const T *)a.x, (Idx)a.ldx, (const T *)a.res, (Idx)a.ldr,
                      (const T *)a.w, (T *)a.y,   (Idx)a.ldy,         (T *)a.h,
                      (Idx)a.ldh,     a.rstd,     (Idx)a.T,           (int)(a.H / (vec ? NV : 1)),
                      (float)(1.0 / (double)a.H), a.eps, p.W, p.R};
  if (p.generic) {
    const int64_t grid = a.T < (int64_t)dev.sms * 16 ? a.T : (int64_t)dev.sms * 16;
    cudaError_t le = launch_pdl(rmsnorm_fwd_generic<T, Idx, ADD>, dim3((unsigned)grid), dim3(256),
                                0, s, k, (Idx)a.H);
    if (le != cudaSuccess) return le;
    return cudaGetLastError();
  }
  // Rows of one warp's plan, and (without the residual) of two warps' plan:
  // the per-warp cp.async pipeline at every batch size; bf16 rows of one
  // warp take its lean form, with or without the residual (the backward's
  // recomputation of r follows the same order).
  if constexpr (sizeof(T) == 2) {
    if (vec && p.W == 1) {
      switch (p.V) {
        case 1: return fwd_lean_v<Idx, 1, ADD>(k, dev, s);
        case 2: return fwd_lean_v<Idx, 2, ADD>(k, dev, s);
        case 3: return fwd_lean_v<Idx, 3, ADD>(k, dev, s);
        case 4: return fwd_lean_v<Idx, 4, ADD>(k, dev, s);
        default: break;
      }
    }
  }
  if (vec && p.W == 1) {
    switch (p.V) {
      case 1: return fwd_pipe_v<T, Idx, NV, 1, 1, ADD>(k, dev, s);
      case 2: return fwd_pipe_v<T, Idx, NV, 2, 1, ADD>(k, dev, s);
      case 3: return fwd_pipe_v<T, Idx, NV, 3, 1, ADD>(k, dev, s);
      case 4: return fwd_pipe_v<T, Idx, NV, 4, 1, ADD>(k, dev, s);
      default: break;
    }
  }
  if constexpr (!ADD)
    if (vec && p.W == 2 && p.V == 4) return fwd_pipe_v<T, Idx, NV, 4, 2, ADD>(k, dev, s);
  // The staged pipeline pays off once every row group streams a dozen rows
  // or more; smaller batches finish sooner with one row per group and the
  // hardware scheduler refilling SMs (rmsnorm_fwd_rows).
  if (vec && a.T >= (int64_t)12 * p.R * 2 * dev.sms) {
    const StagedPlan sp = plan_rmsnorm_staged(p, a.H, (int)sizeof(T), ADD ? 2 : 1, dev);
    if (sp.S > 0) return fwd_planned<T, Idx, NV, ADD>(p, &sp, k, dev, s);
  }
  return vec ? fwd_planned<T, Idx, NV, ADD>(p, nullptr, k, dev, s)
             : fwd_planned<T, Idx, 1, ADD>(p, nullptr, k, dev, s);
}

template <typename T, typename Idx>
cudaError_t fwd_add_or_not(bool vec, const RmsNormFwdArgs &a, const DeviceInfo &dev,
                           cudaStream_t s) {
  return a.res ? fwd_typed<T, Idx, true>(vec, a, dev, s) : fwd_typed<T, Idx, false>(vec, a, dev, s);
}

}  // namespace

cudaError_t launch_rmsnorm_fwd(DType dt, bool vec, bool wide, const RmsNormFwdArgs &a,
                               const DeviceInfo &dev, cudaStream_t s) {
  if (dt == DType::F32)
    return wide ? fwd_add_or_not<float, int64_t>(vec, a, dev, s)
                : fwd_add_or_not<float, int32_t>(vec, a, dev, s);
  return wide ? fwd_add_or_not<bf16, int64_t>(vec, a, dev, s)
              : fwd_add_or_not<bf16, int32_t>(vec, a, dev, s);
}

}  // namespace ftk
