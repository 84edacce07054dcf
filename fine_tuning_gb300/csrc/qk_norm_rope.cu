// Per-head RMSNorm of Q and K (the q_norm / k_norm of Qwen3-style attention)
// fused with the rotary embedding, forward and backward, over a packed batch
// of variable-length sequences.
//
// For token t at position p and every head vector v (D values) of Q (weight
// wq [D]) or K (weight wk [D]):
//   r   = 1 / sqrt(mean_i v_i^2 + eps)
//   n_i = v_i r w_i                      (fp32, never rounded)
//   out = rotate-half RoPE of n at p      (inv_freq from theta or a table)
// Backward, from the output gradient g:
//   dn  = the rotation by -phi of g
//   c   = sum_i dn_i w_i v_i
//   dv  = r w dn - r^3 v c / D,  dw_i += dn_i v_i r  (over tokens and heads)
// Sources: the fused QK-RoPE kernel of "Unsloth prétend accélérer 5 fois
// l'entraînement des LLM avec de nouveaux noyaux Triton et un auto-packing"
// (seventnews.com) and optimisation (1) of "Chronicals" (arXiv 2601.02609,
// abstract); the norm in front of the rotation is this library's variant.
//
// Warp per token (the layout of qk_rope_warp): half a head is NV = D/2N
// packets and NV divides 32, so lane (slot, j) owns packet j of both halves
// of heads slot, slot + S, ... (S = 32 / NV).  A head's sum of squares is a
// shuffle reduction over its NV lanes.  cos/sin of the token's D/2 angles
// are computed once into the warp's shared-memory slice.  Both directions
// are persistent and walk (token, head pass) pairs, each lane copying its
// packets of the passes ahead into a per-warp shared-memory ring with
// cp.async while it computes the current one.  The backward keeps each
// lane's dwq and dwk column sums in registers, the CTA combines its warps in
// a fixed order into one partial row [2D], and dw_reduce sums the rows in a
// fixed order: bitwise reproducible.  Shapes whose half head does not split
// evenly over lanes, or unaligned rows, take the element-wise kernels (lane
// i owns pairs i, i + 32, ...).
#include "common.cuh"
#include "dw_reduce.cuh"
#include "launch.h"
#include "pair_math.cuh"
#include "rope_common.cuh"

namespace ftk {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxBlocksPerSm = 4;
constexpr int kPairsPerLane = kRopeMaxHalf / 32;  // element-wise kernels

template <typename T, typename Idx> struct NormRopeParams {
  const T *q;  // pre-norm Q / K
  Idx ld_q;
  const T *k;
  Idx ld_k;
  const T *gq;  // backward: gradient of the outputs
  Idx ld_gq;
  const T *gk;
  Idx ld_gk;
  T *oq;  // forward: outputs; backward: gradient of the pre-norm Q / K
  Idx ld_oq;
  T *ok;
  Idx ld_ok;
  const T *wq, *wk;
  float *rq, *rk;  // r per (token, head): written by the forward, read by the backward (nullable)
  float *ws;       // backward: [gridDim.x][2D] partial rows (dwq | dwk)
  const int32_t *cu;
  int B;
  Idx rows;
  int Hq, Hkv, D;
  float eps, inv_d;
};

// Sum over the NV lanes (a power of two dividing 32) that share a slot.
__device__ __forceinline__ float slot_sum(float v, int NV) {
  for (int o = NV >> 1; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float2 slot_sum2(float2 v, int NV) {
  for (int o = NV >> 1; o > 0; o >>= 1) {
    v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
    v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
  }
  return v;
}

// cos and sgn*sin of the token's D/2 angles into the warp's table.
__device__ __forceinline__ void token_table(float2 *wt, const float2 *freq, int half, int p,
                                            float sgn, int lane) {
  for (int i = lane; i < half; i += 32) {
    const float2 f = freq[i];
    float c, sn;
    rope_cos_sin(p, f.x, f.y, &c, &sn);
    wt[i] = make_float2(c, sgn * sn);
  }
}

// The backward warp kernel's staging: per warp kBwdBufs buffers of 5 x 32
// 16-byte slots (gradient halves, pre-norm halves, r; slot c of lane l at
// c * 32 + l, so a warp's accesses to one slot are contiguous); the loads
// run kBwdBufs - 1 head passes ahead of the arithmetic.
constexpr int kBwdSlots = 5, kBwdBufs = 2;
constexpr int kFwdPipeBlocks = 4;  // CTAs per SM the pipelined forward is compiled for
constexpr size_t kBwdStageBytes = sizeof(uint4) * kWarps * kBwdBufs * kBwdSlots * 32;

// The forward, persistent: each warp walks tokens t, t +
// P * kWarps, ... and each token's heads in passes of S heads (lane (slot,
// j) normalises and rotates packet j of both halves of head slot + S p).
// Each lane copies its packets of the next pass into a per-warp
// shared-memory buffer with cp.async while it computes the current pass,
// so the loads of consecutive passes and tokens overlap the arithmetic.
constexpr int kFwdSlots = 2, kFwdBufs = 4;
constexpr size_t kFwdStageBytes = sizeof(uint4) * kWarps * kFwdBufs * kFwdSlots * 32;

// Per token, the warp folds the norm weights into the rotation: for column
// i (first-half weight w1 = w[i], second-half w2 = w[D/2 + i], angle phi)
//   out_i        = r (x1 w1 cos - x2 w2 sin) = r (x1 A - x2 B)
//   out_{D/2+i}  = r (x2 w2 cos + x1 w1 sin) = r (x2 C + x1 E)
// with (A, B, C, E) = (w1 cos, w2 sin, w2 cos, w1 sin) for Q and for K.  The
// entry of column i sits at (i mod N) NV + i / N, so the NV lanes of a head
// reading their packets' e-th columns touch consecutive entries.
template <typename T, typename Idx, int N>
__global__ void __launch_bounds__(kThreads, kFwdPipeBlocks)
qk_norm_rope_fwd_pipe(const NormRopeParams<T, Idx> a, const __grid_constant__ RopeFreqs fr) {
  // [warps][2][D/2] float4 weighted tables (Q, then K), then the staging
  // buffers
  extern __shared__ float4 tab4[];
  __shared__ float2 freq[kRopeMaxHalf];
  __shared__ float wf[4][kRopeMaxHalf];  // wq first half, wq second, wk first, wk second
  const int D = a.D, half = D >> 1, NV = half / N, S = 32 / NV, NH = a.Hq + a.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = lane % NV, slot = lane / NV;
  float4 *wtq = tab4 + warp * 2 * half, *wtk = wtq + half;
  uint4 *stg = reinterpret_cast<uint4 *>(tab4 + kWarps * 2 * half) +
               warp * (kFwdBufs * kFwdSlots * 32);

  for (int i = threadIdx.x; i < half; i += blockDim.x) freq[i] = make_float2(fr.hi[i], fr.lo[i]);
  pdl_wait();
  pdl_trigger();
  if (rope_skipped(fr)) return;  // malformed cu_seqlens: every output untouched
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    wf[0][i] = a.Hq > 0 ? to_float(a.wq[i]) : 0.f;
    wf[1][i] = a.Hq > 0 ? to_float(a.wq[half + i]) : 0.f;
    wf[2][i] = a.Hkv > 0 ? to_float(a.wk[i]) : 0.f;
    wf[3][i] = a.Hkv > 0 ? to_float(a.wk[half + i]) : 0.f;
  }
  __syncthreads();  // the frequency and weight tables

  const Idx step = (Idx)gridDim.x * kWarps;
  const int passes = (NH + S - 1) / S;  // head passes per token, the same on every lane
  auto stage = [&](Idx tt, int p, int b) {
    const int h = slot + p * S;
    if (tt < a.rows && h < NH) {
      const T *vp = (h < a.Hq ? a.q + tt * a.ld_q + (Idx)h * D
                              : a.k + tt * a.ld_k + (Idx)(h - a.Hq) * D) +
                    j * N;
      uint4 *d = stg + b * kFwdSlots * 32 + lane;
      cp_async16(d, vp);
      cp_async16(d + 32, vp + half);
    }
    cp_async_commit();  // one group per pass on every lane, empty or not
  };
  Idx t = (Idx)blockIdx.x * kWarps + warp, t2 = t;
  int p = 0, p2 = 0, b = 0;
  auto advance = [&](Idx &tt, int &pp) {
    if (++pp == passes) {
      pp = 0;
      tt += step;
    }
  };
  stage(t2, p2, 0);
  for (int i = 1; i < kFwdBufs - 1; ++i) {
    advance(t2, p2);
    stage(t2, p2, i);
  }
  while (t < a.rows) {  // warp-uniform
    advance(t2, p2);
    stage(t2, p2, b == 0 ? kFwdBufs - 1 : b - 1);  // the next passes' loads fly meanwhile
    if (p == 0) {
      __syncwarp();  // the previous token's tables have been read
      const int pos = position_of<Idx>(t, a.cu, a.B);
      for (int i = lane; i < half; i += 32) {
        const float2 f = freq[i];
        float c, sn;
        rope_cos_sin(pos, f.x, f.y, &c, &sn);
        const int at = (i % N) * NV + i / N;
        wtq[at] = make_float4(wf[0][i] * c, wf[1][i] * sn, wf[1][i] * c, wf[0][i] * sn);
        wtk[at] = make_float4(wf[2][i] * c, wf[3][i] * sn, wf[3][i] * c, wf[2][i] * sn);
      }
      __syncwarp();
    }
    cp_async_wait<kFwdBufs - 1>();  // this lane's copies for (t, p) have landed
    const int h = slot + p * S;
    const bool act = h < NH, isq = h < a.Hq;
    Packet<T, N> x1, x2;
    float ss = 0.f;
    if (act) {
      const uint4 *d = stg + b * kFwdSlots * 32 + lane;
      *reinterpret_cast<uint4 *>(&x1) = d[0];
      *reinterpret_cast<uint4 *>(&x2) = d[32];
#pragma unroll
      for (int e = 0; e < N; ++e) {
        const float u1 = x1.get(e), u2 = x2.get(e);
        ss = fmaf(u1, u1, fmaf(u2, u2, ss));
      }
    }
    ss = slot_sum(ss, NV);  // every lane takes part
    if (act) {
      const float r = rsqrtf(fmaf(ss, a.inv_d, a.eps));
      const float4 *tw = (isq ? wtq : wtk) + j;
      Packet<T, N> o1, o2;
#pragma unroll
      for (int e = 0; e < N; e += 2) {
        const float4 t0 = tw[e * NV], t1 = tw[(e + 1) * NV];
        const float a0 = x1.get(e), b0 = x2.get(e), a1 = x1.get(e + 1), b1 = x2.get(e + 1);
        o1.set2(e, r * fmaf(a0, t0.x, -b0 * t0.y), r * fmaf(a1, t1.x, -b1 * t1.y));
        o2.set2(e, r * fmaf(b0, t0.z, a0 * t0.w), r * fmaf(b1, t1.z, a1 * t1.w));
      }
      T *dst = isq ? a.oq + t * a.ld_oq + (Idx)h * D : a.ok + t * a.ld_ok + (Idx)(h - a.Hq) * D;
      store_packet<T, N>(dst + (Idx)j * N, o1);
      store_packet<T, N>(dst + half + (Idx)j * N, o2);
      if (j == 0) {
        if (isq && a.rq) a.rq[t * a.Hq + h] = r;
        if (!isq && a.rk) a.rk[t * a.Hkv + (h - a.Hq)] = r;
      }
    }
    advance(t, p);
    b = b + 1 == kFwdBufs ? 0 : b + 1;
  }
  cp_async_wait<0>();
}

// bf16 heads whose half is 8 NV values, NV a power of two dividing 32: the
// lean form of qk_norm_rope_fwd_pipe, as qk_rope_lean is of qk_rope_pipe:
// the same token order (warp w of G takes tokens w, w + G, ...), the weighted
// rotation table laid out for fp32 pairs and the rotation on pairs.  A head's sum of squares
// keeps the scalar order of the other forms, so r (saved, or recomputed by
// the backward) is the same bits, and every output is rounded exactly like
// qk_norm_rope_fwd_pipe's: the two kernels agree bit for bit.
// Shared memory: per warp four tables of 4 NV entries, for lane j's column
// pair m (columns 8 j + 2 m and 8 j + 2 m + 1) at m NV + j:
//   0: (A, A', B, B') for Q   1: (C, C', E, E') for Q   2, 3: the same for K
// with (A, B, C, E) = (w1 cos, w2 sin, w2 cos, w1 sin) of the column (primed:
// the pair's second column); then the per-warp staging ring.
template <int NV> constexpr size_t fwd_lean_tab_bytes() {
  return sizeof(float4) * kWarps * 4 * 4 * NV;
}

constexpr int kFwdLeanBlocks = 3;  // CTAs per SM the lean forward is compiled for

template <typename Idx, int NV>
__global__ void __launch_bounds__(kThreads, kFwdLeanBlocks)
qk_norm_rope_fwd_lean(const NormRopeParams<bf16, Idx> a, const __grid_constant__ RopeFreqs fr) {
  constexpr int N = 8, half = N * NV, D = 2 * half, S = 32 / NV;
  extern __shared__ float4 dyn[];
  __shared__ float2 freq[half];
  __shared__ float wf[4][half];  // wq first half, wq second, wk first, wk second
  __shared__ int32_t cu_s[kCuInShared];
  const int NH = a.Hq + a.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = lane % NV, slot = lane / NV;
  float4 *const tab = dyn + warp * 4 * 4 * NV;  // [4][4 NV]
  uint4 *const stg = reinterpret_cast<uint4 *>(dyn + kWarps * 4 * 4 * NV) +
                     warp * (kFwdBufs * kFwdSlots * 32) + lane;

  for (int i = threadIdx.x; i < half; i += blockDim.x) freq[i] = make_float2(fr.hi[i], fr.lo[i]);
  pdl_wait();
  pdl_trigger();
  if (rope_skipped(fr)) return;  // malformed cu_seqlens: every output untouched
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    wf[0][i] = a.Hq > 0 ? to_float(a.wq[i]) : 0.f;
    wf[1][i] = a.Hq > 0 ? to_float(a.wq[half + i]) : 0.f;
    wf[2][i] = a.Hkv > 0 ? to_float(a.wk[i]) : 0.f;
    wf[3][i] = a.Hkv > 0 ? to_float(a.wk[half + i]) : 0.f;
  }
  const bool cu_staged = a.B < kCuInShared;
  if (cu_staged)
    for (int i = threadIdx.x; i <= a.B; i += blockDim.x) cu_s[i] = __ldg(a.cu + i);
  __syncthreads();  // the frequency, weight and boundary tables; no block barrier follows
  const int32_t *bounds = cu_staged ? cu_s : a.cu;

  // this warp's tokens: t, t + G, ... below rows
  const Idx G = (Idx)gridDim.x * kWarps;
  Idx t = (Idx)blockIdx.x * kWarps + warp;
  if (t >= a.rows) return;
  const int passes = (NH + S - 1) / S;

  Idx t2 = t;
  int p2 = 0, b2 = 0;
  const bf16 *q2 = a.q + t2 * a.ld_q + j * N, *k2 = a.k + t2 * a.ld_k + j * N - (Idx)a.Hq * D;
  auto stage = [&]() {
    const int h = slot + p2 * S;
    if (t2 < a.rows && h < NH) {
      const bf16 *v = (h < a.Hq ? q2 : k2) + (Idx)h * D;
      uint4 *d = stg + b2 * (kFwdSlots * 32);
      cp_async16(d, v);
      cp_async16(d + 32, v + half);
    }
    cp_async_commit();  // one group per pass on every lane, empty or not
    if (++p2 == passes) {
      p2 = 0;
      t2 += G;
      q2 += G * a.ld_q;
      k2 += G * a.ld_k;
    }
    b2 = b2 + 1 == kFwdBufs ? 0 : b2 + 1;
  };
#pragma unroll
  for (int i = 0; i < kFwdBufs - 1; ++i) stage();

  bf16 *oqr = a.oq + t * a.ld_oq + j * N, *okr = a.ok + t * a.ld_ok + j * N - (Idx)a.Hq * D;
  int p = 0, b = 0;
  while (t < a.rows) {  // warp-uniform
    stage();
    if (p == 0) {
      const int pos = position_of<Idx>(t, bounds, a.B);
      __syncwarp();  // the previous token's tables have been read
      float *tf = reinterpret_cast<float *>(tab);
#pragma unroll
      for (int i = lane; i < half; i += 32) {
        const float2 f = freq[i];
        float c, sn;
        rope_cos_sin(pos, f.x, f.y, &c, &sn);
        const int at = 4 * (((i % N) >> 1) * NV + i / N) + (i & 1);
        tf[at] = wf[0][i] * c;                          // Q: A
        tf[at + 2] = wf[1][i] * sn;                     // Q: B
        tf[4 * 4 * NV + at] = wf[1][i] * c;             // Q: C
        tf[4 * 4 * NV + at + 2] = wf[0][i] * sn;        // Q: E
        tf[2 * 4 * 4 * NV + at] = wf[2][i] * c;         // K: A
        tf[2 * 4 * 4 * NV + at + 2] = wf[3][i] * sn;    // K: B
        tf[3 * 4 * 4 * NV + at] = wf[3][i] * c;         // K: C
        tf[3 * 4 * 4 * NV + at + 2] = wf[2][i] * sn;    // K: E
      }
      __syncwarp();
    }
    cp_async_wait<kFwdBufs - 1>();  // this lane's copies for (t, p) have landed
    const int h = slot + p * S;
    const bool act = h < NH, isq = h < a.Hq;
    float2 xa[4], xb[4];
    float ss = 0.f;
    if (act) {
      const uint4 *d = stg + b * (kFwdSlots * 32);
      unpack8(d[0], xa);
      unpack8(d[32], xb);
#pragma unroll
      for (int m = 0; m < 4; ++m) {  // the scalar order of the other forms, column by column
        ss = fmaf(xa[m].x, xa[m].x, fmaf(xb[m].x, xb[m].x, ss));
        ss = fmaf(xa[m].y, xa[m].y, fmaf(xb[m].y, xb[m].y, ss));
      }
    }
    ss = slot_sum(ss, NV);  // every lane takes part
    if (act) {
      const float r = rsqrtf(fmaf(ss, a.inv_d, a.eps));
      const float2 r2 = make_float2(r, r);
      const float4 *tab_ab = tab + (isq ? 0 : 2) * 4 * NV + j;
      const float4 *tab_ce = tab_ab + 4 * NV;
      uint32_t o1[4], o2[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float4 ab = tab_ab[m * NV], ce = tab_ce[m * NV];
        const float2 A2 = make_float2(ab.x, ab.y), B2 = make_float2(ab.z, ab.w);
        const float2 C2 = make_float2(ce.x, ce.y), E2 = make_float2(ce.z, ce.w);
        const float2 bB = __fmul2_rn(xb[m], B2), aE = __fmul2_rn(xa[m], E2);
        // r (a A - b B) and r (b C + a E), each fma rounded once as in the scalar form
        o1[m] = bf2_pack(__fmul2_rn(r2, __ffma2_rn(xa[m], A2, make_float2(-bB.x, -bB.y))));
        o2[m] = bf2_pack(__fmul2_rn(r2, __ffma2_rn(xb[m], C2, aE)));
      }
      bf16 *dst = (isq ? oqr : okr) + (Idx)h * D;
      *reinterpret_cast<uint4 *>(dst) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
      *reinterpret_cast<uint4 *>(dst + half) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
      if (j == 0) {
        if (isq && a.rq) a.rq[t * a.Hq + h] = r;
        if (!isq && a.rk) a.rk[t * a.Hkv + (h - a.Hq)] = r;
      }
    }
    if (++p == passes) {
      p = 0;
      t += G;
      oqr += G * a.ld_oq;
      okr += G * a.ld_ok;
    }
    b = b + 1 == kFwdBufs ? 0 : b + 1;
  }
  cp_async_wait<0>();
}

// The CTA's dwq | dwk partial row: sum over the warp's lanes that hold the
// same packet j (lane % NV == j), then over the CTA's warps in order, into
// ws[blockIdx.x].
template <int N>
__device__ __forceinline__ void write_partial(float (&acc)[4][N], float *part, float *ws, int D,
                                              int NV, int j, int lane, int warp) {
  const int nwarps = (int)(blockDim.x >> 5);
  const int half = D >> 1;
#pragma unroll
  for (int g = 0; g < 4; ++g)
#pragma unroll
    for (int e = 0; e < N; ++e)
      for (int o = NV; o < 32; o <<= 1) acc[g][e] += __shfl_xor_sync(0xffffffffu, acc[g][e], o);
  if (lane < NV) {  // lane == j: the warp's first lane with this packet
    float *mine = part + warp * 2 * D;  // [warps][2D]
#pragma unroll
    for (int e = 0; e < N; ++e) {
      mine[j * N + e] = acc[0][e];
      mine[half + j * N + e] = acc[1][e];
      mine[D + j * N + e] = acc[2][e];
      mine[D + half + j * N + e] = acc[3][e];
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c < 2 * D; c += blockDim.x) {
    float s = 0.f;
    for (int w = 0; w < nwarps; ++w) s += part[w * 2 * D + c];
    ws[(size_t)blockIdx.x * 2 * D + c] = s;
  }
}

template <typename T, typename Idx, int N, bool HAS_RSTD>
__global__ void __launch_bounds__(kThreads, 2)
qk_norm_rope_bwd_warp(const NormRopeParams<T, Idx> a, const __grid_constant__ RopeFreqs fr) {
  // [warps][D/2] (cos, -sin), then [warps][2D] fp32 partials, then the
  // staging buffers (16-byte aligned: D is a multiple of 8 here)
  extern __shared__ float2 tab[];
  __shared__ float2 freq[kRopeMaxHalf];
  __shared__ int32_t cu_s[kCuInShared];
  const int D = a.D, half = D >> 1, NV = half / N, S = 32 / NV, NH = a.Hq + a.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = lane % NV, slot = lane / NV;
  float *part = reinterpret_cast<float *>(tab + kWarps * half);

  for (int i = threadIdx.x; i < half; i += blockDim.x) freq[i] = make_float2(fr.hi[i], fr.lo[i]);
  pdl_wait();
  pdl_trigger();
  if (rope_skipped(fr)) return;  // malformed cu_seqlens: every output untouched
  // the sequence boundaries in shared memory when they fit (every token's
  // position is a binary search over them); read after the barrier below
  const bool cu_staged = a.B < kCuInShared;
  if (cu_staged)
    for (int i = threadIdx.x; i <= a.B; i += blockDim.x) cu_s[i] = __ldg(a.cu + i);
  const int32_t *bounds = cu_staged ? cu_s : a.cu;
  // the norm weights are re-read per head (L1 hits) rather than held in
  // registers, which go to the four accumulators below
  float acc[4][N];  // dwq first half, dwq second half, dwk first half, dwk second half
#pragma unroll
  for (int g = 0; g < 4; ++g)
#pragma unroll
    for (int e = 0; e < N; ++e) acc[g][e] = 0.f;
  __syncthreads();  // the frequency table and the boundaries

  float2 *wt = tab + warp * half;
  uint4 *stg =
      reinterpret_cast<uint4 *>(part + kWarps * 2 * D) + warp * (kBwdBufs * kBwdSlots * 32);
  const Idx step = (Idx)gridDim.x * kWarps;
  const int passes = (NH + S - 1) / S;  // head passes per token, the same on every lane
  // Copies this lane's packets of (token tt, head pass p) into buffer b: both
  // halves of the output gradient and of the pre-norm input, and r.  Every
  // lane commits one group per pass, empty or not.
  auto stage = [&](Idx tt, int p, int b) {
    const int h = slot + p * S;
    if (tt < a.rows && h < NH) {
      const bool isq = h < a.Hq;
      const int hk = h - a.Hq;
      const T *gp = (isq ? a.gq + tt * a.ld_gq + (Idx)h * D : a.gk + tt * a.ld_gk + (Idx)hk * D) +
                    j * N;
      const T *vp =
          (isq ? a.q + tt * a.ld_q + (Idx)h * D : a.k + tt * a.ld_k + (Idx)hk * D) + j * N;
      uint4 *d = stg + b * kBwdSlots * 32 + lane;
      cp_async16(d, gp);
      cp_async16(d + 32, gp + half);
      cp_async16(d + 64, vp);
      cp_async16(d + 96, vp + half);
      if (HAS_RSTD) cp_async4(d + 128, isq ? a.rq + tt * a.Hq + h : a.rk + tt * a.Hkv + hk);
    }
    cp_async_commit();
  };
  // (cos, -sin) of this lane's columns are read from the table per head
  // rather than held in registers
  const float4 *cs_j = reinterpret_cast<const float4 *>(wt) + j;
  // (t, p): the pass computed now; (t2, p2): the last pass staged
  auto advance = [&](Idx &tt, int &pp) {
    if (++pp == passes) {
      pp = 0;
      tt += step;
    }
  };
  Idx t = (Idx)blockIdx.x * kWarps + warp, t2 = t;
  int p = 0, p2 = 0, b = 0;
  stage(t2, p2, 0);
  for (int i = 1; i < kBwdBufs - 1; ++i) {
    advance(t2, p2);
    stage(t2, p2, i);
  }
  while (t < a.rows) {  // warp-uniform
    advance(t2, p2);
    // the pass kBwdBufs - 1 ahead goes into the buffer computed last time
    stage(t2, p2, b == 0 ? kBwdBufs - 1 : b - 1);
    if (p == 0) {
      __syncwarp();  // the previous token's table has been read
      // (cos, -sin) of columns j N + e and j N + e + 1 (e even) in one
      // 16-byte entry at (e / 2) NV + j: a head's lanes read consecutive
      // entries
      const int pos = position_of<Idx>(t, bounds, a.B);
      for (int c = lane; c < half; c += 32) {
        const float2 f = freq[c];
        float cv, sn;
        rope_cos_sin(pos, f.x, f.y, &cv, &sn);
        const int e = c % N;
        wt[2 * ((e >> 1) * NV + c / N) + (e & 1)] = make_float2(cv, -sn);
      }
      __syncwarp();
    }
    cp_async_wait<kBwdBufs - 1>();  // this lane's copies for (t, p) have landed
    {
      const int h = slot + p * S;
      const bool act = h < NH;
      const bool isq = h < a.Hq;
      const int hk = h - a.Hq;
      Packet<T, N> g1, g2, v1, v2, w1, w2;
      float r = 0.f;
      if (act) {
        const uint4 *d = stg + b * kBwdSlots * 32 + lane;
        const T *wp = (isq ? a.wq : a.wk) + j * N;
        *reinterpret_cast<uint4 *>(&g1) = d[0];
        *reinterpret_cast<uint4 *>(&g2) = d[32];
        *reinterpret_cast<uint4 *>(&v1) = d[64];
        *reinterpret_cast<uint4 *>(&v2) = d[96];
        w1 = load_packet<T, N>(wp);
        w2 = load_packet<T, N>(wp + half);
        if (HAS_RSTD) r = *reinterpret_cast<const float *>(d + 128);
      }
      float dn1[N], dn2[N];
      float2 cs = make_float2(0.f, 0.f);  // (sum dn w v, sum v v)
      if (act) {
#pragma unroll
        for (int e = 0; e < N; ++e) {
          const float a1 = g1.get(e), a2 = g2.get(e);
          const float4 c4 = cs_j[(e >> 1) * NV];
          const float2 c = (e & 1) ? make_float2(c4.z, c4.w) : make_float2(c4.x, c4.y);
          dn1[e] = fmaf(a1, c.x, -a2 * c.y);
          dn2[e] = fmaf(a2, c.x, a1 * c.y);
          const float u1 = v1.get(e), u2 = v2.get(e);
          cs.x = fmaf(dn1[e] * w1.get(e), u1, fmaf(dn2[e] * w2.get(e), u2, cs.x));
          if (!HAS_RSTD) cs.y = fmaf(u1, u1, fmaf(u2, u2, cs.y));
        }
      }
      if (HAS_RSTD)
        cs.x = slot_sum(cs.x, NV);
      else
        cs = slot_sum2(cs, NV);
      if (act) {
        if (!HAS_RSTD) r = rsqrtf(fmaf(cs.y, a.inv_d, a.eps));
        const float am = r * r * r * cs.x * a.inv_d;
        Packet<T, N> o1, o2;
        // fixed accumulator indices (a runtime index would put acc in
        // local memory): a q head adds to 0 and 1, a k head to 2 and 3
        const float rq_ = isq ? r : 0.f, rk_ = isq ? 0.f : r;
#pragma unroll
        for (int e = 0; e < N; ++e) {
          const float u1 = v1.get(e), u2 = v2.get(e);
          o1.set(e, fmaf(-am, u1, r * w1.get(e) * dn1[e]));
          o2.set(e, fmaf(-am, u2, r * w2.get(e) * dn2[e]));
          const float p1 = dn1[e] * u1, p2 = dn2[e] * u2;
          acc[0][e] = fmaf(p1, rq_, acc[0][e]);
          acc[1][e] = fmaf(p2, rq_, acc[1][e]);
          acc[2][e] = fmaf(p1, rk_, acc[2][e]);
          acc[3][e] = fmaf(p2, rk_, acc[3][e]);
        }
        T *dst = isq ? a.oq + t * a.ld_oq + (Idx)h * D : a.ok + t * a.ld_ok + (Idx)hk * D;
        store_packet<T, N>(dst + (Idx)j * N, o1);
        store_packet<T, N>(dst + half + (Idx)j * N, o2);
      }
    }
    advance(t, p);
    b = b + 1 == kBwdBufs ? 0 : b + 1;
  }
  cp_async_wait<0>();
  write_partial<N>(acc, part, a.ws, D, NV, j, lane, warp);
}

// bf16 heads whose half is 8 NV values, NV a power of two dividing 32: the
// lean form of qk_norm_rope_bwd_warp (same token order, staging and
// reductions), with the inverse rotation, the norm's gradient and the dw sums
// on fp32 pairs and the norm weights as fp32 in shared memory.  sum v^2 (r
// recomputed) keeps the forward's scalar order, so a recomputed r equals the
// saved one bit for bit; sum dn w v runs as one pair chain per lane.
// Shared memory: [warps][4 NV] float4 (cos, cos', -sin, -sin') of lane j's
// column pair m at m NV + j; then [warps][2D] fp32 partials; then the
// per-warp staging ring.
template <int NV> constexpr size_t bwd_lean_tab_bytes() { return sizeof(float4) * kWarps * 4 * NV; }

template <typename Idx, int NV, bool HAS_RSTD>
__global__ void __launch_bounds__(kThreads, 2)
qk_norm_rope_bwd_lean(const NormRopeParams<bf16, Idx> a, const __grid_constant__ RopeFreqs fr) {
  constexpr int N = 8, half = N * NV, D = 2 * half, S = 32 / NV;
  extern __shared__ float4 dyn[];
  __shared__ float2 freq[half];
  __shared__ float wfl[4][half];  // wq first half, wq second, wk first, wk second
  __shared__ int32_t cu_s[kCuInShared];
  const int NH = a.Hq + a.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = lane % NV, slot = lane / NV;
  float4 *const tab = dyn + warp * 4 * NV;
  float *const part = reinterpret_cast<float *>(dyn + kWarps * 4 * NV);  // [warps][2D]
  uint4 *const stg = reinterpret_cast<uint4 *>(part + kWarps * 2 * D) +
                     warp * (kBwdBufs * kBwdSlots * 32) + lane;

  for (int i = threadIdx.x; i < half; i += blockDim.x) freq[i] = make_float2(fr.hi[i], fr.lo[i]);
  pdl_wait();
  pdl_trigger();
  if (rope_skipped(fr)) return;  // malformed cu_seqlens: every output untouched
  for (int i = threadIdx.x; i < half; i += blockDim.x) {
    wfl[0][i] = a.Hq > 0 ? to_float(a.wq[i]) : 0.f;
    wfl[1][i] = a.Hq > 0 ? to_float(a.wq[half + i]) : 0.f;
    wfl[2][i] = a.Hkv > 0 ? to_float(a.wk[i]) : 0.f;
    wfl[3][i] = a.Hkv > 0 ? to_float(a.wk[half + i]) : 0.f;
  }
  const bool cu_staged = a.B < kCuInShared;
  if (cu_staged)
    for (int i = threadIdx.x; i <= a.B; i += blockDim.x) cu_s[i] = __ldg(a.cu + i);
  __syncthreads();  // the frequency, weight and boundary tables
  const int32_t *bounds = cu_staged ? cu_s : a.cu;

  float2 acc[4][4];  // dwq first half, dwq second half, dwk first half, dwk second half
#pragma unroll
  for (int g = 0; g < 4; ++g)
#pragma unroll
    for (int m = 0; m < 4; ++m) acc[g][m] = make_float2(0.f, 0.f);

  // tokens t, t + G, ... (every warp runs the loop, then the CTA combines)
  const Idx G = (Idx)gridDim.x * kWarps;
  Idx t = (Idx)blockIdx.x * kWarps + warp;
  const int passes = (NH + S - 1) / S;
  Idx t2 = t;
  int p2 = 0, b2 = 0;
  auto stage = [&]() {
    const int h = slot + p2 * S;
    if (t2 < a.rows && h < NH) {
      const bool isq = h < a.Hq;
      const int hk = h - a.Hq;
      const bf16 *gp =
          (isq ? a.gq + t2 * a.ld_gq + (Idx)h * D : a.gk + t2 * a.ld_gk + (Idx)hk * D) + j * N;
      const bf16 *vp =
          (isq ? a.q + t2 * a.ld_q + (Idx)h * D : a.k + t2 * a.ld_k + (Idx)hk * D) + j * N;
      uint4 *d = stg + b2 * (kBwdSlots * 32);
      cp_async16(d, gp);
      cp_async16(d + 32, gp + half);
      cp_async16(d + 64, vp);
      cp_async16(d + 96, vp + half);
      if (HAS_RSTD) cp_async4(d + 128, isq ? a.rq + t2 * a.Hq + h : a.rk + t2 * a.Hkv + hk);
    }
    cp_async_commit();  // one group per pass on every lane, empty or not
    if (++p2 == passes) {
      p2 = 0;
      t2 += G;
    }
    b2 = b2 + 1 == kBwdBufs ? 0 : b2 + 1;
  };
#pragma unroll
  for (int i = 0; i < kBwdBufs - 1; ++i) stage();
  int p = 0, b = 0;
  while (t < a.rows) {  // warp-uniform
    stage();
    if (p == 0) {
      const int pos = position_of<Idx>(t, bounds, a.B);
      __syncwarp();  // the previous token's table has been read
      float *tf = reinterpret_cast<float *>(tab);
#pragma unroll
      for (int i = lane; i < half; i += 32) {
        const float2 f = freq[i];
        float cv, sn;
        rope_cos_sin(pos, f.x, f.y, &cv, &sn);
        const int at = 4 * (((i % N) >> 1) * NV + i / N) + (i & 1);
        tf[at] = cv;
        tf[at + 2] = -sn;
      }
      __syncwarp();
    }
    cp_async_wait<kBwdBufs - 1>();  // this lane's copies for (t, p) have landed
    const int h = slot + p * S;
    const bool act = h < NH, isq = h < a.Hq;
    const uint4 *d = stg + b * (kBwdSlots * 32);
    float2 dn1[4], dn2[4], v1[4], v2[4];
    float r = 0.f, ss = 0.f;
    float2 c2 = make_float2(0.f, 0.f);
    const float *w1s = wfl[isq ? 0 : 2] + j * N, *w2s = wfl[isq ? 1 : 3] + j * N;
    if (act) {
      float2 g1[4], g2[4];
      unpack8(d[0], g1);
      unpack8(d[32], g2);
      unpack8(d[64], v1);
      unpack8(d[96], v2);
      if (HAS_RSTD) r = *reinterpret_cast<const float *>(d + 128);
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float4 cs = tab[m * NV + j];
        const float2 C2 = make_float2(cs.x, cs.y), NS2 = make_float2(cs.z, cs.w);
        // the rotation by -phi: dn1 = g1 cos + g2 sin, dn2 = g2 cos - g1 sin
        const float2 t1 = __fmul2_rn(g2[m], NS2), t2 = __fmul2_rn(g1[m], NS2);
        dn1[m] = __ffma2_rn(g1[m], C2, make_float2(-t1.x, -t1.y));
        dn2[m] = __ffma2_rn(g2[m], C2, t2);
        const float2 W1 = *reinterpret_cast<const float2 *>(w1s + 2 * m);
        const float2 W2 = *reinterpret_cast<const float2 *>(w2s + 2 * m);
        c2 = __ffma2_rn(__fmul2_rn(dn1[m], W1), v1[m],
                        __ffma2_rn(__fmul2_rn(dn2[m], W2), v2[m], c2));
        if (!HAS_RSTD) {  // the forward's order, column by column
          ss = fmaf(v1[m].x, v1[m].x, fmaf(v2[m].x, v2[m].x, ss));
          ss = fmaf(v1[m].y, v1[m].y, fmaf(v2[m].y, v2[m].y, ss));
        }
      }
    }
    float cx = c2.x + c2.y;
    if (HAS_RSTD) {
      cx = slot_sum(cx, NV);
    } else {
      const float2 cs = slot_sum2(make_float2(cx, ss), NV);
      cx = cs.x;
      ss = cs.y;
    }
    if (act) {
      if (!HAS_RSTD) r = rsqrtf(fmaf(ss, a.inv_d, a.eps));
      const float am = r * r * r * cx * a.inv_d;
      const float2 r2 = make_float2(r, r), nam2 = make_float2(-am, -am);
      // fixed accumulator indices (a runtime index would put acc in local
      // memory): a q head adds to 0 and 1, a k head to 2 and 3
      const float2 rq2 = isq ? r2 : make_float2(0.f, 0.f), rk2 = isq ? make_float2(0.f, 0.f) : r2;
      uint32_t o1[4], o2[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float2 W1 = *reinterpret_cast<const float2 *>(w1s + 2 * m);
        const float2 W2 = *reinterpret_cast<const float2 *>(w2s + 2 * m);
        // dv = r w dn - r^3 v c / D;  dw += dn v r
        o1[m] = bf2_pack(__ffma2_rn(nam2, v1[m], __fmul2_rn(__fmul2_rn(r2, W1), dn1[m])));
        o2[m] = bf2_pack(__ffma2_rn(nam2, v2[m], __fmul2_rn(__fmul2_rn(r2, W2), dn2[m])));
        const float2 p1 = __fmul2_rn(dn1[m], v1[m]), q1 = __fmul2_rn(dn2[m], v2[m]);
        acc[0][m] = __ffma2_rn(p1, rq2, acc[0][m]);
        acc[1][m] = __ffma2_rn(q1, rq2, acc[1][m]);
        acc[2][m] = __ffma2_rn(p1, rk2, acc[2][m]);
        acc[3][m] = __ffma2_rn(q1, rk2, acc[3][m]);
      }
      bf16 *dst = (isq ? a.oq + t * a.ld_oq + (Idx)h * D
                       : a.ok + t * a.ld_ok + (Idx)(h - a.Hq) * D) + j * N;
      *reinterpret_cast<uint4 *>(dst) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
      *reinterpret_cast<uint4 *>(dst + half) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
    }
    if (++p == passes) {
      p = 0;
      t += G;
    }
    b = b + 1 == kBwdBufs ? 0 : b + 1;
  }
  cp_async_wait<0>();
  float accf[4][N];
#pragma unroll
  for (int g = 0; g < 4; ++g)
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      accf[g][2 * m] = acc[g][m].x;
      accf[g][2 * m + 1] = acc[g][m].y;
    }
  write_partial<N>(accf, part, a.ws, D, NV, j, lane, warp);
}

// Element-wise forms: one warp per token, heads one after another, lane i
// owning the pairs i, i + 32, ... of every head.
template <typename T, typename Idx>
__global__ void __launch_bounds__(kThreads)
qk_norm_rope_fwd_generic(const NormRopeParams<T, Idx> a, const __grid_constant__ RopeFreqs fr) {
  extern __shared__ float2 tab[];
  __shared__ float2 freq[kRopeMaxHalf];
  const int D = a.D, half = D >> 1, NH = a.Hq + a.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Idx t = (Idx)blockIdx.x * kWarps + warp;
  for (int i = threadIdx.x; i < half; i += blockDim.x) freq[i] = make_float2(fr.hi[i], fr.lo[i]);
  pdl_wait();
  pdl_trigger();
  if (rope_skipped(fr)) return;  // malformed cu_seqlens: every output untouched
  __syncthreads();
  if (t >= a.rows) return;
  float2 *wt = tab + warp * half;
  token_table(wt, freq, half, position_of<Idx>(t, a.cu, a.B), 1.0f, lane);
  __syncwarp();
  for (int h = 0; h < NH; ++h) {
    const bool isq = h < a.Hq;
    const int hk = h - a.Hq;
    const T *v = isq ? a.q + t * a.ld_q + (Idx)h * D : a.k + t * a.ld_k + (Idx)hk * D;
    const T *w = isq ? a.wq : a.wk;
    // the sum of squares in the backward's order (pairs), so that r
    // recomputed there is bit-identical
    float ss = 0.f;
#pragma unroll
    for (int m = 0; m < kPairsPerLane; ++m) {
      const int i = lane + 32 * m;
      if (i < half) {
        const float u1 = to_float(v[i]), u2 = to_float(v[i + half]);
        ss = fmaf(u1, u1, fmaf(u2, u2, ss));
      }
    }
    ss = warp_sum(ss);
    const float r = rsqrtf(fmaf(ss, a.inv_d, a.eps));
    T *o = isq ? a.oq + t * a.ld_oq + (Idx)h * D : a.ok + t * a.ld_ok + (Idx)hk * D;
    float n1[kPairsPerLane], n2[kPairsPerLane];
#pragma unroll
    for (int m = 0; m < kPairsPerLane; ++m) {
      const int i = lane + 32 * m;
      if (i < half) {
        n1[m] = to_float(v[i]) * r * to_float(w[i]);
        n2[m] = to_float(v[i + half]) * r * to_float(w[i + half]);
      }
    }
    __syncwarp();  // every lane has read the head before any lane writes it (o may be v)
#pragma unroll
    for (int m = 0; m < kPairsPerLane; ++m) {
      const int i = lane + 32 * m;
      if (i < half) {
        const float2 c = wt[i];
        o[i] = from_float<T>(fmaf(n1[m], c.x, -n2[m] * c.y));
        o[i + half] = from_float<T>(fmaf(n2[m], c.x, n1[m] * c.y));
      }
    }
    if (lane == 0) {
      if (isq && a.rq) a.rq[t * a.Hq + h] = r;
      if (!isq && a.rk) a.rk[t * a.Hkv + hk] = r;
    }
  }
}

template <typename T, typename Idx, bool HAS_RSTD>
__global__ void __launch_bounds__(kThreads)
qk_norm_rope_bwd_generic(const NormRopeParams<T, Idx> a, const __grid_constant__ RopeFreqs fr) {
  extern __shared__ float2 tab[];  // [warps][D/2], then [warps][2D] fp32 partials
  __shared__ float2 freq[kRopeMaxHalf];
  const int D = a.D, half = D >> 1, NH = a.Hq + a.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float *part = reinterpret_cast<float *>(tab + kWarps * half);
  for (int i = threadIdx.x; i < half; i += blockDim.x) freq[i] = make_float2(fr.hi[i], fr.lo[i]);
  pdl_wait();
  pdl_trigger();
  if (rope_skipped(fr)) return;  // malformed cu_seqlens: every output untouched
  float acc[4][kPairsPerLane];
#pragma unroll
  for (int g = 0; g < 4; ++g)
#pragma unroll
    for (int m = 0; m < kPairsPerLane; ++m) acc[g][m] = 0.f;
  __syncthreads();
  float2 *wt = tab + warp * half;
  const Idx step = (Idx)gridDim.x * kWarps;
  for (Idx t = (Idx)blockIdx.x * kWarps + warp; t < a.rows; t += step) {
    __syncwarp();
    token_table(wt, freq, half, position_of<Idx>(t, a.cu, a.B), -1.0f, lane);
    __syncwarp();
    for (int h = 0; h < NH; ++h) {
      const bool isq = h < a.Hq;
      const int hk = h - a.Hq;
      const T *g = isq ? a.gq + t * a.ld_gq + (Idx)h * D : a.gk + t * a.ld_gk + (Idx)hk * D;
      const T *v = isq ? a.q + t * a.ld_q + (Idx)h * D : a.k + t * a.ld_k + (Idx)hk * D;
      const T *w = isq ? a.wq : a.wk;
      float dn1[kPairsPerLane], dn2[kPairsPerLane];
      float2 cs = make_float2(0.f, 0.f);
#pragma unroll
      for (int m = 0; m < kPairsPerLane; ++m) {
        const int i = lane + 32 * m;
        if (i < half) {
          const float2 c = wt[i];
          const float a1 = to_float(g[i]), a2 = to_float(g[i + half]);
          dn1[m] = fmaf(a1, c.x, -a2 * c.y);
          dn2[m] = fmaf(a2, c.x, a1 * c.y);
          const float u1 = to_float(v[i]), u2 = to_float(v[i + half]);
          cs.x = fmaf(dn1[m] * to_float(w[i]), u1, fmaf(dn2[m] * to_float(w[i + half]), u2, cs.x));
          cs.y = fmaf(u1, u1, fmaf(u2, u2, cs.y));
        }
      }
      cs = warp_sum2(cs);
      const float r = HAS_RSTD ? (isq ? a.rq[t * a.Hq + h] : a.rk[t * a.Hkv + hk])
                               : rsqrtf(fmaf(cs.y, a.inv_d, a.eps));
      const float am = r * r * r * cs.x * a.inv_d;
      T *o = isq ? a.oq + t * a.ld_oq + (Idx)h * D : a.ok + t * a.ld_ok + (Idx)hk * D;
      const int g0 = isq ? 0 : 2;
      __syncwarp();  // every lane has read the head before any lane writes it (o may be g)
#pragma unroll
      for (int m = 0; m < kPairsPerLane; ++m) {
        const int i = lane + 32 * m;
        if (i < half) {
          const float u1 = to_float(v[i]), u2 = to_float(v[i + half]);
          o[i] = from_float<T>(fmaf(-am, u1, r * to_float(w[i]) * dn1[m]));
          o[i + half] = from_float<T>(fmaf(-am, u2, r * to_float(w[i + half]) * dn2[m]));
          acc[g0][m] = fmaf(dn1[m] * u1, r, acc[g0][m]);
          acc[g0 + 1][m] = fmaf(dn2[m] * u2, r, acc[g0 + 1][m]);
        }
      }
    }
  }
  float *mine = part + warp * 2 * D;
#pragma unroll
  for (int m = 0; m < kPairsPerLane; ++m) {
    const int i = lane + 32 * m;
    if (i < half) {
      mine[i] = acc[0][m];
      mine[half + i] = acc[1][m];
      mine[D + i] = acc[2][m];
      mine[D + half + i] = acc[3][m];
    }
  }
  __syncthreads();
  for (int c = threadIdx.x; c < 2 * D; c += blockDim.x) {
    float s = 0.f;
    for (int w = 0; w < kWarps; ++w) s += part[w * 2 * D + c];
    a.ws[(size_t)blockIdx.x * 2 * D + c] = s;
  }
}

template <typename T, typename Idx>
NormRopeParams<T, Idx> params_of(const QkNormRopeArgs &a) {
  return NormRopeParams<T, Idx>{
      (const T *)a.q,  (Idx)a.ld_q,  (const T *)a.k,  (Idx)a.ld_k,  (const T *)a.gq,
      (Idx)a.ld_gq,    (const T *)a.gk, (Idx)a.ld_gk, (T *)a.oq,     (Idx)a.ld_oq,
      (T *)a.ok,       (Idx)a.ld_ok, (const T *)a.wq, (const T *)a.wk, a.rq,
      a.rk,            a.ws,         a.cu,            a.B,           (Idx)a.T,
      a.Hq,            a.Hkv,        a.D,             a.eps,         (float)(1.0 / (double)a.D)};
}

cudaError_t finish_launch(cudaError_t e) { return e != cudaSuccess ? e : cudaGetLastError(); }

template <typename Idx, int NV>
cudaError_t fwd_lean_launch(const QkNormRopeArgs &a, const RopeFreqs &fr, const DeviceInfo &dev,
                            cudaStream_t s) {
  auto kern = qk_norm_rope_fwd_lean<Idx, NV>;
  const size_t smem = fwd_lean_tab_bytes<NV>() + kFwdStageBytes;
  const int occ = blocks_per_sm((const void *)kern, kThreads, smem, dev, kFwdLeanBlocks);
  int64_t P = ceil_div(a.T, (int64_t)kWarps);
  if (P > (int64_t)dev.sms * occ) P = (int64_t)dev.sms * occ;
  return finish_launch(launch_pdl(kern, dim3((unsigned)P), dim3(kThreads), smem, s,
                                  params_of<bf16, Idx>(a), fr));
}

template <typename T, typename Idx>
cudaError_t fwd_typed(bool warp_path, const QkNormRopeArgs &a, const RopeFreqs &fr,
                      const DeviceInfo &dev, cudaStream_t s) {
  constexpr int NV = VecWidth<T>::value;
  if constexpr (sizeof(T) == 2) {
    if (warp_path) {
      switch (a.D / 2 / NV) {
        case 1: return fwd_lean_launch<Idx, 1>(a, fr, dev, s);
        case 2: return fwd_lean_launch<Idx, 2>(a, fr, dev, s);
        case 4: return fwd_lean_launch<Idx, 4>(a, fr, dev, s);
        case 8: return fwd_lean_launch<Idx, 8>(a, fr, dev, s);
        case 16: return fwd_lean_launch<Idx, 16>(a, fr, dev, s);
        case 32: return fwd_lean_launch<Idx, 32>(a, fr, dev, s);
        default: break;
      }
    }
  }
  if (warp_path) {
    auto kern = qk_norm_rope_fwd_pipe<T, Idx, NV>;
    const size_t smem = sizeof(float4) * (size_t)kWarps * 2 * (a.D / 2) + kFwdStageBytes;
    const int occ = blocks_per_sm((const void *)kern, kThreads, smem, dev, kMaxBlocksPerSm);
    int64_t P = ceil_div(a.T, (int64_t)kWarps);
    if (P > (int64_t)dev.sms * occ) P = (int64_t)dev.sms * occ;
    return finish_launch(
        launch_pdl(kern, dim3((unsigned)P), dim3(kThreads), smem, s, params_of<T, Idx>(a), fr));
  }
  const size_t smem = sizeof(float2) * (size_t)kWarps * (a.D / 2);
  return finish_launch(launch_pdl(qk_norm_rope_fwd_generic<T, Idx>,
                                  dim3((unsigned)ceil_div(a.T, (int64_t)kWarps)), dim3(kThreads),
                                  smem, s, params_of<T, Idx>(a), fr));
}

template <typename Idx, int NV>
cudaError_t bwd_lean_launch(const QkNormRopeArgs &a, const RopeFreqs &fr, const DeviceInfo &dev,
                            cudaStream_t s) {
  const size_t smem = bwd_lean_tab_bytes<NV>() + sizeof(float) * (size_t)kWarps * 2 * a.D +
                      kBwdStageBytes;
  const bool rstd = a.rq != nullptr || a.rk != nullptr;
  // the grid (and with it the order of dwq's and dwk's sums) must not depend
  // on whether r is saved: size it for the less resident of the two forms
  const int occ_s = blocks_per_sm((const void *)qk_norm_rope_bwd_lean<Idx, NV, true>, kThreads,
                                  smem, dev, kMaxBlocksPerSm);
  const int occ_r = blocks_per_sm((const void *)qk_norm_rope_bwd_lean<Idx, NV, false>, kThreads,
                                  smem, dev, kMaxBlocksPerSm);
  const int occ = occ_s < occ_r ? occ_s : occ_r;
  int64_t P = ceil_div(a.T, (int64_t)kWarps);
  if (P > (int64_t)dev.sms * occ) P = (int64_t)dev.sms * occ;
  if (P > a.ws_rows) P = a.ws_rows;
  const NormRopeParams<bf16, Idx> k = params_of<bf16, Idx>(a);
  const dim3 grid((unsigned)P), block(kThreads);
  cudaError_t e = rstd ? launch_pdl(qk_norm_rope_bwd_lean<Idx, NV, true>, grid, block, smem, s,
                                    k, fr)
                       : launch_pdl(qk_norm_rope_bwd_lean<Idx, NV, false>, grid, block, smem, s,
                                    k, fr);
  if (e != cudaSuccess) return e;
  if (a.dwq || a.dwk) {
    e = launch_dw_reduce(a.ws, P, 2 * (int64_t)a.D, 2 * (int64_t)a.D, a.dwq, a.D, a.dwk, s,
                         a.skip);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

template <typename T, typename Idx>
cudaError_t bwd_typed(bool warp_path, const QkNormRopeArgs &a, const RopeFreqs &fr,
                      const DeviceInfo &dev, cudaStream_t s) {
  constexpr int NV = VecWidth<T>::value;
  if constexpr (sizeof(T) == 2) {
    if (warp_path) {
      switch (a.D / 2 / NV) {
        case 1: return bwd_lean_launch<Idx, 1>(a, fr, dev, s);
        case 2: return bwd_lean_launch<Idx, 2>(a, fr, dev, s);
        case 4: return bwd_lean_launch<Idx, 4>(a, fr, dev, s);
        case 8: return bwd_lean_launch<Idx, 8>(a, fr, dev, s);
        case 16: return bwd_lean_launch<Idx, 16>(a, fr, dev, s);
        case 32: return bwd_lean_launch<Idx, 32>(a, fr, dev, s);
        default: break;
      }
    }
  }
  const size_t smem = sizeof(float2) * (size_t)kWarps * (a.D / 2) +
                      sizeof(float) * (size_t)kWarps * 2 * a.D + (warp_path ? kBwdStageBytes : 0);
  const bool rstd = a.rq != nullptr || a.rk != nullptr;
  // the grid (and with it the order of dwq's and dwk's sums) must not depend
  // on whether r is saved: size it for the less resident of the two forms
  const void *k_saved = warp_path ? (const void *)qk_norm_rope_bwd_warp<T, Idx, NV, true>
                                  : (const void *)qk_norm_rope_bwd_generic<T, Idx, true>;
  const void *k_recomp = warp_path ? (const void *)qk_norm_rope_bwd_warp<T, Idx, NV, false>
                                   : (const void *)qk_norm_rope_bwd_generic<T, Idx, false>;
  const int occ_s = blocks_per_sm(k_saved, kThreads, smem, dev, kMaxBlocksPerSm);
  const int occ_r = blocks_per_sm(k_recomp, kThreads, smem, dev, kMaxBlocksPerSm);
  const int occ = occ_s < occ_r ? occ_s : occ_r;
  int64_t P = ceil_div(a.T, (int64_t)kWarps);
  if (P > (int64_t)dev.sms * occ) P = (int64_t)dev.sms * occ;
  if (P > a.ws_rows) P = a.ws_rows;
  const NormRopeParams<T, Idx> k = params_of<T, Idx>(a);
  const dim3 grid((unsigned)P), block(kThreads);
  cudaError_t e;
  if (warp_path)
    e = rstd ? launch_pdl(qk_norm_rope_bwd_warp<T, Idx, NV, true>, grid, block, smem, s, k, fr)
             : launch_pdl(qk_norm_rope_bwd_warp<T, Idx, NV, false>, grid, block, smem, s, k, fr);
  else
    e = rstd ? launch_pdl(qk_norm_rope_bwd_generic<T, Idx, true>, grid, block, smem, s, k, fr)
             : launch_pdl(qk_norm_rope_bwd_generic<T, Idx, false>, grid, block, smem, s, k, fr);
  if (e != cudaSuccess) return e;
  // dwq from columns [0, D) of the partial rows, dwk from [D, 2D): one launch
  if (a.dwq || a.dwk) {
    e = launch_dw_reduce(a.ws, P, 2 * (int64_t)a.D, 2 * (int64_t)a.D, a.dwq, a.D, a.dwk, s,
                         a.skip);
    if (e != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace

int64_t qk_norm_rope_partial_rows(int64_t T, const DeviceInfo &dev) {
  const int64_t cap = (int64_t)dev.sms * kMaxBlocksPerSm;
  const int64_t need = ceil_div(T, (int64_t)kWarps);
  return need < cap ? need : cap;
}

cudaError_t launch_qk_norm_rope(DType dt, bool vec, bool wide, const QkNormRopeArgs &a,
                                const DeviceInfo &dev, cudaStream_t s) {
  const RopeFreqs fr = make_rope_freqs(a.D, a.theta, a.inv_freq, a.skip);
  // the warp kernels need half a head to split evenly over a power-of-two
  // number of lanes (NV divides 32)
  const int n = dt == DType::F32 ? VecWidth<float>::value : VecWidth<bf16>::value;
  const int nv = vec ? a.D / 2 / n : 0;
  const bool warp_path = vec && nv >= 1 && nv <= 32 && (nv & (nv - 1)) == 0;
#define FTK_NR(T, Idx) \
  return a.backward ? bwd_typed<T, Idx>(warp_path, a, fr, dev, s) \
                    : fwd_typed<T, Idx>(warp_path, a, fr, dev, s);
  if (dt == DType::F32) {
    if (wide) { FTK_NR(float, int64_t) }
    FTK_NR(float, int32_t)
  }
  if (wide) { FTK_NR(bf16, int64_t) }
  FTK_NR(bf16, int32_t)
#undef FTK_NR
}

}  // namespace ftk
