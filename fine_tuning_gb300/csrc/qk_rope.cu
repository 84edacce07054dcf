// In-place rotary position embedding of Q and K together, rotate-half
// layout, over a packed batch of variable-length sequences.
//
// Sources: "Unsloth prétend accélérer 5 fois l'entraînement des LLM avec de
// nouveaux noyaux Triton et un auto-packing" (seventnews.com): Q and K are
// rotated by ONE kernel instead of two, variable-length RoPE, fully in place
// (no clone, no contiguous transpose); blocks are launched for groups of
// heads; LONG_INDEXING (64-bit offsets) for 500k-token runs; packing keeps
// the sequence-length metadata so positions restart in every sequence.
// Chronicals (arXiv 2601.02609), abstract, optimisation (1): fused QK-RoPE.
//
// For token t of sequence b, p = t - cu[b]; for i < D/2,
// phi_i = p * theta^(-2i/D) and every head vector v of Q and K becomes
//   v[i] <- v[i] cos phi_i - v[i+D/2] sin phi_i
//   v[i+D/2] <- v[i+D/2] cos phi_i + v[i] sin phi_i
// (backward: phi -> -phi, the transpose).  A caller may pass its own table
// of inverse frequencies instead of theta^(-2i/D) (a scaled RoPE such as
// the llama3 rule; the table is built on the host, rope_freqs.cu); the
// kernels only ever see f_i = inv_freq_i / 2pi.
//
// Heads whose half splits over a power-of-two number of lanes (every model
// measured) take qk_rope_pipe: persistent warps walk (token, head pass)
// pairs, each lane streaming its packets of the passes ahead through a
// per-warp cp.async ring.  The other forms remain for the remaining head
// sizes: qk_rope_staged (a TMA ring of whole tokens), qk_rope_warp (one warp
// per token) and qk_rope_kernel, where a CTA owns TOK consecutive tokens
// and, per token, TPT = NV * S threads (NV packet slots across one half of a
// head times S head slots; the thread with (slot s, packet j) rotates
// packet j of heads s, s+S, s+2S, ..., HPT heads per pass).  Every form finds
// a token's position by a binary search of the sequence boundaries
// (cu_seqlens, read on the device: no host synchronisation), kept in shared
// memory when they fit, and computes cos/sin of the token's D/2 angles once
// into shared memory, shared by every head of the token.  No cos/sin table
// is read from HBM.
//
// The angle is formed in turns, phi / 2pi = p * f_i with f_i split on the
// host into two floats (hi + lo, ~48 significant bits); p is split into a
// multiple of 4096 and a remainder so each partial product is exact or
// nearly so (Dekker's two-product via fma), the integer turns are dropped
// from every term, and sincospif() of the remaining fraction gives cos and
// sin.  The angle error stays near 1e-7 rad at p = 5e5, where a plain fp32
// p * inv_freq would be off by up to ~0.03 rad.
#include <cmath>

#include "common.cuh"
#include "launch.h"
#include "pair_math.cuh"
#include "rope_common.cuh"

namespace ftk {

namespace {

constexpr int kCtaThreads = 256;

template <typename T, typename Idx, int N, int HPT>
__global__ void __launch_bounds__(kCtaThreads, 3)
qk_rope_kernel(T *q, Idx ld_q, T *k, Idx ld_k, const int32_t *__restrict__ cu, int B,
               Idx rows, int Hq, int NH, int D, int S, int NV, int TOK, float sgn,
               const __grid_constant__ RopeFreqs fr) {
  extern __shared__ float2 cs[];  // [TOK][D/2] (cos, sgn*sin)
  __shared__ float2 freq[kRopeMaxHalf];  // (hi, lo) turns per position
  __shared__ int32_t cu_s[kCuInShared];
  pdl_wait();
  pdl_trigger();
  if (rope_skipped(fr)) return;  // malformed cu_seqlens: q, k untouched

  const int half = D >> 1;
  const int TPT = NV * S;
  const int tl = threadIdx.x / TPT;
  const int rem = threadIdx.x - tl * TPT;
  const int slot = rem / NV, j = rem - slot * NV;
  const Idx t = (Idx)blockIdx.x * TOK + tl;
  const bool active = tl < TOK && t < rows;
  T *const qrow = q + t * ld_q + (Idx)j * N;
  T *const krow = k + t * ld_k + (Idx)j * N - (Idx)Hq * D;
  auto head = [&](int h) -> T * { return (h < Hq ? qrow : krow) + (Idx)h * D; };

  // loads of this thread's first HPT heads go out first ...
  Packet<T, N> a[HPT], b[HPT];
#pragma unroll
  for (int m = 0; m < HPT; ++m) {
    const int h = m * S + slot;
    if (active && h < NH) {
      a[m] = load_packet<T, N>(head(h));
      b[m] = load_packet<T, N>(head(h) + half);
    }
  }

  // ... and while they are in flight: frequencies and sequence boundaries
  // into shared memory (one coalesced read each), then positions and
  // cos/sin of every (token, frequency) of the CTA
  for (int i = threadIdx.x; i < half; i += blockDim.x) freq[i] = make_float2(fr.hi[i], fr.lo[i]);
  const bool cu_staged = B < kCuInShared;
  if (cu_staged)
    for (int i = threadIdx.x; i <= B; i += blockDim.x) cu_s[i] = __ldg(cu + i);
  __syncthreads();
  const int32_t *bounds = cu_staged ? cu_s : cu;
  for (int e = threadIdx.x; e < TOK * half; e += blockDim.x) {
    const int tt = e / half, i = e - tt * half;
    const Idx tok = (Idx)blockIdx.x * TOK + tt;
    const int p = tok < rows ? position_of<Idx>(tok, bounds, B) : 0;
    const float2 f = freq[i];
    float c, s;
    rope_cos_sin(p, f.x, f.y, &c, &s);
    cs[e] = make_float2(c, sgn * s);
  }
  __syncthreads();

  if (!active) return;
  const float2 *row_cs = cs + tl * half + j * N;
  float cv[N], sv[N];
#pragma unroll
  for (int e = 0; e < N; ++e) {
    const float2 v = row_cs[e];
    cv[e] = v.x;
    sv[e] = v.y;
  }

  for (int h0 = 0;; h0 += HPT * S) {
#pragma unroll
    for (int m = 0; m < HPT; ++m) {
      const int h = h0 + m * S + slot;
      if (h < NH) {
        Packet<T, N> oa, ob;
#pragma unroll
        for (int e = 0; e < N; ++e) {
          const float x1 = a[m].get(e), x2 = b[m].get(e);
          oa.set(e, fmaf(x1, cv[e], -x2 * sv[e]));
          ob.set(e, fmaf(x2, cv[e], x1 * sv[e]));
        }
        store_packet<T, N>(head(h), oa);
        store_packet<T, N>(head(h) + half, ob);
      }
    }
    // heads beyond the first HPT * S (wide rows only)
    const int next = h0 + HPT * S;
    if (next >= NH) break;
#pragma unroll
    for (int m = 0; m < HPT; ++m) {
      const int h = next + m * S + slot;
      if (h < NH) {
        a[m] = load_packet<T, N>(head(h));
        b[m] = load_packet<T, N>(head(h) + half);
      }
    }
  }
}

// 16-byte aligned rows: a persistent grid of independent row groups.  A
// group (W warps) owns a ring of S shared-memory stages; a stage holds TB
// whole tokens (their Q rows, then their K rows).  The group's leader lane
// bulk-loads the group's blocks ahead (cp.async.bulk completing on the
// stage's mbarrier); while a block lands the group computes the block's
// positions and cos/sin; the warps rotate it in shared memory; the leader
// bulk-stores it back in place, and at the start of the next iteration, once
// that store has read the stage, refills the stage with the group's block S
// iterations ahead (so with S = 2 one block loads while the other rotates).  Groups
// synchronise only among their own warps, so the R groups of a CTA (and the
// CTAs of an SM) overlap each other's latencies.
template <typename T, typename Idx, int N>
__global__ void __launch_bounds__(kCtaThreads)
qk_rope_staged(T *q, Idx ld_q, T *k, Idx ld_k, const int32_t *__restrict__ cu, int B, Idx rows,
               int Hq, int Hkv, int D, int TB, int S, int W, int R, float sgn,
               uint32_t off_cs, uint32_t off_stage, uint32_t stage_bytes, unsigned *status,
               long long wait_limit, const __grid_constant__ RopeFreqs fr) {
  extern __shared__ __align__(128) unsigned char sbuf[];
  __shared__ float2 freq[kRopeMaxHalf];
  __shared__ int32_t cu_s[kCuInShared];

  const int half = D >> 1, NV = half / N, NH = Hq + Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = warp / W, wig = warp - grp * W;
  const int gi = wig * 32 + lane, G = W * 32;
  const bool leader = gi == 0;
  const int HS = G / NV;  // head slots of the group (NV <= G: the launcher checks)
  const int j = gi % NV, slot = gi / NV;
  uint64_t *bars = reinterpret_cast<uint64_t *>(sbuf) + grp * S;               // [R][S]
  float2 *cs = reinterpret_cast<float2 *>(sbuf + off_cs) + (size_t)grp * TB * half;  // [R][TB][half]
  unsigned char *ring = sbuf + off_stage + (size_t)grp * S * stage_bytes;      // [R][S][stage]

  const Idx nblocks = (rows + TB - 1) / TB;
  const size_t qrow_b = (size_t)Hq * D * sizeof(T), krow_b = (size_t)Hkv * D * sizeof(T);
  const bool q_contig = ld_q == (Idx)Hq * D, k_contig = ld_k == (Idx)Hkv * D;

  if (leader)
    for (int i = 0; i < S; ++i) mbar_init(&bars[i], 1);
  for (int i = threadIdx.x; i < half; i += blockDim.x) freq[i] = make_float2(fr.hi[i], fr.lo[i]);
  pdl_wait();
  pdl_trigger();
  if (rope_skipped(fr)) return;  // malformed cu_seqlens: q, k untouched
  const bool cu_staged = B < kCuInShared;
  if (cu_staged)
    for (int i = threadIdx.x; i <= B; i += blockDim.x) cu_s[i] = __ldg(cu + i);
  if (threadIdx.x == 0) fence_mbar_init();
  __syncthreads();
  const int32_t *bounds = cu_staged ? cu_s : cu;

  auto ntok = [&](Idx b) -> int {
    const Idx left = rows - b * TB;
    return (int)(left < (Idx)TB ? left : (Idx)TB);
  };
  // block b <-> stage s: Q rows [TB][Hq*D] then K rows [TB][Hkv*D]
  auto load = [&](int s, Idx b) {
    const Idx t0 = b * TB;
    const int nt = ntok(b);
    unsigned char *st = ring + (size_t)s * stage_bytes;
    mbar_arrive_expect_tx(&bars[s], (uint32_t)(nt * (qrow_b + krow_b)));
    if (qrow_b) {
      if (q_contig)
        bulk_copy_g2s(st, q + t0 * ld_q, (uint32_t)(nt * qrow_b), &bars[s]);
      else
        for (int i = 0; i < nt; ++i)
          bulk_copy_g2s(st + i * qrow_b, q + (t0 + i) * ld_q, (uint32_t)qrow_b, &bars[s]);
    }
    if (krow_b) {
      unsigned char *sk = st + (size_t)TB * qrow_b;
      if (k_contig)
        bulk_copy_g2s(sk, k + t0 * ld_k, (uint32_t)(nt * krow_b), &bars[s]);
      else
        for (int i = 0; i < nt; ++i)
          bulk_copy_g2s(sk + i * krow_b, k + (t0 + i) * ld_k, (uint32_t)krow_b, &bars[s]);
    }
  };
  auto store = [&](int s, Idx b) {
    const Idx t0 = b * TB;
    const int nt = ntok(b);
    const unsigned char *st = ring + (size_t)s * stage_bytes;
    if (qrow_b) {
      if (q_contig)
        bulk_copy_s2g(q + t0 * ld_q, st, (uint32_t)(nt * qrow_b));
      else
        for (int i = 0; i < nt; ++i)
          bulk_copy_s2g(q + (t0 + i) * ld_q, st + i * qrow_b, (uint32_t)qrow_b);
    }
    if (krow_b) {
      const unsigned char *sk = st + (size_t)TB * qrow_b;
      if (k_contig)
        bulk_copy_s2g(k + t0 * ld_k, sk, (uint32_t)(nt * krow_b));
      else
        for (int i = 0; i < nt; ++i)
          bulk_copy_s2g(k + (t0 + i) * ld_k, sk + i * krow_b, (uint32_t)krow_b);
    }
    bulk_commit_group();
  };
  auto group_sync = [&]() {
    if (W > 1)
      group_barrier(grp, G);
    else
      __syncwarp();
  };

  const Idx first = (Idx)blockIdx.x * R + grp;
  const Idx stride = (Idx)gridDim.x * R;
  int issued = 0;
  if (leader)
    for (int i = 0; i < S; ++i) {
      const Idx b = first + (Idx)i * stride;
      if (b >= nblocks) break;
      load(i, b);
      ++issued;
    }

  bool live = true;
  int it = 0;
  for (Idx b = first; b < nblocks; b += stride, ++it) {
    const int s = it % S;
    const Idx t0 = b * TB;
    const int nt = ntok(b);
    if (leader && it >= 1) {
      // the previous block's store has read its stage: refill that stage
      // with the block S iterations after it, before working on this one
      bulk_wait_group_read<0>();
      const Idx nb = b - stride + (Idx)S * stride;
      if (nb < nblocks) {
        load((it - 1) % S, nb);
        ++issued;
      }
    }
    // cos/sin of this block while its rows land
    for (int e = gi; e < nt * half; e += G) {
      const int tt = e / half, i = e - tt * half;
      const int p = position_of<Idx>(t0 + tt, bounds, B);
      const float2 f = freq[i];
      float c, sn;
      rope_cos_sin(p, f.x, f.y, &c, &sn);
      cs[e] = make_float2(c, sgn * sn);
    }
    if (live) live = mbar_wait_bounded(&bars[s], (uint32_t)((it / S) & 1), wait_limit, status);
    group_sync();
    unsigned char *st = ring + (size_t)s * stage_bytes;
    // lane (slot, j): packet j of heads slot, slot + HS, ... of every token;
    // its N cos/sin pairs are read once per token
    if (slot < HS) {
      for (int tt = 0; tt < nt; ++tt) {
        const float2 *c2 = cs + tt * half + j * N;
        float cv[N], sv[N];
#pragma unroll
        for (int e = 0; e < N; ++e) {
          const float2 r = c2[e];
          cv[e] = r.x;
          sv[e] = r.y;
        }
        T *qt = reinterpret_cast<T *>(st) + (size_t)tt * Hq * D + j * N;
        T *kt = reinterpret_cast<T *>(st + (size_t)TB * qrow_b) + ((size_t)tt * Hkv - Hq) * D + j * N;
#pragma unroll 2
        for (int h = slot; h < NH; h += HS) {
          T *v = (h < Hq ? qt : kt) + (size_t)h * D;
          const Packet<T, N> pa = *reinterpret_cast<const Packet<T, N> *>(v);
          const Packet<T, N> pb = *reinterpret_cast<const Packet<T, N> *>(v + half);
          Packet<T, N> oa, ob;
#pragma unroll
          for (int e = 0; e < N; ++e) {
            const float x1 = pa.get(e), x2 = pb.get(e);
            oa.set(e, fmaf(x1, cv[e], -x2 * sv[e]));
            ob.set(e, fmaf(x2, cv[e], x1 * sv[e]));
          }
          *reinterpret_cast<Packet<T, N> *>(v) = oa;
          *reinterpret_cast<Packet<T, N> *>(v + half) = ob;
        }
      }
    }
    fence_proxy_async_smem();  // this thread's stage writes before the bulk store reads them
    group_sync();
    if (leader) store(s, b);
  }
  if (leader) {
    if (!live)  // let loads still in flight land (bounded) before the CTA exits
      for (int i = it; i < issued; ++i)
        mbar_wait_bounded(&bars[i % S], (uint32_t)((i / S) & 1), wait_limit, status);
    bulk_wait_group_all();
  }
}

// One warp per token (half a head fits in the warp's lanes, NV <= 32): lane
// (slot, j) rotates packet j of heads slot, slot + S, ... (S = 32 / NV).
// The warp's head loads go out first; all lanes then find the token's
// position (the same cu_seqlens addresses, so the loads are broadcast) and
// compute its cos/sin table into the warp's own shared-memory slice;
// __syncwarp orders the table, so apart from the one barrier that publishes
// the frequency table at the start, warps never wait on each other.
template <typename T, typename Idx, int N, int HPT>
__global__ void __launch_bounds__(kCtaThreads, 3)
qk_rope_warp(T *q, Idx ld_q, T *k, Idx ld_k, const int32_t *__restrict__ cu, int B, Idx rows,
             int Hq, int NH, int D, float sgn, const __grid_constant__ RopeFreqs fr) {
  extern __shared__ float2 tab[];  // [warps][D/2] (cos, sgn*sin)
  __shared__ float2 freq[kRopeMaxHalf];
  const int half = D >> 1, NV = half / N, S = 32 / NV;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = lane % NV, slot = lane / NV;
  const Idx t = (Idx)blockIdx.x * (blockDim.x >> 5) + warp;
  const bool active = t < rows && slot < S;
  T *const qrow = q + t * ld_q + (Idx)j * N;
  T *const krow = k + t * ld_k + (Idx)j * N - (Idx)Hq * D;
  auto head = [&](int h) -> T * { return (h < Hq ? qrow : krow) + (Idx)h * D; };

  for (int i = threadIdx.x; i < half; i += blockDim.x) freq[i] = make_float2(fr.hi[i], fr.lo[i]);
  pdl_wait();
  pdl_trigger();
  if (rope_skipped(fr)) return;  // malformed cu_seqlens: q, k untouched
  Packet<T, N> a[HPT], b[HPT];
#pragma unroll
  for (int m = 0; m < HPT; ++m) {
    const int h = slot + m * S;
    if (active && h < NH) {
      a[m] = load_packet<T, N>(head(h));
      b[m] = load_packet<T, N>(head(h) + half);
    }
  }
  __syncthreads();  // the frequency table
  if (t >= rows) return;

  const int p = position_of<Idx>(t, cu, B);
  float2 *wt = tab + warp * half;
  for (int i = lane; i < half; i += 32) {
    const float2 f = freq[i];
    float c, sn;
    rope_cos_sin(p, f.x, f.y, &c, &sn);
    wt[i] = make_float2(c, sgn * sn);
  }
  __syncwarp();
  if (slot >= S) return;
  float cv[N], sv[N];
#pragma unroll
  for (int e = 0; e < N; ++e) {
    const float2 v = wt[j * N + e];
    cv[e] = v.x;
    sv[e] = v.y;
  }
  for (int h0 = 0;; h0 += HPT * S) {
#pragma unroll
    for (int m = 0; m < HPT; ++m) {
      const int h = h0 + slot + m * S;
      if (h < NH) {
        Packet<T, N> oa, ob;
#pragma unroll
        for (int e = 0; e < N; ++e) {
          const float x1 = a[m].get(e), x2 = b[m].get(e);
          oa.set(e, fmaf(x1, cv[e], -x2 * sv[e]));
          ob.set(e, fmaf(x2, cv[e], x1 * sv[e]));
        }
        store_packet<T, N>(head(h), oa);
        store_packet<T, N>(head(h) + half, ob);
      }
    }
    const int next = h0 + HPT * S;
    if (next >= NH) break;
#pragma unroll
    for (int m = 0; m < HPT; ++m) {
      const int h = next + slot + m * S;
      if (h < NH) {
        a[m] = load_packet<T, N>(head(h));
        b[m] = load_packet<T, N>(head(h) + half);
      }
    }
  }
}

// Persistent and pipelined, for every batch whose half head splits over a
// power-of-two number of lanes: each warp walks (token, head pass) pairs
// (tokens t, t + P * 8, ...; a pass is S heads, lane (slot, j) rotating
// packet j of both halves of head slot + S p), and each lane copies its
// packets of the next kPipeBufs - 1 passes into a per-warp shared-memory
// ring with cp.async while it rotates the current pass in registers and
// writes it back in place.
constexpr int kPipeSlots = 2, kPipeBufs = 4, kPipeBlocks = 4;
constexpr size_t kPipeStageBytes =
    sizeof(uint4) * (kCtaThreads / 32) * kPipeBufs * kPipeSlots * 32;

template <typename T, typename Idx, int N>
__global__ void __launch_bounds__(kCtaThreads, kPipeBlocks)
qk_rope_pipe(T *q, Idx ld_q, T *k, Idx ld_k, const int32_t *__restrict__ cu, int B, Idx rows,
             int Hq, int NH, int D, float sgn, const __grid_constant__ RopeFreqs fr) {
  static_assert(N % 2 == 0, "pairs of columns per table entry");
  constexpr int kWarps = kCtaThreads / 32;
  // [warps][D/2] (cos, sgn sin), then the staging ring (16-byte aligned:
  // D is a multiple of 8 here)
  extern __shared__ float2 tab[];
  __shared__ float2 freq[kRopeMaxHalf];
  __shared__ int32_t cu_s[kCuInShared];
  const int half = D >> 1, NV = half / N, S = 32 / NV;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = lane % NV, slot = lane / NV;
  // the token's table: (cos, sgn sin) of columns j N + e and j N + e + 1 (e
  // even) in one 16-byte entry at (e / 2) NV + j, so the NV lanes of a head
  // read consecutive entries
  float4 *wt = reinterpret_cast<float4 *>(tab + warp * half);
  uint4 *stg = reinterpret_cast<uint4 *>(tab + kWarps * half) + warp * (kPipeBufs * kPipeSlots * 32);
  auto head = [&](Idx tt, int h) -> T * {
    return (h < Hq ? q + tt * ld_q + (Idx)h * D : k + tt * ld_k + (Idx)(h - Hq) * D) + j * N;
  };

  for (int i = threadIdx.x; i < half; i += blockDim.x) freq[i] = make_float2(fr.hi[i], fr.lo[i]);
  pdl_wait();
  pdl_trigger();
  if (rope_skipped(fr)) return;  // malformed cu_seqlens: q, k untouched
  // the sequence boundaries in shared memory when they fit: every token's
  // position is a binary search over them
  const bool cu_staged = B < kCuInShared;
  if (cu_staged)
    for (int i = threadIdx.x; i <= B; i += blockDim.x) cu_s[i] = __ldg(cu + i);
  __syncthreads();  // the frequency table and the boundaries
  const int32_t *bounds = cu_staged ? cu_s : cu;

  const Idx step = (Idx)gridDim.x * kWarps;
  const int passes = (NH + S - 1) / S;  // head passes per token, the same on every lane
  auto stage = [&](Idx tt, int p, int b) {
    const int h = slot + p * S;
    if (tt < rows && h < NH) {
      const T *v = head(tt, h);
      uint4 *d = stg + b * kPipeSlots * 32 + lane;
      cp_async16(d, v);
      cp_async16(d + 32, v + half);
    }
    cp_async_commit();  // one group per pass on every lane, empty or not
  };
  auto advance = [&](Idx &tt, int &pp) {
    if (++pp == passes) {
      pp = 0;
      tt += step;
    }
  };
  const float4 *cs_j = wt + j;
  Idx t = (Idx)blockIdx.x * kWarps + warp, t2 = t;
  int p = 0, p2 = 0, b = 0;
  stage(t2, p2, 0);
  for (int i = 1; i < kPipeBufs - 1; ++i) {
    advance(t2, p2);
    stage(t2, p2, i);
  }
  while (t < rows) {  // warp-uniform
    advance(t2, p2);
    stage(t2, p2, b == 0 ? kPipeBufs - 1 : b - 1);  // the next passes' loads fly meanwhile
    if (p == 0) {
      __syncwarp();  // the previous token's table has been read
      const int pos = position_of<Idx>(t, bounds, B);
      float2 *w2 = reinterpret_cast<float2 *>(wt);
      for (int i = lane; i < half; i += 32) {
        const float2 f = freq[i];
        float c, sn;
        rope_cos_sin(pos, f.x, f.y, &c, &sn);
        const int e = i % N;
        w2[2 * ((e >> 1) * NV + i / N) + (e & 1)] = make_float2(c, sgn * sn);
      }
      __syncwarp();
    }
    cp_async_wait<kPipeBufs - 1>();  // this lane's copies for (t, p) have landed
    const int h = slot + p * S;
    if (h < NH) {
      const uint4 *d = stg + b * kPipeSlots * 32 + lane;
      Packet<T, N> x1, x2, o1, o2;
      *reinterpret_cast<uint4 *>(&x1) = d[0];
      *reinterpret_cast<uint4 *>(&x2) = d[32];
#pragma unroll
      for (int e = 0; e < N; e += 2) {
        const float4 c = cs_j[(e >> 1) * NV];  // (cos, sin) of columns e and e + 1
        const float a0 = x1.get(e), b0 = x2.get(e), a1 = x1.get(e + 1), b1 = x2.get(e + 1);
        o1.set2(e, fmaf(a0, c.x, -b0 * c.y), fmaf(a1, c.z, -b1 * c.w));
        o2.set2(e, fmaf(b0, c.x, a0 * c.y), fmaf(b1, c.z, a1 * c.w));
      }
      T *v = head(t, h);
      store_packet<T, N>(v, o1);
      store_packet<T, N>(v + half, o2);
    }
    advance(t, p);
    b = b + 1 == kPipeBufs ? 0 : b + 1;
  }
  cp_async_wait<0>();
}

// bf16 heads whose half is 8 NV values, NV a power of two dividing 32 (D =
// 16 .. 512): the lean form of qk_rope_pipe, with the same per-warp
// cp.async ring of head passes, the same (cos, sin) table per token and the
// same token order (warp w of G takes tokens w, w + G, ...: the grid sweeps
// the batch one contiguous window at a time, which measured 1-2.5% faster on
// every workload than giving each warp a contiguous run of tokens).  The
// rotation runs on fp32 pairs, each half rounded exactly like the scalar
// fma(a, c, -(b s)) of qk_rope_pipe, so the two kernels agree bit for bit;
// row addresses advance by G rows per token.  The table entry of lane (slot, j)
// for columns 8 j + 2 m, 8 j + 2 m + 1 holds (cos, cos, sgn sin, sgn sin)
// at m NV + j, so the NV lanes of a head read consecutive 16-byte entries.
template <typename Idx, int NV>
__global__ void __launch_bounds__(kCtaThreads, kPipeBlocks)
qk_rope_lean(bf16 *q, Idx ld_q, bf16 *k, Idx ld_k, const int32_t *__restrict__ cu, int B,
             Idx rows, int Hq, int NH, float sgn, const __grid_constant__ RopeFreqs fr) {
  constexpr int N = 8, half = N * NV, D = 2 * half, S = 32 / NV;
  constexpr int kWarps = kCtaThreads / 32;
  __shared__ float4 tab_all[kWarps][4 * NV];
  __shared__ float2 freq[half];
  __shared__ int32_t cu_s[kCuInShared];
  extern __shared__ uint4 stg_all[];  // [warps][kPipeBufs][2][32]
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int j = lane % NV, slot = lane / NV;
  float4 *const tab = tab_all[warp];
  uint4 *const stg = stg_all + warp * (kPipeBufs * 2 * 32) + lane;

  for (int i = threadIdx.x; i < half; i += blockDim.x) freq[i] = make_float2(fr.hi[i], fr.lo[i]);
  pdl_wait();
  pdl_trigger();
  if (rope_skipped(fr)) return;  // malformed cu_seqlens: q, k untouched
  const bool cu_staged = B < kCuInShared;
  if (cu_staged)
    for (int i = threadIdx.x; i <= B; i += blockDim.x) cu_s[i] = __ldg(cu + i);
  __syncthreads();  // the frequency table and the boundaries; no block barrier follows
  const int32_t *bounds = cu_staged ? cu_s : cu;

  // this warp's tokens: t, t + G, ... below rows
  const Idx G = (Idx)gridDim.x * kWarps;
  Idx t = (Idx)blockIdx.x * kWarps + warp;
  if (t >= rows) return;
  const int passes = (NH + S - 1) / S;  // head passes per token, the same on every lane

  // the stager runs kPipeBufs - 1 passes ahead with its own row pointers
  Idx t2 = t;
  int p2 = 0, b2 = 0;
  const bf16 *q2 = q + t2 * ld_q + j * N, *k2 = k + t2 * ld_k + j * N - (Idx)Hq * D;
  auto stage = [&]() {
    const int h = slot + p2 * S;
    if (t2 < rows && h < NH) {
      const bf16 *v = (h < Hq ? q2 : k2) + (Idx)h * D;
      uint4 *d = stg + b2 * 64;
      cp_async16(d, v);
      cp_async16(d + 32, v + half);
    }
    cp_async_commit();  // one group per pass on every lane, empty or not
    if (++p2 == passes) {
      p2 = 0;
      t2 += G;
      q2 += G * ld_q;
      k2 += G * ld_k;
    }
    b2 = b2 + 1 == kPipeBufs ? 0 : b2 + 1;
  };
#pragma unroll
  for (int i = 0; i < kPipeBufs - 1; ++i) stage();

  bf16 *qr = q + t * ld_q + j * N, *kr = k + t * ld_k + j * N - (Idx)Hq * D;
  int b = 0;
  for (; t < rows; t += G, qr += G * ld_q, kr += G * ld_k) {  // warp-uniform
    // the token's table, built by the warp; every lane then keeps the four
    // entries of its columns in registers for all of the token's head passes
    const int pos = position_of<Idx>(t, bounds, B);
    __syncwarp();  // the previous token's table has been read
    float *tf = reinterpret_cast<float *>(tab);
#pragma unroll
    for (int i = lane; i < half; i += 32) {
      const float2 f = freq[i];
      float c, sn;
      rope_cos_sin(pos, f.x, f.y, &c, &sn);
      float *ent = tf + 4 * (((i % N) >> 1) * NV + i / N) + (i & 1);
      ent[0] = c;
      ent[2] = sgn * sn;
    }
    __syncwarp();
    float2 c2[4], s2[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const float4 cs = tab[m * NV + j];
      c2[m] = make_float2(cs.x, cs.y);
      s2[m] = make_float2(cs.z, cs.w);
    }
    for (int p = 0; p < passes; ++p) {
      stage();  // the next passes' loads fly meanwhile
      cp_async_wait<kPipeBufs - 1>();  // this lane's copies for (t, p) have landed
      const int h = slot + p * S;
      if (h < NH) {
        const uint4 *d = stg + b * 64;
        const uint4 xa = d[0], xb = d[32];
        const uint32_t wa[4] = {xa.x, xa.y, xa.z, xa.w}, wb[4] = {xb.x, xb.y, xb.z, xb.w};
        uint32_t o1[4], o2[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const float2 a = bf2_unpack(wa[m]), bb = bf2_unpack(wb[m]);
          const float2 bs = __fmul2_rn(bb, s2[m]), as = __fmul2_rn(a, s2[m]);
          o1[m] = bf2_pack(__ffma2_rn(a, c2[m], make_float2(-bs.x, -bs.y)));
          o2[m] = bf2_pack(__ffma2_rn(bb, c2[m], as));
        }
        bf16 *v = (h < Hq ? qr : kr) + (Idx)h * D;
        *reinterpret_cast<uint4 *>(v) = make_uint4(o1[0], o1[1], o1[2], o1[3]);
        *reinterpret_cast<uint4 *>(v + half) = make_uint4(o2[0], o2[1], o2[2], o2[3]);
      }
      b = b + 1 == kPipeBufs ? 0 : b + 1;
    }
  }
  cp_async_wait<0>();
}

template <typename Idx, int NV>
cudaError_t rope_lean_launch(const RopeArgs &a, const RopeFreqs &fr, const DeviceInfo &dev,
                             cudaStream_t s) {
  constexpr int kWarps = kCtaThreads / 32;
  const size_t smem = kPipeStageBytes;
  auto kern = qk_rope_lean<Idx, NV>;
  const int occ = blocks_per_sm((const void *)kern, kCtaThreads, smem, dev, kPipeBlocks);
  int64_t P = ceil_div(a.T, (int64_t)kWarps);
  if (P > (int64_t)dev.sms * occ) P = (int64_t)dev.sms * occ;
  cudaError_t e = launch_pdl(kern, dim3((unsigned)P), dim3(kCtaThreads), smem, s, (bf16 *)a.q,
                             (Idx)a.ld_q, (bf16 *)a.k, (Idx)a.ld_k, a.cu, a.B, (Idx)a.T, a.Hq,
                             a.Hq + a.Hkv, a.backward ? -1.0f : 1.0f, fr);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T, typename Idx, int N>
cudaError_t rope_pipe_launch(const RopeArgs &a, const RopeFreqs &fr, const DeviceInfo &dev,
                             cudaStream_t s) {
  constexpr int kWarps = kCtaThreads / 32;
  const int NH = a.Hq + a.Hkv;
  const size_t smem = sizeof(float2) * (size_t)kWarps * (a.D / 2) + kPipeStageBytes;
  auto kern = qk_rope_pipe<T, Idx, N>;
  const int occ = blocks_per_sm((const void *)kern, kCtaThreads, smem, dev, kPipeBlocks);
  int64_t P = ceil_div(a.T, (int64_t)kWarps);
  if (P > (int64_t)dev.sms * occ) P = (int64_t)dev.sms * occ;
  cudaError_t e = launch_pdl(kern, dim3((unsigned)P), dim3(kCtaThreads), smem, s, (T *)a.q,
                             (Idx)a.ld_q, (T *)a.k, (Idx)a.ld_k, a.cu, a.B, (Idx)a.T, a.Hq, NH,
                             a.D, a.backward ? -1.0f : 1.0f, fr);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T, typename Idx, int N>
cudaError_t rope_warp_launch(const RopeArgs &a, const RopeFreqs &fr, cudaStream_t s) {
  const int NH = a.Hq + a.Hkv, half = a.D / 2, NV = half / N, S = 32 / NV;
  const int per_lane = (NH + S - 1) / S;
  constexpr int kWarps = kCtaThreads / 32;
  const dim3 grid((unsigned)ceil_div(a.T, (int64_t)kWarps));
  const size_t smem = sizeof(float2) * (size_t)kWarps * half;
  const float sgn = a.backward ? -1.0f : 1.0f;
#define FTK_ROPE_WARP(H)                                                                     \
  {                                                                                          \
    cudaError_t le_ = launch_pdl(qk_rope_warp<T, Idx, N, H>, grid, dim3(kCtaThreads), smem, s, \
                                 (T *)a.q, (Idx)a.ld_q, (T *)a.k, (Idx)a.ld_k, a.cu, a.B,     \
                                 (Idx)a.T, a.Hq, NH, a.D, sgn, fr);                          \
    if (le_ != cudaSuccess) return le_;                                                      \
    return cudaGetLastError();                                                               \
  }
  if (per_lane <= 1) FTK_ROPE_WARP(1)
  if (per_lane <= 2 || N >= 8) FTK_ROPE_WARP(2)
  FTK_ROPE_WARP(4)
#undef FTK_ROPE_WARP
}

template <typename T, typename Idx, int N, int HPT>
cudaError_t rope_launch(const RopeArgs &a, const RopeFreqs &fr, cudaStream_t s) {
  const int NH = a.Hq + a.Hkv;
  const int half = a.D / 2;
  const int NV = half / N;
  int S = (NH + HPT - 1) / HPT;
  if (S * NV > kCtaThreads) S = kCtaThreads / NV > 0 ? kCtaThreads / NV : 1;
  const int TPT = NV * S;
  int TOK = kCtaThreads / TPT;
  if (TOK < 1) TOK = 1;
  const int threads = TOK * TPT;
  const size_t smem = sizeof(float2) * (size_t)TOK * half;
  const int64_t grid = ceil_div(a.T, (int64_t)TOK);
  {
    cudaError_t le_ = launch_pdl(qk_rope_kernel<T, Idx, N, HPT>, dim3((unsigned)grid), dim3(threads), smem, s, 
      (T *)a.q, (Idx)a.ld_q, (T *)a.k, (Idx)a.ld_k, a.cu, a.B, (Idx)a.T, a.Hq, NH, a.D, S, NV,
      TOK, a.backward ? -1.0f : 1.0f, fr);
    if (le_ != cudaSuccess) return le_;
  }
  return cudaGetLastError();
}

// Heads per thread: as many packets in flight as fit in the 80 registers
// that let three CTAs share an SM (bf16 16-byte packets: 2 heads; fp32: 4;
// element-wise: 8).
template <typename T, typename Idx, int N>
cudaError_t rope_heads(const RopeArgs &a, const RopeFreqs &fr, cudaStream_t s) {
  constexpr int kMaxHpt = N >= 8 ? 2 : (N >= 4 ? 4 : 8);
  const int NH = a.Hq + a.Hkv;
  if (NH <= 1) return rope_launch<T, Idx, N, 1>(a, fr, s);
  if constexpr (kMaxHpt == 2) {
    return rope_launch<T, Idx, N, 2>(a, fr, s);
  } else {
    if (NH <= 2) return rope_launch<T, Idx, N, 2>(a, fr, s);
    if constexpr (kMaxHpt == 4) {
      return rope_launch<T, Idx, N, 4>(a, fr, s);
    } else {
      if (NH <= 4) return rope_launch<T, Idx, N, 4>(a, fr, s);
      return rope_launch<T, Idx, N, 8>(a, fr, s);
    }
  }
}

template <typename T, typename Idx, int N>
cudaError_t rope_staged_launch(const RopeArgs &a, const RopeFreqs &fr, const DeviceInfo &dev,
                               cudaStream_t s, bool *launched) {
  *launched = false;
  const int NH = a.Hq + a.Hkv, half = a.D / 2, NV = half / N;
  const size_t tok_bytes = (size_t)NH * a.D * sizeof(T);
  // ~8 KiB of whole tokens per stage; W warps per group so that each lane
  // rotates ~8 packet pairs per block; R groups per CTA (<= 256 threads).
  int TB = (int)(8192 / tok_bytes);
  TB = TB < 1 ? 1 : (TB > 16 ? 16 : TB);
  int W = (int)ceil_div((int64_t)TB * NH * NV, (int64_t)256);
  W = W < 1 ? 1 : (W > 8 ? 8 : W);
  const int R = 8 / W > 0 ? 8 / W : 1;
  const size_t stage_bytes = (size_t)TB * tok_bytes;
  // ~150 KiB of stages per SM over two CTAs, 2..6 stages per group
  int S = (int)(76800 / ((size_t)R * stage_bytes));
  S = S < 2 ? 2 : (S > 6 ? 6 : S);
  const size_t static_smem = sizeof(float2) * kRopeMaxHalf + sizeof(int32_t) * kCuInShared;
  size_t off_cs = 0, off_stage = 0, smem = 0;
  for (; S >= 2; --S) {
    off_cs = ((size_t)R * S * 8 + 15) / 16 * 16;
    off_stage = (off_cs + (size_t)R * TB * half * sizeof(float2) + 127) / 128 * 128;
    smem = off_stage + (size_t)R * S * stage_bytes;
    if (smem + static_smem <= (size_t)dev.max_smem_optin) break;
  }
  if (S < 2 || stage_bytes >= (1u << 20) || NV > 32 * W) return cudaSuccess;  // register kernel
  auto kern = qk_rope_staged<T, Idx, N>;
  const int threads = 32 * W * R;
  const int occ = blocks_per_sm((const void *)kern, threads, smem, dev, 8);
  const int64_t nblocks = ceil_div(a.T, (int64_t)TB);
  int64_t P = (int64_t)dev.sms * occ;
  // the pipeline pays off once every group streams several blocks; smaller
  // batches go to the one-pass register kernel
  if (nblocks < (int64_t)6 * P * R) return cudaSuccess;
  unsigned *status = nullptr;
  cudaError_t e = device_status_ptr(dev, &status);
  if (e != cudaSuccess) return e;
  {
    cudaError_t le_ = launch_pdl(kern, dim3((unsigned)P), dim3(threads), smem, s, 
      (T *)a.q, (Idx)a.ld_q, (T *)a.k, (Idx)a.ld_k, a.cu, a.B, (Idx)a.T, a.Hq, a.Hkv, a.D, TB, S,
      W, R, a.backward ? -1.0f : 1.0f, (uint32_t)off_cs, (uint32_t)off_stage,
      (uint32_t)stage_bytes, status, kWaitLimitCycles, fr);
    if (le_ != cudaSuccess) return le_;
  }
  *launched = true;
  return cudaGetLastError();
}

template <typename T, typename Idx>
cudaError_t rope_typed(bool vec, const RopeArgs &a, const RopeFreqs &fr, const DeviceInfo &dev,
                       cudaStream_t s) {
  constexpr int NV = VecWidth<T>::value;
  if (vec) {
    const int nv = a.D / 2 / NV;
    if constexpr (sizeof(T) == 2) {
      switch (nv) {
        case 1: return rope_lean_launch<Idx, 1>(a, fr, dev, s);
        case 2: return rope_lean_launch<Idx, 2>(a, fr, dev, s);
        case 4: return rope_lean_launch<Idx, 4>(a, fr, dev, s);
        case 8: return rope_lean_launch<Idx, 8>(a, fr, dev, s);
        case 16: return rope_lean_launch<Idx, 16>(a, fr, dev, s);
        case 32: return rope_lean_launch<Idx, 32>(a, fr, dev, s);
        default: break;
      }
    }
    if (nv >= 1 && nv <= 32 && (nv & (nv - 1)) == 0) return rope_pipe_launch<T, Idx, NV>(a, fr, dev, s);
    bool launched = false;
    cudaError_t e = rope_staged_launch<T, Idx, NV>(a, fr, dev, s, &launched);
    if (e != cudaSuccess || launched) return e;
    if (a.D / 2 / NV <= 32) return rope_warp_launch<T, Idx, NV>(a, fr, s);
    return rope_heads<T, Idx, NV>(a, fr, s);
  }
  if (a.D / 2 <= 32) return rope_warp_launch<T, Idx, 1>(a, fr, s);
  return rope_heads<T, Idx, 1>(a, fr, s);
}

}  // namespace

cudaError_t launch_qk_rope(DType dt, bool vec, bool wide, const RopeArgs &a,
                           const DeviceInfo &dev, cudaStream_t s) {
  const RopeFreqs fr = make_rope_freqs(a.D, a.theta, a.inv_freq, a.skip);
  if (dt == DType::F32)
    return wide ? rope_typed<float, int64_t>(vec, a, fr, dev, s)
                : rope_typed<float, int32_t>(vec, a, fr, dev, s);
  return wide ? rope_typed<bf16, int64_t>(vec, a, fr, dev, s)
              : rope_typed<bf16, int32_t>(vec, a, fr, dev, s);
}

}  // namespace ftk
