// Pieces shared by the RoPE kernels (qk_rope.cu, qk_norm_rope.cu): the
// frequency table, the extended-precision angle, and the position lookup in
// cu_seqlens.
//
// The angle is formed in turns, phi / 2pi = p * f_i with f_i split on the
// host into two floats (hi + lo, ~48 significant bits); p is split into a
// multiple of 4096 and a remainder so each partial product is exact or
// nearly so (Dekker's two-product via fma), the integer turns are dropped
// from every term, and sincospif() of the remaining fraction gives cos and
// sin.
#pragma once

#include <cmath>

#include "common.cuh"
#include "launch.h"

namespace ftk {

namespace {

struct RopeFreqs {
  float hi[kRopeMaxHalf];
  float lo[kRopeMaxHalf];
  // nullable: a word written by the sequence-boundary check; when it is
  // non-zero the kernel returns before touching q or k
  const uint32_t *skip;
};

// True when the boundary check that ran before this kernel found the batch's
// cu_seqlens malformed.  Read after the grid-dependency wait (the check is
// the preceding kernel) and past L1; uniform across a CTA, so an early
// return skips no barrier another thread waits on.
__device__ __forceinline__ bool rope_skipped(const RopeFreqs &fr) {
  return fr.skip != nullptr && __ldcg(fr.skip) != 0u;
}

constexpr int kCuInShared = 2048;  // cu_seqlens entries a CTA stages in shared memory

__device__ __forceinline__ float frac_turns(float a) { return a - rintf(a); }

// cos and sin of 2*pi*p*(fhi + flo).
__device__ __forceinline__ void rope_cos_sin(int p, float fhi, float flo, float *c, float *s) {
  const float ph = (float)(p & ~4095);  // exact: at most 19 significant bits
  const float pl = (float)(p & 4095);   // exact
  const float a1 = __fmul_rn(ph, fhi);
  const float e1 = fmaf(ph, fhi, -a1);  // ph*fhi = a1 + e1 exactly
  const float a2 = __fmul_rn(pl, fhi);
  const float e2 = fmaf(pl, fhi, -a2);  // pl*fhi = a2 + e2 exactly
  const float a3 = __fmul_rn(ph, flo);
  const float a4 = __fmul_rn(pl, flo);
  float r = frac_turns(a1) + frac_turns(a2);
  r += frac_turns(a3) + frac_turns(e1);
  r += e2 + a4;
  r = frac_turns(r);
  sincospif(2.0f * r, s, c);
}

// Sequence of token t: largest b < B with cu[b] <= t (zero-length sequences
// are skipped because their boundary repeats).  Clamped to [0, B-1], so a
// malformed cu can only give wrong positions, never a wrong address.
// `cu` is a generic pointer: the CTA's shared-memory copy when it fits,
// else the device array itself.
template <typename Idx>
__device__ __forceinline__ int sequence_of(Idx t, const int32_t *cu, int B) {
  int lo = 1, hi = B;  // first i in [1, B] with cu[i] > t
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    if ((Idx)cu[mid] <= t)
      lo = mid + 1;
    else
      hi = mid - 1;
  }
  const int b = lo - 1;
  return b < 0 ? 0 : (b > B - 1 ? B - 1 : b);
}

template <typename Idx>
__device__ __forceinline__ int position_of(Idx t, const int32_t *cu, int B) {
  const int b = sequence_of<Idx>(t, cu, B);
  return (int)(t - (Idx)cu[b]);
}

// f_i = inv_freq_i / (2 pi) in double, split into two floats; inv_freq_i is
// theta^(-2i/D), or the caller's (scaled) table when inv_freq is set.
inline RopeFreqs make_rope_freqs(int D, double theta, const double *inv_freq,
                                 const uint32_t *skip = nullptr) {
  RopeFreqs fr;
  fr.skip = skip;
  const int half = D / 2;
  for (int i = 0; i < kRopeMaxHalf; ++i) {
    if (i < half) {
      const double inv = inv_freq ? inv_freq[i] : std::pow(theta, -2.0 * (double)i / (double)D);
      const double f = inv / 6.283185307179586476925;
      const float hi = (float)f;
      fr.hi[i] = hi;
      fr.lo[i] = (float)(f - (double)hi);
    } else {
      fr.hi[i] = fr.lo[i] = 0.f;
    }
  }
  return fr;
}

}  // namespace

}  // namespace ftk
