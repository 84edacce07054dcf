// fp32 pair arithmetic for the lean bf16 kernels (rmsnorm_{fwd,bwd}_lean,
// qk_rope_lean, qk_norm_rope_{fwd,bwd}_lean) and the row sums and output
// step of the multi-warp RMSNorm kernels: bf16 <-> fp32 pairs, and the row
// sum of squares in the order the forward and backward kernels share.
//
// Those kernels do their fp32 arithmetic on pairs (Blackwell's two-wide fp32
// multiply and fused multiply-add; each half is rounded exactly like the
// scalar instruction), unpack each bf16 once and pack two per conversion,
// which cuts the instruction count per row or token by a third or more
// against scalar code.
#pragma once

#include "common.cuh"

namespace ftk {

namespace {

// The two bf16 of a 32-bit word as an fp32 pair (exact: bf16 is the top half
// of an fp32).
__device__ __forceinline__ float2 bf2_unpack(uint32_t u) {
  return make_float2(__uint_as_float(u << 16), __uint_as_float(u & 0xffff0000u));
}

// An fp32 pair rounded to nearest even, two bf16 in one word.
__device__ __forceinline__ uint32_t bf2_pack(float2 v) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(v.x, v.y);
  return *reinterpret_cast<const uint32_t *>(&h);
}

__device__ __forceinline__ void unpack8(const uint4 &u, float2 (&f)[4]) {
  f[0] = bf2_unpack(u.x);
  f[1] = bf2_unpack(u.y);
  f[2] = bf2_unpack(u.z);
  f[3] = bf2_unpack(u.w);
}

__device__ __forceinline__ uint4 pack8(const float2 (&f)[4]) {
  return make_uint4(bf2_pack(f[0]), bf2_pack(f[1]), bf2_pack(f[2]), bf2_pack(f[3]));
}

// The lean row order of sum_j x_j^2: each lane runs one pair chain over its
// packets in column order (even columns in .x, odd in .y, each step a fused
// multiply-add), adds the pair's halves, and the warp adds the lanes with
// the xor butterfly.  The forward and the backward's recomputation both go
// through these two functions, so a recomputed r equals the saved one bit for
// bit.
__device__ __forceinline__ void lean_sumsq_step(float2 &acc, float2 x) {
  acc = __ffma2_rn(x, x, acc);
}
__device__ __forceinline__ float lean_lane_total(float2 acc) { return acc.x + acc.y; }

// The multi-warp RMSNorm kernels (rmsnorm_{fwd,bwd}_{pipe,rows,staged}) sum
// a lane's squares through these two: for 8-wide bf16 packets the lean pair
// chain above (even columns in .x, odd in .y, halves added at the end), for
// any other packet one scalar chain in .x.  Every forward and backward of a
// row plan goes through them, so a recomputed r equals the saved one and
// the residual-add forward equals the plain norm of its h, bit for bit.
template <typename T, int N>
__device__ __forceinline__ void sumsq_packet(float2 &acc, const Packet<T, N> &v) {
  if constexpr (sizeof(T) == 2 && N == 8) {
    float2 f[4];
    unpack8(*reinterpret_cast<const uint4 *>(&v), f);
#pragma unroll
    for (int p = 0; p < 4; ++p) lean_sumsq_step(acc, f[p]);
  } else {
#pragma unroll
    for (int e = 0; e < N; ++e) {
      const float f = v.get(e);
      acc.x = fmaf(f, f, acc.x);
    }
  }
}
template <typename T, int N> __device__ __forceinline__ float sumsq_total(float2 acc) {
  if constexpr (sizeof(T) == 2 && N == 8) {
    return lean_lane_total(acc);
  } else {
    return acc.x;
  }
}

// The RMSNorm forward's output packet (x r) w for the multi-warp kernels
// (rmsnorm_fwd_{pipe,rows,staged}): on fp32 pairs when PAIR is set and the
// packet is 8 bf16, else per element.  Both forms round every product like
// the scalar expression, so they give the same bits.
template <typename T, int N, bool PAIR>
__device__ __forceinline__ Packet<T, N> scale_packet(const Packet<T, N> x, float r,
                                                     const Packet<T, N> w) {
  Packet<T, N> o;
  if constexpr (PAIR && sizeof(T) == 2 && N == 8) {
    float2 xf[4], wf[4];
    unpack8(*reinterpret_cast<const uint4 *>(&x), xf);
    unpack8(*reinterpret_cast<const uint4 *>(&w), wf);
    const float2 r2 = make_float2(r, r);
#pragma unroll
    for (int p = 0; p < 4; ++p) xf[p] = __fmul2_rn(__fmul2_rn(xf[p], r2), wf[p]);
    *reinterpret_cast<uint4 *>(&o) = pack8(xf);
  } else {
#pragma unroll
    for (int e = 0; e < N; ++e) o.set(e, (x.get(e) * r) * w.get(e));
  }
  return o;
}

}  // namespace

}  // namespace ftk
