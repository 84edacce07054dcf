// Device-side helpers shared by the ftk kernels: 16-byte packets of bf16 or
// fp32 values, fp32 conversion, cache-hinted global loads/stores and warp
// reductions.  Everything here is plain CUDA C++ for sm_103a.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ftk {

using bf16 = __nv_bfloat16;

// Elements of T in one 16-byte vector.
template <typename T> struct VecWidth;
template <> struct VecWidth<float> { static constexpr int value = 4; };
template <> struct VecWidth<bf16> { static constexpr int value = 8; };

__device__ __forceinline__ float to_float(float v) { return v; }
__device__ __forceinline__ float to_float(bf16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_float(float v);
template <> __device__ __forceinline__ float from_float<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_float<bf16>(float v) {
  return __float2bfloat16_rn(v);
}

// N consecutive elements of T moved as one access (16 bytes for the
// vectorised kernels, one element for the element-wise ones).
template <typename T, int N> struct alignas(sizeof(T) * N) Packet {
  T v[N];

  __device__ __forceinline__ float get(int i) const { return to_float(v[i]); }
  __device__ __forceinline__ void set(int i, float f) { v[i] = from_float<T>(f); }
};

// 16-byte packets go through explicit vector accesses so that the compiler
// always emits one 128-bit instruction; smaller packets are plain copies.
template <typename T, int N>
__device__ __forceinline__ Packet<T, N> load_packet(const T *p) {
  Packet<T, N> r;
  if constexpr (sizeof(T) * N == 16) {
    *reinterpret_cast<uint4 *>(&r) = *reinterpret_cast<const uint4 *>(p);
  } else {
    r = *reinterpret_cast<const Packet<T, N> *>(p);
  }
  return r;
}

// Streaming load: data read exactly once, not worth keeping in L1.
template <typename T, int N>
__device__ __forceinline__ Packet<T, N> load_packet_stream(const T *p) {
  Packet<T, N> r;
  if constexpr (sizeof(T) * N == 16) {
    uint4 u;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(u.x), "=r"(u.y), "=r"(u.z), "=r"(u.w)
                 : "l"(p));
    *reinterpret_cast<uint4 *>(&r) = u;
  } else {
    r = *reinterpret_cast<const Packet<T, N> *>(p);
  }
  return r;
}

template <typename T, int N>
__device__ __forceinline__ void store_packet(T *p, const Packet<T, N> &r) {
  if constexpr (sizeof(T) * N == 16) {
    *reinterpret_cast<uint4 *>(p) = *reinterpret_cast<const uint4 *>(&r);
  } else {
    *reinterpret_cast<Packet<T, N> *>(p) = r;
  }
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float2 warp_sum2(float2 v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
    v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
  }
  return v;
}

template <typename T, typename U> __host__ __device__ constexpr T ceil_div(T a, U b) {
  return (a + b - 1) / b;
}

}  // namespace ftk
