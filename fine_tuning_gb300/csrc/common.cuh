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
  // elements i and i+1 (i even) in one conversion
  __device__ __forceinline__ void set2(int i, float a, float b) {
    if constexpr (sizeof(T) == 2 && N % 2 == 0) {
      *reinterpret_cast<__nv_bfloat162 *>(&v[i]) = __floats2bfloat162_rn(a, b);
    } else {
      set(i, a);
      if (i + 1 < N) set(i + 1, b);
    }
  }
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

// ---------------------------------------------------------------------------
// Bulk-copy (TMA) pipeline pieces: mbarriers in shared memory, 1-D bulk
// copies global -> shared completing on an mbarrier, bounded waits.

// Bits of the library's device status word.
constexpr unsigned kStatusWaitTimeout = 1u;  // a pipeline wait gave up

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
}

// Makes initialised mbarriers visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's earlier shared-memory accesses before later
// bulk-copy writes into the same buffer.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// bytes: multiple of 16; src and dst 16-byte aligned.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Per-thread asynchronous copies into shared memory (cp.async; 16 bytes
// bypassing L1, or 4 bytes), committed and waited for in groups.
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int K> __device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(K) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for phase `parity` of `bar` for at most `limit` SM clock cycles.
// On expiry it records kStatusWaitTimeout in *status (device memory) and
// returns false; the caller then stops waiting and finishes without hanging.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  long long limit, unsigned *status) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - t0 > limit) {
      atomicOr(status, kStatusWaitTimeout);
      return false;
    }
  }
  return true;
}

// Bulk copy shared -> global, tracked by this thread's bulk async-groups.
__device__ __forceinline__ void bulk_copy_s2g(void *dst, const void *src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
               "r"(smem_addr(src)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until at most N of this thread's bulk groups still read shared memory.
template <int N> __device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Waits until all of this thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_group_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Programmatic dependent launch.  Every ftk kernel calls pdl_wait() before
// its first global memory access: when it was launched as a programmatic
// dependent of the previous kernel in the stream, this waits until that
// kernel has completed and its writes are visible (otherwise it returns at
// once).  pdl_trigger() then lets the next kernel in the stream be launched
// as soon as every CTA of this one has started, so its launch and prologue
// overlap this kernel's tail; it still waits for this kernel's completion
// before touching memory.
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" :::);
}

// Named barrier over `threads` threads (a multiple of 32) with id 1..15.
__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Named barrier 1 + g (g < 4) of a CTA's row group g, over `threads` threads.
// Each case names its barrier by a constant, so a kernel that uses only this
// form reserves barriers 0-4; a barrier id computed at run time makes the
// compiler reserve all 16, which caps an SM at 4 resident CTAs of the kernel.
// Groups that synchronise have W >= 2 warps, hence at most 8 / W = 4 per CTA.
__device__ __forceinline__ void group_barrier(int g, int threads) {
  switch (g) {
    case 0: asm volatile("bar.sync 1, %0;" ::"r"(threads) : "memory"); break;
    case 1: asm volatile("bar.sync 2, %0;" ::"r"(threads) : "memory"); break;
    case 2: asm volatile("bar.sync 3, %0;" ::"r"(threads) : "memory"); break;
    default: asm volatile("bar.sync 4, %0;" ::"r"(threads) : "memory"); break;
  }
}

}  // namespace ftk
