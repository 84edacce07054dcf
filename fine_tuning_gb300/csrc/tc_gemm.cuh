// A persistent bf16 GEMM on the 5th-generation tensor cores (tcgen05) with a
// pluggable epilogue: C[m, n] = sum_k A[m, k] B[n, k], A [M, K] and B [N, K]
// both row-major (K contiguous), fp32 accumulation in tensor memory.  The
// epilogue sees each output row in 32-column slices and never writes the
// accumulator tile as such unless it wants to; the cross-entropy kernels
// (cce.cu) use it to fold a softmax into the contraction.
//
// One CTA per SM, 10 warps:
//   warp 0      one elected lane issues TMA loads (cp.async.bulk.tensor, 128-
//               byte swizzle) of the A tile [128 x 64] and the B tile
//               [BN x 64] of every k-step into a ring of 4 stages;
//   warp 1      allocates 2 x BN columns of tensor memory; one elected lane
//               issues tcgen05.mma (M = 128, N = BN, K = 16, four per stage)
//               and commits each stage back to the producer and each
//               finished tile to the epilogue;
//   warps 2..9  read the tile's rows from tensor memory (tcgen05.ld, warp w
//               owns lanes 32 (w % 4) ...; warps 2..5 the first half of the
//               columns, 6..9 the second) and run the epilogue, while the
//               next tile accumulates in the other tensor-memory buffer.
//               Two warps per sub-partition keep the epilogue's exp and
//               conversion work from holding the tensor core back.
// Tiles go to CTAs round-robin, M fastest, so the CTAs working at any moment
// share the same B tile (B streams from HBM about once; A stays in L2).
// Every wait is bounded: on timeout a status bit is set and the roles wind
// down, waiting (bounded) for their own copies and MMAs before the tensor
// memory is freed.
#pragma once

#include <cuda.h>

#include "common.cuh"
#include "launch.h"

namespace ftk {
namespace tc {

constexpr int BM = 128;          // rows of a tile (tensor-memory lanes)
constexpr int BK = 64;           // k-step: 64 bf16 = one 128-byte swizzle row
constexpr uint32_t kSmemBudget = 227 * 1024 - 2048;  // stages + barriers + alignment slack
constexpr int kThreads = 320;    // 10 warps
constexpr int kEpiThreads = 256;  // 8 epilogue warps: 4 lane quarters x 2 column halves
constexpr uint32_t kTmemCols = 512;  // two accumulators of up to 256 columns

constexpr uint32_t kScratchWords = 32 * 32;  // an epilogue warp's staging tile: 32 x 32 words

constexpr int kMnBlock = 64;           // MN-major operands: 64-element (128-byte) column blocks
constexpr uint32_t kMnBoxBytes = kMnBlock * BK * 2;  // one such block of a k-step: 8 KB

// Operand majors of a GEMM: K-major (K contiguous, the natural layout of
// A [M, K] and B [N, K]) or MN-major (M or N contiguous: A stored [K, M], B
// stored [K, N]).
enum Major : int { kKMajor = 0, kAMn = 1, kBMn = 2 };

// SCRATCH: whether each epilogue warp gets a 4 KB shared-memory tile to
// regroup its values before storing them.  MAJ: the operand majors.  An
// MN-major operand is staged as 64-element blocks of BK rows (8 KB each),
// block j at j x 8 KB; a K-major one as rows of BK elements.
template <int BN, bool SCRATCH, int MAJ = kKMajor> struct Layout {
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN: a multiple of 32 up to 256");
  static constexpr int b_blocks = (BN + kMnBlock - 1) / kMnBlock;
  static constexpr uint32_t a_bytes = BM * BK * 2;  // the same in both majors
  static constexpr uint32_t b_bytes = (MAJ & kBMn) ? b_blocks * kMnBoxBytes : BN * BK * 2;
  static constexpr uint32_t stage_bytes = a_bytes + b_bytes;  // a multiple of 1024
  static constexpr uint32_t scratch_bytes = SCRATCH ? (kEpiThreads / 32) * kScratchWords * 4 : 0;
  // 4 stages (a fifth, where it fits, measured no faster)
  static constexpr int stages_fit = (int)((kSmemBudget - scratch_bytes) / stage_bytes);
  static constexpr int kStages = stages_fit > 4 ? 4 : stages_fit;
  static_assert(kStages >= 2, "two stages must fit");
  static constexpr uint32_t scratch_offset = kStages * stage_bytes;
  static constexpr uint32_t bar_offset = scratch_offset + scratch_bytes;
  // full[S], empty[S], acc_full[2], acc_empty[2], drain; then the tensor
  // memory address and an abort flag
  static constexpr uint32_t smem_bytes = bar_offset + (2 * kStages + 5) * 8 + 16 + 1024;
  static_assert(smem_bytes <= 227 * 1024, "shared memory per CTA");
};

// ---------------------------------------------------------------- PTX

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: rows of 128 bytes, 8-row atoms 1024 bytes apart (stride
// byte offset), leading byte offset unused (1), descriptor version 1,
// layout 2 = 128-byte swizzle.  The tile must start on a 1024-byte boundary.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t addr) {
  return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
         ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// The same for an MN-major tile: each k row holds 64 M (or N) elements in
// 128 bytes, 8-row swizzle atoms of 1024 bytes follow each other along k
// (stride byte offset 1024), and the 64-element blocks along M (or N) are
// kMnBoxBytes apart (leading byte offset).
__device__ __forceinline__ uint64_t desc_sw128_mn(uint32_t addr) {
  return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)(kMnBoxBytes >> 4) << 16) |
         ((uint64_t)(1024 >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, N = BN, M = 128;
// bit 15 / 16 mark A / B as MN-major.
template <int BN, int MAJ> __device__ __forceinline__ constexpr uint32_t idesc_bf16() {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((MAJ & kAMn) ? 1u << 15 : 0u) |
         ((MAJ & kBMn) ? 1u << 16 : 0u) | ((uint32_t)(BN >> 3) << 17) |
         ((uint32_t)(BM >> 4) << 24);
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_addr(bar))
      : "memory");
}

// 32 consecutive fp32 columns of this thread's tensor-memory lane; the
// wait is in the same statement so no use of v can be placed before it.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

// ---------------------------------------------------------------- kernel

// Epi provides:
//   static constexpr bool kScratch;                 wants a staging tile
//   struct Row;                                     per-row state
//   __device__ void begin(Row&, int m, int n0) const;
//   __device__ void slice(Row&, int m, int n, const float (&x)[32],
//                         uint32_t *scr) const;      columns n .. n + 31
//   __device__ void end(Row&, int m, int n0, int half) const;
//                                                   after the tile is released
// A row of a tile is seen by two threads, one per column half (half 0:
// the first ceil(BN/64) slices of 32 columns, half 1 the rest), each with
// its own Row.  m may be >= M (rows past the end of A read as zero): the
// epilogue masks.  slice is called by all 32 lanes of a warp together
// (lane i holding row m - lane + i), so it may exchange values between
// lanes; scr is the warp's own 32 x 32-word shared-memory tile (null unless
// kScratch), which keeps nothing between calls that the epilogue does not
// put there itself.
// ta / tb: tensor maps with 64-element inner boxes; a K-major operand's
// box is [BM or BN rows x 64 k], an MN-major one's [64 k rows x 64].
template <int BN, class Epi, int MAJ>
__global__ void __launch_bounds__(kThreads, 1)
tc_gemm(const __grid_constant__ CUtensorMap ta, const __grid_constant__ CUtensorMap tb, int M,
        int N, int K, const Epi epi, unsigned *status, long long wait_limit) {
  using L = Layout<BN, Epi::kScratch, MAJ>;
  constexpr int kStages = L::kStages;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  unsigned char *sm = smem_raw + ((1024 - (raw & 1023)) & 1023);  // 1024-aligned tiles
  const uint32_t sbase = smem_addr(sm);
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + L::bar_offset);
  uint64_t *empty = full + kStages;
  uint64_t *acc_full = empty + kStages;
  uint64_t *acc_empty = acc_full + 2;
  uint64_t *drain = acc_empty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = (M + BM - 1) / BM, nt = (N + BN - 1) / BN;
  const int ntiles = mt * nt;
  const int nk = (K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], kEpiThreads);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x) {
        const int m0 = (tile % mt) * BM, n0 = (tile / mt) * BN;
        // MN-major blocks that start past the matrix are not loaded: they
        // feed only rows >= M or columns >= N, which the epilogue drops
        const int a_blk = (MAJ & kAMn) ? (M - m0 > kMnBlock ? 2 : 1) : 0;
        int b_blk = 0;
        if (MAJ & kBMn) {
          b_blk = (N - n0 + kMnBlock - 1) / kMnBlock;
          if (b_blk > L::b_blocks) b_blk = L::b_blocks;
        }
        const uint32_t tx = ((MAJ & kAMn) ? a_blk * kMnBoxBytes : L::a_bytes) +
                            ((MAJ & kBMn) ? b_blk * kMnBoxBytes : L::b_bytes);
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kStages;
          if (*abort_flag ||
              !mbar_wait_bounded(&empty[s], ((it / kStages) & 1) ^ 1, wait_limit, status)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          const uint32_t st = sbase + s * L::stage_bytes;
          const uint32_t bar = smem_addr(&full[s]);
          mbar_arrive_expect_tx(&full[s], tx);
          if (MAJ & kAMn) {
            for (int j = 0; j < a_blk; ++j)
              tma_load_2d(st + j * kMnBoxBytes, &ta, m0 + j * kMnBlock, kb * BK, bar);
          } else {
            tma_load_2d(st, &ta, kb * BK, m0, bar);
          }
          if (MAJ & kBMn) {
            for (int j = 0; j < b_blk; ++j)
              tma_load_2d(st + L::a_bytes + j * kMnBoxBytes, &tb, n0 + j * kMnBlock, kb * BK,
                          bar);
          } else {
            tma_load_2d(st + L::a_bytes, &tb, kb * BK, n0, bar);
          }
        }
      }
      // loads still in flight land before the CTA can exit: wait for the
      // last kStages issued stages (consumed ones complete at once)
      for (int i = it - kStages; i < it; ++i)
        if (i >= 0) mbar_wait_bounded(&full[i % kStages], (i / kStages) & 1, wait_limit, status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16<BN, MAJ>();
      // descriptor step per 16 k: 32 bytes along a K-major row, 16 rows of
      // 128 bytes down an MN-major block (in 16-byte units)
      constexpr uint64_t a_step = (MAJ & kAMn) ? (16 * 128) >> 4 : 2;
      constexpr uint64_t b_step = (MAJ & kBMn) ? (16 * 128) >> 4 : 2;
      int it = 0, tcount = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < ntiles; tile += gridDim.x, ++tcount) {
        const int b = tcount & 1;
        if (*abort_flag ||
            !mbar_wait_bounded(&acc_empty[b], ((tcount >> 1) & 1) ^ 1, wait_limit, status)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(b * BN);
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kStages;
          if (*abort_flag ||
              !mbar_wait_bounded(&full[s], (it / kStages) & 1, wait_limit, status)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = sbase + s * L::stage_bytes;
          const uint64_t ad = (MAJ & kAMn) ? desc_sw128_mn(st) : desc_sw128(st);
          const uint64_t bd = (MAJ & kBMn) ? desc_sw128_mn(st + L::a_bytes)
                                           : desc_sw128(st + L::a_bytes);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_bf16(d, ad + a_step * kk, bd + b_step * kk, idesc, (kb | kk) != 0);
          umma_commit(&empty[s]);  // the stage is free once these MMAs have read it
        }
        if (ok) umma_commit(&acc_full[b]);
      }
      // every MMA issued has completed before the tensor memory is freed
      umma_commit(drain);
      mbar_wait_bounded(drain, 0, wait_limit, status);
    }
  } else {
    // ------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // the tensor-memory lanes this warp may read
    const int half = (warp - 2) >> 2;
    constexpr int kSlices = BN / 32, kFirst = (kSlices + 1) / 2;
    const int c_begin = half ? kFirst * 32 : 0, c_end = half ? BN : kFirst * 32;
    const int r = quarter * 32 + lane;
    uint32_t *scr = Epi::kScratch
                        ? reinterpret_cast<uint32_t *>(sm + L::scratch_offset) +
                              (warp - 2) * kScratchWords
                        : nullptr;
    int tcount = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x, ++tcount) {
      const int b = tcount & 1;
      bool go = !*abort_flag &&
                mbar_wait_bounded(&acc_full[b], (tcount >> 1) & 1, wait_limit, status);
      // the tensor-memory loads below are warp-collective: the whole warp
      // goes on, or the whole warp stops
      go = __all_sync(0xffffffffu, go);
      if (!go) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const int m = (tile % mt) * BM + r, n0 = (tile / mt) * BN;
      typename Epi::Row row;
      epi.begin(row, m, n0);
      const uint32_t base = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(b * BN);
#pragma unroll 1
      for (int c = c_begin; c < c_end; c += 32) {
        uint32_t v[32];
        tmem_ld32(base + (uint32_t)c, v);
        float x[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(v[e]);
        epi.slice(row, m, n0 + c, x, scr);
      }
      tc_fence_before();
      mbar_arrive(&acc_empty[b]);  // the buffer may take the next tile
      epi.end(row, m, n0, half);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- host

// A row-major bf16 matrix [rows, cols] with a row stride of ld elements
// (ld % 8 == 0, base 16-byte aligned), read in boxes of box_rows x 64 with
// the 128-byte swizzle; reads past rows / cols return zeros.  A K-major
// operand is [M or N rows, K cols] with box_rows = BM or BN; an MN-major one
// [K rows, M or N cols] with box_rows = BK (a box starts at a column that is
// a multiple of 8).
cudaError_t make_tmap_bf16(CUtensorMap *map, const void *base, int64_t rows, int64_t cols,
                           int64_t ld, int box_rows);

// Launches tc_gemm on min(#tiles, #SMs) persistent CTAs (plain launch: the
// kernel holds all of an SM's tensor memory while it runs).
template <int BN, int MAJ, class Epi>
cudaError_t launch_tc_gemm(const CUtensorMap &ta, const CUtensorMap &tb, int M, int N, int K,
                           const Epi &epi, const DeviceInfo &dev, cudaStream_t s) {
  using L = Layout<BN, Epi::kScratch, MAJ>;
  auto kern = tc_gemm<BN, Epi, MAJ>;
  static bool raised[64] = {};
  if (dev.device >= 0 && dev.device < 64 && !raised[dev.device]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L::smem_bytes);
    if (e != cudaSuccess) return e;
    raised[dev.device] = true;
  }
  unsigned *status = nullptr;
  cudaError_t e = device_status_ptr(dev, &status);
  if (e != cudaSuccess) return e;
  const int64_t tiles = (int64_t)((M + BM - 1) / BM) * ((N + BN - 1) / BN);
  if (tiles == 0) return cudaSuccess;
  const int grid = (int)(tiles < dev.sms ? tiles : dev.sms);
  kern<<<grid, kThreads, L::smem_bytes, s>>>(ta, tb, M, N, K, epi, status, kWaitLimitCycles);
  return cudaGetLastError();
}

}  // namespace tc
}  // namespace ftk
