// A persistent bf16 GEMM on the 5th-generation tensor cores (tcgen05) with a
// pluggable epilogue: C[m, n] = sum_k A[m, k] B[n, k], fp32 accumulation in
// tensor memory.  Either operand is read K-major (A stored [M, K], B [N, K])
// or MN-major (A stored [K, M], B [K, N]), so no operand is ever transposed
// in memory.  The epilogue sees each output row in 32-column slices and
// never writes the accumulator tile as such unless it wants to; the
// cross-entropy kernels (cce.cu) use it to fold a softmax into the
// contraction.  One launch may run two problems of the same epilogue type
// (a grouped GEMM): their tiles share one persistent grid.
//
// One CTA per SM; CTAs run in pairs (clusters of two) that compute one
// 256-row tile together with the 2-SM MMA (tcgen05 cta_group::2, see
// unit_of).  10 warps per CTA:
//   warp 0      one elected lane issues TMA loads (cp.async.bulk.tensor, 128-
//               byte swizzle) of this CTA's A rows [128 x 64] and its half
//               of the B tile [BN/2 x 64] of every k-step into a ring of 6 - 7
//               stages, completing on the leader CTA's barrier;
//   warp 1      allocates 2 x 256 columns of tensor memory in both CTAs; in
//               the leader, one elected lane issues tcgen05.mma (M = 256,
//               N = BN, K = 16, four per stage) and commits each stage back
//               to both producers and each finished tile to both epilogues;
//   warps 2..9  read the CTA's 128 rows of the tile from tensor memory
//               (tcgen05.ld, warp w owns lanes 32 (w % 4) ...; warps 2..5 the
//               first half of the columns, 6..9 the second) and run the
//               epilogue, while the next tile accumulates in the other
//               tensor-memory buffer.  Two warps per sub-partition keep the
//               epilogue's exp and conversion work from holding the tensor
//               core back.
// Units (pairs of M-tiles) go to CTA pairs round-robin.  Within a problem
// they run M fastest when B is the larger operand (the pairs working at any
// moment share a B tile, so B streams from HBM about once while A stays in
// L2) and N fastest when A is (the same with the roles swapped).
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

// Operand majors of a problem: K-major (K contiguous, the natural layout of
// A [M, K] and B [N, K]) or MN-major (M or N contiguous: A stored [K, M], B
// stored [K, N]).
enum Major : int { kKMajor = 0, kAMn = 1, kBMn = 2 };

// SCRATCH: whether each epilogue warp gets a 4 KB shared-memory tile to
// regroup its values before storing them.  A stage holds this CTA's A tile
// [128 x 64] (16 KB in either major) and room for its half of the B tile in
// either major: BN / 2 rows of 128 bytes (K-major) or ceil(BN / 128) blocks
// of 64 elements x BK rows, 8 KB each, block j at j x 8 KB (MN-major).
template <int BN, bool SCRATCH> struct Layout {
  static_assert(BN % 32 == 0 && BN >= 64 && BN <= 256, "BN: a multiple of 32, 64 .. 256");
  static constexpr int kHalf = BN / 2;  // B rows (or columns) per CTA
  static constexpr int b_blocks = (kHalf + kMnBlock - 1) / kMnBlock;
  static constexpr uint32_t a_bytes = BM * BK * 2;
  static constexpr uint32_t b_bytes_k = kHalf * BK * 2;
  static constexpr uint32_t b_bytes = b_blocks * kMnBoxBytes;  // >= b_bytes_k
  static constexpr uint32_t stage_bytes = a_bytes + b_bytes;  // a multiple of 1024
  static constexpr uint32_t scratch_bytes = SCRATCH ? (kEpiThreads / 32) * kScratchWords * 4 : 0;
  static constexpr int stages_fit = (int)((kSmemBudget - scratch_bytes) / stage_bytes);
  static constexpr int kStages = stages_fit > 8 ? 8 : stages_fit;
  static_assert(kStages >= 2, "two stages must fit");
  static constexpr uint32_t scratch_offset = kStages * stage_bytes;
  static constexpr uint32_t bar_offset = scratch_offset + scratch_bytes;
  // full[S], empty[S], acc_full[2], acc_empty[2], drain; then the tensor
  // memory address and an abort flag
  static constexpr uint32_t smem_bytes = bar_offset + (2 * kStages + 5) * 8 + 16 + 1024;
  static_assert(smem_bytes <= 227 * 1024, "shared memory per CTA");
};

// One GEMM of a launch.  ta / tb: tensor maps with 64-element inner boxes;
// a K-major operand's box is [BM (A) or BN / 2 (B, loaded in two halves)
// rows x 64 k], an MN-major one's [64 k rows x 64].  Filled in by
// make_problem.
template <class Epi> struct Problem {
  CUtensorMap ta, tb;  // 64-byte aligned
  Epi epi;
  int M, N, K;
  int maj;     // Major bits
  int mt, nt;  // tiles along M and N
  int n_fast;  // 1: units run N fastest
  int units;   // ceil(mt / 2) x nt pairs of M-tiles (see unit_of)
};

template <class Epi> struct Group {
  Problem<Epi> p[2];
  int count;  // 1 or 2 problems
  int units;  // over all problems
};

// ---------------------------------------------------------------- PTX

// A TMA tile load into this CTA's shared memory whose bytes complete on the
// mbarrier at cluster address bar, which may be the peer CTA's.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".cta_group::2 [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// The tcgen05 instructions of this kernel all act on the CTA pair
// (cta_group::2).  Allocation and release: one warp in each of the two
// CTAs, collectively; the same columns in both CTAs' tensor memory.
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(slot)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
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

// Instruction descriptor, kind::f16: D fp32, A and B bf16, N = BN, M = 256
// (the CTA pair's tile); bit 15 / 16 mark A / B as MN-major.
template <int BN> __device__ __forceinline__ uint32_t idesc_bf16(int maj) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((maj & kAMn) ? 1u << 15 : 0u) |
         ((maj & kBMn) ? 1u << 16 : 0u) | ((uint32_t)(BN >> 3) << 17) |
         ((uint32_t)((2 * BM) >> 4) << 24);
}

// D [256 x BN] (+)= A B^T for the pair, issued by one thread of the leader
// (rank 0): A rows 0..127 from the leader's shared memory, 128..255 from
// the peer's, both at descriptor a; B rows (N) 0..BN/2-1 from the leader's,
// the rest from the peer's, at descriptor b; each CTA's tensor memory gets
// its own 128 rows.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrives once on the mbarrier at the same offset in every CTA of mask when
// the pair's earlier MMAs have completed.
__device__ __forceinline__ void umma_commit(uint64_t *bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_addr(bar)),
      "h"(mask)
      : "memory");
}

// 64 consecutive fp32 columns of this thread's tensor-memory lane, in one
// load and one wait (in the same statement, so no use of v can be placed
// before the wait).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&v)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, "
      "%45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, "
      "%62, %63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]),
        "=r"(v[32]), "=r"(v[33]), "=r"(v[34]), "=r"(v[35]), "=r"(v[36]), "=r"(v[37]),
        "=r"(v[38]), "=r"(v[39]), "=r"(v[40]), "=r"(v[41]), "=r"(v[42]), "=r"(v[43]),
        "=r"(v[44]), "=r"(v[45]), "=r"(v[46]), "=r"(v[47]), "=r"(v[48]), "=r"(v[49]),
        "=r"(v[50]), "=r"(v[51]), "=r"(v[52]), "=r"(v[53]), "=r"(v[54]), "=r"(v[55]),
        "=r"(v[56]), "=r"(v[57]), "=r"(v[58]), "=r"(v[59]), "=r"(v[60]), "=r"(v[61]),
        "=r"(v[62]), "=r"(v[63])
      : "r"(taddr)
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


// Brings the box of map at (x, y) into L2 without copying it anywhere.
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap *map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y)
               : "memory");
}

// ---------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of both CTAs of the cluster; also a barrier within the CTA.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The cluster address of the same shared-memory object in CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void *p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}

// mbarrier arrive on a cluster address (this CTA's or the peer's).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar)
               : "memory");
}

// ---------------------------------------------------------------- tiles

// The CTAs run in clusters of two, a pair that computes one 256-row tile
// with the 2-SM MMA: a unit of work is M-tiles 2 p (the leader, rank 0) and
// 2 p + 1 (rank 1) of one N-tile.  Each CTA stages its own 128 rows of A and
// one half of B, so a CTA holds 32 KB per k-step instead of 48 and the ring
// gets 6 - 7 stages deep.
//
// What a role needs to walk one problem's units, read once from the kernel
// parameters into registers.
struct Seq {
  int mp, nt, n_fast, maj, nk, first;  // mp: M-tile pairs; first: the problem's first unit
};

template <int G, class Epi>
__device__ __forceinline__ void load_seqs(const Group<Epi> &g, Seq (&q)[G]) {
#pragma unroll
  for (int i = 0; i < G; ++i) {
    q[i].mp = (g.p[i].mt + 1) >> 1;
    q[i].nt = g.p[i].nt;
    q[i].n_fast = g.p[i].n_fast;
    q[i].maj = g.p[i].maj;
    q[i].nk = (g.p[i].K + BK - 1) / BK;
    q[i].first = i ? g.p[0].units : 0;
  }
}

// The problem (0 or G - 1) of the group's unit u and its origin: the
// leader's first row m0 (rank 1 starts at m0 + 128) and first column n0; s
// receives the problem's Seq.  (Selects, not an indexed array, keep
// everything in registers.)
template <int BN, int G>
__device__ __forceinline__ int unit_of(const Seq (&q)[G], int u, int &m0, int &n0, Seq &s) {
  const int pi = (G > 1 && u >= q[G - 1].first) ? G - 1 : 0;
  s = pi ? q[G - 1] : q[0];
  const int v = u - s.first;
  const int pm = s.n_fast ? v / s.nt : v % s.mp;
  const int pn = s.n_fast ? v - pm * s.nt : v / s.mp;
  m0 = 2 * pm * BM;
  n0 = pn * BN;
  return pi;
}

// What CTA `rank` of the pair loads per k-step of a unit: its A rows
// (none if they start past M; MN-major: the 64-row blocks that start below
// M) and its half of B (none if it starts past N; MN-major: the blocks that
// start below N).  In bytes, and as block counts for the MN-major forms.
template <int BN, bool SCRATCH> struct Share {
  int a_blk, b_blk;  // K-major: 1 or 0
  uint32_t bytes;
  __device__ __forceinline__ Share(int maj, int M, int N, int m0, int n0, uint32_t rank) {
    using L = Layout<BN, SCRATCH>;
    const int ma = m0 + (int)rank * BM, nb = n0 + (int)rank * L::kHalf;
    a_blk = ma >= M ? 0 : (maj & kAMn) ? (M - ma > kMnBlock ? 2 : 1) : 1;
    if (nb >= N) {
      b_blk = 0;
    } else if (maj & kBMn) {
      b_blk = (N - nb + kMnBlock - 1) / kMnBlock;
      if (b_blk > L::b_blocks) b_blk = L::b_blocks;
    } else {
      b_blk = 1;
    }
    bytes = (uint32_t)a_blk * ((maj & kAMn) ? kMnBoxBytes : L::a_bytes) +
            (uint32_t)b_blk * ((maj & kBMn) ? kMnBoxBytes : L::b_bytes_k);
  }
};

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
// its own Row.  m may be >= M (rows past the end of A read as zero, or as
// anything in a tile that lies wholly past M): the epilogue masks.  slice is
// called by all 32 lanes of a warp together (lane i holding row m - lane +
// i), so it may exchange values between lanes; scr is the warp's own 32 x
// 32-word shared-memory tile (null unless kScratch), which keeps nothing
// between calls that the epilogue does not put there itself.
//
// Pair protocol (rank 0 = leader, which alone issues MMAs):
//   full[s]       the leader's: one arrival (its producer, expecting both
//                 CTAs' bytes) plus the bytes of both CTAs' loads;
//   empty[s]      each CTA's: one arrival from the leader's MMA commit;
//   acc_full[b]   each CTA's: one arrival from the leader's MMA commit;
//   acc_empty[b]  the leader's: one arrival per epilogue warp of both CTAs.
// Before a CTA leaves, every arrival its barriers will get from the other
// CTA has come, and the leader's MMAs (which write both CTAs' tensor memory)
// have completed.
template <int BN, int G, class Epi>
__global__ void __launch_bounds__(kThreads, 1)
tc_gemm(const __grid_constant__ Group<Epi> g, unsigned *status, long long wait_limit) {
  using L = Layout<BN, Epi::kScratch>;
  using Sh = Share<BN, Epi::kScratch>;
  constexpr int kStages = L::kStages;
  constexpr int kEpiWarps = kEpiThreads / 32;
  constexpr uint16_t kBoth = 0x3, kLeader = 0x1;
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  // the dynamic window starts at the same offset in both CTAs, so the
  // tiles and barriers below sit at the same offsets in each
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
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int cid = (int)(blockIdx.x >> 1), ncl = (int)(gridDim.x >> 1);
  const int nunits = g.units;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 2 * kEpiWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers exist before either targets the other's
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint32_t full0 = cluster_addr(full, 0);  // the leader's full[0]
      Seq q[G];
      load_seqs<G>(g, q);
      int it = 0;
      bool ok = true;
      for (int u = cid; ok && u < nunits; u += ncl) {
        int m0, n0;
        Seq sq;
        const int pi = unit_of<BN, G>(q, u, m0, n0, sq);
        const Problem<Epi> &P = pi ? g.p[G - 1] : g.p[0];
        const int maj = sq.maj, nk = sq.nk;
        const CUtensorMap *ta = &P.ta, *tb = &P.tb;
        const Sh mine(maj, P.M, P.N, m0, n0, rank);
        const uint32_t tx = leader ? mine.bytes + Sh(maj, P.M, P.N, m0, n0, 1).bytes : 0;
        const int ma = m0 + (int)rank * BM, nb = n0 + (int)rank * L::kHalf;
        // When units run M fastest, the pairs working at a time share two or
        // three B tiles, and every pair starts a new one together: the pair
        // whose next unit opens an N-tile (M-pair 0) fetches that tile's B
        // half into L2 one unit ahead, so the others find it there.
        if (u + ncl < nunits) {
          int pm0, pn0;
          Seq sn;
          const int pj = unit_of<BN, G>(q, u + ncl, pm0, pn0, sn);
          if (!sn.n_fast && pm0 == 0 && !(sn.maj & kBMn)) {
            const Problem<Epi> &Pn = pj ? g.p[G - 1] : g.p[0];
            const int nbn = pn0 + (int)rank * L::kHalf;
            if (nbn < Pn.N)
              for (int kb = 0; kb < sn.nk; ++kb) tma_prefetch_2d(&Pn.tb, kb * BK, nbn);
          }
        }
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kStages;
          if (*abort_flag ||
              !mbar_wait_bounded(&empty[s], ((it / kStages) & 1) ^ 1, wait_limit, status)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          const uint32_t st = sbase + s * L::stage_bytes;
          const uint32_t bar = full0 + 8u * (uint32_t)s;
          if (leader) mbar_arrive_expect_tx(&full[s], tx);
          if (maj & kAMn) {
            for (int j = 0; j < mine.a_blk; ++j)
              tma_load_2d(st + j * kMnBoxBytes, ta, ma + j * kMnBlock, kb * BK, bar);
          } else if (mine.a_blk) {
            tma_load_2d(st, ta, kb * BK, ma, bar);
          }
          if (maj & kBMn) {
            for (int j = 0; j < mine.b_blk; ++j)
              tma_load_2d(st + L::a_bytes + j * kMnBoxBytes, tb, nb + j * kMnBlock, kb * BK, bar);
          } else if (mine.b_blk) {
            tma_load_2d(st + L::a_bytes, tb, kb * BK, nb, bar);
          }
        }
      }
      // before the CTA may leave: the leader sees every load of both CTAs
      // land (the last kStages stages; earlier ones were consumed), and each
      // CTA sees the leader's MMAs release every stage it filled
      if (leader)
        for (int i = it - kStages; i < it; ++i)
          if (i >= 0) mbar_wait_bounded(&full[i % kStages], (i / kStages) & 1, wait_limit, status);
      for (int i = it - kStages; i < it; ++i)
        if (i >= 0) mbar_wait_bounded(&empty[i % kStages], (i / kStages) & 1, wait_limit, status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      Seq q[G];
      load_seqs<G>(g, q);
      int it = 0, tcount = 0;
      bool ok = true;
      for (int u = cid; ok && u < nunits; u += ncl, ++tcount) {
        int m0, n0;
        Seq sq;
        unit_of<BN, G>(q, u, m0, n0, sq);
        const int maj = sq.maj, nk = sq.nk;
        const uint32_t idesc = idesc_bf16<BN>(maj);
        // descriptor step per 16 k: 32 bytes along a K-major row, 16 rows
        // of 128 bytes down an MN-major block (in 16-byte units)
        const uint64_t a_step = (maj & kAMn) ? (16 * 128) >> 4 : 2;
        const uint64_t b_step = (maj & kBMn) ? (16 * 128) >> 4 : 2;
        // the descriptors without their start address, per operand major
        const uint64_t a_hi = (maj & kAMn) ? desc_sw128_mn(0) : desc_sw128(0);
        const uint64_t b_hi = (maj & kBMn) ? desc_sw128_mn(0) : desc_sw128(0);
        const int b = tcount & 1;
        if (*abort_flag ||
            !mbar_wait_bounded(&acc_empty[b], ((tcount >> 1) & 1) ^ 1, wait_limit, status)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(b * 256);
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
          const uint64_t ad = a_hi | (uint64_t)(((st) & 0x3FFFF) >> 4);
          const uint64_t bd = b_hi | (uint64_t)(((st + L::a_bytes) & 0x3FFFF) >> 4);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_bf16(d, ad + a_step * kk, bd + b_step * kk, idesc, (kb | kk) != 0);
          umma_commit(&empty[s], kBoth);  // both CTAs may refill stage s
        }
        if (ok) umma_commit(&acc_full[b], kBoth);
      }
      // every MMA issued has completed (both CTAs' tensor memory is final),
      // and both CTAs' epilogues have released the last two tiles
      umma_commit(drain, kLeader);
      mbar_wait_bounded(drain, 0, wait_limit, status);
      for (int t = tcount - 2; t < tcount; ++t)
        if (t >= 0) mbar_wait_bounded(&acc_empty[t & 1], (t >> 1) & 1, wait_limit, status);
    }
  } else {
    // ------------------------------------------------------ epilogue
    const int quarter = warp & 3;  // the tensor-memory lanes this warp may read
    const int half = (warp - 2) >> 2;
    constexpr int kSlices = BN / 32, kFirst = (kSlices + 1) / 2;
    const int c_begin = half ? kFirst * 32 : 0, c_end = half ? BN : kFirst * 32;
    const int r = (int)rank * BM + quarter * 32 + lane;
    const uint32_t acc_empty0 = cluster_addr(acc_empty, 0);  // the leader's
    uint32_t *scr = Epi::kScratch
                        ? reinterpret_cast<uint32_t *>(sm + L::scratch_offset) +
                              (warp - 2) * kScratchWords
                        : nullptr;
    Seq q[G];
    load_seqs<G>(g, q);
    int tcount = 0;
    for (int u = cid; u < nunits; u += ncl, ++tcount) {
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
      int m0, n0;
      Seq sq;
      // a copy: the epilogue's fields live in registers for the whole tile
      const Epi epi = unit_of<BN, G>(q, u, m0, n0, sq) ? g.p[G - 1].epi : g.p[0].epi;
      const int m = m0 + r;
      typename Epi::Row row;
      epi.begin(row, m, n0);
      const uint32_t base = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(b * 256);
      // 64 columns per tensor-memory round trip, then a last 32 if the
      // half has an odd number of slices
      int c = c_begin;
#pragma unroll 1
      for (; c + 64 <= c_end; c += 64) {
        uint32_t v[64];
        tmem_ld64(base + (uint32_t)c, v);
        float x[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(v[e]);
        epi.slice(row, m, n0 + c, x, scr);
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(v[32 + e]);
        epi.slice(row, m, n0 + c + 32, x, scr);
      }
      if (c < c_end) {
        uint32_t v[32];
        tmem_ld32(base + (uint32_t)c, v);
        float x[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) x[e] = __uint_as_float(v[e]);
        epi.slice(row, m, n0 + c, x, scr);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(acc_empty0 + 8u * (uint32_t)b);  // the buffer is free
      epi.end(row, m, n0, half);
    }
  }
  tc_fence_before();
  cluster_sync();  // the leader's MMAs are complete: both may free tensor memory
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_sync();  // neither CTA leaves while the other may still reach it
}

// ---------------------------------------------------------------- host

// A row-major bf16 matrix [rows, cols] with a row stride of ld elements
// (ld % 8 == 0, base 16-byte aligned), read in boxes of box_rows x 64 with
// the 128-byte swizzle; reads past rows / cols return zeros.  A K-major
// operand is [M or N rows, K cols] (box_rows BM for A, BN / 2 for B); an
// MN-major one [K rows, M or N cols] with box_rows = BK (a box starts at a
// column that is a multiple of 8).
cudaError_t make_tmap_bf16(CUtensorMap *map, const void *base, int64_t rows, int64_t cols,
                           int64_t ld, int box_rows);

// Fills P for C [M, N] = A B^T with the given operand majors: a is A stored
// [M, lda] (K-major) or [K, lda] (MN-major), b likewise [N, ldb] or [K, ldb].
template <class Epi>
cudaError_t make_problem(Problem<Epi> &P, int bn, const void *a, int64_t lda, const void *b,
                         int64_t ldb, int M, int N, int K, int maj, const Epi &epi) {
  cudaError_t e = (maj & kAMn) ? make_tmap_bf16(&P.ta, a, K, M, lda, BK)
                               : make_tmap_bf16(&P.ta, a, M, K, lda, BM);
  if (e != cudaSuccess) return e;
  e = (maj & kBMn) ? make_tmap_bf16(&P.tb, b, K, N, ldb, BK)
                   : make_tmap_bf16(&P.tb, b, N, K, ldb, bn / 2);
  if (e != cudaSuccess) return e;
  P.epi = epi;
  P.M = M;
  P.N = N;
  P.K = K;
  P.maj = maj;
  P.mt = (M + BM - 1) / BM;
  P.nt = (N + bn - 1) / bn;
  P.n_fast = N < M ? 1 : 0;  // stream the larger operand once
  P.units = ((P.mt + 1) / 2) * P.nt;
  return cudaSuccess;
}

// Launches tc_gemm over the group's G problems (g.count == G, all with tile
// width BN): CTA pairs (clusters of two), as many as fit on the device at
// once (at most one per unit), persistent (the kernel holds all of an SM's
// tensor memory while it runs).
template <int BN, int G, class Epi>
cudaError_t launch_tc_gemm(Group<Epi> &g, const DeviceInfo &dev, cudaStream_t s) {
  static_assert(G == 1 || G == 2, "one or two problems");
  using L = Layout<BN, Epi::kScratch>;
  auto kern = tc_gemm<BN, G, Epi>;
  static int max_clusters[64] = {};
  if (dev.device < 0 || dev.device >= 64) return cudaErrorInvalidDevice;
  if (g.count != G) return cudaErrorInvalidValue;
  g.units = 0;
  for (int i = 0; i < G; ++i) g.units += g.p[i].units;
  if (g.units == 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::smem_bytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!max_clusters[dev.device]) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)L::smem_bytes);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3((unsigned)(dev.sms & ~1));
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (n < 1) return cudaErrorInvalidConfiguration;  // no pair of CTAs fits at all
    max_clusters[dev.device] = n;
  }
  unsigned *status = nullptr;
  cudaError_t e = device_status_ptr(dev, &status);
  if (e != cudaSuccess) return e;
  const int ncl = g.units < max_clusters[dev.device] ? g.units : max_clusters[dev.device];
  cfg.gridDim = dim3((unsigned)(2 * ncl));
  long long limit = kWaitLimitCycles;
  return cudaLaunchKernelEx(&cfg, kern, g, status, limit);
}

}  // namespace tc
}  // namespace ftk
