// Cross-entropy of the LM head without materialised logits ("Chronicals",
// arXiv 2601.02609, abstract, optimisation (2): Cut Cross-Entropy; an online
// softmax keeps the logits from ever sitting in memory at once).
//
//   z = h W^T,  lse[t] = log sum_v e^z[t,v],
//   loss = (1/N) sum_{valid t} (lse[t] - z[t, y_t])   (valid: 0 <= y_t < V)
//   dz = (g/N)(softmax(z) - onehot(y)),  dh = dz W,  dW = dz^T h
//
// Forward: one tcgen05 GEMM over the whole vocabulary whose epilogue folds
// each 128 x 256 logit tile into per-row (max, sum of exp) partials and
// picks out the target logit, so no logit reaches HBM; a warp per row then
// merges the partials into lse and the row losses, and one CTA sums them in
// a fixed order.
// Backward, per vocabulary chunk of C columns (cce_bwd_chunk: 4,096 to 16,384,
// sized so that the chunk's tiles fill whole waves of the SMs): a GEMM whose
// epilogue turns the recomputed logits into dz (bf16 [T, C]: 185 MB for
// 8,192 tokens and 11,264 columns, about the ~135 MB the page quotes for its
// logits), then dh += dz W_c and dW_c = dz^T h as one grouped GEMM that
// reads dz, W_c and h where they lie (MN-major where a transpose is
// needed).  dh accumulates in fp32 and is rounded to bf16 by the last
// chunk's epilogue.
#include <cudaTypedefs.h>

#include <cmath>

#include "tc_gemm.cuh"

namespace ftk {

namespace tc {

cudaError_t make_tmap_bf16(CUtensorMap *map, const void *base, int64_t rows, int64_t cols,
                           int64_t ld, int box_rows) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  const cuuint32_t elem[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base),
                            dims, strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace tc

namespace {

constexpr int kChunkMin = 4096;   // vocabulary columns per backward chunk: chosen in
constexpr int kChunkMax = 16384;  // [kChunkMin, kChunkMax] by cce_bwd_chunk
constexpr int kFwdBN = 256;      // logit tile width of the forward / dz GEMMs
constexpr float kLog2e = 1.4426950408889634f;

// ------------------------------------------------------------ epilogues

// 2^x by the hardware approximation (PTX ex2.approx.ftz.f32: relative error
// about 2^-22, 2^-inf = +0).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Forward: per-row (max, sum e^(z - max)) over a half tile's columns < V,
// and the target logit when the slice holds it.  part holds 2 partials per
// row per tile (one per column half).
struct EpiLse {
  const int32_t *y;
  int T, V, nparts;
  float2 *part;  // [T][nparts]
  float *tgt;    // [T]
  static constexpr bool kScratch = false;
  struct Row {
    float m, s;
    int y;
  };
  __device__ void begin(Row &r, int m, int) const {
    r.m = -INFINITY;
    r.s = 0.f;
    r.y = m < T ? y[m] : -1;
  }
  __device__ void slice(Row &r, int m, int n, const float (&x)[32], uint32_t *) const {
    if ((unsigned)(r.y - n) < 32u && m < T) {  // the target logit is in this slice
      float zt = 0.f;
#pragma unroll
      for (int e = 0; e < 32; ++e) zt = (e == r.y - n) ? x[e] : zt;
      tgt[m] = zt;
    }
    const bool full = n + 32 <= V;
    float cm;
    if (full) {
      float t[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) t[e] = fmaxf(x[e], x[e + 16]);
#pragma unroll
      for (int w = 8; w > 0; w >>= 1)
#pragma unroll
        for (int e = 0; e < w; ++e) t[e] = fmaxf(t[e], t[e + w]);
      cm = t[0];
    } else {
      cm = -INFINITY;
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (n + e < V) cm = fmaxf(cm, x[e]);
      if (cm == -INFINITY) return;  // every column past V
    }
    if (cm > r.m) {
      r.s *= ex2((r.m - cm) * kLog2e);
      r.m = cm;
    }
    const float ml = r.m * kLog2e;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    if (full) {
#pragma unroll
      for (int e = 0; e < 32; ++e) acc[e & 3] += ex2(fmaf(x[e], kLog2e, -ml));
    } else {
#pragma unroll
      for (int e = 0; e < 32; ++e)
        if (n + e < V) acc[e & 3] += ex2(fmaf(x[e], kLog2e, -ml));
    }
    r.s += (acc[0] + acc[1]) + (acc[2] + acc[3]);
  }
  __device__ void end(Row &r, int m, int n0, int half) const {
    if (m < T) part[(size_t)m * nparts + 2 * (n0 / kFwdBN) + half] = make_float2(r.m, r.s);
  }
};

// Backward, one vocabulary chunk [c0, c0 + Cv): dz = gs (e^(z - lse) - [v == y])
// stored as bf16 row-major [T][ldz].  The values go through the warp's
// shared-memory tile, two slices at a time, so that each store covers whole
// 128-byte lines (64 columns of a row); this pairing needs 64-column aligned
// halves of a tile, i.e. the 256-wide tiles.
static_assert(kFwdBN == 256, "the dz epilogue pairs slices within 128-column halves");
struct EpiGrad {
  const int32_t *y;
  const float *lse, *gscale;
  int T, V, Cv, c0;
  bf16 *dz;
  int64_t ldz;  // ldz % 8 == 0 and dz 16-byte aligned
  static constexpr bool kScratch = true;
  struct Row {
    float l2, gs;
    int yl;
  };
  __device__ void begin(Row &r, int m, int) const {
    r.l2 = 0.f;
    r.gs = 0.f;
    r.yl = -1;
    if (m < T) {
      const int yv = y[m];
      const bool valid = yv >= 0 && yv < V;
      r.l2 = lse[m] * kLog2e;
      r.gs = valid ? *gscale : 0.f;
      r.yl = valid ? yv - c0 : -1;
    }
  }
  // Rows past T carry gs = 0 and are not stored.  This slice is the first
  // (words 0..15 of each staged row) or second (words 16..31) of a
  // 64-column pair; 16-byte chunk j of staged row i sits at j ^ (i & 7), so
  // the row-wise writes and the line-wise reads are free of bank conflicts.
  __device__ void slice(Row &r, int m, int n, const float (&x)[32], uint32_t *scr) const {
    const int lane = threadIdx.x & 31;
    const int hit = r.yl - n;  // the target's column in this slice, if in [0, 32)
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
      float g0 = ex2(fmaf(x[e], kLog2e, -r.l2));
      float g1 = ex2(fmaf(x[e + 1], kLog2e, -r.l2));
      if ((unsigned)hit < 32u) {
        g0 -= (e == hit) ? 1.f : 0.f;
        g1 -= (e + 1 == hit) ? 1.f : 0.f;
      }
      const __nv_bfloat162 b2 = __floats2bfloat162_rn(g0 * r.gs, g1 * r.gs);
      pk[e >> 1] = *reinterpret_cast<const uint32_t *>(&b2);
    }
    const int second = (n >> 5) & 1;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<uint4 *>(scr + lane * 32 + (((4 * second + q) ^ (lane & 7)) << 2)) =
          make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
    if (second) {
      __syncwarp();
      flush(m - lane, n - 32, scr);
      __syncwarp();  // the tile is free for the next pair
    }
  }
  // the staged rows mb .. mb + 31, columns n .. n + 63: pass i stores rows
  // 4 i .. 4 i + 3, lane -> row 4 i + lane / 8, 8 columns from 8 (lane % 8)
  __device__ void flush(int mb, int n, const uint32_t *scr) const {
    const int lane = threadIdx.x & 31, j = lane & 7, col = n + 8 * j;
    const bool full = n + 64 <= Cv;
#pragma unroll 2
    for (int i = 0; i < 8; ++i) {
      const int rr = 4 * i + (lane >> 3), row = mb + rr;
      const uint4 v = *reinterpret_cast<const uint4 *>(scr + rr * 32 + ((j ^ (rr & 7)) << 2));
      if (row >= T) continue;
      bf16 *dst = dz + (size_t)row * ldz + col;
      if (full) {
        *reinterpret_cast<uint4 *>(dst) = v;
      } else {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        unsigned short *d = reinterpret_cast<unsigned short *>(dst);
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (col + e < Cv) d[e] = (unsigned short)(w[e >> 1] >> (16 * (e & 1)));
      }
    }
  }
  __device__ void end(Row &, int, int, int) const {}
};

// Plain output: C[m][n] (+= the fp32 value already there), written as fp32
// or rounded to bf16.  A thread holds one row of a slice; the warp first
// regroups its 32 x 32 values in shared memory so that every store (and
// every read of the old value) covers whole 128-byte lines of a few rows
// instead of 16 bytes of 32 rows.
struct EpiStore {
  float *c;         // fp32 [M][ldc]: read when acc_in, written unless cb
  bf16 *cb;         // nullable: write bf16 [M][ldcb] instead
  int64_t ldc, ldcb;
  int M, N;
  bool acc_in;
  bool vc, vb;      // 16-byte vector access is aligned for c / cb (base and stride)
  static constexpr bool kScratch = true;
  struct Row {};
  __device__ void begin(Row &, int, int) const {}
  // scr holds row i of the slice at words 32 i .. 32 i + 31, its 16-byte
  // chunk j at position j ^ (i & 7): both the row-wise writes and the
  // line-wise reads below are free of bank conflicts.
  __device__ void slice(Row &, int m, int n, const float (&x)[32], uint32_t *scr) const {
    const int lane = threadIdx.x & 31;
    const int mb = m - lane;  // the row of lane 0
    float *sf = reinterpret_cast<float *>(scr);
#pragma unroll
    for (int j = 0; j < 8; ++j)
      *reinterpret_cast<float4 *>(sf + lane * 32 + ((j ^ (lane & 7)) << 2)) =
          make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
    __syncwarp();
    const bool full = n + 32 <= N;
    if (!cb) {
      // pass i: rows 4 i .. 4 i + 3, lane -> row 4 i + lane / 8, columns 4 (lane % 8) ..
      const int j = lane & 7, col = n + 4 * j;
#pragma unroll 2
      for (int i = 0; i < 8; ++i) {
        const int rr = 4 * i + (lane >> 3), row = mb + rr;
        float4 v = *reinterpret_cast<const float4 *>(sf + rr * 32 + ((j ^ (rr & 7)) << 2));
        if (row >= M) continue;
        float *dst = c + (size_t)row * ldc + col;
        if (full && vc) {
          if (acc_in) {
            const float4 o = *reinterpret_cast<const float4 *>(dst);
            v.x += o.x;
            v.y += o.y;
            v.z += o.z;
            v.w += o.w;
          }
          *reinterpret_cast<float4 *>(dst) = v;
        } else {
          const float e4[4] = {v.x, v.y, v.z, v.w};
          for (int e = 0; e < 4; ++e)
            if (col + e < N) dst[e] = acc_in ? dst[e] + e4[e] : e4[e];
        }
      }
    } else {
      // pass i: rows 8 i .. 8 i + 7, lane -> row 8 i + lane / 4, columns 8 (lane % 4) ..
      const int j = 2 * (lane & 3), col = n + 4 * j;
#pragma unroll 2
      for (int i = 0; i < 4; ++i) {
        const int rr = 8 * i + (lane >> 2), row = mb + rr;
        const float4 a = *reinterpret_cast<const float4 *>(sf + rr * 32 + ((j ^ (rr & 7)) << 2));
        const float4 b =
            *reinterpret_cast<const float4 *>(sf + rr * 32 + (((j + 1) ^ (rr & 7)) << 2));
        if (row >= M) continue;
        float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        const float *src = c + (size_t)row * ldc + col;
        bf16 *dst = cb + (size_t)row * ldcb + col;
        if (full && vb && (!acc_in || vc)) {
          if (acc_in) {
            const float4 o0 = reinterpret_cast<const float4 *>(src)[0];
            const float4 o1 = reinterpret_cast<const float4 *>(src)[1];
            v[0] += o0.x;
            v[1] += o0.y;
            v[2] += o0.z;
            v[3] += o0.w;
            v[4] += o1.x;
            v[5] += o1.y;
            v[6] += o1.z;
            v[7] += o1.w;
          }
          __align__(16) __nv_bfloat162 o[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) o[q] = __floats2bfloat162_rn(v[2 * q], v[2 * q + 1]);
          *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(o);
        } else {
          for (int e = 0; e < 8; ++e)
            if (col + e < N) dst[e] = __float2bfloat16_rn(acc_in ? v[e] + src[e] : v[e]);
        }
      }
    }
    __syncwarp();  // the tile is free for the next slice
  }
  __device__ void end(Row &, int, int, int) const {}
};

// ------------------------------------------------------------ small kernels

// lse and the row loss from the forward partials: one warp per row.
__global__ void __launch_bounds__(256)
cce_row_lse(const float2 *__restrict__ part, int ntn, const float *__restrict__ tgt,
            const int32_t *__restrict__ y, int T, int V, float *__restrict__ lse,
            float *__restrict__ row_loss) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + warp;
  if (t >= T) return;
  const float2 *p = part + (size_t)t * ntn;
  float m = -INFINITY;
  for (int j = lane; j < ntn; j += 32) m = fmaxf(m, p[j].x);
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float s = 0.f;
  for (int j = lane; j < ntn; j += 32) {
    const float2 q = p[j];
    if (q.y > 0.f) s += q.y * exp2f((q.x - m) * kLog2e);
  }
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if (lane == 0) {
    const float l = m + logf(s);
    lse[t] = l;
    const int yv = y[t];
    row_loss[t] = (yv >= 0 && yv < V) ? l - tgt[t] : 0.f;
  }
}

// loss = sum of the row losses / N, in a fixed order (one CTA); also the
// backward's scale g / N when g is given.
__global__ void __launch_bounds__(1024)
cce_finish(const float *__restrict__ row_loss, const int32_t *__restrict__ y, int T, int V,
           float *__restrict__ loss, const float *__restrict__ g, float *__restrict__ gscale) {
  __shared__ float ps[1024];
  __shared__ int pn[1024];
  float s = 0.f;
  int n = 0;
  for (int t = threadIdx.x; t < T; t += blockDim.x) {
    const int yv = y[t];
    if (yv >= 0 && yv < V) {
      ++n;
      if (row_loss) s += row_loss[t];
    }
  }
  ps[threadIdx.x] = s;
  pn[threadIdx.x] = n;
  __syncthreads();
  for (int w = blockDim.x >> 1; w > 0; w >>= 1) {
    if ((int)threadIdx.x < w) {
      ps[threadIdx.x] += ps[threadIdx.x + w];
      pn[threadIdx.x] += pn[threadIdx.x + w];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const int N = pn[0];
    if (loss) *loss = N > 0 ? ps[0] / (float)N : 0.f;
    if (gscale) *gscale = N > 0 ? *g / (float)N : 0.f;
  }
}

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

bool vec16(const void *p) { return ((uintptr_t)p & 15) == 0; }

// The tile width of a GEMM whose N is the hidden size: one that divides it
// if there is one, else 256 (ragged last tile).
int pick_bn(int64_t n) {
  if (n % 256 == 0) return 256;
  if (n % 224 == 0) return 224;
  if (n % 192 == 0) return 192;
  return 256;
}

template <int G, class Epi>
cudaError_t launch_group(int bn, tc::Group<Epi> &g, const DeviceInfo &dev, cudaStream_t s) {
  switch (bn) {
    case 256: return tc::launch_tc_gemm<256, G>(g, dev, s);
    case 224: return tc::launch_tc_gemm<224, G>(g, dev, s);
    case 192: return tc::launch_tc_gemm<192, G>(g, dev, s);
    default: return cudaErrorInvalidConfiguration;
  }
}

// Estimated tensor-core time of the backward with chunks of Cv columns, in
// k-steps of one CTA pair, for `pairs` persistent pairs: per chunk, the dz
// GEMM (waves of equal units) and the grouped dh + dW GEMM (units dealt
// round-robin: dh units of ceil(Cv/64) steps first, then dW units of
// ceil(T/64) steps; the busiest pair sets the time), plus a fixed cost per
// launch.  A unit is two 128-row tiles of one N-tile (tc_gemm.cuh).
double chunk_cost(int64_t T, int64_t H, int64_t Cv, int pairs) {
  constexpr double kLaunchSteps = 30.0;  // ~10 us of launch, fill and drain
  const int64_t mp = ((T + 127) / 128 + 1) / 2, kh = (H + 63) / 64;
  const int64_t grad_units = mp * ((Cv + kFwdBN - 1) / kFwdBN);
  const double grad = (double)((grad_units + pairs - 1) / pairs) * (double)kh;
  const int bn = pick_bn(H);
  const int64_t nt = (H + bn - 1) / bn;
  const int64_t n_dh = mp * nt, n_dw = (((Cv + 127) / 128 + 1) / 2) * nt, n = n_dh + n_dw;
  const double c_dh = (double)((Cv + 63) / 64) * bn / 256.0;
  const double c_dw = (double)((T + 63) / 64) * bn / 256.0;
  double worst = 0.0;
  for (int i = 0; i < pairs && i < n; ++i) {
    const int64_t mine = (n - i + pairs - 1) / pairs;                 // units i, i + pairs, ...
    const int64_t dh = i < n_dh ? (n_dh - i + pairs - 1) / pairs : 0;  // of them below n_dh
    const double t = (double)dh * c_dh + (double)(mine - dh) * c_dw;
    worst = t > worst ? t : worst;
  }
  return grad + worst + 2.0 * kLaunchSteps;
}

}  // namespace

// The backward's chunk width on a device with `sms` SMs: V rounded up to 64
// when it fits one chunk, else the multiple of 256 in [kChunkMin,
// kChunkMax] with the least estimated time (ties to the smaller chunk).
int64_t cce_bwd_chunk(int64_t T, int64_t H, int64_t V, int sms) {
  if (V <= kChunkMax) return round_up(V, 64);
  const int pairs = sms / 2 > 0 ? sms / 2 : 1;
  int64_t best = kChunkMin;
  double best_cost = 0.0;
  for (int64_t C = kChunkMin; C <= kChunkMax; C += 256) {
    const int64_t full = V / C, rest = V - full * C;
    double cost = (double)full * chunk_cost(T, H, C, pairs);
    if (rest) cost += chunk_cost(T, H, rest, pairs);
    if (C == kChunkMin || cost < best_cost) {
      best = C;
      best_cost = cost;
    }
  }
  return best;
}

// ------------------------------------------------------------ plain GEMM

cudaError_t launch_gemm_bf16(const void *a, int64_t lda, bool a_mn, const void *b, int64_t ldb,
                             bool b_mn, float *c, int64_t ldc, int64_t M, int64_t N, int64_t K,
                             const DeviceInfo &dev, cudaStream_t s) {
  const EpiStore st{c, nullptr, ldc, 0, (int)M, (int)N, false, vec16(c) && ldc % 4 == 0, false};
  const int bn = pick_bn(N);
  tc::Group<EpiStore> g;
  g.count = 1;
  cudaError_t e = tc::make_problem(g.p[0], bn, a, lda, b, ldb, (int)M, (int)N, (int)K,
                                   (a_mn ? tc::kAMn : 0) | (b_mn ? tc::kBMn : 0), st);
  if (e != cudaSuccess) return e;
  return launch_group<1>(bn, g, dev, s);
}

// ------------------------------------------------------------ workspaces

size_t cce_fwd_workspace_bytes(int64_t T, int64_t V) {
  const int64_t nparts = 2 * ((V + kFwdBN - 1) / kFwdBN);
  return (size_t)(round_up(T * nparts * 8, 256) + round_up(T * 4, 256) * 2);
}

size_t cce_bwd_workspace_bytes(int64_t T, int64_t H, int64_t V) {
  // room for the widest chunk pick_chunk may choose on any device
  const int64_t C = V <= kChunkMax ? round_up(V, 64) : kChunkMax;
  const int64_t bytes = 256                     // g / N
                        + round_up(T * C * 2, 256)  // dz of one chunk
                        + round_up(T * H, 64) * 4;  // dh in fp32
  return (size_t)bytes + 3 * 256;               // alignment of each piece
}

namespace {

struct Carve {
  unsigned char *p;
  template <class X> X *take(size_t bytes) {
    X *r = reinterpret_cast<X *>(p);
    p += (bytes + 255) / 256 * 256;
    return r;
  }
};

}  // namespace

cudaError_t launch_cce_fwd(const CceArgs &a, const DeviceInfo &dev, cudaStream_t s) {
  const int T = (int)a.T, H = (int)a.H, V = (int)a.V;
  const int nparts = 2 * ((V + kFwdBN - 1) / kFwdBN);  // two column halves per tile
  Carve w{(unsigned char *)a.ws};
  float2 *part = w.take<float2>((size_t)T * nparts * 8);
  float *tgt = w.take<float>((size_t)T * 4);
  float *row_loss = w.take<float>((size_t)T * 4);
  tc::Group<EpiLse> g;
  g.count = 1;
  cudaError_t e = tc::make_problem(g.p[0], kFwdBN, a.h, a.ldh, a.w, a.ldw, T, V, H, tc::kKMajor,
                                   EpiLse{a.y, T, V, nparts, part, tgt});
  if (e != cudaSuccess) return e;
  e = tc::launch_tc_gemm<kFwdBN, 1>(g, dev, s);
  if (e != cudaSuccess) return e;
  cce_row_lse<<<(T + 7) / 8, 256, 0, s>>>(part, nparts, tgt, a.y, T, V, a.lse, row_loss);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cce_finish<<<1, 1024, 0, s>>>(row_loss, a.y, T, V, a.loss, nullptr, nullptr);
  return cudaGetLastError();
}

// A second stream per device for the backward's dW GEMMs, and the events
// that order it against the caller's stream (created once, kept).
cudaError_t launch_cce_bwd(const CceArgs &a, const DeviceInfo &dev, cudaStream_t s) {
  const int T = (int)a.T, H = (int)a.H, V = (int)a.V;
  const int64_t C = cce_bwd_chunk(T, H, V, dev.sms);
  Carve w{(unsigned char *)a.ws};
  float *gscale = w.take<float>(256);
  bf16 *dz = w.take<bf16>((size_t)T * C * 2);
  float *dh32 = w.take<float>((size_t)round_up((int64_t)T * H, 64) * 4);

  cce_finish<<<1, 1024, 0, s>>>(nullptr, a.y, T, V, nullptr, a.dloss, gscale);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int bn_h = pick_bn(H);
  // Per chunk, two launches on the caller's stream: dz, then dh (+)= dz W_c
  // and dW_c = dz^T h as one grouped GEMM (their tiles fill each other's
  // partial waves).  Neither W nor h is ever transposed: the GEMMs that
  // need W_c^T, dz^T or h^T read them MN-major.
  for (int64_t c0 = 0; c0 < V; c0 += C) {
    const int Cv = (int)(V - c0 < C ? V - c0 : C);
    const bool first = c0 == 0, last = c0 + C >= V;
    const bf16 *wc = (const bf16 *)a.w + c0 * a.ldw;
    // dz [T x Cv] for columns [c0, c0 + Cv): A = h [T x H], B = W_c [Cv x H]
    tc::Group<EpiGrad> gg;
    gg.count = 1;
    e = tc::make_problem(gg.p[0], kFwdBN, a.h, a.ldh, wc, a.ldw, T, Cv, H, tc::kKMajor,
                         EpiGrad{a.y, a.lse, gscale, T, V, Cv, (int)c0, dz, C});
    if (e != cudaSuccess) return e;
    e = tc::launch_tc_gemm<kFwdBN, 1>(gg, dev, s);
    if (e != cudaSuccess) return e;
    tc::Group<EpiStore> gs;
    gs.count = 2;
    // dh (+)= dz W_c: A = dz [T x Cv] K-major; B = W_c^T, MN-major from
    // W_c [Cv x H]; K = Cv.  fp32 partial sums, bf16 from the last chunk.
    const EpiStore sh{dh32, last ? (bf16 *)a.dh : nullptr, (int64_t)H, a.lddh, T, H, !first,
                      H % 4 == 0, vec16(a.dh) && a.lddh % 8 == 0};
    e = tc::make_problem(gs.p[0], bn_h, dz, C, wc, a.ldw, T, H, Cv, tc::kBMn, sh);
    if (e != cudaSuccess) return e;
    // dW_c = dz^T h: A = dz^T, MN-major from dz [T x Cv]; B = h^T,
    // MN-major from h [T x H]; K = T
    const EpiStore sw{a.dw + c0 * a.lddw, nullptr, a.lddw, 0, Cv, H, false,
                      vec16(a.dw) && a.lddw % 4 == 0, false};
    e = tc::make_problem(gs.p[1], bn_h, dz, C, a.h, a.ldh, Cv, H, T, tc::kAMn | tc::kBMn, sw);
    if (e != cudaSuccess) return e;
    e = launch_group<2>(bn_h, gs, dev, s);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace ftk
