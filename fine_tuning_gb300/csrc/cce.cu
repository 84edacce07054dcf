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
// Backward, per vocabulary chunk of kChunk columns: a GEMM whose epilogue
// turns the recomputed logits into dz (bf16), written row-major and
// transposed (T kChunk bf16 each: 134 MB for 8,192 tokens, the ~135 MB the
// page quotes for its logits); then dh += dz W_c and dW_c = dz^T h as two
// more GEMMs with both
// operands K-major (W_c and h are transposed once by a plain kernel).  dh
// accumulates in fp32 and is rounded to bf16 by the last chunk's epilogue.
// The dW GEMMs run on a second stream with double-buffered chunk buffers,
// overlapping the next chunk's work and filling each launch's last wave.
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

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

constexpr int kChunk = 8192;     // vocabulary columns per backward chunk
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
  struct Row {
    float m, s;
    int y;
  };
  __device__ void begin(Row &r, int m, int) const {
    r.m = -INFINITY;
    r.s = 0.f;
    r.y = m < T ? y[m] : -1;
  }
  __device__ void slice(Row &r, int m, int n, const float (&x)[32]) const {
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
// stored as bf16 row-major [T][ldz] and transposed [Cv][ldzt].
struct EpiGrad {
  const int32_t *y;
  const float *lse, *gscale;
  int T, V, Cv, c0;
  bf16 *dz, *dzt;
  int64_t ldz, ldzt;
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
  __device__ void slice(Row &r, int m, int n, const float (&x)[32]) const {
    // every lane of the warp gets here (rows past T carry gs = 0): the
    // paired transposed stores below exchange values between lanes
    const bool ok = m < T;
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
    const bool full = n + 32 <= Cv;
    if (full && __all_sync(0xffffffffu, ok)) {
      bf16 *row = dz + (size_t)m * ldz + n;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        reinterpret_cast<uint4 *>(row)[q] =
            make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      // dz^T: lanes 2k and 2k + 1 hold rows m and m + 1 (consecutive); for
      // columns (2i, 2i + 1) the even lane writes column 2i and the odd lane
      // column 2i + 1, each as one 4-byte pair of rows, after swapping the
      // value the other one needs
      const bool odd = (threadIdx.x & 1) != 0;
      unsigned short *col = reinterpret_cast<unsigned short *>(dzt);
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const uint32_t lo = pk[i] & 0xFFFFu, hi = pk[i] >> 16;  // columns 2i, 2i + 1
        const uint32_t got = __shfl_xor_sync(0xffffffffu, odd ? lo : hi, 1);
        const uint32_t pair = odd ? (got | (hi << 16)) : (lo | (got << 16));
        const int c = n + 2 * i + (odd ? 1 : 0);
        *reinterpret_cast<uint32_t *>(col + (size_t)c * ldzt + (m & ~1)) = pair;
      }
    } else if (ok) {
      unsigned short *rs = reinterpret_cast<unsigned short *>(dz + (size_t)m * ldz + n);
      unsigned short *col = reinterpret_cast<unsigned short *>(dzt) + (size_t)n * ldzt + m;
      for (int e = 0; e < 32 && n + e < Cv; ++e) {
        const unsigned short v = (unsigned short)(pk[e >> 1] >> (16 * (e & 1)));
        rs[e] = v;
        col[(size_t)e * ldzt] = v;
      }
    }
  }
  __device__ void end(Row &, int, int, int) const {}
};

// Plain output: C[m][n] (+= the fp32 value already there), written as fp32
// or rounded to bf16.
struct EpiStore {
  float *c;         // fp32 [M][ldc]: read when acc_in, written unless cb
  bf16 *cb;         // nullable: write bf16 [M][ldcb] instead
  int64_t ldc, ldcb;
  int M, N;
  bool acc_in;
  bool vc, vb;      // 16-byte vector access is aligned for c / cb (base and stride)
  struct Row {};
  __device__ void begin(Row &, int, int) const {}
  __device__ void slice(Row &, int m, int n, const float (&x)[32]) const {
    if (m >= M) return;
    float v[32];
    const float *src = c + (size_t)m * ldc + n;
    const bool full = n + 32 <= N;
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = x[e];
    if (acc_in) {
      if (full && vc) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 a = reinterpret_cast<const float4 *>(src)[q];
          v[4 * q] += a.x;
          v[4 * q + 1] += a.y;
          v[4 * q + 2] += a.z;
          v[4 * q + 3] += a.w;
        }
      } else {
        for (int e = 0; e < 32 && n + e < N; ++e) v[e] += src[e];
      }
    }
    if (cb) {
      bf16 *dst = cb + (size_t)m * ldcb + n;
      __align__(16) bf16 o[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) o[e] = __float2bfloat16_rn(v[e]);
      if (full && vb) {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          reinterpret_cast<uint4 *>(dst)[q] = reinterpret_cast<const uint4 *>(o)[q];
      } else {
        for (int e = 0; e < 32 && n + e < N; ++e) dst[e] = o[e];
      }
    } else {
      float *dst = c + (size_t)m * ldc + n;
      if (full && vc) {
#pragma unroll
        for (int q = 0; q < 8; ++q)
          reinterpret_cast<float4 *>(dst)[q] =
              make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
      } else {
        for (int e = 0; e < 32 && n + e < N; ++e) dst[e] = v[e];
      }
    }
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

// out[c][r] = in[r][c] for r < R, c < C (bf16), 32 x 32 tiles via shared memory.
__global__ void __launch_bounds__(256)
transpose_bf16(const bf16 *__restrict__ in, int64_t ldi, int R, int C, bf16 *__restrict__ out,
               int64_t ldo) {
  __shared__ bf16 tile[32][34];
  const int r0 = blockIdx.y * 32, c0 = blockIdx.x * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  for (int i = ty; i < 32; i += 8) {
    const int r = r0 + i, c = c0 + tx;
    if (r < R && c < C) tile[i][tx] = in[(size_t)r * ldi + c];
  }
  __syncthreads();
  for (int i = ty; i < 32; i += 8) {
    const int c = c0 + i, r = r0 + tx;
    if (r < R && c < C) out[(size_t)c * ldo + r] = tile[tx][i];
  }
}

cudaError_t transpose(const bf16 *in, int64_t ldi, int R, int C, bf16 *out, int64_t ldo,
                      cudaStream_t s) {
  if (R == 0 || C == 0) return cudaSuccess;
  const dim3 grid((unsigned)((C + 31) / 32), (unsigned)((R + 31) / 32));
  transpose_bf16<<<grid, 256, 0, s>>>(in, ldi, R, C, out, ldo);
  return cudaGetLastError();
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

template <class Epi>
cudaError_t gemm_bn(int bn, const CUtensorMap &ta, const void *b_base, int64_t b_rows,
                    int64_t b_cols, int64_t ldb, int M, int N, int K, const Epi &epi,
                    const DeviceInfo &dev, cudaStream_t s) {
  alignas(64) CUtensorMap tb;
  cudaError_t e = tc::make_tmap_bf16(&tb, b_base, b_rows, b_cols, ldb, bn);
  if (e != cudaSuccess) return e;
  switch (bn) {
    case 256: return tc::launch_tc_gemm<256>(ta, tb, M, N, K, epi, dev, s);
    case 224: return tc::launch_tc_gemm<224>(ta, tb, M, N, K, epi, dev, s);
    case 192: return tc::launch_tc_gemm<192>(ta, tb, M, N, K, epi, dev, s);
    default: return cudaErrorInvalidConfiguration;
  }
}

}  // namespace

// ------------------------------------------------------------ plain GEMM

cudaError_t launch_gemm_bf16(const void *a, int64_t lda, const void *b, int64_t ldb, float *c,
                             int64_t ldc, int64_t M, int64_t N, int64_t K, const DeviceInfo &dev,
                             cudaStream_t s) {
  alignas(64) CUtensorMap ta;
  cudaError_t e = tc::make_tmap_bf16(&ta, a, M, K, lda, tc::BM);
  if (e != cudaSuccess) return e;
  EpiStore st{c, nullptr, ldc, 0, (int)M, (int)N, false, vec16(c) && ldc % 4 == 0, false};
  return gemm_bn(pick_bn(N), ta, b, N, K, ldb, (int)M, (int)N, (int)K, st, dev, s);
}

// ------------------------------------------------------------ workspaces

size_t cce_fwd_workspace_bytes(int64_t T, int64_t V) {
  const int64_t nparts = 2 * ((V + kFwdBN - 1) / kFwdBN);
  return (size_t)(round_up(T * nparts * 8, 256) + round_up(T * 4, 256) * 2);
}

size_t cce_bwd_workspace_bytes(int64_t T, int64_t H, int64_t V) {
  const int64_t C = V < kChunk ? round_up(V, 64) : kChunk;
  const int64_t ldt = round_up(T, 64);
  const int64_t bytes = 256                   // g / N
                        + H * ldt * 2         // h^T
                        + 2 * H * C * 2       // W_c^T, two buffers
                        + 2 * T * C * 2       // dz, two buffers
                        + 2 * C * ldt * 2     // dz^T, two buffers
                        + round_up(T * H, 64) * 4;  // dh in fp32
  return (size_t)bytes + 9 * 256;             // alignment of each piece
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
  alignas(64) CUtensorMap ta;
  cudaError_t e = tc::make_tmap_bf16(&ta, a.h, T, H, a.ldh, tc::BM);
  if (e != cudaSuccess) return e;
  EpiLse epi{a.y, T, V, nparts, part, tgt};
  e = gemm_bn(kFwdBN, ta, a.w, V, H, a.ldw, T, V, H, epi, dev, s);
  if (e != cudaSuccess) return e;
  cce_row_lse<<<(T + 7) / 8, 256, 0, s>>>(part, nparts, tgt, a.y, T, V, a.lse, row_loss);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  cce_finish<<<1, 1024, 0, s>>>(row_loss, a.y, T, V, a.loss, nullptr, nullptr);
  return cudaGetLastError();
}

// A second stream per device for the backward's dW GEMMs, and the events
// that order it against the caller's stream (created once, kept).
struct SideStream {
  cudaStream_t s = nullptr;
  cudaEvent_t ready[2] = {}, done[2] = {};
};

cudaError_t side_stream(int device, SideStream **out) {
  static std::mutex mu;
  static SideStream side[64];
  if (device < 0 || device >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  SideStream &x = side[device];
  if (!x.s) {
    cudaError_t e = cudaStreamCreateWithFlags(&x.s, cudaStreamNonBlocking);
    for (int b = 0; e == cudaSuccess && b < 2; ++b) {
      e = cudaEventCreateWithFlags(&x.ready[b], cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&x.done[b], cudaEventDisableTiming);
    }
    if (e != cudaSuccess) {
      x.s = nullptr;
      return e;
    }
  }
  *out = &x;
  return cudaSuccess;
}

cudaError_t launch_cce_bwd(const CceArgs &a, const DeviceInfo &dev, cudaStream_t s) {
  const int T = (int)a.T, H = (int)a.H, V = (int)a.V;
  const int64_t C = V < kChunk ? round_up(V, 64) : kChunk;
  const int64_t ldt = round_up(T, 64);
  Carve w{(unsigned char *)a.ws};
  float *gscale = w.take<float>(256);
  bf16 *ht = w.take<bf16>((size_t)H * ldt * 2);
  bf16 *wt[2], *dz[2], *dzt[2];
  for (int b = 0; b < 2; ++b) {
    wt[b] = w.take<bf16>((size_t)H * C * 2);
    dz[b] = w.take<bf16>((size_t)T * C * 2);
    dzt[b] = w.take<bf16>((size_t)C * ldt * 2);
  }
  float *dh32 = w.take<float>((size_t)round_up((int64_t)T * H, 64) * 4);
  SideStream *side = nullptr;
  cudaError_t e = side_stream(dev.device, &side);
  if (e != cudaSuccess) return e;

  cce_finish<<<1, 1024, 0, s>>>(nullptr, a.y, T, V, nullptr, a.dloss, gscale);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  e = transpose((const bf16 *)a.h, a.ldh, T, H, ht, ldt, s);
  if (e != cudaSuccess) return e;
  alignas(64) CUtensorMap th, tdz, tdzt;
  e = tc::make_tmap_bf16(&th, a.h, T, H, a.ldh, tc::BM);
  if (e != cudaSuccess) return e;
  const int bn_h = pick_bn(H);
  // chunk c uses buffer c & 1: the caller's stream makes dz, dz^T and W_c^T
  // and runs dh; the side stream runs dW_c once the chunk's buffers are
  // ready, overlapping dh(c) and the next chunk's dz; a buffer is reused
  // only after its dW has read it.  Only events recorded in this call are
  // waited on, so the whole sequence can be captured into a graph.
  bool pending[2] = {false, false};
  int c = 0;
  for (int64_t c0 = 0; c0 < V; c0 += C, ++c) {
    const int b = c & 1;
    const int Cv = (int)(V - c0 < C ? V - c0 : C);
    const bool first = c0 == 0, last = c0 + C >= V;
    const bf16 *wc = (const bf16 *)a.w + c0 * a.ldw;
    if (pending[b]) {
      e = cudaStreamWaitEvent(s, side->done[b], 0);
      if (e != cudaSuccess) return e;
    }
    // dz for columns [c0, c0 + Cv)
    EpiGrad g{a.y, a.lse, gscale, T, V, Cv, (int)c0, dz[b], dzt[b], C, ldt};
    e = gemm_bn(kFwdBN, th, wc, Cv, H, a.ldw, T, Cv, H, g, dev, s);
    if (e != cudaSuccess) return e;
    e = transpose(wc, a.ldw, Cv, H, wt[b], C, s);
    if (e != cudaSuccess) return e;
    e = cudaEventRecord(side->ready[b], s);
    if (e != cudaSuccess) return e;
    // dW_c = dz^T h on the side stream: A = dz^T [Cv x T], B = h^T [H x T]
    e = cudaStreamWaitEvent(side->s, side->ready[b], 0);
    if (e != cudaSuccess) return e;
    e = tc::make_tmap_bf16(&tdzt, dzt[b], Cv, T, ldt, tc::BM);
    if (e != cudaSuccess) return e;
    EpiStore sw{a.dw + c0 * a.lddw, nullptr, a.lddw, 0, Cv, H, false,
                vec16(a.dw) && a.lddw % 4 == 0, false};
    e = gemm_bn(bn_h, tdzt, ht, H, T, ldt, Cv, H, T, sw, dev, side->s);
    if (e != cudaSuccess) return e;
    e = cudaEventRecord(side->done[b], side->s);
    if (e != cudaSuccess) return e;
    pending[b] = true;
    // dh (+)= dz W_c on the caller's stream: A = dz [T x Cv], B = W_c^T [H x Cv]
    e = tc::make_tmap_bf16(&tdz, dz[b], T, Cv, C, tc::BM);
    if (e != cudaSuccess) return e;
    EpiStore sh{dh32, last ? (bf16 *)a.dh : nullptr, (int64_t)H, a.lddh, T, H, !first,
                H % 4 == 0, vec16(a.dh) && a.lddh % 8 == 0};
    e = gemm_bn(bn_h, tdz, wt[b], H, Cv, C, T, H, Cv, sh, dev, s);
    if (e != cudaSuccess) return e;
  }
  // join: the caller's stream waits for every dW still in flight
  for (int b = 0; b < 2; ++b)
    if (pending[b]) {
      e = cudaStreamWaitEvent(s, side->done[b], 0);
      if (e != cudaSuccess) return e;
    }
  return cudaSuccess;
}

}  // namespace ftk
