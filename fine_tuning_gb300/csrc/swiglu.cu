// SwiGLU forward and backward, elementwise over T rows of I features
// (Chronicals, arXiv 2601.02609, abstract, optimisation (1): fused SwiGLU;
// the page gives no formula, these are the standard definitions):
//   forward:   h  = silu(g) * u = g * s * u,   s = sigmoid(g) = 1 / (1 + e^-g)
//   backward:  dg = dh * u * s * (1 + g * (1 - s)),   du = dh * g * s
// The backward can also re-emit h (EMIT_H), computed exactly as the forward
// computes it, for a caller that keeps g and u but not h (the down
// projection's weight gradient needs h); that costs one extra write instead
// of storing h in the forward and reading it back.
//
// Every input element is read once and every output written once.  A thread
// moves U 16-byte packets of each operand per launch, all loads issued before
// any arithmetic so that U * (operands) packets are in flight per thread.
// Rows may be strided (ld >= I) so a fused [T, 2I] gate_up buffer can be
// passed as two views; the contiguous case skips the row arithmetic.
#include "common.cuh"
#include "launch.h"

namespace ftk {

namespace {

constexpr int kThreads = 256;

// sigmoid(g) and 1 - sigmoid(g) from e = exp(-|g|), which never overflows:
// for g >= 0, s = 1/(1+e) and 1-s = e/(1+e); for g < 0 the two swap.  Both
// stay accurate where the other form would round to 0 or 1.
// fp32 storage uses expf and the correctly rounded reciprocal; bf16 storage
// (8 significant bits) uses the hardware approximations __expf and
// __fdividef, whose ~1e-6 relative error is far below bf16's 2^-9, at a
// third of the instructions (the forward pass is otherwise issue-bound).
template <typename T>
__device__ __forceinline__ void sigmoid2(float g, float *s, float *one_minus_s) {
  float e, r;
  if constexpr (sizeof(T) == 4) {
    e = expf(-fabsf(g));
    r = __frcp_rn(1.0f + e);
  } else {
    e = __expf(-fabsf(g));
    r = __fdividef(1.0f, 1.0f + e);  // 1 + e lies in (1, 2]
  }
  const float er = e * r;
  *s = g >= 0.0f ? r : er;
  *one_minus_s = g >= 0.0f ? er : r;
}

// Packet v of a [rows, ip packets] view -> element offset in a row-strided buffer.
template <typename Idx, int N, bool CONTIG>
__device__ __forceinline__ Idx packet_offset(Idx v, Idx ip, Idx ld) {
  if (CONTIG) return v * N;
  const Idx row = v / ip;
  return row * ld + (v - row * ip) * N;
}

template <typename T, typename Idx, int N, int U, bool CONTIG>
__global__ void __launch_bounds__(kThreads)
swiglu_fwd_kernel(const T *g, const T *u, Idx ld_gu, T *h, Idx ld_h, Idx npk, Idx ip) {
  pdl_wait();
  pdl_trigger();
  const Idx base = (Idx)blockIdx.x * (kThreads * U) + threadIdx.x;
  Packet<T, N> gv[U], uv[U];
#pragma unroll
  for (int k = 0; k < U; ++k) {
    const Idx v = base + k * kThreads;
    if (v < npk) {
      const Idx o = packet_offset<Idx, N, CONTIG>(v, ip, ld_gu);
      gv[k] = load_packet_stream<T, N>(g + o);
      uv[k] = load_packet_stream<T, N>(u + o);
    }
  }
#pragma unroll
  for (int k = 0; k < U; ++k) {
    const Idx v = base + k * kThreads;
    if (v < npk) {
      Packet<T, N> o;
      auto h_of = [&](int e) {
        const float gf = gv[k].get(e);
        float sg, sc;
        sigmoid2<T>(gf, &sg, &sc);
        return gf * sg * uv[k].get(e);
      };
      if constexpr (N % 2 == 0) {
#pragma unroll
        for (int e = 0; e < N; e += 2) o.set2(e, h_of(e), h_of(e + 1));
      } else {
#pragma unroll
        for (int e = 0; e < N; ++e) o.set(e, h_of(e));
      }
      store_packet<T, N>(h + packet_offset<Idx, N, CONTIG>(v, ip, ld_h), o);
    }
  }
}

template <typename T, typename Idx, int N, int U, bool CONTIG, bool EMIT_H>
__global__ void __launch_bounds__(kThreads)
swiglu_bwd_kernel(const T *dh, Idx ld_dh, const T *g, const T *u, Idx ld_gu, T *dg, T *du,
                  Idx ld_dgu, T *h, Idx ld_h, Idx npk, Idx ip) {
  pdl_wait();
  pdl_trigger();
  const Idx base = (Idx)blockIdx.x * (kThreads * U) + threadIdx.x;
  Packet<T, N> hv[U], gv[U], uv[U];
#pragma unroll
  for (int k = 0; k < U; ++k) {
    const Idx v = base + k * kThreads;
    if (v < npk) {
      const Idx o = packet_offset<Idx, N, CONTIG>(v, ip, ld_gu);
      hv[k] = load_packet_stream<T, N>(dh + packet_offset<Idx, N, CONTIG>(v, ip, ld_dh));
      gv[k] = load_packet_stream<T, N>(g + o);
      uv[k] = load_packet_stream<T, N>(u + o);
    }
  }
#pragma unroll
  for (int k = 0; k < U; ++k) {
    const Idx v = base + k * kThreads;
    if (v < npk) {
      Packet<T, N> og, ou, oh;
      float dgv[N], duv[N], hv_out[N];
#pragma unroll
      for (int e = 0; e < N; ++e) {
        const float gf = gv[k].get(e), uf = uv[k].get(e), hf = hv[k].get(e);
        float s, sc;
        sigmoid2<T>(gf, &s, &sc);
        dgv[e] = hf * uf * (s * fmaf(gf, sc, 1.0f));
        duv[e] = hf * (gf * s);
        if (EMIT_H) hv_out[e] = gf * s * uf;  // the forward's expression
      }
      if constexpr (N % 2 == 0) {
#pragma unroll
        for (int e = 0; e < N; e += 2) {
          og.set2(e, dgv[e], dgv[e + 1]);
          ou.set2(e, duv[e], duv[e + 1]);
          if (EMIT_H) oh.set2(e, hv_out[e], hv_out[e + 1]);
        }
      } else {
#pragma unroll
        for (int e = 0; e < N; ++e) {
          og.set(e, dgv[e]);
          ou.set(e, duv[e]);
          if (EMIT_H) oh.set(e, hv_out[e]);
        }
      }
      const Idx o = packet_offset<Idx, N, CONTIG>(v, ip, ld_dgu);
      store_packet<T, N>(dg + o, og);
      store_packet<T, N>(du + o, ou);
      if (EMIT_H) store_packet<T, N>(h + packet_offset<Idx, N, CONTIG>(v, ip, ld_h), oh);
    }
  }
}

template <typename T, typename Idx, int N, int U, bool CONTIG>
cudaError_t fwd_launch(const SwigluFwdArgs &a, cudaStream_t s) {
  const Idx ip = (Idx)(a.I / N);
  const Idx npk = (Idx)a.T * ip;
  const int64_t grid = ceil_div((int64_t)npk, (int64_t)kThreads * U);
  {
    cudaError_t le_ = launch_pdl(swiglu_fwd_kernel<T, Idx, N, U, CONTIG>, dim3((unsigned)grid), dim3(kThreads), 0, s,
                                 (const T *)a.g, (const T *)a.u, (Idx)a.ld_gu, (T *)a.h, (Idx)a.ld_h, npk, ip);
    if (le_ != cudaSuccess) return le_;
  }
  return cudaGetLastError();
}

template <typename T, typename Idx, int N, int U, bool CONTIG, bool EMIT_H>
cudaError_t bwd_launch_form(const SwigluBwdArgs &a, cudaStream_t s) {
  const Idx ip = (Idx)(a.I / N);
  const Idx npk = (Idx)a.T * ip;
  const int64_t grid = ceil_div((int64_t)npk, (int64_t)kThreads * U);
  cudaError_t e = launch_pdl(swiglu_bwd_kernel<T, Idx, N, U, CONTIG, EMIT_H>,
                             dim3((unsigned)grid), dim3(kThreads), 0, s, (const T *)a.dh,
                             (Idx)a.ld_dh, (const T *)a.g, (const T *)a.u, (Idx)a.ld_gu,
                             (T *)a.dg, (T *)a.du, (Idx)a.ld_dgu, (T *)a.h, (Idx)a.ld_h, npk, ip);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <typename T, typename Idx, int N, int U, bool CONTIG>
cudaError_t bwd_launch(const SwigluBwdArgs &a, cudaStream_t s) {
  return a.h ? bwd_launch_form<T, Idx, N, U, CONTIG, true>(a, s)
             : bwd_launch_form<T, Idx, N, U, CONTIG, false>(a, s);
}

}  // namespace

cudaError_t launch_swiglu_fwd(DType dt, bool vec, bool wide, const SwigluFwdArgs &a,
                              const DeviceInfo &, cudaStream_t s) {
  constexpr int U = 4;
  const bool contig = a.ld_gu == a.I && a.ld_h == a.I;
#define FTK_SWIGLU_FWD(T, Idx)                                                     \
  if (vec) {                                                                       \
    constexpr int NV = VecWidth<T>::value;                                         \
    return contig ? fwd_launch<T, Idx, NV, U, true>(a, s)                          \
                  : fwd_launch<T, Idx, NV, U, false>(a, s);                        \
  }                                                                                \
  return contig ? fwd_launch<T, Idx, 1, U, true>(a, s) : fwd_launch<T, Idx, 1, U, false>(a, s);
  if (dt == DType::F32) {
    if (wide) { FTK_SWIGLU_FWD(float, int64_t) }
    FTK_SWIGLU_FWD(float, int32_t)
  }
  if (wide) { FTK_SWIGLU_FWD(bf16, int64_t) }
  FTK_SWIGLU_FWD(bf16, int32_t)
#undef FTK_SWIGLU_FWD
}

cudaError_t launch_swiglu_bwd(DType dt, bool vec, bool wide, const SwigluBwdArgs &a,
                              const DeviceInfo &, cudaStream_t s) {
  constexpr int U = 2;
  const bool contig =
      a.ld_dh == a.I && a.ld_gu == a.I && a.ld_dgu == a.I && (!a.h || a.ld_h == a.I);
#define FTK_SWIGLU_BWD(T, Idx)                                                     \
  if (vec) {                                                                       \
    constexpr int NV = VecWidth<T>::value;                                         \
    return contig ? bwd_launch<T, Idx, NV, U, true>(a, s)                          \
                  : bwd_launch<T, Idx, NV, U, false>(a, s);                        \
  }                                                                                \
  return contig ? bwd_launch<T, Idx, 1, U, true>(a, s) : bwd_launch<T, Idx, 1, U, false>(a, s);
  if (dt == DType::F32) {
    if (wide) { FTK_SWIGLU_BWD(float, int64_t) }
    FTK_SWIGLU_BWD(float, int32_t)
  }
  if (wide) { FTK_SWIGLU_BWD(bf16, int64_t) }
  FTK_SWIGLU_BWD(bf16, int32_t)
#undef FTK_SWIGLU_BWD
}

}  // namespace ftk
