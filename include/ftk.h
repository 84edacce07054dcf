/*
 * ftk.h: C ABI of the fused per-token layer ops of LLM fine-tuning
 * (RMSNorm, SwiGLU, in-place varlen QK-RoPE; forward and backward),
 * implemented as hand-written CUDA kernels for GB300 (sm_103a).
 *
 * Where each op comes from:
 *   - "Chronicals: A High-Performance Framework for LLM Fine-Tuning with
 *     3.51x Speedup over Unsloth" (arXiv 2601.02609), abstract,
 *     optimisation (1): fused RMSNorm, SwiGLU and QK-RoPE kernels that cut
 *     memory traffic.  The page names the ops but prints no formula; the
 *     standard definitions written beside each call below are used.
 *   - "Unsloth prétend accélérer 5 fois l'entraînement des LLM avec de
 *     nouveaux noyaux Triton et un auto-packing" (seventnews.com): the
 *     paragraph on the fused QK RoPE kernel (Q and K rotated by ONE kernel,
 *     in place, variable-length sequences), the paragraph on LONG_INDEXING
 *     (64-bit offsets for 500k-token contexts) and the paragraph on
 *     auto-packing (one 1-D token tensor plus sequence-length metadata).
 *   - "Unsloth und NVIDIA optimieren LLM-Training um zusätzliche 25%"
 *     (lumeric.app), item (1): packed-sequence metadata kept on the device so
 *     no GPU-to-CPU synchronisation is needed; these calls read cu_seqlens on
 *     the device and never synchronise.
 *
 * Conventions shared by every call:
 *   - Pointers without a "host" note are DEVICE pointers.  The caller owns
 *     every buffer; the library never allocates, frees or keeps a buffer.
 *   - Every call is asynchronous on `stream` (NULL = the legacy default
 *     stream) and never synchronises the host.
 *   - Argument errors are detected on the host before anything is launched
 *     and returned as a status; nothing is written then.  A failed launch
 *     returns FTK_ERR_CUDA (the CUDA error text is kept per thread, see
 *     ftk_last_cuda_error).
 *   - Storage dtype is FTK_F32 or FTK_BF16; arithmetic is always fp32, bf16
 *     results are rounded to nearest even once on store.
 *   - Tensors are row-major.  A row stride `ld*` counts ELEMENTS between the
 *     starts of consecutive token rows; it must be >= the row length.
 *   - Element offsets switch from 32-bit to 64-bit arithmetic automatically
 *     when any offset reached by a call can exceed 2^31 - 1.
 *   - 16-byte aligned pointers, and row lengths and strides that are a
 *     multiple of 16 bytes, take the vectorised kernels; anything else takes
 *     the element-wise kernels (still on the GPU, same results).
 *   - T = 0 (or I = 0) is a valid empty call: FTK_OK, nothing launched.
 */
#ifndef FTK_H_
#define FTK_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FTK_API __attribute__((visibility("default")))
#else
#define FTK_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* the CUDA runtime's cudaStream_t is `struct CUstream_st *` */
typedef struct CUstream_st *ftk_stream_t;

typedef enum {
    FTK_OK = 0,
    FTK_ERR_NULL = 1,      /* a required pointer is NULL */
    FTK_ERR_SHAPE = 2,     /* a size or stride is negative / inconsistent */
    FTK_ERR_ALIGN = 3,     /* a pointer is not aligned to its element size */
    FTK_ERR_DTYPE = 4,     /* unknown dtype */
    FTK_ERR_WORKSPACE = 5, /* workspace missing or smaller than required */
    FTK_ERR_CUDA = 6,      /* a CUDA call failed (see ftk_last_cuda_error) */
    FTK_ERR_ALIAS = 7      /* two buffers overlap where that is not allowed */
} ftk_status;

typedef enum { FTK_F32 = 0, FTK_BF16 = 1 } ftk_dtype;

/* ------------------------------------------------------------- RMSNorm */

/* Forward RMSNorm of T token rows of H features ("Chronicals", arXiv
 * 2601.02609, abstract, optimisation (1): the fused RMSNorm kernel, one of
 * the three fusions that remove most of the step's memory traffic; the page
 * names the op, the formula is the standard RMSNorm):
 *   r[t]   = 1 / sqrt( (1/H) sum_j x[t,j]^2 + eps )
 *   y[t,j] = x[t,j] * r[t] * w[j]
 * x [T, ldx], y [T, ldy] (dtype), w [H] (dtype, contiguous),
 * rstd [T] fp32 contiguous, nullable: receives r[t] for the backward pass.
 * y may alias x exactly (ldy == ldx) for an in-place norm. */
FTK_API ftk_status ftk_rmsnorm_fwd(const void *x, int64_t ldx, const void *w, void *y,
                           int64_t ldy, float *rstd, int64_t T, int64_t H,
                           float eps, ftk_dtype dtype, ftk_stream_t stream);

/* Bytes of device workspace ftk_rmsnorm_bwd needs for T rows of H features
 * of `dtype` on the CURRENT device (it depends on the device's SM count).
 * Returns 0 when T or H is 0 or the arguments are invalid. */
FTK_API size_t ftk_rmsnorm_bwd_workspace_bytes(int64_t T, int64_t H,
                                               ftk_dtype dtype);

/* Backward RMSNorm (gradient of sum(dy * y) for the forward above; the
 * backward half of the fused RMSNorm of "Chronicals", arXiv 2601.02609,
 * abstract, optimisation (1)):
 *   c[t]    = sum_j dy[t,j] w[j] x[t,j]
 *   dx[t,j] = r[t] w[j] dy[t,j] - r[t]^3 x[t,j] c[t] / H
 *   dw[j]   = sum_t dy[t,j] x[t,j] r[t]          (fp32, OVERWRITTEN)
 * dy [T, lddy], x [T, ldx], dx [T, lddx] (dtype); w [H] (dtype); dw [H]
 * fp32; rstd [T] fp32 from the forward pass, or NULL to recompute r from x
 * and eps.  workspace: >= ftk_rmsnorm_bwd_workspace_bytes(T, H, dtype) bytes,
 * 16-byte aligned, contents ignored and clobbered.  dw is the sum of
 * per-CTA fp32 partials reduced in a fixed order by a second kernel, so it
 * is bitwise reproducible run to run on the same device.  dx may alias dy
 * exactly (same pointer and stride). */
FTK_API ftk_status ftk_rmsnorm_bwd(const void *dy, int64_t lddy, const void *x,
                           int64_t ldx, const void *w, const float *rstd,
                           void *dx, int64_t lddx, float *dw, void *workspace,
                           size_t workspace_bytes, int64_t T, int64_t H,
                           float eps, ftk_dtype dtype, ftk_stream_t stream);

/* Same operation, arguments and results as ftk_rmsnorm_bwd, for callers
 * that cannot allocate device memory (for example code that runs inside a
 * fixed memory pool or a runtime that forbids cudaMalloc after start-up, or
 * a plugin that is handed only input and output pointers).  The pages have
 * no counterpart: it exists for those callers only.  Instead of a workspace
 * it uses a 4 MiB scratch array built into the library (held by every device
 * that loads the library until the process exits); it allocates nothing.
 *   - H must be <= 1,048,576 (one row of fp32 partial sums must fit in the
 *     scratch), else FTK_ERR_WORKSPACE; larger H values leave fewer partial
 *     rows, hence fewer CTAs, than ftk_rmsnorm_bwd would use.
 *   - The first call on a device looks up the scratch array's device
 *     address and caches it; make that first call before any stream
 *     capture.
 *   - Every call on a device shares the scratch and leaves its contents
 *     behind; nothing in it needs clearing (each call writes every partial
 *     row it sums).  Calls that overlap on the GPU race on it: serialise
 *     them. */
FTK_API ftk_status ftk_rmsnorm_bwd_noalloc(const void *dy, int64_t lddy, const void *x,
                                           int64_t ldx, const void *w, const float *rstd,
                                           void *dx, int64_t lddx, float *dw, int64_t T,
                                           int64_t H, float eps, ftk_dtype dtype,
                                           ftk_stream_t stream);

/* Forward RMSNorm with the pre-norm block's residual add fused in front
 * (the variant of optimisation (1) of "Chronicals", arXiv 2601.02609,
 * abstract, in which the norm also performs the add of the residual stream
 * that precedes it; the page prints no formula):
 *   h[t,j] = x[t,j] + res[t,j]    added in fp32, rounded to dtype, STORED
 *   then ftk_rmsnorm_fwd of h:  r[t] from h,  y[t,j] = h[t,j] * r[t] * w[j]
 * The norm reads the stored (rounded) h, so the results equal a separate add
 * followed by ftk_rmsnorm_fwd, bit for bit.  x [T, ldx], res [T, ldr],
 * h [T, ldh], y [T, ldy] (dtype); w [H] (dtype); rstd [T] fp32, nullable.
 * h may alias x or res exactly (same pointer and stride) to update the
 * residual stream in place; y must not overlap any other argument.
 * Each row of x and res is read once and h, y written once. */
FTK_API ftk_status ftk_rmsnorm_add_fwd(const void *x, int64_t ldx, const void *res,
                                       int64_t ldr, const void *w, void *h, int64_t ldh,
                                       void *y, int64_t ldy, float *rstd, int64_t T,
                                       int64_t H, float eps, ftk_dtype dtype,
                                       ftk_stream_t stream);

/* Backward of ftk_rmsnorm_add_fwd.  The gradient reaching h is dh (from the
 * later users of the residual stream) plus the norm's backward at h; it is
 * the gradient of x and of res alike, returned once as dx:
 *   c[t]    = sum_j dy[t,j] w[j] h[t,j]
 *   dx[t,j] = dh[t,j] + r[t] w[j] dy[t,j] - r[t]^3 h[t,j] c[t] / H
 *   dw[j]   = sum_t dy[t,j] h[t,j] r[t]          (fp32, OVERWRITTEN)
 * dy [T, lddy], dh [T, lddh], h [T, ldh] (the forward's stored h),
 * dx [T, lddx] (dtype); w, rstd, dw, workspace and the workspace size as in
 * ftk_rmsnorm_bwd (ftk_rmsnorm_bwd_workspace_bytes gives it; rstd NULL
 * recomputes r from h).  dx may alias dy or dh exactly; it must not overlap
 * h, w, rstd, dw or the workspace.  dw is bitwise reproducible run to run. */
FTK_API ftk_status ftk_rmsnorm_add_bwd(const void *dy, int64_t lddy, const void *dh,
                                       int64_t lddh, const void *h, int64_t ldh,
                                       const void *w, const float *rstd, void *dx,
                                       int64_t lddx, float *dw, void *workspace,
                                       size_t workspace_bytes, int64_t T, int64_t H,
                                       float eps, ftk_dtype dtype, ftk_stream_t stream);

/* -------------------------------------------------------------- SwiGLU */

/* Forward SwiGLU, elementwise over T rows of I features ("Chronicals",
 * arXiv 2601.02609, abstract, optimisation (1): the fused SwiGLU kernel;
 * the page names the op, the formula is the standard gated SiLU):
 *   h = silu(g) * u = g * sigmoid(g) * u,   sigmoid(g) = 1 / (1 + e^-g)
 * g, u: [T, ld_gu] (so a fused [T, 2I] gate_up projection can be passed as
 * g = gu, u = gu + I, ld_gu = 2I); h: [T, ld_h]. */
FTK_API ftk_status ftk_swiglu_fwd(const void *g, const void *u, int64_t ld_gu, void *h,
                          int64_t ld_h, int64_t T, int64_t I, ftk_dtype dtype,
                          ftk_stream_t stream);

/* Backward SwiGLU (gradient of sum(dh * h); the backward half of the fused
 * SwiGLU of "Chronicals", arXiv 2601.02609, abstract, optimisation (1)),
 * s = sigmoid(g):
 *   dg = dh * u * s * (1 + g * (1 - s)),   du = dh * g * s
 * dh: [T, ld_dh]; g, u: [T, ld_gu]; dg, du: [T, ld_dgu].  dg may alias g and
 * du may alias u exactly (same pointer, ld_dgu == ld_gu): every element is
 * read before it is written by the same thread. */
FTK_API ftk_status ftk_swiglu_bwd(const void *dh, int64_t ld_dh, const void *g,
                          const void *u, int64_t ld_gu, void *dg, void *du,
                          int64_t ld_dgu, int64_t T, int64_t I,
                          ftk_dtype dtype, ftk_stream_t stream);

/* ftk_swiglu_bwd that also re-emits the forward's h (optimisation (1) of
 * "Chronicals", arXiv 2601.02609, abstract: the fused SwiGLU; re-emitting h
 * is this library's variant): besides dg and du it writes
 *   h = g * sigmoid(g) * u,
 * computed exactly as ftk_swiglu_fwd computes it (bit-identical), so a
 * training step can drop h after the forward and get it back here, where
 * the down projection's weight gradient needs it.  h: [T, ld_h], written
 * once.  h may replace dh, g or u exactly (same pointer and stride) but must
 * not overlap dg or du; the other arguments and rules are ftk_swiglu_bwd's. */
FTK_API ftk_status ftk_swiglu_bwd_h(const void *dh, int64_t ld_dh, const void *g,
                                    const void *u, int64_t ld_gu, void *dg, void *du,
                                    int64_t ld_dgu, void *h, int64_t ld_h, int64_t T,
                                    int64_t I, ftk_dtype dtype, ftk_stream_t stream);

/* ------------------------------------------------------------- QK-RoPE */

/* In-place rotary embedding of Q and K together, rotate-half (NeoX) layout,
 * over a packed batch of B variable-length sequences (the fused QK RoPE
 * paragraph of "Unsloth prétend accélérer 5 fois l'entraînement des LLM
 * avec de nouveaux noyaux Triton et un auto-packing", seventnews.com: Q and
 * K in ONE kernel, variable-length, fully in place with no clone or
 * transpose; its LONG_INDEXING paragraph for the 64-bit offsets of
 * 500k-token contexts; "Chronicals", arXiv 2601.02609, abstract,
 * optimisation (1): fused QK-RoPE.  The pages print no formula; this is the
 * standard rotate-half RoPE):
 *   token t of sequence b (cu_seqlens[b] <= t < cu_seqlens[b+1]) sits at
 *   position p = t - cu_seqlens[b]; for i < D/2, phi = p * theta^(-2i/D);
 *   every head vector v of Q and K at t becomes
 *     v[i]       <- v[i] cos(phi) - v[i+D/2] sin(phi)
 *     v[i+D/2]   <- v[i+D/2] cos(phi) + v[i] sin(phi)
 * q: [T, ld_q] holding Hq heads of D contiguous values per token,
 * k: [T, ld_k] holding Hkv heads (any GQA ratio: Hq, Hkv >= 0, Hq + Hkv
 * >= 1; q may be NULL when Hq == 0 and k when Hkv == 0).  q and k must not
 * overlap; they may be interleaved slices of one fused QKV buffer.
 * cu_seqlens: DEVICE int32 [B+1], cu[0] = 0, non-decreasing, cu[B] = T; read on the device, never copied to the host.  Tokens outside
 * every sequence are impossible when that holds; if it does not, results are
 * unspecified but every access stays inside q and k (ftk_check_seqlens and
 * the *_checked calls below validate it on the device and skip the
 * rotation instead).  0 < D <= 512, D even.
 * The angle is formed in extended precision (position times a two-float
 * split of theta^(-2i/D) / 2pi), so it is accurate to ~1e-7 rad at
 * positions beyond 500k; no cos/sin table is read. */
FTK_API ftk_status ftk_qk_rope_fwd(void *q, int64_t ld_q, void *k, int64_t ld_k,
                           const int32_t *cu_seqlens, int32_t B, int64_t T,
                           int32_t Hq, int32_t Hkv, int32_t D, double theta,
                           ftk_dtype dtype, ftk_stream_t stream);

/* Backward of the above on dq, dk in place: the same rotation by -phi (the
 * transpose of the forward rotation; the pages' fused QK-RoPE serves the
 * training step, whose backward pass needs this).  Same arguments and
 * rules. */
FTK_API ftk_status ftk_qk_rope_bwd(void *dq, int64_t ld_q, void *dk, int64_t ld_k,
                           const int32_t *cu_seqlens, int32_t B, int64_t T,
                           int32_t Hq, int32_t Hkv, int32_t D, double theta,
                           ftk_dtype dtype, ftk_stream_t stream);

/* The rotation above with the caller's inverse frequencies in place of
 * theta^(-2i/D):  phi_i = p * inv_freq[i].  Any scaled RoPE whose angle is
 * position times a per-dimension frequency (linear, "llama3", NTK-style)
 * comes down to such a table; the pages apply no scaling, this is the
 * library's variant of the same kernels.  inv_freq: HOST double [D/2], read
 * during the call only (it may be freed on return); each entry must lie in
 * [0, 1] (every such rule only slows theta's frequencies, and theta^0 = 1),
 * else FTK_ERR_SHAPE.  The angle keeps the same ~1e-7 rad accuracy.  Other
 * arguments and rules are ftk_qk_rope_fwd's / ftk_qk_rope_bwd's. */
FTK_API ftk_status ftk_qk_rope_freq_fwd(void *q, int64_t ld_q, void *k, int64_t ld_k,
                                        const int32_t *cu_seqlens, int32_t B, int64_t T,
                                        int32_t Hq, int32_t Hkv, int32_t D,
                                        const double *inv_freq, ftk_dtype dtype,
                                        ftk_stream_t stream);
FTK_API ftk_status ftk_qk_rope_freq_bwd(void *dq, int64_t ld_q, void *dk, int64_t ld_k,
                                        const int32_t *cu_seqlens, int32_t B, int64_t T,
                                        int32_t Hq, int32_t Hkv, int32_t D,
                                        const double *inv_freq, ftk_dtype dtype,
                                        ftk_stream_t stream);

/* The "llama3" scaled table (the rule published with Llama 3.1, used by the
 * Llama-3.2 models) for ftk_qk_rope_freq_*.  Host code; inv_freq: HOST
 * double [D/2], written.  With base_i = theta^(-2i/D), wavelength
 * lambda_i = 2 pi / base_i and L = original_max_position:
 *   lambda_i < L / high_freq_factor:  inv_freq[i] = base_i
 *   lambda_i > L / low_freq_factor:   inv_freq[i] = base_i / factor
 *   otherwise, s = (L / lambda_i - low_freq_factor)
 *                  / (high_freq_factor - low_freq_factor):
 *                                     inv_freq[i] = s base_i + (1 - s) base_i / factor
 * Needs D even in [2, 512], theta > 1, factor >= 1, 0 < low_freq_factor <
 * high_freq_factor, L > 0 (all finite), else FTK_ERR_SHAPE.  Llama-3.2:
 * theta 5e5, factor 32, low 1, high 4, L 8192. */
FTK_API ftk_status ftk_rope_llama3_inv_freq(int32_t D, double theta, double factor,
                                            double low_freq_factor, double high_freq_factor,
                                            double original_max_position, double *inv_freq);

/* ------------------------------------ checked sequence boundaries (RoPE) */

/* Bits of the word ftk_check_seqlens writes (0: the boundaries are valid). */
#define FTK_SEQLENS_BAD_START 1u  /* cu[0] != 0 */
#define FTK_SEQLENS_DECREASING 2u /* some cu[b+1] < cu[b] */
#define FTK_SEQLENS_BAD_END 4u    /* cu[B] != T */

/* Validates a packed batch's sequence boundaries where they live, on the
 * device, without a host synchronisation ("Unsloth und NVIDIA optimieren
 * LLM-Training um zusätzliche 25%", lumeric.app, item (1): the packed
 * metadata stays on the GPU; the auto-packing paragraph of the Unsloth item
 * on seventnews.com makes it the contract between packer and kernels).
 * cu_seqlens: DEVICE int32 [B+1]; status: DEVICE uint32, caller-owned,
 * OVERWRITTEN (after the check completes, in stream order) with the
 * FTK_SEQLENS_* bits found: cu[0] == 0, cu non-decreasing, cu[B] == T.  With
 * those three, every boundary lies in [0, T].  One small kernel (one CTA);
 * nothing traps or faults on bad input.  Check once per batch, then pass
 * `status` to the checked RoPE calls of every layer.  B >= 0, T >= 0, else
 * FTK_ERR_SHAPE; NULL pointers give FTK_ERR_NULL; status must not overlap
 * cu_seqlens (FTK_ERR_ALIAS) and both need 4-byte alignment. */
FTK_API ftk_status ftk_check_seqlens(const int32_t *cu_seqlens, int32_t B, int64_t T,
                                     uint32_t *status, ftk_stream_t stream);

/* ftk_qk_rope_fwd / ftk_qk_rope_bwd (inv_freq NULL: theta's table) or
 * ftk_qk_rope_freq_fwd / _bwd (inv_freq set, HOST double [D/2]), guarded by
 * the word ftk_check_seqlens wrote for this batch: every CTA reads
 * *seqlens_status (DEVICE uint32, read-only here) after the preceding work on
 * the stream has finished, and when it is non-zero the kernel returns
 * without touching q or k.  A caller may also set the word itself to skip
 * the rotation.  Host-side rules and errors are those of the unchecked calls,
 * plus FTK_ERR_NULL for a NULL seqlens_status (T > 0).  The fused QK-norm
 * rotation has the same mode (ftk_qk_norm_rope_{fwd,bwd}_checked, below). */
FTK_API ftk_status ftk_qk_rope_fwd_checked(void *q, int64_t ld_q, void *k, int64_t ld_k,
                                           const int32_t *cu_seqlens, int32_t B, int64_t T,
                                           int32_t Hq, int32_t Hkv, int32_t D, double theta,
                                           const double *inv_freq,
                                           const uint32_t *seqlens_status, ftk_dtype dtype,
                                           ftk_stream_t stream);
FTK_API ftk_status ftk_qk_rope_bwd_checked(void *dq, int64_t ld_q, void *dk, int64_t ld_k,
                                           const int32_t *cu_seqlens, int32_t B, int64_t T,
                                           int32_t Hq, int32_t Hkv, int32_t D, double theta,
                                           const double *inv_freq,
                                           const uint32_t *seqlens_status, ftk_dtype dtype,
                                           ftk_stream_t stream);

/* ------------------------------------- QK-RMSNorm fused into the QK-RoPE */

/* Per-head RMSNorm of Q and K (the q_norm / k_norm of Qwen3-style attention)
 * followed by the rotation of ftk_qk_rope_fwd, in one pass over Q and K.
 * The pages fuse the QK-RoPE (the fused QK RoPE paragraph of the Unsloth
 * item on seventnews.com; "Chronicals", arXiv 2601.02609, abstract,
 * optimisation (1)); the norm in front of it is this library's variant.
 * For token t at position p (as in ftk_qk_rope_fwd) and every head vector v
 * of D values of Q (weight wq) or K (weight wk):
 *   r[t,h] = 1 / sqrt( (1/D) sum_i v_i^2 + eps )
 *   n_i    = v_i r w_i                    (fp32; not rounded)
 *   out    = n rotated by phi_i = p * inv_freq_i (rotate-half pairs)
 * inv_freq: HOST double [D/2] (entries in [0, 1]), or NULL for
 * theta^(-2i/D).  q [T, ld_q] of Hq heads, k [T, ld_k] of Hkv heads;
 * q_out [T, ld_qo], k_out [T, ld_ko]: each may BE its input (same pointer and
 * stride) for an in-place update, but then the backward needs a copy of the
 * pre-norm values.  wq, wk: [D] (dtype).  rstd_q [T, Hq], rstd_k [T, Hkv]:
 * fp32 contiguous, nullable, receive r.  q, wq, q_out may be NULL when
 * Hq == 0, and the k arguments when Hkv == 0.  cu_seqlens, B, T, D (even, <=
 * 512) as in ftk_qk_rope_fwd; eps >= 0. */
FTK_API ftk_status ftk_qk_norm_rope_fwd(const void *q, int64_t ld_q, const void *k, int64_t ld_k,
                                        const void *wq, const void *wk, void *q_out,
                                        int64_t ld_qo, void *k_out, int64_t ld_ko,
                                        float *rstd_q, float *rstd_k,
                                        const int32_t *cu_seqlens, int32_t B, int64_t T,
                                        int32_t Hq, int32_t Hkv, int32_t D, double theta,
                                        const double *inv_freq, float eps, ftk_dtype dtype,
                                        ftk_stream_t stream);

/* Bytes of device workspace ftk_qk_norm_rope_bwd needs for T tokens and
 * head dimension D on the CURRENT device; 0 for invalid arguments. */
FTK_API size_t ftk_qk_norm_rope_bwd_workspace_bytes(int64_t T, int32_t D, ftk_dtype dtype);

/* Backward of ftk_qk_norm_rope_fwd.  From the output gradients dq_out,
 * dk_out and the PRE-norm q, k:
 *   dn     = dq_out (or dk_out) rotated by -phi (the transpose)
 *   c      = sum_i dn_i w_i v_i
 *   dq     = r w dn - r^3 v c / D             (likewise dk)
 *   dwq[i] = sum over tokens and Q heads of dn_i v_i r   (fp32, OVERWRITTEN;
 *            dwk likewise over K heads)
 * rstd_q/rstd_k from the forward, or both NULL to recompute r from v and
 * eps.  dq [T, ld_dq] may be dq_out itself (same pointer and stride), dk
 * likewise; no other output may overlap anything.  workspace: >=
 * ftk_qk_norm_rope_bwd_workspace_bytes(T, D, dtype) bytes, 16-byte aligned.
 * dwq and dwk are sums of per-CTA fp32 partials added in a fixed order:
 * bitwise reproducible run to run.  Other rules as in the forward. */
FTK_API ftk_status ftk_qk_norm_rope_bwd(const void *dq_out, int64_t ld_gq, const void *dk_out,
                                        int64_t ld_gk, const void *q, int64_t ld_q,
                                        const void *k, int64_t ld_k, const void *wq,
                                        const void *wk, const float *rstd_q,
                                        const float *rstd_k, void *dq, int64_t ld_dq, void *dk,
                                        int64_t ld_dk, float *dwq, float *dwk, void *workspace,
                                        size_t workspace_bytes, const int32_t *cu_seqlens,
                                        int32_t B, int64_t T, int32_t Hq, int32_t Hkv, int32_t D,
                                        double theta, const double *inv_freq, float eps,
                                        ftk_dtype dtype, ftk_stream_t stream);

/* ftk_qk_norm_rope_fwd / ftk_qk_norm_rope_bwd guarded by the word
 * ftk_check_seqlens wrote for this batch (the checked mode of the plain
 * rotation above, for the fused QK-norm): every kernel of the call reads
 * *seqlens_status (DEVICE uint32, read-only here) after the preceding work on
 * the stream has finished, and when it is non-zero returns without writing
 * any output: q_out, k_out, rstd_q, rstd_k (forward); dq, dk, dwq, dwk and
 * the workspace (backward).  Host-side rules and errors are those of the
 * unchecked calls, plus FTK_ERR_NULL for a NULL seqlens_status (T > 0) and
 * FTK_ERR_ALIAS when the word overlaps an output. */
FTK_API ftk_status ftk_qk_norm_rope_fwd_checked(
    const void *q, int64_t ld_q, const void *k, int64_t ld_k, const void *wq, const void *wk,
    void *q_out, int64_t ld_qo, void *k_out, int64_t ld_ko, float *rstd_q, float *rstd_k,
    const int32_t *cu_seqlens, int32_t B, int64_t T, int32_t Hq, int32_t Hkv, int32_t D,
    double theta, const double *inv_freq, float eps, const uint32_t *seqlens_status,
    ftk_dtype dtype, ftk_stream_t stream);
FTK_API ftk_status ftk_qk_norm_rope_bwd_checked(
    const void *dq_out, int64_t ld_gq, const void *dk_out, int64_t ld_gk, const void *q,
    int64_t ld_q, const void *k, int64_t ld_k, const void *wq, const void *wk,
    const float *rstd_q, const float *rstd_k, void *dq, int64_t ld_dq, void *dk, int64_t ld_dk,
    float *dwq, float *dwk, void *workspace, size_t workspace_bytes, const int32_t *cu_seqlens,
    int32_t B, int64_t T, int32_t Hq, int32_t Hkv, int32_t D, double theta,
    const double *inv_freq, float eps, const uint32_t *seqlens_status, ftk_dtype dtype,
    ftk_stream_t stream);

/* ------------------------------------------------------ tensor-core GEMM */

/* C = A B^T on the 5th-generation tensor cores: A bf16 [M, lda], B bf16
 * [N, ldb] (both K contiguous), C fp32 [M, ldc] (overwritten), fp32
 * accumulation in tensor memory.  The contraction the cross-entropy calls
 * below are built on, exposed for reuse and testing; the pages have no
 * counterpart.  A and B 16-byte aligned with lda, ldb multiples of 8;
 * K >= 1 (FTK_ERR_SHAPE for K = 0 with M, N > 0); C must not overlap A or B. */
FTK_API ftk_status ftk_gemm_bf16(const void *a, int64_t lda, const void *b, int64_t ldb,
                                 float *c, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                 ftk_stream_t stream);

/* The same with either operand stored the other way round: a_mn != 0 reads
 * A from a bf16 [K, lda] array (A[m, k] = a[k * lda + m], M contiguous) and
 * b_mn != 0 reads B from [K, ldb] (B[n, k] = b[k * ldb + n]); the tensor
 * cores take such operands as they are, with no transposed copy.  The
 * alignment and error rules are those of ftk_gemm_bf16, with lda >= M
 * (ldb >= N) for an MN-major operand. */
FTK_API ftk_status ftk_gemm_bf16_ex(const void *a, int64_t lda, int a_mn, const void *b,
                                    int64_t ldb, int b_mn, float *c, int64_t ldc, int64_t M,
                                    int64_t N, int64_t K, ftk_stream_t stream);

/* ---------------------------------------------------- Cut Cross-Entropy */

/* Cross-entropy loss of a linear LM head without materialised logits
 * ("Chronicals", arXiv 2601.02609, abstract, optimisation (2): Cut
 * Cross-Entropy, an online softmax that keeps the [T, V] logits out of
 * memory, 5 GB down to 135 MB for its run):
 *   z[t,v] = sum_j h[t,j] W[v,j]        (bf16 operands, fp32 accumulation)
 *   lse[t] = log sum_v exp(z[t,v])
 *   loss   = (1/N) sum_{valid t} (lse[t] - z[t, y_t]),  N = #valid tokens
 * A token is valid when 0 <= y[t] < V (so -100, or any negative value, marks
 * one to ignore); N = 0 gives loss 0.  bf16 only (FTK_ERR_DTYPE otherwise):
 * the contraction runs on the tensor cores (tcgen05).
 * h [T, ldh] and W [V, ldw] (bf16, 16-byte aligned, ldh and ldw multiples of
 * 8); y int32 [T]; loss: ONE fp32 on the device; lse fp32 [T] (keep it for
 * the backward).  workspace: >= ftk_cce_fwd_workspace_bytes(T, V) bytes,
 * 256-byte aligned.  No output may overlap an input or another output.  The
 * loss is summed in a fixed order: bitwise reproducible run to run. */
FTK_API size_t ftk_cce_fwd_workspace_bytes(int64_t T, int64_t V);
FTK_API ftk_status ftk_cce_fwd(const void *h, int64_t ldh, const void *w, int64_t ldw,
                               const int32_t *y, int64_t T, int64_t H, int64_t V, float *loss,
                               float *lse, void *workspace, size_t workspace_bytes,
                               ftk_dtype dtype, ftk_stream_t stream);

/* Backward of ftk_cce_fwd for an upstream gradient g of the loss (dloss:
 * ONE fp32 on the device):
 *   dz[t,v] = (g/N) (softmax(z[t])_v - [v == y_t])   (valid t; 0 otherwise)
 *   dh = dz W  -> bf16 [T, lddh],     dW = dz^T h  -> fp32 [V, lddw]
 * dz is rounded to bf16 before the two contractions (the tensor cores take
 * bf16 operands); they accumulate in fp32.  The logits are recomputed a
 * vocabulary chunk at a time (ftk_cce_bwd_chunk columns, 4,096 to 16,384,
 * or all of V when V <= 16,384), two launches per chunk.  lse from the
 * forward.  workspace: >= ftk_cce_bwd_workspace_bytes(T, H, V) bytes,
 * 256-byte aligned (enough for any chunk width).  dh and dW are
 * overwritten; no output may overlap an input or another output.
 * dh is summed over the chunks in a fixed order and dW written once per
 * element: both are bitwise reproducible run to run. */
FTK_API size_t ftk_cce_bwd_workspace_bytes(int64_t T, int64_t H, int64_t V);

/* The vocabulary chunk width ftk_cce_bwd uses on a device with `sms` SMs:
 * the one (a multiple of 256) whose dz and dh + dW launches fill the SMs'
 * waves best by a static estimate.  Host-only; 0 for a non-positive
 * argument. */
FTK_API int64_t ftk_cce_bwd_chunk(int64_t T, int64_t H, int64_t V, int32_t sms);
FTK_API ftk_status ftk_cce_bwd(const void *h, int64_t ldh, const void *w, int64_t ldw,
                               const int32_t *y, const float *lse, const float *dloss,
                               int64_t T, int64_t H, int64_t V, void *dh, int64_t lddh,
                               float *dw, int64_t lddw, void *workspace,
                               size_t workspace_bytes, ftk_dtype dtype, ftk_stream_t stream);

/* -------------------------------------------------------------- packing */

/* Best-Fit-Decreasing packing of n sequences into bins of `capacity` tokens
 * ("Chronicals", arXiv 2601.02609, abstract, optimisation (4): Best-Fit
 * Decreasing sequence packing recovers the compute padding wastes).  Host
 * code; every pointer is a HOST pointer.
 *   Sequences are taken longest first (equal lengths: lower index first);
 *   each goes to the open bin with the least room that still holds it
 *   (equal room: lower bin index), else to a new bin.
 * lengths: int32 [n], each in [0, capacity].  Outputs, caller-allocated:
 * bin_of: int32 [n], the bin of each sequence; order: int64 [n], the
 * sequence indices bin by bin, each bin's in the order they were placed
 * (concatenating them gives the packed batch); bin_start: int64 [n + 1]
 * (room for the worst case of one bin per sequence), bin b holds
 * order[bin_start[b] .. bin_start[b+1]); *n_bins: the number of bins.
 * A length outside [0, capacity] gives FTK_ERR_SHAPE and writes nothing.
 * O(n log n) time, O(n) memory (the descending order is a counting sort
 * only while capacity <= 4 n + 1024). */
FTK_API ftk_status ftk_bfd_pack(const int32_t *lengths, int64_t n, int32_t capacity,
                                int32_t *bin_of, int64_t *order, int64_t *bin_start,
                                int64_t *n_bins);

/* ------------------------------------------------------------ utilities */

/* Bits of the device status word. */
#define FTK_DEVSTAT_WAIT_TIMEOUT 1u /* a kernel's pipeline wait ran out */

/* The device status word of the current device, into *flags (host
 * pointer); cleared afterwards when clear != 0.  Kernels that stream data
 * through shared memory wait on barriers for bulk copies; every such wait
 * gives up after ~1 s of SM clock, sets FTK_DEVSTAT_WAIT_TIMEOUT and lets
 * the kernel finish instead of hanging.  A set bit means some launch since
 * the last clear produced invalid results.  This call synchronises with
 * the device (it reads device memory). */
FTK_API ftk_status ftk_device_status(uint32_t *flags, int clear);

/* Launches one CTA that waits, bounded by limit_cycles SM clock cycles, on
 * a barrier nothing will ever complete, so the timeout path runs for real:
 * afterwards ftk_device_status reports FTK_DEVSTAT_WAIT_TIMEOUT.  For
 * testing failure detection; faults and hangs nothing. */
FTK_API ftk_status ftk_selftest_wait_timeout(int64_t limit_cycles, ftk_stream_t stream);

/* Static text for a status code. */
FTK_API const char *ftk_status_str(ftk_status status);

/* Text of the last CUDA error seen by a call on this host thread ("" if
 * none).  The pointer stays valid until the next call on the thread. */
FTK_API const char *ftk_last_cuda_error(void);

/* Library version, e.g. "0.1.0". */
FTK_API const char *ftk_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FTK_H_ */
