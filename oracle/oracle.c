/*
 * CPU oracle for the fused per-token layer ops: RMSNorm, SwiGLU and the
 * in-place varlen QK-RoPE, forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this file:
 * it is used by tests/, by __graft_entry__.smoke() and by bench.py's
 * cpu_baseline / reference leg, and it shares no source with the CUDA
 * library (no header, helper, table or constant generator in common).
 *
 * Everything is plain double precision.  Inputs arrive as doubles that hold
 * the stored (fp32 or bf16) values exactly; outputs stay in double.  Each
 * function is the textbook definition of its op written out loop by loop, in
 * the pages' terms:
 *
 *   - Chronicals: A High-Performance Framework for LLM Fine-Tuning with 3.51x
 *     Speedup over Unsloth (arXiv 2601.02609), abstract, optimisation (1):
 *     fused RMSNorm, SwiGLU and QK-RoPE kernels.  The page names the ops but
 *     prints no formula, so the standard definitions are used.
 *   - "Unsloth prétend accélérer 5 fois l'entraînement des LLM avec de
 *     nouveaux noyaux Triton et un auto-packing" (seventnews.com), paragraph
 *     on the fused QK RoPE kernel (Q and K rotated by one in-place kernel,
 *     variable-length RoPE) and paragraph on auto-packing (sequences packed
 *     into one 1-D token tensor with their length metadata kept).
 *
 * Besides each output, several functions can also return the element's
 * condition scale: the sum of the absolute values of the terms that form
 * the output.  The parity tests measure the error of a cancelling output
 * against that scale.
 *
 * Pins: every function is checked, without a second implementation, by
 * tests/test_oracle_pins.py (closed forms, invariants, finite differences,
 * a textbook special case).
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_API __attribute__((visibility("default")))

/* Threads an OpenMP loop of this library runs on (1 without OpenMP). */
ORACLE_API int oracle_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Runs the following OpenMP loops of this library on n threads (n >= 1;
 * a no-op without OpenMP); returns the previous count.  Only the timing of
 * the oracle uses it: the loops' results do not depend on the thread count. */
ORACLE_API int oracle_set_threads(int n)
{
    const int prev = oracle_threads();
#ifdef _OPENMP
    if (n >= 1)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
    return prev;
}

/* ---------------------------------------------------------------- RMSNorm */

/* y[t,j] = x[t,j] * r[t] * w[j],  r[t] = 1 / sqrt(mean_j x[t,j]^2 + eps).
 * rstd (nullable) receives r[t]. */
ORACLE_API void oracle_rmsnorm_fwd(const double *x, const double *w, double *y,
                                   double *rstd, int64_t T, int64_t H,
                                   double eps)
{
    int64_t t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < T; ++t) {
        const double *xr = x + t * H;
        double ss = 0.0;
        for (int64_t j = 0; j < H; ++j)
            ss += xr[j] * xr[j];
        double r = 1.0 / sqrt(ss / (double)H + eps);
        for (int64_t j = 0; j < H; ++j)
            y[t * H + j] = xr[j] * r * w[j];
        if (rstd)
            rstd[t] = r;
    }
}

/* Gradient of sum(dy * y) for y = rmsnorm(x, w):
 *   c[t]    = sum_j dy[t,j] w[j] x[t,j]
 *   dx[t,j] = r[t] w[j] dy[t,j] - r[t]^3 x[t,j] c[t] / H
 *   dw[j]   = sum_t dy[t,j] x[t,j] r[t]
 * dx_scale[t,j] = r|w dy| + r^3 |x| (sum_j |dy w x|) / H   (nullable)
 * dw_scale[j]   = sum_t |dy x r|                           (nullable)     */
ORACLE_API void oracle_rmsnorm_bwd(const double *dy, const double *x,
                                   const double *w, double *dx, double *dw,
                                   double *dx_scale, double *dw_scale,
                                   int64_t T, int64_t H, double eps)
{
    double *r = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1));
    int64_t t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < T; ++t) {
        const double *xr = x + t * H, *dyr = dy + t * H;
        double ss = 0.0, c = 0.0, cabs = 0.0;
        for (int64_t j = 0; j < H; ++j) {
            ss += xr[j] * xr[j];
            c += dyr[j] * w[j] * xr[j];
            cabs += fabs(dyr[j] * w[j] * xr[j]);
        }
        double rt = 1.0 / sqrt(ss / (double)H + eps);
        r[t] = rt;
        for (int64_t j = 0; j < H; ++j) {
            double a = rt * w[j] * dyr[j];
            double b = rt * rt * rt * xr[j] * c / (double)H;
            dx[t * H + j] = a - b;
            if (dx_scale)
                dx_scale[t * H + j] =
                    fabs(a) + rt * rt * rt * fabs(xr[j]) * cabs / (double)H;
        }
    }
    /* column sums, rows in order 0..T-1; blocks of columns run in parallel */
    const int64_t CB = 64;
    int64_t nb = (H + CB - 1) / CB, b;
#pragma omp parallel for schedule(static)
    for (b = 0; b < nb; ++b) {
        double acc[64], accabs[64];
        int64_t j0 = b * CB, j1 = j0 + CB < H ? j0 + CB : H;
        for (int64_t j = j0; j < j1; ++j)
            acc[j - j0] = accabs[j - j0] = 0.0;
        for (int64_t tt = 0; tt < T; ++tt)
            for (int64_t j = j0; j < j1; ++j) {
                double v = dy[tt * H + j] * x[tt * H + j] * r[tt];
                acc[j - j0] += v;
                accabs[j - j0] += fabs(v);
            }
        for (int64_t j = j0; j < j1; ++j) {
            dw[j] = acc[j - j0];
            if (dw_scale)
                dw_scale[j] = accabs[j - j0];
        }
    }
    free(r);
}

/* ---------------------------------------------- RMSNorm with residual add */

/* The storage rounding of a sum: the two stored values are added in fp32
 * (the precision the kernels add in), then the fp32 sum is rounded to the
 * storage type: kept (storage 0 = fp32), rounded to nearest even on its low
 * 16 bits (storage 1 = bf16), or not rounded at all (storage 2 = exact, the
 * double sum; used by the finite-difference pins). */
static double stored_sum(double a, double b, int storage)
{
    if (storage == 2)
        return a + b;
    float f = (float)a + (float)b;
    if (storage == 0)
        return (double)f;
    union {
        float f;
        uint32_t u;
    } v;
    v.f = f;
    uint32_t lsb = (v.u >> 16) & 1u;
    v.u = (v.u + 0x7FFFu + lsb) & 0xFFFF0000u;
    return (double)v.f;
}

/* Pre-norm residual step: h = x + res, stored (see stored_sum), then
 * y = rmsnorm(h) * w with r[t] = 1/sqrt(mean_j h[t,j]^2 + eps).
 * h, y, rstd are outputs (rstd nullable). */
ORACLE_API void oracle_rmsnorm_add_fwd(const double *x, const double *res,
                                       const double *w, double *h, double *y,
                                       double *rstd, int64_t T, int64_t H,
                                       double eps, int storage)
{
    int64_t n = T * H, i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < n; ++i)
        h[i] = stored_sum(x[i], res[i], storage);
    oracle_rmsnorm_fwd(h, w, y, rstd, T, H, eps);
}

/* Backward of the step above: the gradient reaching h is dh (from the
 * residual stream) plus the norm's backward of dy, and it is the gradient of
 * both x and res:  dx = dh + (r w dy - r^3 h c / H),  dw as in
 * oracle_rmsnorm_bwd.  dx_scale adds |dh| to the norm's scale (nullable). */
ORACLE_API void oracle_rmsnorm_add_bwd(const double *dy, const double *dh,
                                       const double *h, const double *w,
                                       double *dx, double *dw, double *dx_scale,
                                       double *dw_scale, int64_t T, int64_t H,
                                       double eps)
{
    oracle_rmsnorm_bwd(dy, h, w, dx, dw, dx_scale, dw_scale, T, H, eps);
    int64_t n = T * H, i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < n; ++i) {
        dx[i] += dh[i];
        if (dx_scale)
            dx_scale[i] += fabs(dh[i]);
    }
}

/* ----------------------------------------------------------------- SwiGLU */

static double sigmoid(double g) { return 1.0 / (1.0 + exp(-g)); }

/* h = silu(g) * u = g * sigmoid(g) * u, elementwise over n values. */
ORACLE_API void oracle_swiglu_fwd(const double *g, const double *u, double *h,
                                  int64_t n)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < n; ++i)
        h[i] = g[i] * sigmoid(g[i]) * u[i];
}

/* Gradient of sum(dh * h), s = sigmoid(g):
 *   dg = dh u s (1 + g (1 - s)),   du = dh g s
 * dg_scale = |dh u s| (1 + |g (1 - s)|)   (nullable)                      */
ORACLE_API void oracle_swiglu_bwd(const double *dh, const double *g,
                                  const double *u, double *dg, double *du,
                                  double *dg_scale, int64_t n)
{
    int64_t i;
#pragma omp parallel for schedule(static)
    for (i = 0; i < n; ++i) {
        double s = sigmoid(g[i]);
        double a = dh[i] * u[i] * s;
        dg[i] = a * (1.0 + g[i] * (1.0 - s));
        du[i] = dh[i] * g[i] * s;
        if (dg_scale)
            dg_scale[i] = fabs(a) * (1.0 + fabs(g[i] * (1.0 - s)));
    }
}

/* ------------------------------------------------------------ QK-RoPE */

/* Position of global token t inside its packed sequence: t - cu[b] for the
 * sequence b with cu[b] <= t < cu[b+1].  Zero-length sequences (repeated
 * boundaries) hold no token and are passed over by the scan. */
static int64_t position_of(int64_t t, const int32_t *cu, int32_t B)
{
    for (int32_t b = 0; b < B; ++b)
        if ((int64_t)cu[b] <= t && t < (int64_t)cu[b + 1])
            return t - (int64_t)cu[b];
    return -1; /* t outside the batch: the caller rejects this */
}

/* Rotate-half RoPE of one head vector v[0..D) at position p:
 *   phi_i = p * inv_freq[i],  i < D/2
 *   (v_i, v_{i+D/2}) <- (v_i cos phi - v_{i+D/2} sin phi,
 *                        v_{i+D/2} cos phi + v_i sin phi)
 * sign = -1 rotates by -phi (the transpose, used by the backward pass).
 * Condition scale of each output: its two terms' magnitudes, plus
 * ANGLE_WEIGHT times its sensitivity to the angle (the derivative's terms,
 * |v_i sin| + |v_{i+D/2} cos| for the first output): no finite-precision
 * angle is exact, and near cos phi = 0 an output still moves by |v| per
 * radian of angle error although its own terms are ~0.  The weight is the
 * angle error allowed (1e-6 rad, the accuracy a GPU angle formed in
 * extended precision reaches at every position below 524,288) over the
 * relative bar the scale is multiplied by in fp32 (1e-5). */
#define ANGLE_WEIGHT 0.1
static void rotate_head(const double *v, double *out, double *scale,
                        int64_t p, int32_t D, const double *inv_freq, int sign)
{
    int32_t half = D / 2;
    for (int32_t i = 0; i < half; ++i) {
        double phi = (double)sign * (double)p * inv_freq[i];
        double c = cos(phi), s = sin(phi);
        double a = v[i], b = v[i + half];
        out[i] = a * c - b * s;
        out[i + half] = b * c + a * s;
        if (scale) {
            double cc = fabs(c) + ANGLE_WEIGHT * fabs(s);
            double ss = fabs(s) + ANGLE_WEIGHT * fabs(c);
            scale[i] = fabs(a) * cc + fabs(b) * ss;
            scale[i + half] = fabs(b) * cc + fabs(a) * ss;
        }
    }
}

/* Q and K of n packed tokens rotated together with the inverse frequencies
 * inv_freq[D/2].  Row r of q/k is global token tok[r] (tok may be NULL: row
 * r is token r).  q: [n, Hq, D], k: [n, Hkv, D] (contiguous), cu: int32
 * [B+1] sequence boundaries.  sign = +1 forward, -1 backward.  Returns 0,
 * or -1 if a token lies outside the batch or D is odd.  q_scale/k_scale are
 * nullable. */
ORACLE_API int oracle_qk_rope_freq(const double *q, const double *k, double *q_out,
                                   double *k_out, double *q_scale, double *k_scale,
                                   const int64_t *tok, int64_t n, const int32_t *cu,
                                   int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                                   const double *inv_freq, int sign)
{
    if (D % 2 != 0)
        return -1;
    int bad = 0;
    int64_t r;
#pragma omp parallel for schedule(static) reduction(| : bad)
    for (r = 0; r < n; ++r) {
        int64_t t = tok ? tok[r] : r;
        int64_t p = position_of(t, cu, B);
        if (p < 0) {
            bad = 1;
            continue;
        }
        for (int32_t h = 0; h < Hq; ++h) {
            int64_t o = (r * Hq + h) * D;
            rotate_head(q + o, q_out + o, q_scale ? q_scale + o : NULL, p, D,
                        inv_freq, sign);
        }
        for (int32_t h = 0; h < Hkv; ++h) {
            int64_t o = (r * Hkv + h) * D;
            rotate_head(k + o, k_out + o, k_scale ? k_scale + o : NULL, p, D,
                        inv_freq, sign);
        }
    }
    return bad ? -1 : 0;
}

/* The unscaled inverse frequencies: inv_freq[i] = theta^(-2i/D). */
ORACLE_API void oracle_rope_inv_freq(int32_t D, double theta, double *inv_freq)
{
    for (int32_t i = 0; i < D / 2; ++i)
        inv_freq[i] = pow(theta, -2.0 * (double)i / (double)D);
}

/* The plain rotation (no scaling): oracle_qk_rope_freq with theta's table. */
ORACLE_API int oracle_qk_rope(const double *q, const double *k, double *q_out,
                              double *k_out, double *q_scale, double *k_scale,
                              const int64_t *tok, int64_t n, const int32_t *cu,
                              int32_t B, int32_t Hq, int32_t Hkv, int32_t D,
                              double theta, int sign)
{
    if (D % 2 != 0 || D <= 0)
        return -1;
    double *f = (double *)malloc(sizeof(double) * (size_t)(D / 2));
    if (!f)
        return -1;
    oracle_rope_inv_freq(D, theta, f);
    int rc = oracle_qk_rope_freq(q, k, q_out, k_out, q_scale, k_scale, tok, n, cu, B,
                                 Hq, Hkv, D, f, sign);
    free(f);
    return rc;
}

/* "llama3" rope scaling, the rule published with Llama 3.1 for stretching a
 * model trained on contexts of L = original_max_position tokens: with the
 * wavelength of dimension i, lambda_i = 2 pi / inv_freq_i,
 *   lambda_i < L / high_freq_factor  (fast-turning):  inv_freq_i unchanged;
 *   lambda_i > L / low_freq_factor   (slow-turning):  inv_freq_i / factor;
 *   in between: a blend,  s = (L / lambda_i - low_freq_factor)
 *                            / (high_freq_factor - low_freq_factor),
 *               (1 - s) * inv_freq_i / factor + s * inv_freq_i.
 * Returns 0, or -1 for D odd / non-positive or high_freq_factor <=
 * low_freq_factor. */
ORACLE_API int oracle_rope_llama3_inv_freq(int32_t D, double theta, double factor,
                                           double low_freq_factor,
                                           double high_freq_factor,
                                           double original_max_position,
                                           double *inv_freq)
{
    if (D <= 0 || D % 2 != 0 || !(high_freq_factor > low_freq_factor))
        return -1;
    const double two_pi = 6.283185307179586476925;
    const double L = original_max_position;
    oracle_rope_inv_freq(D, theta, inv_freq);
    for (int32_t i = 0; i < D / 2; ++i) {
        double f = inv_freq[i];
        double lambda = two_pi / f;
        if (lambda < L / high_freq_factor)
            continue;
        if (lambda > L / low_freq_factor) {
            inv_freq[i] = f / factor;
            continue;
        }
        double s = (L / lambda - low_freq_factor) / (high_freq_factor - low_freq_factor);
        inv_freq[i] = (1.0 - s) * f / factor + s * f;
    }
    return 0;
}

/* Positions alone (for the packing tests): pos[r] = position of tok[r]. */
ORACLE_API int oracle_positions(int64_t *pos, const int64_t *tok, int64_t n,
                                const int32_t *cu, int32_t B)
{
    for (int64_t r = 0; r < n; ++r) {
        pos[r] = position_of(tok ? tok[r] : r, cu, B);
        if (pos[r] < 0)
            return -1;
    }
    return 0;
}
