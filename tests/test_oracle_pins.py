"""Pins of the CPU oracle against what the mathematics fixes.

None of these re-types an oracle formula.  Each checks one of: a closed form
worked by hand, an invariant of the op, central finite differences of the
oracle's own (separately pinned) forward pass, or a textbook special case
(complex multiplication for D=2 RoPE).  Together they are chosen so that a
dropped term, a wrong sign, a wrong frequency index or pairing, an
off-by-one position or a transposed operand in the oracle fails at least one.
"""
import cmath
import math

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(12345)


# ---------------------------------------------------------------- RMSNorm fwd

@pytest.mark.parametrize("c", [2.0, -3.0, 0.5])
@pytest.mark.parametrize("eps", [1e-6, 0.25])
def test_rmsnorm_constant_row(c, eps):
    # x = c * 1  ->  mean x^2 = c^2  ->  y = w c / sqrt(c^2 + eps)
    H = 37
    w = 1.0 + 0.1 * RNG.standard_normal(H)
    y, r = oracle.rmsnorm_fwd(np.full((1, H), c), w, eps)
    np.testing.assert_allclose(y[0], w * c / math.sqrt(c * c + eps), rtol=1e-14)
    np.testing.assert_allclose(r[0], 1 / math.sqrt(c * c + eps), rtol=1e-14)
    if eps == 1e-6:  # returns w (with the sign of c) as eps -> 0
        np.testing.assert_allclose(y[0], w * math.copysign(1, c), rtol=eps / c ** 2)


def test_rmsnorm_hand_example():
    # x = (3, 4): mean square = 25/2; w = (1, 2)
    y, r = oracle.rmsnorm_fwd(np.array([[3.0, 4.0]]), np.array([1.0, 2.0]), 0.0)
    s = math.sqrt(12.5)
    np.testing.assert_allclose(y[0], [3 / s, 8 / s], rtol=1e-15)
    np.testing.assert_allclose(r[0], 1 / s, rtol=1e-15)


def test_rmsnorm_eps_inside_root():
    # x = (1, 1), eps = 1: r = 1/sqrt(1 + 1), not 1/(1 + 1) or 1/sqrt(1) + 1
    y, r = oracle.rmsnorm_fwd(np.ones((1, 2)), np.ones(2), 1.0)
    np.testing.assert_allclose(r[0], 1 / math.sqrt(2), rtol=1e-15)


def test_rmsnorm_scale_invariance_and_rows_independent():
    x = RNG.standard_normal((6, 33))
    w = 1.0 + 0.1 * RNG.standard_normal(33)
    y, _ = oracle.rmsnorm_fwd(x, w, 0.0)
    y2, _ = oracle.rmsnorm_fwd(7.5 * x, w, 0.0)
    np.testing.assert_allclose(y2, y, rtol=1e-13)
    perm = RNG.permutation(6)
    y3, _ = oracle.rmsnorm_fwd(x[perm], w, 0.0)
    np.testing.assert_allclose(y3, y[perm], rtol=0, atol=0)
    # unit RMS of every output row when w = 1, eps = 0
    y4, _ = oracle.rmsnorm_fwd(x, np.ones(33), 0.0)
    np.testing.assert_allclose(np.sqrt((y4 ** 2).mean(axis=1)), 1.0, rtol=1e-13)


# ------------------------------------------------ finite-difference helpers

def _central_fd(f, arr, h_rel=1e-6):
    """d f / d arr by central differences, f: array -> scalar (float64)."""
    g = np.zeros_like(arr)
    flat, gflat = arr.reshape(-1), g.reshape(-1)
    for i in range(flat.size):
        h = h_rel * max(1.0, abs(flat[i]))
        old = flat[i]
        flat[i] = old + h
        fp = f(arr)
        flat[i] = old - h
        fm = f(arr)
        flat[i] = old
        gflat[i] = (fp - fm) / (2 * h)
    return g


def _fd_close(fd, an, rel=1e-7):
    scale = max(1.0, float(np.abs(an).max()))
    assert np.abs(fd - an).max() <= rel * scale * 10, (np.abs(fd - an).max(), scale)


# ---------------------------------------------------------------- RMSNorm bwd

@pytest.mark.parametrize("eps", [1e-6, 0.3])
def test_rmsnorm_bwd_matches_finite_differences(eps):
    T, H = 5, 12
    x = RNG.standard_normal((T, H))
    w = 1.0 + 0.1 * RNG.standard_normal(H)
    ghat = RNG.standard_normal((T, H))

    def loss_x(xx):
        return float((ghat * oracle.rmsnorm_fwd(xx, w, eps)[0]).sum())

    def loss_w(ww):
        return float((ghat * oracle.rmsnorm_fwd(x, ww, eps)[0]).sum())

    dx, dw = oracle.rmsnorm_bwd(ghat, x, w, eps)
    _fd_close(_central_fd(loss_x, x.copy()), dx)
    _fd_close(_central_fd(loss_w, w.copy()), dw)


def test_rmsnorm_bwd_scales_bound_values():
    T, H = 9, 40
    x, dy = RNG.standard_normal((T, H)), RNG.standard_normal((T, H))
    w = 1.0 + 0.1 * RNG.standard_normal(H)
    dx, dw, dxs, dws = oracle.rmsnorm_bwd(dy, x, w, 1e-6, scales=True)
    assert np.all(np.abs(dx) <= dxs * (1 + 1e-12))
    assert np.all(np.abs(dw) <= dws * (1 + 1e-12))
    # the scale form does not change the values
    dx2, dw2 = oracle.rmsnorm_bwd(dy, x, w, 1e-6)
    np.testing.assert_array_equal(dx, dx2)
    np.testing.assert_array_equal(dw, dw2)


def test_rmsnorm_bwd_zero_upstream():
    x = RNG.standard_normal((3, 8))
    dx, dw = oracle.rmsnorm_bwd(np.zeros((3, 8)), x, np.ones(8), 1e-6)
    assert not dx.any() and not dw.any()


def test_oracle_results_do_not_depend_on_thread_count():
    # the timing leg runs the oracle on one thread and on all of them
    x, dy = RNG.standard_normal((300, 200)), RNG.standard_normal((300, 200))
    w = 1 + 0.1 * RNG.standard_normal(200)
    prev = oracle.set_threads(1)
    try:
        one = oracle.rmsnorm_bwd(dy, x, w, 1e-6)
        oracle.set_threads(max(prev, 4))
        many = oracle.rmsnorm_bwd(dy, x, w, 1e-6)
    finally:
        oracle.set_threads(prev)
    assert oracle.threads() == prev
    assert np.array_equal(one[0], many[0]) and np.array_equal(one[1], many[1])


# ---------------------------------------------------------------- SwiGLU

def test_swiglu_special_values():
    u = np.array([1.7, -0.3, 2.0, 5.0])
    # silu(0) = 0
    assert np.all(oracle.swiglu_fwd(np.zeros(4), u) == 0)
    # sigmoid(ln 3) = 3/4 exactly in real arithmetic
    g = np.full(4, math.log(3.0))
    np.testing.assert_allclose(oracle.swiglu_fwd(g, u), 0.75 * math.log(3.0) * u, rtol=1e-15)
    # silu(g) -> g as g -> +inf and -> 0 as g -> -inf
    np.testing.assert_allclose(oracle.swiglu_fwd(np.full(4, 40.0), u), 40.0 * u, rtol=1e-15)
    assert np.all(np.abs(oracle.swiglu_fwd(np.full(4, -40.0), u)) < 1e-15)
    # swiglu_bwd at g = 0: sigmoid(0) = 1/2 -> dg = dh u / 2, du = 0
    dh = np.array([0.5, -2.0, 1.0, 3.0])
    dg, du = oracle.swiglu_bwd(dh, np.zeros(4), u)
    np.testing.assert_allclose(dg, dh * u / 2, rtol=1e-15)
    assert not du.any()


def test_swiglu_bwd_matches_finite_differences():
    n = 23
    g, u, dh = RNG.standard_normal(n) * 2, RNG.standard_normal(n), RNG.standard_normal(n)
    dg, du = oracle.swiglu_bwd(dh, g, u)
    fd_g = _central_fd(lambda gg: float((dh * oracle.swiglu_fwd(gg, u)).sum()), g.copy())
    fd_u = _central_fd(lambda uu: float((dh * oracle.swiglu_fwd(g, uu)).sum()), u.copy())
    _fd_close(fd_g, dg)
    _fd_close(fd_u, du)
    dg2, du2, dgs = oracle.swiglu_bwd(dh, g, u, scales=True)
    np.testing.assert_array_equal(dg, dg2)
    assert np.all(np.abs(dg) <= dgs * (1 + 1e-12))


# ---------------------------------------------------------------- QK-RoPE

def _single(q, k, p, theta, sign=+1):
    """Rotate one token at position p (a one-sequence batch of p+1 tokens)."""
    n = p + 1
    qq = np.zeros((n,) + q.shape)
    kk = np.zeros((n,) + k.shape)
    qq[p], kk[p] = q, k
    qo, ko = oracle.qk_rope(qq[p:p + 1], kk[p:p + 1], [0, n], theta, sign, tok=[p])
    return qo[0], ko[0]


def test_rope_hand_example_d4():
    # D = 4, theta = 100: pair 0 = (x0, x2) turns by p * 1, pair 1 = (x1, x3)
    # turns by p * 100^(-1/2) = p / 10.  Position 1.
    e = np.eye(4)
    k0 = np.zeros((1, 4))
    out = [_single(e[i][None, :], k0, 1, 100.0)[0][0] for i in range(4)]
    c1, s1, c2, s2 = math.cos(1), math.sin(1), math.cos(0.1), math.sin(0.1)
    np.testing.assert_allclose(out[0], [c1, 0, s1, 0], atol=1e-15)
    np.testing.assert_allclose(out[1], [0, c2, 0, s2], atol=1e-15)
    np.testing.assert_allclose(out[2], [-s1, 0, c1, 0], atol=1e-15)
    np.testing.assert_allclose(out[3], [0, -s2, 0, c2], atol=1e-15)
    # the backward rotation is the transpose
    back = _single(e[0][None, :], k0, 1, 100.0, sign=-1)[0][0]
    np.testing.assert_allclose(back, [c1, 0, -s1, 0], atol=1e-15)


@pytest.mark.parametrize("p", [0, 1, 7, 1000, 524287])
def test_rope_d2_is_complex_multiplication(p):
    # D = 2: the single frequency is theta^0 = 1, so (a, b) -> (a + ib) e^{ip}
    a, b = 0.8, -1.3
    z = complex(a, b) * cmath.exp(1j * p)
    qo, _ = _single(np.array([[a, b]]), np.zeros((1, 2)), p, 1e6)
    np.testing.assert_allclose(qo[0], [z.real, z.imag], rtol=0, atol=1e-12)


def _packed_case(D=16, Hq=4, Hkv=2, lens=(5, 17, 0, 32, 10)):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    q = RNG.standard_normal((T, Hq, D))
    k = RNG.standard_normal((T, Hkv, D))
    return cu, q, k


def test_rope_identity_at_sequence_starts_and_positions():
    cu, q, k = _packed_case()
    qo, ko = oracle.qk_rope(q, k, cu, 1e4)
    starts = sorted(set(int(c) for c in cu[:-1]) - {int(cu[-1])})
    for t in starts:
        np.testing.assert_array_equal(qo[t], q[t])
        np.testing.assert_array_equal(ko[t], k[t])
    pos = oracle.positions(cu)
    expect = np.concatenate([np.arange(l) for l in np.diff(cu)])
    np.testing.assert_array_equal(pos, expect)
    # no other token is left unrotated
    rotated = [t for t in range(int(cu[-1])) if t not in starts]
    assert all(np.abs(qo[t] - q[t]).max() > 0 for t in rotated)


def test_rope_preserves_pair_norms():
    cu, q, k = _packed_case(D=64, Hq=3, Hkv=1, lens=(100,))
    qo, ko = oracle.qk_rope(q, k, cu, 1e6)
    h = 32
    for a, b in ((q, qo), (k, ko)):
        n_in = a[..., :h] ** 2 + a[..., h:] ** 2
        n_out = b[..., :h] ** 2 + b[..., h:] ** 2
        np.testing.assert_allclose(n_out, n_in, rtol=1e-13)


def test_rope_relative_position_and_gqa():
    # q_m . k_n depends only on m - n inside one sequence; q-head h reads
    # kv-head floor(h * Hkv / Hq)
    D, Hq, Hkv = 16, 4, 2
    L = 64
    cu = np.array([0, 3, 3 + L], dtype=np.int32)
    T = 3 + L
    qv = RNG.standard_normal((Hq, D))
    kv = RNG.standard_normal((Hkv, D))
    q = np.broadcast_to(qv, (T, Hq, D)).copy()
    k = np.broadcast_to(kv, (T, Hkv, D)).copy()
    qo, ko = oracle.qk_rope(q, k, cu, 1e4)

    def score(m, n, h):
        return float(qo[3 + m, h] @ ko[3 + n, h * Hkv // Hq])

    for h in range(Hq):
        for (m, n), s in (((9, 4), 11), ((20, 20), 30), ((5, 17), 40)):
            assert abs(score(m, n, h) - score(m + s, n + s, h)) < 1e-12
    # tokens of the first sequence restart at position 0 in the second one
    np.testing.assert_array_equal(qo[3], q[3])
    np.testing.assert_allclose(qo[1], qo[4], rtol=0, atol=0)


def test_rope_packing_invariance():
    lens = (5, 17, 0, 32, 10)
    cu, q, k = _packed_case(lens=lens)
    qo, ko = oracle.qk_rope(q, k, cu, 1e4)
    for b in range(len(lens)):
        s, e = int(cu[b]), int(cu[b + 1])
        if s == e:
            continue
        qs, ks = oracle.qk_rope(q[s:e], k[s:e], [0, e - s], 1e4)
        np.testing.assert_array_equal(qs, qo[s:e])
        np.testing.assert_array_equal(ks, ko[s:e])


def test_rope_bwd_is_transpose_and_inverse():
    cu, q, k = _packed_case(D=32)
    gq = RNG.standard_normal(q.shape)
    gk = RNG.standard_normal(k.shape)
    qo, ko = oracle.qk_rope(q, k, cu, 5e5, +1)
    gqb, gkb = oracle.qk_rope(gq, gk, cu, 5e5, -1)
    # <R x, y> = <x, R^T y>
    lhs = float((qo * gq).sum() + (ko * gk).sum())
    rhs = float((q * gqb).sum() + (k * gkb).sum())
    assert abs(lhs - rhs) < 1e-11 * max(1.0, abs(lhs))
    # R^T R = I
    qi, ki = oracle.qk_rope(qo, ko, cu, 5e5, -1)
    np.testing.assert_allclose(qi, q, atol=1e-13)
    np.testing.assert_allclose(ki, k, atol=1e-13)


def test_rope_scale_bounds_output_and_is_unchanged_by_it():
    cu, q, k = _packed_case(D=32)
    qo, ko = oracle.qk_rope(q, k, cu, 1e4)
    qs_, ks_, qsc, ksc = oracle.qk_rope(q, k, cu, 1e4, scales=True)
    np.testing.assert_array_equal(qo, qs_)
    np.testing.assert_array_equal(ko, ks_)
    assert np.all(np.abs(qo) <= qsc * (1 + 1e-12))
    assert np.all(np.abs(ko) <= ksc * (1 + 1e-12))


def test_rope_scale_covers_the_angle_sensitivity_of_the_complex_product():
    # D = 2 is multiplication by e^{i p} (inv_freq = theta^0 = 1), whose
    # derivative in the angle is i times the product: the real output moves
    # by |Im| per radian and the imaginary one by |Re|.  The scale must hold
    # each output's magnitude plus a tenth of that motion (a 1e-6 rad angle
    # error against the 1e-5 fp32 relative bar), and with the angle error
    # that large the perturbed product must stay inside the fp32 bar.
    rng = np.random.default_rng(5)
    T = 4000
    q = rng.standard_normal((T, 1, 2))
    cu = [0, T]
    qo, _, qsc, _ = oracle.qk_rope(q, np.zeros((T, 0, 2)), cu, 1e4, scales=True)
    z = (q[:, 0, 0] + 1j * q[:, 0, 1]) * np.exp(1j * np.arange(T))
    re, im = qo[:, 0, 0], qo[:, 0, 1]
    np.testing.assert_allclose(re + 1j * im, z, atol=1e-12)
    assert np.all(qsc[:, 0, 0] >= (np.abs(re) + 0.1 * np.abs(im)) * (1 - 1e-12))
    assert np.all(qsc[:, 0, 1] >= (np.abs(im) + 0.1 * np.abs(re)) * (1 - 1e-12))
    zp = (q[:, 0, 0] + 1j * q[:, 0, 1]) * np.exp(1j * (np.arange(T) + 1e-6))
    assert np.all(np.abs(zp.real - re) <= 1e-5 * qsc[:, 0, 0] + 1e-15)
    assert np.all(np.abs(zp.imag - im) <= 1e-5 * qsc[:, 0, 1] + 1e-15)
    # an angle error ten times larger falls outside it somewhere
    zb = (q[:, 0, 0] + 1j * q[:, 0, 1]) * np.exp(1j * (np.arange(T) + 1e-5))
    assert np.any(np.abs(zb.real - re) > 1e-5 * qsc[:, 0, 0])


def test_rope_sampled_rows_equal_full():
    cu, q, k = _packed_case()
    qo, ko = oracle.qk_rope(q, k, cu, 1e4)
    tok = np.array([63, 0, 22, 21, 5])
    qs, ks = oracle.qk_rope(q[tok], k[tok], cu, 1e4, tok=tok)
    np.testing.assert_array_equal(qs, qo[tok])
    np.testing.assert_array_equal(ks, ko[tok])


def test_rope_rejects_out_of_batch_token():
    cu, q, k = _packed_case()
    with pytest.raises(ValueError):
        oracle.qk_rope(q[:1], k[:1], cu, 1e4, tok=[int(cu[-1])])


# ------------------------------------------------ RoPE with a frequency table

@pytest.mark.parametrize("p", [0, 3, 40000])
def test_rope_freq_d2_is_complex_multiplication(p):
    # D = 2 with an arbitrary frequency f: (a, b) -> (a + ib) e^{i p f}
    f, a, b = 0.37, -0.6, 1.9
    z = complex(a, b) * cmath.exp(1j * p * f)
    qo, _ = oracle.qk_rope_freq(np.array([[[a, b]]]), np.zeros((1, 1, 2)), [0, p + 1], [f],
                                tok=[p])
    np.testing.assert_allclose(qo[0, 0], [z.real, z.imag], rtol=0, atol=1e-12)
    back, _ = oracle.qk_rope_freq(np.array([[[a, b]]]), np.zeros((1, 1, 2)), [0, p + 1], [f],
                                  sign=-1, tok=[p])
    zb = complex(a, b) * cmath.exp(-1j * p * f)
    np.testing.assert_allclose(back[0, 0], [zb.real, zb.imag], rtol=0, atol=1e-12)


def test_rope_inv_freq_closed_forms():
    # theta^(-2i/D): 1 at i = 0, theta^(-1/2) at i = D/4, a geometric sequence
    f = oracle.rope_inv_freq(128, 5e5)
    assert f[0] == 1.0
    assert math.isclose(f[32], 5e5 ** -0.5, rel_tol=1e-15)
    np.testing.assert_allclose(f[1:] / f[:-1], 5e5 ** (-2 / 128), rtol=1e-13)


def test_rope_freq_table_drives_each_pair():
    # pair i turns by p * f[i]: with f = e_1 (only pair 1 turns) a unit vector
    # in pair 0 stays put and one in pair 1 turns by p
    D, p = 8, 5
    f = np.array([0.0, 1.0, 0.0, 0.0])
    e = np.eye(D)
    qo, _ = oracle.qk_rope_freq(e[None, :, :], np.zeros((1, 0, D)), [0, p + 1], f, tok=[p])
    np.testing.assert_allclose(qo[0, 0], e[0], atol=1e-15)
    np.testing.assert_allclose(qo[0, 1], math.cos(p) * e[1] + math.sin(p) * e[5], atol=1e-15)


LLAMA32 = dict(factor=32.0, low_freq_factor=1.0, high_freq_factor=4.0,
               original_max_position=8192.0)


def test_llama3_factor_one_is_unscaled():
    for lo, hi in ((1.0, 4.0), (2.0, 3.0)):
        f = oracle.rope_llama3_inv_freq(64, 5e5, 1.0, lo, hi, 8192.0)
        np.testing.assert_allclose(f, oracle.rope_inv_freq(64, 5e5), rtol=1e-15)


def test_llama3_bands_for_llama32_shapes():
    # D = 64, theta = 5e5: wavelength 2 pi 5e5^(i/32) is below 8192/4 = 2048
    # for i <= 14 (1956 at i = 14), above 8192/1 for i >= 18 (10081 at i =
    # 18), and in between for i = 15, 16, 17 (2949 .. 6692)
    f0 = oracle.rope_inv_freq(64, 5e5)
    f = oracle.rope_llama3_inv_freq(64, 5e5, **LLAMA32)
    assert np.array_equal(f[:15], f0[:15])
    np.testing.assert_allclose(f[18:], f0[18:] / 32, rtol=1e-15)
    mid = f[15:18] / f0[15:18]
    assert np.all(mid > 1 / 32) and np.all(mid < 1)
    # the kept share falls as the wavelength grows
    assert np.all(np.diff(mid) < 0)


def test_llama3_blend_endpoints_and_midpoint():
    # pick L so that dimension i sits exactly on a band edge or halfway: the
    # blend must meet the unscaled frequency at L/lambda = high, the divided
    # one at L/lambda = low, and their mean halfway between
    D, theta, factor, lo, hi = 32, 1e4, 8.0, 1.0, 4.0
    f0 = oracle.rope_inv_freq(D, theta)
    i = 9
    lam = 2 * math.pi / f0[i]
    for L, want in ((hi * lam, f0[i]), (lo * lam, f0[i] / factor),
                    ((lo + hi) / 2 * lam, 0.5 * (f0[i] + f0[i] / factor))):
        f = oracle.rope_llama3_inv_freq(D, theta, factor, lo, hi, L)
        assert math.isclose(f[i], want, rel_tol=1e-12), (L, f[i], want)


def test_llama3_rejects_bad_bands():
    with pytest.raises(ValueError):
        oracle.rope_llama3_inv_freq(64, 5e5, 32.0, 4.0, 4.0, 8192.0)
    with pytest.raises(ValueError):
        oracle.rope_llama3_inv_freq(63, 5e5, 32.0, 1.0, 4.0, 8192.0)


# ------------------------------------------- per-head QK-RMSNorm, then RoPE

def test_qk_norm_rope_unit_rms_inputs_reduce_to_rope():
    # entries of +-1 have mean square 1: with w = 1 and eps = 0 the norm is
    # the identity, so the op is the rotation alone
    cu, q, k = _packed_case(D=16)
    q, k = np.sign(q), np.sign(k)
    f = oracle.rope_inv_freq(16, 1e4)
    qo, ko, rq, rk = oracle.qk_norm_rope_fwd(q, k, np.ones(16), np.ones(16), 0.0, cu, f)
    qr, kr = oracle.qk_rope_freq(q, k, cu, f)
    np.testing.assert_allclose(qo, qr, atol=1e-14)
    np.testing.assert_allclose(ko, kr, atol=1e-14)
    assert np.allclose(rq, 1.0) and np.allclose(rk, 1.0)


def test_qk_norm_rope_head_norms():
    # rotation keeps lengths: with w = 1 each output head vector has squared
    # length D * ms / (ms + eps), ms its input's mean square
    cu, q, k = _packed_case(D=32, Hq=3, Hkv=1)
    eps = 0.25
    f = oracle.rope_inv_freq(32, 1e6)
    qo, ko, _, _ = oracle.qk_norm_rope_fwd(q, k, np.ones(32), np.ones(32), eps, cu, f)
    for v, o in ((q, qo), (k, ko)):
        ms = (v ** 2).mean(axis=-1)
        np.testing.assert_allclose((o ** 2).sum(axis=-1), 32 * ms / (ms + eps), rtol=1e-12)


def test_qk_norm_rope_hand_example_d2():
    # v = (3, 4), w = (1, 2), eps = 0: ms = 12.5, r = 12.5^-1/2, normalised
    # n = (3r, 8r); at p = 0 it is the output, at p = 2 with f = 1 it is
    # turned by 2 rad: (3r + 8r i) e^{2i}
    r = 12.5 ** -0.5
    v = np.array([[[3.0, 4.0]]])
    k0 = np.zeros((1, 0, 2))
    for p, z in ((0, complex(3 * r, 8 * r)), (2, complex(3 * r, 8 * r) * cmath.exp(2j))):
        qo, _, rq, _ = oracle.qk_norm_rope_fwd(v, k0, [1.0, 2.0], [1.0, 2.0], 0.0, [0, p + 1],
                                               [1.0], tok=[p])
        np.testing.assert_allclose(qo[0, 0], [z.real, z.imag], atol=1e-14)
        assert math.isclose(rq[0, 0], r, rel_tol=1e-15)


def test_qk_norm_rope_bwd_matches_finite_differences():
    cu, q, k = _packed_case(D=8, Hq=2, Hkv=1, lens=(3, 0, 4))
    wq, wk = 1 + 0.1 * RNG.standard_normal(8), 1 + 0.1 * RNG.standard_normal(8)
    f = oracle.rope_llama3_inv_freq(8, 1e4, 4.0, 1.0, 4.0, 16.0)
    eps = 1e-3
    dq, dk = RNG.standard_normal(q.shape), RNG.standard_normal(k.shape)

    def loss(q_, k_, wq_, wk_):
        qo, ko, _, _ = oracle.qk_norm_rope_fwd(q_, k_, wq_, wk_, eps, cu, f)
        return float((dq * qo).sum() + (dk * ko).sum())

    gq, gk, gwq, gwk = oracle.qk_norm_rope_bwd(dq, dk, q, k, wq, wk, eps, cu, f)
    h = 1e-6
    for arr, g in ((q, gq), (k, gk), (wq, gwq), (wk, gwk)):
        e = RNG.standard_normal(arr.shape)
        args_p = [q, k, wq, wk]
        args_m = [q, k, wq, wk]
        i = [id(q), id(k), id(wq), id(wk)].index(id(arr))
        args_p[i], args_m[i] = arr + h * e, arr - h * e
        fd = (loss(*args_p) - loss(*args_m)) / (2 * h)
        assert math.isclose(fd, float((g * e).sum()), rel_tol=1e-6, abs_tol=1e-8)


def test_qk_norm_rope_bwd_scales_bound_values():
    cu, q, k = _packed_case(D=16)
    w = 1 + 0.1 * RNG.standard_normal(16)
    f = oracle.rope_inv_freq(16, 1e4)
    dq, dk = RNG.standard_normal(q.shape), RNG.standard_normal(k.shape)
    out = oracle.qk_norm_rope_bwd(dq, dk, q, k, w, w, 1e-6, cu, f, scales=True)
    for v, sc in zip(out[:4], out[4:]):
        assert np.all(np.abs(v) <= sc * (1 + 1e-12))


# ------------------------------------------------- RMSNorm with residual add

def test_rmsnorm_add_reduces_to_rmsnorm():
    # res = 0: h = x exactly (a stored value plus zero), y = rmsnorm(x)
    x = RNG.standard_normal((7, 24)).astype(np.float32).astype(np.float64)
    w = 1.0 + 0.1 * RNG.standard_normal(24)
    h, y, r = oracle.rmsnorm_add_fwd(x, np.zeros_like(x), w, 1e-6, storage="f32")
    y0, r0 = oracle.rmsnorm_fwd(x, w, 1e-6)
    np.testing.assert_array_equal(h, x)
    np.testing.assert_array_equal(y, y0)
    np.testing.assert_array_equal(r, r0)


def test_rmsnorm_add_storage_rounding():
    # bf16 keeps 8 significant bits: ulp(1) = 2^-7.  1 + 2^-8 is a tie between
    # 1 and 1 + 2^-7 and rounds to the even 1; 1 + 3*2^-8 is a tie between
    # 1 + 2^-7 (odd) and 1 + 2^-6 (even) and rounds up; 1 + 2^-8 + 2^-12 is
    # above the tie and rounds up.
    x = np.array([[1.0, 1.0, 1.0, -1.0]])
    res = np.array([[2.0 ** -8, 3 * 2.0 ** -8, 2.0 ** -8 + 2.0 ** -12, -(2.0 ** -8)]])
    h, _, _ = oracle.rmsnorm_add_fwd(x, res, np.ones(4), 1e-6, storage="bf16")
    np.testing.assert_array_equal(h[0], [1.0, 1 + 2.0 ** -6, 1 + 2.0 ** -7, -1.0])
    hf, _, _ = oracle.rmsnorm_add_fwd(x, res, np.ones(4), 1e-6, storage="f32")
    np.testing.assert_array_equal(hf[0], x[0] + res[0])  # exact in fp32
    # fp32 rounding: 1 + 2^-24 is a tie between 1 and 1 + 2^-23 -> 1
    hf, _, _ = oracle.rmsnorm_add_fwd(np.ones((1, 1)), np.full((1, 1), 2.0 ** -24),
                                      np.ones(1), 1e-6, storage="f32")
    assert hf[0, 0] == 1.0


def test_rmsnorm_add_bwd_matches_finite_differences():
    # L = sum(gy * y) + sum(gh * h) with h = x + res unrounded; dL/dx = dL/dres
    T, H = 4, 10
    x, res = RNG.standard_normal((T, H)), RNG.standard_normal((T, H))
    w = 1.0 + 0.1 * RNG.standard_normal(H)
    gy, gh = RNG.standard_normal((T, H)), RNG.standard_normal((T, H))

    def loss(xx, rr, ww):
        h, y, _ = oracle.rmsnorm_add_fwd(xx, rr, ww, 1e-6, storage="exact")
        return float((gy * y).sum() + (gh * h).sum())

    h, _, _ = oracle.rmsnorm_add_fwd(x, res, w, 1e-6, storage="exact")
    dx, dw = oracle.rmsnorm_add_bwd(gy, gh, h, w, 1e-6)
    _fd_close(_central_fd(lambda xx: loss(xx, res, w), x.copy()), dx)
    _fd_close(_central_fd(lambda rr: loss(x, rr, w), res.copy()), dx)
    _fd_close(_central_fd(lambda ww: loss(x, res, ww), w.copy()), dw)
    # linear in the residual gradient
    dx0, dw0 = oracle.rmsnorm_add_bwd(gy, np.zeros_like(gh), h, w, 1e-6)
    np.testing.assert_allclose(dx - dx0, gh, atol=1e-14)
    np.testing.assert_array_equal(dw, dw0)
