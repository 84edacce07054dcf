"""Pins of the cross-entropy oracle (oracle/cce.py) against closed forms,
invariants and finite differences; and of the memory arithmetic the page
quotes for the online-softmax loss (5 GB of fp32 logits down to 135 MB)."""
import math

import numpy as np
import pytest

from oracle import cce

RNG = np.random.default_rng(2024)


def test_zero_head_gives_log_v():
    # W = 0: every logit is 0, lse = log V, loss = log V, dz = (1/V - onehot)/N
    T, H, V = 5, 7, 11
    h = RNG.standard_normal((T, H))
    y = np.array([0, 3, 10, -100, 4])
    loss, lse, n = cce.cce_fwd(h, np.zeros((V, H)), y)
    assert n == 4
    np.testing.assert_allclose(lse, math.log(V), rtol=1e-15)
    assert math.isclose(loss, math.log(V), rel_tol=1e-15)
    dz = cce.dz_rows(h, np.zeros((V, H)), y, 2.0, n)
    want = np.full((T, V), 1.0 / V)
    want[np.arange(T), np.where(y < 0, 0, y)] -= 1.0
    want[3] = 0.0
    np.testing.assert_allclose(dz, want * 2.0 / 4, atol=1e-16)


def test_two_classes_is_logistic_loss():
    # V = 2: loss = log(1 + e^(z_other - z_target)) (softplus of the margin)
    h = np.array([[1.5, -0.5]])
    W = np.array([[0.3, 2.0], [-1.0, 0.7]])
    z = h @ W.T
    for t in (0, 1):
        loss, _, _ = cce.cce_fwd(h, W, [t])
        other = z[0, 1 - t] - z[0, t]
        assert math.isclose(loss, math.log1p(math.exp(other)), rel_tol=1e-14)


def test_common_shift_of_the_head_changes_nothing():
    # adding one vector u to every row of W adds h.u to every logit of a
    # token: loss and dh stay, since each dz row sums to zero
    T, H, V = 6, 5, 9
    h, W = RNG.standard_normal((T, H)), RNG.standard_normal((V, H))
    y = RNG.integers(0, V, T)
    u = RNG.standard_normal(H)
    l1, _, _ = cce.cce_fwd(h, W, y)
    l2, _, _ = cce.cce_fwd(h, W + u, y)
    assert math.isclose(l1, l2, rel_tol=1e-12)
    dh1, _ = cce.cce_bwd(h, W, y)
    dh2, _ = cce.cce_bwd(h, W + u, y)
    np.testing.assert_allclose(dh1, dh2, atol=1e-13)


def test_gradients_match_finite_differences():
    T, H, V = 4, 3, 6
    h, W = RNG.standard_normal((T, H)), RNG.standard_normal((V, H))
    y = np.array([1, -100, 5, 0])
    g = 0.7
    dh, dW = cce.cce_bwd(h, W, y, g)
    eps = 1e-6
    for arr, grad in ((h, dh), (W, dW)):
        e = RNG.standard_normal(arr.shape)
        hp, Wp = (h + eps * e, W) if arr is h else (h, W + eps * e)
        hm, Wm = (h - eps * e, W) if arr is h else (h, W - eps * e)
        fd = g * (cce.cce_fwd(hp, Wp, y)[0] - cce.cce_fwd(hm, Wm, y)[0]) / (2 * eps)
        assert math.isclose(fd, float((grad * e).sum()), rel_tol=1e-7, abs_tol=1e-10)


def test_dw_columns_sum_to_zero_and_sampling_agrees():
    T, H, V = 9, 4, 13
    h, W = RNG.standard_normal((T, H)), RNG.standard_normal((V, H))
    y = RNG.integers(0, V, T)
    y[2] = -100
    dh, dW, dhs, dWs = cce.cce_bwd(h, W, y, scales=True, chunk=4)
    np.testing.assert_allclose(dW.sum(axis=0), 0.0, atol=1e-14)
    assert np.all(np.abs(dh) <= dhs * (1 + 1e-12)) and np.all(np.abs(dW) <= dWs * (1 + 1e-12))
    # the sampled forms (some tokens, some vocabulary rows) equal the full ones
    dh_s, dW_s = cce.cce_bwd(h, W, y, tok=[8, 0, 5], vocab=[12, 3], chunk=2)
    np.testing.assert_allclose(dh_s, dh[[8, 0, 5]], rtol=1e-14, atol=1e-16)
    np.testing.assert_allclose(dW_s, dW[[12, 3]], rtol=1e-13, atol=1e-16)
    assert np.all(dh[2] == 0.0)  # an ignored token gets no gradient


def test_all_ignored():
    h, W = RNG.standard_normal((3, 2)), RNG.standard_normal((4, 2))
    loss, _, n = cce.cce_fwd(h, W, [-100, -100, -100])
    assert n == 0 and loss == 0.0
    dh, dW = cce.cce_bwd(h, W, [-100, -100, -100])
    assert not dh.any() and not dW.any()


def test_memory_arithmetic_of_the_page():
    # Qwen2.5-0.5B (vocabulary 151,936), 8,192 tokens: fp32 logits take
    # ~5 GB; a 4,096-column slice of them takes ~135 MB
    T, V, C = 8192, 151936, 4096
    assert round(T * V * 4 / 1e9, 2) == 4.98
    assert round(T * C * 4 / 1e6) == 134
