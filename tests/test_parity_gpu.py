"""CUDA kernels vs the double-precision oracle on the five seeded workloads.

Small workloads are compared element by element in full.  At full size the
kernels run on the whole batch in the same launch configuration the
benchmark times, and the oracle checks sampled rows/tokens (always including
the first and last ones, so every ragged tail is covered); RMSNorm's dw, a
reduction over every row, is checked in full by summing the oracle's
per-chunk column sums in double.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.tolerance import assert_close, f64
from fine_tuning_gb300 import build, ftk
from fine_tuning_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda"
SMALL = ("tiny_f32", "qwen2.5-0.5b")
LARGE = ("llama-3.2-1b", "qwen3-8b")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ftk.library()
    ftk.device_status(clear=True)
    yield
    torch.cuda.empty_cache()


@pytest.fixture(autouse=True)
def _no_wait_timeouts():
    yield
    # no kernel's bounded pipeline wait may have run out during the test
    assert ftk.device_status(clear=True) == 0


def dt(wl):
    return "f32" if wl.dtype == "f32" else "bf16"


def sample_rows(T, n, seed=7, extra=()):
    if T <= n:
        return np.arange(T)
    rng = np.random.default_rng(seed)
    s = set(rng.choice(T, n, replace=False).tolist()) | {0, 1, T - 2, T - 1} | set(extra)
    return np.array(sorted(x for x in s if 0 <= x < T))


def dw_oracle_chunked(dy, x, w, eps, chunk=16384):
    """Full-batch dw and its scale: oracle column sums per chunk, added in double."""
    T, H = x.shape
    dw = np.zeros(H)
    dws = np.zeros(H)
    wc = w.cpu()
    for a in range(0, T, chunk):
        b = min(T, a + chunk)
        _, p, _, ps = oracle.rmsnorm_bwd(dy[a:b].cpu(), x[a:b].cpu(), wc, eps, scales=True)
        dw += p
        dws += ps
    return dw, dws


# ------------------------------------------------------------------ RMSNorm

def check_rmsnorm(wl, n_rows=None):
    d = W.rmsnorm_inputs(wl, DEV)
    x, w, dy = d["x"], d["w"], d["dy"]
    y, rstd = ftk.rmsnorm_fwd(x, w, wl.eps)
    dx, dw = ftk.rmsnorm_bwd(dy, x, w, rstd, wl.eps)
    dx_re, dw_re = ftk.rmsnorm_bwd(dy, x, w, None, wl.eps)
    torch.cuda.synchronize()
    rows = np.arange(wl.T) if n_rows is None else sample_rows(wl.T, n_rows)
    ri = torch.as_tensor(rows, device=DEV)
    xs, dys = x[ri].cpu(), dy[ri].cpu()
    yr, rr = oracle.rmsnorm_fwd(xs, w.cpu(), wl.eps)
    dxr, _, dxs, _ = oracle.rmsnorm_bwd(dys, xs, w.cpu(), wl.eps, scales=True)
    assert_close("y", y[ri], yr, dtype=dt(wl))
    assert_close("rstd", rstd[ri], rr, dtype="f32")
    assert_close("dx", dx[ri], dxr, dxs, dtype=dt(wl))
    dwr, dws = dw_oracle_chunked(dy, x, w, wl.eps)
    assert_close("dw", dw, dwr, dws, dtype=dt(wl), kind="dw")
    # recomputing rstd in the backward pass reproduces the saved one exactly
    assert torch.equal(dx, dx_re) and torch.equal(dw, dw_re)


@pytest.mark.parametrize("name", SMALL)
def test_rmsnorm_small_full(name):
    check_rmsnorm(W.WORKLOADS[name])


@pytest.mark.parametrize("name", LARGE)
def test_rmsnorm_large_sampled(name):
    check_rmsnorm(W.WORKLOADS[name], n_rows=2048)


@pytest.mark.slow
def test_rmsnorm_524k_sampled():
    check_rmsnorm(W.WORKLOADS["qwen3-32b-524k"], n_rows=1024)


# ------------------------------------------------------------------- SwiGLU

def check_swiglu(wl, n_rows=None):
    d = W.swiglu_inputs(wl, DEV)
    g, u, dh = d["g"], d["u"], d["dh"]
    h = ftk.swiglu_fwd(g, u)
    dg, du = ftk.swiglu_bwd(dh, g, u)
    dg2, du2, h2 = ftk.swiglu_bwd_h(dh, g, u)
    torch.cuda.synchronize()
    # the backward that re-emits h: h exactly as the forward wrote it, and
    # the same dg, du
    assert torch.equal(h2, h) and torch.equal(dg2, dg) and torch.equal(du2, du)
    rows = np.arange(wl.T_swiglu) if n_rows is None else sample_rows(wl.T_swiglu, n_rows)
    ri = torch.as_tensor(rows, device=DEV)
    gs, us, dhs = g[ri].cpu(), u[ri].cpu(), dh[ri].cpu()
    hr = oracle.swiglu_fwd(gs, us)
    dgr, dur, dgs = oracle.swiglu_bwd(dhs, gs, us, scales=True)
    assert_close("h", h[ri], hr, dtype=dt(wl))
    assert_close("dg", dg[ri], dgr, dgs, dtype=dt(wl))
    assert_close("du", du[ri], dur, dtype=dt(wl))


def test_swiglu_tiny_full():
    check_swiglu(W.WORKLOADS["tiny_f32"])


@pytest.mark.parametrize("name", ("qwen2.5-0.5b",) + LARGE)
def test_swiglu_sampled(name):
    check_swiglu(W.WORKLOADS[name], n_rows=512)


@pytest.mark.slow
def test_swiglu_524k_slice_sampled():
    check_swiglu(W.WORKLOADS["qwen3-32b-524k"], n_rows=256)


# ------------------------------------------------------------------ QK-RoPE

LLAMA3 = dict(factor=32.0, low_freq_factor=1.0, high_freq_factor=4.0,
              original_max_position=8192.0)  # the Llama-3.2 rope_scaling


def check_rope(wl, n_tok=None, llama3=False):
    """llama3=True rotates with the llama3-scaled table (the library's own
    table on the GPU, the oracle's table on the CPU)."""
    lens = W.draw_lengths(wl)
    cu = W.cu_seqlens_from_lengths(lens)
    cu_d = torch.as_tensor(cu, device=DEV)
    d = W.rope_inputs(wl, DEV)
    starts = cu[:-1].tolist()
    tok = np.arange(wl.T) if n_tok is None else sample_rows(
        wl.T, n_tok, extra=starts[:64] + [s - 1 for s in starts[1:64]])
    ti = torch.as_tensor(tok, device=DEV)
    q0, k0, dq0, dk0 = (d[n][ti].cpu() for n in ("q", "k", "dq", "dk"))
    if llama3:
        f_gpu = ftk.rope_llama3_inv_freq(wl.D, wl.theta, **LLAMA3)
        f_ref = oracle.rope_llama3_inv_freq(wl.D, wl.theta, **LLAMA3)
        ftk.qk_rope_freq_fwd(d["q"], d["k"], cu_d, f_gpu)
        ftk.qk_rope_freq_bwd(d["dq"], d["dk"], cu_d, f_gpu)
        torch.cuda.synchronize()
        qr, kr, qs, ks = oracle.qk_rope_freq(q0, k0, cu, f_ref, +1, tok=tok, scales=True)
        dqr, dkr, dqs, dks = oracle.qk_rope_freq(dq0, dk0, cu, f_ref, -1, tok=tok, scales=True)
    else:
        ftk.qk_rope_fwd(d["q"], d["k"], cu_d, wl.theta)
        ftk.qk_rope_bwd(d["dq"], d["dk"], cu_d, wl.theta)
        torch.cuda.synchronize()
        qr, kr, qs, ks = oracle.qk_rope(q0, k0, cu, wl.theta, +1, tok=tok, scales=True)
        dqr, dkr, dqs, dks = oracle.qk_rope(dq0, dk0, cu, wl.theta, -1, tok=tok, scales=True)
    assert_close("q", d["q"][ti], qr, qs, dtype=dt(wl))
    assert_close("k", d["k"][ti], kr, ks, dtype=dt(wl))
    assert_close("dq", d["dq"][ti], dqr, dqs, dtype=dt(wl))
    assert_close("dk", d["dk"][ti], dkr, dks, dtype=dt(wl))


@pytest.mark.parametrize("name", SMALL)
def test_rope_small_full(name):
    check_rope(W.WORKLOADS[name])


@pytest.mark.parametrize("name", LARGE)
def test_rope_large_sampled(name):
    check_rope(W.WORKLOADS[name], n_tok=4096)


@pytest.mark.parametrize("name", ("tiny_f32", "qwen2.5-0.5b", "llama-3.2-1b"))
def test_rope_llama3_scaled(name):
    wl = W.WORKLOADS[name]
    check_rope(wl, n_tok=None if wl.T <= 16384 else 4096, llama3=True)


@pytest.mark.slow
def test_rope_llama3_scaled_524k_sampled():
    check_rope(W.WORKLOADS["qwen3-32b-524k"], n_tok=2048, llama3=True)


@pytest.mark.slow
def test_rope_524k_long_index_sampled():
    wl = W.WORKLOADS["qwen3-32b-524k"]
    assert wl.T * wl.Hq * wl.D >= 2 ** 32  # Q has more than 2^31 elements
    check_rope(wl, n_tok=2048)


@pytest.mark.slow
def test_rope_angle_every_position_to_524k():
    """cos/sin of every (position, frequency) pair for p < 524288, D = 128,
    theta = 1e6, in fp32: a unit first half gives (cos phi, sin phi) back.
    The angle must hold 1e-6 rad everywhere (a plain fp32 product of
    position and inverse frequency is off by up to ~3e-2 rad here)."""
    T, D, theta = 524288, 128, 1e6
    q = torch.zeros((T, 1, D), dtype=torch.float32, device=DEV)
    q[:, :, : D // 2] = 1.0
    cu = torch.tensor([0, T], dtype=torch.int32, device=DEV)
    ftk.qk_rope_fwd(q, None, cu, theta)
    got = f64(q[:, 0, :])
    ref_q, _ = oracle.qk_rope(np.concatenate([np.ones((T, 1, D // 2)), np.zeros((T, 1, D // 2))], axis=2),
                              np.zeros((T, 0, D)), [0, T], theta)
    err = np.abs(got - ref_q[:, 0, :]).max()
    assert err <= 1e-6, err
