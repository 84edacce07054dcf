"""Per-head QK-RMSNorm fused into QK-RoPE: CUDA vs the oracle.

The oracle runs its pinned RMSNorm (rows of D) and its pinned table-driven
rotation one after the other in double.  Full comparison on the small
workloads, sampled tokens (always the first and last, and sequence starts)
on the large ones; dwq and dwk, sums over every token and head, in full
against the oracle's chunked sums.  Also: a recomputed r equals the saved
one bit for bit, in-place forms, Q-only / K-only, the element-wise path,
a llama3-scaled table, canaries around every output.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.tolerance import assert_close
from fine_tuning_gb300 import build, ftk
from fine_tuning_gb300 import workloads as W
from test_edge_gpu import Guarded, randn, code
from test_parity_gpu import sample_rows

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ftk.library()
    ftk.device_status(clear=True)
    yield
    torch.cuda.empty_cache()


def dt(wl):
    return "f32" if wl.dtype == "f32" else "bf16"


def dw_oracle_chunked(dq, dk, q, k, wq, wk, eps, cu, f, chunk=4096):
    """dwq, dwk and their scales over every token, the oracle run chunk by
    chunk (rows = global token ids) and added in double."""
    T, D = q.shape[0], q.shape[2]
    acc = [np.zeros(D) for _ in range(4)]
    for a in range(0, T, chunk):
        b = min(T, a + chunk)
        out = oracle.qk_norm_rope_bwd(dq[a:b].cpu(), dk[a:b].cpu(), q[a:b].cpu(), k[a:b].cpu(),
                                      wq.cpu(), wk.cpu(), eps, cu, f, tok=np.arange(a, b),
                                      scales=True)
        for i, v in enumerate((out[2], out[3], out[6], out[7])):
            acc[i] += v
    return acc


def check(wl, n_tok=None, llama3=False, dw=True):
    d = W.qk_norm_rope_inputs(wl, DEV)
    q, k, gq, gk, wq, wk = d["q"], d["k"], d["dq"], d["dk"], d["wq"], d["wk"]
    cu = W.cu_seqlens_from_lengths(W.draw_lengths(wl))
    cu_d = torch.as_tensor(cu, device=DEV)
    if llama3:
        f_gpu = ftk.rope_llama3_inv_freq(wl.D, wl.theta, 32.0, 1.0, 4.0, 8192.0)
        f_ref = oracle.rope_llama3_inv_freq(wl.D, wl.theta, 32.0, 1.0, 4.0, 8192.0)
        kw = dict(inv_freq=f_gpu)
    else:
        f_ref = oracle.rope_inv_freq(wl.D, wl.theta)
        kw = dict(theta=wl.theta)
    eps = wl.eps
    qo, ko, rq, rk = ftk.qk_norm_rope_fwd(q, k, wq, wk, cu_d, eps, **kw)
    dq, dk, dwq, dwk = ftk.qk_norm_rope_bwd(gq, gk, q, k, wq, wk, rq, rk, cu_d, eps, **kw)
    dq2, dk2, dwq2, dwk2 = ftk.qk_norm_rope_bwd(gq, gk, q, k, wq, wk, None, None, cu_d, eps, **kw)
    torch.cuda.synchronize()
    assert ftk.device_status(clear=True) == 0
    starts = cu[:-1].tolist()
    tok = np.arange(wl.T) if n_tok is None else sample_rows(
        wl.T, n_tok, extra=starts[:64] + [s - 1 for s in starts[1:64]])
    ti = torch.as_tensor(tok, device=DEV)
    qr, kr, rqr, rkr, qs, ks = oracle.qk_norm_rope_fwd(q[ti].cpu(), k[ti].cpu(), wq.cpu(),
                                                       wk.cpu(), eps, cu, f_ref, tok=tok,
                                                       scales=True)
    assert_close("q_out", qo[ti], qr, qs, dtype=dt(wl))
    assert_close("k_out", ko[ti], kr, ks, dtype=dt(wl))
    assert_close("rstd_q", rq[ti], rqr, dtype="f32")
    assert_close("rstd_k", rk[ti], rkr, dtype="f32")
    out = oracle.qk_norm_rope_bwd(gq[ti].cpu(), gk[ti].cpu(), q[ti].cpu(), k[ti].cpu(), wq.cpu(),
                                  wk.cpu(), eps, cu, f_ref, tok=tok, scales=True)
    assert_close("dq", dq[ti], out[0], out[4], dtype=dt(wl))
    assert_close("dk", dk[ti], out[1], out[5], dtype=dt(wl))
    if dw:
        dwqr, dwkr, dwqs, dwks = dw_oracle_chunked(gq, gk, q, k, wq, wk, eps, cu, f_ref)
        assert_close("dwq", dwq, dwqr, dwqs, dtype=dt(wl), kind="dw")
        assert_close("dwk", dwk, dwkr, dwks, dtype=dt(wl), kind="dw")
    # r recomputed in the backward equals the saved one
    assert torch.equal(dq, dq2) and torch.equal(dk, dk2)
    assert torch.equal(dwq, dwq2) and torch.equal(dwk, dwk2)


@pytest.mark.parametrize("name", ("tiny_f32", "qwen2.5-0.5b"))
def test_small_full(name):
    check(W.WORKLOADS[name])


@pytest.mark.parametrize("name", ("llama-3.2-1b", "qwen3-8b"))
def test_large_sampled(name):
    check(W.WORKLOADS[name], n_tok=2048)


def test_llama3_table():
    check(W.WORKLOADS["llama-3.2-1b"], n_tok=2048, llama3=True)


@pytest.mark.slow
def test_524k_sampled():
    # dwq / dwk over 524k tokens x 72 heads are left to the smaller cases
    check(W.WORKLOADS["qwen3-32b-524k"], n_tok=1024, dw=False)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("lens,Hq,Hkv,D", [
    ((1,), 4, 2, 16),                      # one token
    ((5, 17, 0, 32, 10), 4, 2, 16),        # zero-length sequences
    ((300, 1, 77), 14, 2, 64),
    ((7, 60, 3), 32, 8, 128),
    ((33, 12), 3, 1, 18),                  # D/2 = 9: element-wise path
    ((40,), 6, 0, 64),                     # Q only
    ((40,), 0, 3, 64),                     # K only
    ((9,), 2, 1, 512),                     # the largest head
    ((60, 41), 4, 4, 32),                  # half a head over two lanes (bf16)
    ((31, 2, 19), 3, 1, 256),              # half a head over sixteen lanes (bf16)
    (tuple((i * 5) % 7 for i in range(2100)), 3, 1, 64),  # > 2,047 sequences: bounds via L1
])
def test_shapes(dtype, lens, Hq, Hkv, D):
    eps = 1e-6
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    cu_d = torch.as_tensor(cu, device=DEV)
    q, k = randn((T, Hq, D), dtype, 61), randn((T, Hkv, D), dtype, 62)
    gq, gk = randn((T, Hq, D), dtype, 63), randn((T, Hkv, D), dtype, 64)
    wq = (1 + 0.1 * randn((D,), torch.float32, 65)).to(dtype)
    wk = (1 + 0.1 * randn((D,), torch.float32, 66)).to(dtype)
    f = oracle.rope_inv_freq(D, 1e4)
    qo, ko = Guarded((T, Hq, D), dtype), Guarded((T, Hkv, D), dtype)
    dq, dk = Guarded((T, Hq, D), dtype), Guarded((T, Hkv, D), dtype)
    qq = q if Hq else None
    kk = k if Hkv else None
    _, _, rq, rk = ftk.qk_norm_rope_fwd(qq, kk, wq if Hq else None, wk if Hkv else None, cu_d,
                                        eps, theta=1e4, q_out=qo.t if Hq else None,
                                        k_out=ko.t if Hkv else None)
    _, _, dwq, dwk = ftk.qk_norm_rope_bwd(gq if Hq else None, gk if Hkv else None, qq, kk,
                                          wq if Hq else None, wk if Hkv else None, rq, rk, cu_d,
                                          eps, theta=1e4, dq=dq.t if Hq else None,
                                          dk=dk.t if Hkv else None)
    torch.cuda.synchronize()
    for g in (qo, ko, dq, dk):
        g.check()
    c = code(dtype)
    qr, kr, rqr, rkr, qs, ks = oracle.qk_norm_rope_fwd(q.cpu(), k.cpu(), wq.cpu(), wk.cpu(), eps,
                                                       cu, f, scales=True)
    out = oracle.qk_norm_rope_bwd(gq.cpu(), gk.cpu(), q.cpu(), k.cpu(), wq.cpu(), wk.cpu(), eps,
                                  cu, f, scales=True)
    if Hq:
        assert_close("q_out", qo.t, qr, qs, dtype=c)
        assert_close("rstd_q", rq, rqr, dtype="f32")
        assert_close("dq", dq.t, out[0], out[4], dtype=c)
        assert_close("dwq", dwq, out[2], out[6], dtype=c, kind="dw")
    else:
        assert dwq is None
    if Hkv:
        assert_close("k_out", ko.t, kr, ks, dtype=c)
        assert_close("rstd_k", rk, rkr, dtype="f32")
        assert_close("dk", dk.t, out[1], out[5], dtype=c)
        assert_close("dwk", dwk, out[3], out[7], dtype=c, kind="dw")


def test_in_place_and_fused_qkv_layout():
    """q and k as interleaved slices of one fused QKV buffer, normalised and
    rotated in place; the backward writes dq, dk over the output gradients."""
    T, Hq, Hkv, D = 257, 16, 4, 128
    lens = (100, 57, 100)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cu_d = torch.as_tensor(cu, device=DEV)
    qkv = randn((T, (Hq + 2 * Hkv) * D), torch.bfloat16, 71)
    q = qkv[:, :Hq * D].view(T, Hq, D)
    k = qkv[:, Hq * D:(Hq + Hkv) * D].view(T, Hkv, D)
    v_before = qkv[:, (Hq + Hkv) * D:].clone()
    wq = (1 + 0.1 * randn((D,), torch.float32, 72)).to(torch.bfloat16)
    wk = (1 + 0.1 * randn((D,), torch.float32, 73)).to(torch.bfloat16)
    q0, k0 = q.clone(), k.clone()
    qs_, ks_, rq, rk = ftk.qk_norm_rope_fwd(q0, k0, wq, wk, cu_d, 1e-6, theta=1e6)
    ftk.qk_norm_rope_fwd(q, k, wq, wk, cu_d, 1e-6, theta=1e6, q_out=q, k_out=k)
    torch.cuda.synchronize()
    assert torch.equal(q, qs_) and torch.equal(k, ks_)
    assert torch.equal(qkv[:, (Hq + Hkv) * D:], v_before)  # V untouched
    gq, gk = randn((T, Hq, D), torch.bfloat16, 74), randn((T, Hkv, D), torch.bfloat16, 75)
    dq_sep, dk_sep, dwq, dwk = ftk.qk_norm_rope_bwd(gq, gk, q0, k0, wq, wk, rq, rk, cu_d, 1e-6,
                                                    theta=1e6)
    ftk.qk_norm_rope_bwd(gq, gk, q0, k0, wq, wk, rq, rk, cu_d, 1e-6, theta=1e6, dq=gq, dk=gk)
    torch.cuda.synchronize()
    assert torch.equal(gq, dq_sep) and torch.equal(gk, dk_sep)


def test_deterministic_dw():
    T, Hq, Hkv, D = 5000, 8, 2, 128
    cu = np.array([0, 1234, 5000], dtype=np.int32)
    cu_d = torch.as_tensor(cu, device=DEV)
    q, k = randn((T, Hq, D), torch.bfloat16, 81), randn((T, Hkv, D), torch.bfloat16, 82)
    gq, gk = randn((T, Hq, D), torch.bfloat16, 83), randn((T, Hkv, D), torch.bfloat16, 84)
    w = torch.ones(D, dtype=torch.bfloat16, device=DEV)
    outs = [ftk.qk_norm_rope_bwd(gq, gk, q, k, w, w, None, None, cu_d, 1e-6, theta=1e6)
            for _ in range(3)]
    for o in outs[1:]:
        assert all(torch.equal(a, b) for a, b in zip(o, outs[0]))


def test_large_batch_fused_qkv_in_place_sampled():
    """A batch large enough that every warp of the persistent kernels walks
    many tokens, read from and written back into interleaved Q / K slices of
    one fused QKV buffer."""
    T, Hq, Hkv, D = 20000, 16, 4, 128
    lens = (5000, 1, 8000, 6999)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    cu_d = torch.as_tensor(cu, device=DEV)
    qkv = randn((T, (Hq + 2 * Hkv) * D), torch.bfloat16, 91)
    q = qkv[:, :Hq * D].view(T, Hq, D)
    k = qkv[:, Hq * D:(Hq + Hkv) * D].view(T, Hkv, D)
    wq = (1 + 0.1 * randn((D,), torch.float32, 92)).to(torch.bfloat16)
    wk = (1 + 0.1 * randn((D,), torch.float32, 93)).to(torch.bfloat16)
    q0, k0 = q.clone(), k.clone()
    qo, ko, rq, rk = ftk.qk_norm_rope_fwd(q0, k0, wq, wk, cu_d, 1e-6, theta=1e6)
    ftk.qk_norm_rope_fwd(q, k, wq, wk, cu_d, 1e-6, theta=1e6, q_out=q, k_out=k)
    gq, gk = randn((T, Hq, D), torch.bfloat16, 94), randn((T, Hkv, D), torch.bfloat16, 95)
    dq, dk, dwq, dwk = ftk.qk_norm_rope_bwd(gq, gk, q0, k0, wq, wk, rq, rk, cu_d, 1e-6,
                                            theta=1e6)
    torch.cuda.synchronize()
    assert ftk.device_status(clear=True) == 0
    assert torch.equal(q, qo) and torch.equal(k, ko)
    tok = sample_rows(T, 512, extra=list(cu[:-1]) + [c - 1 for c in cu[1:]])
    ti = torch.as_tensor(tok, device=DEV)
    f = oracle.rope_inv_freq(D, 1e6)
    qr, kr, _, _, qs, ks = oracle.qk_norm_rope_fwd(q0[ti].cpu(), k0[ti].cpu(), wq.cpu(),
                                                   wk.cpu(), 1e-6, cu, f, tok=tok, scales=True)
    assert_close("q_out", qo[ti], qr, qs)
    assert_close("k_out", ko[ti], kr, ks)
    out = oracle.qk_norm_rope_bwd(gq[ti].cpu(), gk[ti].cpu(), q0[ti].cpu(), k0[ti].cpu(),
                                  wq.cpu(), wk.cpu(), 1e-6, cu, f, tok=tok, scales=True)
    assert_close("dq", dq[ti], out[0], out[4])
    assert_close("dk", dk[ti], out[1], out[5])
    dwqr, dwkr, dwqs, dwks = dw_oracle_chunked(gq, gk, q0, k0, wq, wk, 1e-6, cu, f)
    assert_close("dwq", dwq, dwqr, dwqs, kind="dw")
    assert_close("dwk", dwk, dwkr, dwks, kind="dw")
