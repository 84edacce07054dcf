"""RMSNorm with the pre-norm residual add fused in front, CUDA vs the oracle.

h = x + res is stored once (added in fp32, rounded to the storage type), so
the kernel's h must equal the oracle's bit for bit; y, rstd, dx and dw are
compared within the usual tolerances.  The fused forward must also give
exactly what the plain norm gives on the stored h (same per-thread columns,
same summation order), and the recomputed-rstd backward exactly what the
saved-rstd one gives.  Layouts: strided rows, element-wise rows, rows too
long for registers, misaligned rows, and every allowed in-place alias,
with canaries around each output.
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


@pytest.fixture(autouse=True)
def _no_wait_timeouts():
    yield
    assert ftk.device_status(clear=True) == 0


def dt(wl):
    return "f32" if wl.dtype == "f32" else "bf16"


def dw_oracle_chunked(dy, dh, h, w, eps, chunk=16384):
    T, H = h.shape
    dw, dws = np.zeros(H), np.zeros(H)
    wc = w.cpu()
    for a in range(0, T, chunk):
        b = min(T, a + chunk)
        _, p, _, ps = oracle.rmsnorm_add_bwd(dy[a:b].cpu(), dh[a:b].cpu(), h[a:b].cpu(), wc, eps,
                                             scales=True)
        dw += p
        dws += ps
    return dw, dws


def check_add_norm(wl, n_rows=None):
    d = W.rmsnorm_add_inputs(wl, DEV)
    x, res, w, dy, dh = d["x"], d["res"], d["w"], d["dy"], d["dh"]
    h, y, rstd = ftk.rmsnorm_add_fwd(x, res, w, wl.eps)
    dx, dw = ftk.rmsnorm_add_bwd(dy, dh, h, w, rstd, wl.eps)
    dx_re, dw_re = ftk.rmsnorm_add_bwd(dy, dh, h, w, None, wl.eps)
    y_plain, rstd_plain = ftk.rmsnorm_fwd(h, w, wl.eps)
    torch.cuda.synchronize()
    rows = np.arange(wl.T) if n_rows is None else sample_rows(wl.T, n_rows)
    ri = torch.as_tensor(rows, device=DEV)
    hr, yr, rr = oracle.rmsnorm_add_fwd(x[ri].cpu(), res[ri].cpu(), w.cpu(), wl.eps,
                                        storage=dt(wl))
    assert np.array_equal(h[ri].cpu().double().numpy(), hr), "stored h differs"
    assert_close("y", y[ri], yr, dtype=dt(wl))
    assert_close("rstd", rstd[ri], rr, dtype="f32")
    dxr, _, dxs, _ = oracle.rmsnorm_add_bwd(dy[ri].cpu(), dh[ri].cpu(), h[ri].cpu(), w.cpu(),
                                            wl.eps, scales=True)
    assert_close("dx", dx[ri], dxr, dxs, dtype=dt(wl))
    dwr, dws = dw_oracle_chunked(dy, dh, h, w, wl.eps)
    assert_close("dw", dw, dwr, dws, dtype=dt(wl), kind="dw")
    # the fused forward is the plain norm of the stored h, bit for bit
    assert torch.equal(y, y_plain) and torch.equal(rstd, rstd_plain)
    # a recomputed rstd equals the saved one
    assert torch.equal(dx, dx_re) and torch.equal(dw, dw_re)


@pytest.mark.parametrize("name", ("tiny_f32", "qwen2.5-0.5b"))
def test_add_norm_small_full(name):
    check_add_norm(W.WORKLOADS[name])


@pytest.mark.parametrize("name", ("llama-3.2-1b", "qwen3-8b"))
def test_add_norm_large_sampled(name):
    check_add_norm(W.WORKLOADS[name], n_rows=2048)


@pytest.mark.slow
def test_add_norm_524k_sampled():
    check_add_norm(W.WORKLOADS["qwen3-32b-524k"], n_rows=1024)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T,H,skew", [
    (1, 896, 0),        # one token
    (37, 896, 0),       # ragged T, vector path
    (29, 900, 0),       # H not a multiple of the packet: element-wise path
    (17, 64, 2),        # misaligned rows (bf16): element-wise path
    (5, 20000, 0),      # row too long for registers: CTA-per-row kernels
    (300, 5120, 0),     # multi-warp rows
    (4000, 2048, 0),    # enough rows for the staged pipeline
    (999, 768, 0),      # one-warp rows of three packets per lane (bf16)
    (513, 256, 0),      # one-warp rows of one packet per lane (bf16)
    (3001, 512, 0),     # one-warp rows of two packets per lane (bf16), many rows per warp
])
def test_add_norm_shapes(dtype, T, H, skew):
    eps = 1e-6
    skew = skew if dtype == torch.bfloat16 else 0
    x = randn((T, H), dtype, 11)
    res = (2 * randn((T, H), torch.float32, 12)).to(dtype)
    w = (1 + 0.1 * randn((H,), torch.float32, 13)).to(dtype)
    dy, dh = randn((T, H), dtype, 14), randn((T, H), dtype, 15)
    xin = Guarded((T, H), dtype, skew=skew, fill=x).t
    hg, yg = Guarded((T, H), dtype, skew=skew), Guarded((T, H), dtype)
    rg, dxg, dwg = Guarded((T,), torch.float32), Guarded((T, H), dtype), Guarded((H,), torch.float32)
    ftk.rmsnorm_add_fwd(xin, res, w, eps, h=hg.t, y=yg.t, rstd=rg.t)
    ftk.rmsnorm_add_bwd(dy, dh, hg.t, w, rg.t, eps, dx=dxg.t, dw=dwg.t)
    torch.cuda.synchronize()
    for gd in (hg, yg, rg, dxg, dwg):
        gd.check()
    hr, yr, rr = oracle.rmsnorm_add_fwd(x.cpu(), res.cpu(), w.cpu(), eps, storage=code(dtype))
    assert np.array_equal(hg.t.cpu().double().numpy(), hr)
    assert_close("y", yg.t, yr, dtype=code(dtype))
    assert_close("rstd", rg.t, rr, dtype="f32")
    dxr, dwr, dxs, dws = oracle.rmsnorm_add_bwd(dy.cpu(), dh.cpu(), hg.t.cpu(), w.cpu(), eps,
                                                scales=True)
    assert_close("dx", dxg.t, dxr, dxs, dtype=code(dtype))
    assert_close("dw", dwg.t, dwr, dws, dtype=code(dtype), kind="dw")


@pytest.mark.parametrize("T,H", [(64, 2048), (3000, 1024), (7, 900)])
def test_add_norm_in_place(T, H):
    """h written over res (the residual stream updated in place) or over x;
    dx written over dh or over dy; strided rows."""
    eps, ld = 1e-5, H + 64
    dtype = torch.bfloat16
    x = randn((T, H), dtype, 21)
    res_base = (2 * randn((T, ld), torch.float32, 22)).to(dtype)
    res = res_base[:, :H]
    w = (1 + 0.1 * randn((H,), torch.float32, 23)).to(dtype)
    x_ref, res_ref = x.cpu(), res.cpu()
    h_sep, y_sep, r_sep = ftk.rmsnorm_add_fwd(x, res, w, eps)
    # over res
    h1, y1, r1 = ftk.rmsnorm_add_fwd(x, res, w, eps, h=res)
    torch.cuda.synchronize()
    assert h1.data_ptr() == res.data_ptr()
    assert torch.equal(res, h_sep) and torch.equal(y1, y_sep) and torch.equal(r1, r_sep)
    # the columns past H of the strided buffer are untouched
    tail = (2 * randn((T, ld), torch.float32, 22)).to(dtype)[:, H:]
    assert torch.equal(res_base[:, H:], tail)
    # over x
    x2 = x.clone()
    ftk.rmsnorm_add_fwd(x2, res_ref.to(DEV), w, eps, h=x2)
    torch.cuda.synchronize()
    assert torch.equal(x2, h_sep)
    hr, _, _ = oracle.rmsnorm_add_fwd(x_ref, res_ref, w.cpu(), eps, storage="bf16")
    assert np.array_equal(h_sep.cpu().double().numpy(), hr)

    dy, dh = randn((T, H), dtype, 24), randn((T, H), dtype, 25)
    dx_sep, dw_sep = ftk.rmsnorm_add_bwd(dy, dh, h_sep, w, r_sep, eps)
    dh2, dy2 = dh.clone(), dy.clone()
    ftk.rmsnorm_add_bwd(dy, dh2, h_sep, w, r_sep, eps, dx=dh2)
    ftk.rmsnorm_add_bwd(dy2, dh, h_sep, w, r_sep, eps, dx=dy2)
    torch.cuda.synchronize()
    assert torch.equal(dh2, dx_sep) and torch.equal(dy2, dx_sep)
    dxr, dwr, dxs, dws = oracle.rmsnorm_add_bwd(dy.cpu(), dh.cpu(), h_sep.cpu(), w.cpu(), eps,
                                                scales=True)
    assert_close("dx", dx_sep, dxr, dxs)
    assert_close("dw", dw_sep, dwr, dws, kind="dw")


def test_add_norm_rejects_bad_alias():
    buf = torch.zeros(9 * 64, dtype=torch.bfloat16, device=DEV)
    x = buf[:512].view(8, 64)
    shifted = buf[8:520].view(8, 64)                  # overlaps x, but is not x
    res = torch.zeros_like(x)
    w = torch.ones(64, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(ftk.FtkError):
        ftk.rmsnorm_add_fwd(x, res, w, 1e-6, y=res)     # y over an input
    with pytest.raises(ftk.FtkError):
        ftk.rmsnorm_add_fwd(x, res, w, 1e-6, h=shifted)  # h partly over x
    dy, dh = torch.zeros_like(x), torch.zeros_like(x)
    with pytest.raises(ftk.FtkError):
        ftk.rmsnorm_add_bwd(dy, dh, res, w, None, 1e-6, dx=res)  # dx over h
