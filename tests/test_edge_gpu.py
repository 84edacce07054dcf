"""Edge cases, layouts and invariants of the CUDA path, against the oracle.

Every output buffer here sits between 4 KiB canary regions that must come
back untouched (a stand-in for an out-of-bounds checker).  Covered: empty
and one-token batches, ragged sizes that take the element-wise kernels,
misaligned pointers, rows too long for the register plan, strided rows,
fused gate_up / QKV buffers, in-place aliases, zero-length sequences,
64-bit offsets against 32-bit ones, packing invariance, determinism.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.tolerance import assert_close, f64
from fine_tuning_gb300 import build, ftk

pytestmark = pytest.mark.gpu
DEV = "cuda"
CANARY = 4096


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ftk.library()


class Guarded:
    """A [*shape] tensor at byte offset `skew` inside canary-filled memory."""

    def __init__(self, shape, dtype, skew=0, fill=None):
        es = torch.empty((), dtype=dtype).element_size()
        n = int(np.prod(shape))
        self.pad = CANARY // es
        self.skew = skew // es
        self.raw = torch.empty(2 * self.pad + n + self.skew, dtype=dtype, device=DEV)
        self.raw.view(torch.uint8).fill_(0xA5)
        self.canary = self.raw.clone()
        self.t = self.raw[self.pad + self.skew: self.pad + self.skew + n].view(shape)
        if fill is not None:
            self.t.copy_(fill)

    def check(self):
        lo = self.pad + self.skew
        hi = lo + self.t.numel()
        a = self.raw.view(torch.uint8)
        c = self.canary.view(torch.uint8)
        es = self.raw.element_size()
        assert torch.equal(a[: lo * es], c[: lo * es]), "canary before the buffer was written"
        assert torch.equal(a[hi * es:], c[hi * es:]), "canary after the buffer was written"


def randn(shape, dtype, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return torch.randn(shape, generator=g, device=DEV, dtype=torch.float32).to(dtype)


def code(dtype):
    return "f32" if dtype == torch.float32 else "bf16"


# ------------------------------------------------------------------ RMSNorm

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T,H,skew", [
    (1, 896, 0),        # one token
    (37, 896, 0),       # ragged T, vector path
    (29, 900, 0),       # H not a multiple of the packet: element-wise path
    (17, 64, 2),        # misaligned rows: element-wise path (bf16 skew of one element)
    (5, 20000, 0),      # row too long for registers: CTA-per-row kernels
    (300, 5120, 0),     # multi-warp rows
    (3, 8, 0),          # tiny rows
    (4099, 512, 0),     # rows of one warp, many rows per warp (pipelined kernels)
    (2053, 1024, 0),    # one-warp rows of four packets per lane (bf16)
    (999, 768, 0),      # one-warp rows of three packets per lane (bf16)
    (513, 256, 0),      # one-warp rows of one packet per lane (bf16)
    (1027, 2048, 0),    # two-warp rows (bf16), ragged T
    (5, 2048, 0),       # fewer rows than row groups
])
def test_rmsnorm_shapes(dtype, T, H, skew):
    eps = 1e-6
    x = randn((T, H), dtype, 1)
    w = 1 + 0.1 * randn((H,), torch.float32, 2)
    w = w.to(dtype)
    dy = randn((T, H), dtype, 3)
    yg = Guarded((T, H), dtype, skew=skew if dtype == torch.bfloat16 else 0)
    rg = Guarded((T,), torch.float32)
    dxg = Guarded((T, H), dtype)
    dwg = Guarded((H,), torch.float32)
    xin = Guarded((T, H), dtype, skew=skew if dtype == torch.bfloat16 else 0, fill=x).t
    ftk.rmsnorm_fwd(xin, w, eps, y=yg.t, rstd=rg.t)
    ftk.rmsnorm_bwd(dy, xin, w, rg.t, eps, dx=dxg.t, dw=dwg.t)
    torch.cuda.synchronize()
    for gd in (yg, rg, dxg, dwg):
        gd.check()
    yr, rr = oracle.rmsnorm_fwd(x.cpu(), w.cpu(), eps)
    dxr, dwr, dxs, dws = oracle.rmsnorm_bwd(dy.cpu(), x.cpu(), w.cpu(), eps, scales=True)
    assert_close("y", yg.t, yr, dtype=code(dtype))
    assert_close("rstd", rg.t, rr, dtype="f32")
    assert_close("dx", dxg.t, dxr, dxs, dtype=code(dtype))
    assert_close("dw", dwg.t, dwr, dws, dtype=code(dtype), kind="dw")


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T,H", [(37, 896), (29, 900), (4099, 512), (2053, 1024), (1027, 2048),
                                 (300, 5120), (5, 20000), (999, 768), (513, 256)])
def test_rmsnorm_bwd_rstd_modes_agree(dtype, T, H):
    # dx and dw are the same bits whether rstd is saved or recomputed: the
    # recomputed rstd repeats the forward's sum, and the grid (so dw's
    # summation order) does not depend on the mode
    x, dy = randn((T, H), dtype, 31), randn((T, H), dtype, 32)
    w = (1 + 0.1 * randn((H,), torch.float32, 33)).to(dtype)
    _, rstd = ftk.rmsnorm_fwd(x, w, 1e-6)
    dx1, dw1 = ftk.rmsnorm_bwd(dy, x, w, rstd, 1e-6)
    dx2, dw2 = ftk.rmsnorm_bwd(dy, x, w, None, 1e-6)
    torch.cuda.synchronize()
    assert torch.equal(dx1, dx2) and torch.equal(dw1, dw2)


def test_rmsnorm_strided_and_in_place():
    T, H, ld = 50, 2048, 2048 + 64
    base = randn((T, ld), torch.bfloat16, 5)
    x = base[:, :H]
    w = (1 + 0.1 * randn((H,), torch.float32, 6)).to(torch.bfloat16)
    x_ref = x.cpu()
    y, rstd = ftk.rmsnorm_fwd(x, w, 1e-5)
    yr, rr = oracle.rmsnorm_fwd(x_ref, w.cpu(), 1e-5)
    assert_close("y strided", y, yr)
    # in place: y written over x
    ftk.rmsnorm_fwd(x, w, 1e-5, y=x)
    torch.cuda.synchronize()
    assert torch.equal(x, y)
    assert torch.equal(base[:, H:].cpu(), randn((T, ld), torch.bfloat16, 5)[:, H:].cpu())
    # dx written over dy
    dy = randn((T, H), torch.bfloat16, 7)
    dy_ref = dy.cpu()
    dx, dw = ftk.rmsnorm_bwd(dy, x_ref.cuda(), w, None, 1e-5, dx=dy)
    dxr, dwr, dxs, dws = oracle.rmsnorm_bwd(dy_ref, x_ref, w.cpu(), 1e-5, scales=True)
    assert_close("dx in place", dy, dxr, dxs)
    assert_close("dw", dw, dwr, dws, kind="dw")


def test_rmsnorm_empty_is_a_no_op():
    x = torch.empty((0, 896), dtype=torch.bfloat16, device=DEV)
    w = torch.ones(896, dtype=torch.bfloat16, device=DEV)
    y, rstd = ftk.rmsnorm_fwd(x, w, 1e-6)
    dx, dw = ftk.rmsnorm_bwd(x, x, w, rstd, 1e-6, dw=torch.full((896,), 3.0, device=DEV))
    assert y.shape == (0, 896) and dw.eq(3.0).all()


def test_rmsnorm_wide_index_matches_narrow():
    """Row stride large enough that offsets pass 2^31 (64-bit kernels): the
    results must equal the 32-bit kernels' bit for bit."""
    T, H = 4, 896
    ld = (1 << 31) // (T - 1) + 64
    ld -= ld % 8
    big = torch.zeros(((T - 1) * ld + H,), dtype=torch.bfloat16, device=DEV)
    x = torch.as_strided(big, (T, H), (ld, 1))
    xs = randn((T, H), torch.bfloat16, 9)
    x.copy_(xs)
    w = (1 + 0.1 * randn((H,), torch.float32, 10)).to(torch.bfloat16)
    y_wide, r_wide = ftk.rmsnorm_fwd(x, w, 1e-6)
    y_nar, r_nar = ftk.rmsnorm_fwd(xs, w, 1e-6)
    dyb = torch.zeros_like(big)
    dy = torch.as_strided(dyb, (T, H), (ld, 1))
    dys = randn((T, H), torch.bfloat16, 11)
    dy.copy_(dys)
    dx_w, dw_w = ftk.rmsnorm_bwd(dy, x, w, r_wide, 1e-6)
    dx_n, dw_n = ftk.rmsnorm_bwd(dys, xs, w, r_nar, 1e-6)
    torch.cuda.synchronize()
    assert torch.equal(y_wide, y_nar) and torch.equal(r_wide, r_nar)
    assert torch.equal(dx_w, dx_n) and torch.equal(dw_w, dw_n)


def test_rmsnorm_deterministic():
    T, H = 4096, 2048
    x, dy = randn((T, H), torch.bfloat16, 12), randn((T, H), torch.bfloat16, 13)
    w = torch.ones(H, dtype=torch.bfloat16, device=DEV)
    outs = [ftk.rmsnorm_bwd(dy, x, w, None, 1e-6) for _ in range(3)]
    for dx, dw in outs[1:]:
        assert torch.equal(dx, outs[0][0]) and torch.equal(dw, outs[0][1])


# ------------------------------------------------------------------- SwiGLU

@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("T,I", [(1, 8), (3, 4864), (37, 1000), (5, 13), (129, 4104)])
def test_swiglu_shapes(dtype, T, I):
    g, u, dh = (randn((T, I), dtype, s) for s in (21, 22, 23))
    hg, dgg, dug = Guarded((T, I), dtype), Guarded((T, I), dtype), Guarded((T, I), dtype)
    ftk.swiglu_fwd(g, u, h=hg.t)
    ftk.swiglu_bwd(dh, g, u, dg=dgg.t, du=dug.t)
    torch.cuda.synchronize()
    for gd in (hg, dgg, dug):
        gd.check()
    hr = oracle.swiglu_fwd(g.cpu(), u.cpu())
    dgr, dur, dgs = oracle.swiglu_bwd(dh.cpu(), g.cpu(), u.cpu(), scales=True)
    assert_close("h", hg.t, hr, dtype=code(dtype))
    assert_close("dg", dgg.t, dgr, dgs, dtype=code(dtype))
    assert_close("du", dug.t, dur, dtype=code(dtype))
    # the backward that re-emits h, into guarded buffers of its own
    h2, dg2, du2 = Guarded((T, I), dtype), Guarded((T, I), dtype), Guarded((T, I), dtype)
    ftk.swiglu_bwd_h(dh, g, u, dg=dg2.t, du=du2.t, h=h2.t)
    torch.cuda.synchronize()
    for gd in (h2, dg2, du2):
        gd.check()
    assert torch.equal(h2.t, hg.t) and torch.equal(dg2.t, dgg.t) and torch.equal(du2.t, dug.t)


def test_swiglu_fused_gate_up_and_in_place():
    T, I = 77, 4864
    gu = randn((T, 2 * I), torch.bfloat16, 31)
    g, u = gu[:, :I], gu[:, I:]
    g0, u0 = g.cpu(), u.cpu()
    dh = randn((T, I), torch.bfloat16, 32)
    h = ftk.swiglu_fwd(g, u)
    assert_close("h fused", h, oracle.swiglu_fwd(g0, u0))
    dgr, dur, dgs = oracle.swiglu_bwd(dh.cpu(), g0, u0, scales=True)
    ftk.swiglu_bwd(dh, g, u, dg=g, du=u)  # gradients written over gate_up
    torch.cuda.synchronize()
    assert_close("dg in place", g, dgr, dgs)
    assert_close("du in place", u, dur)


def test_swiglu_bwd_h_fused_gate_up_in_place():
    """Fused [T, 2I] gate_up: dg, du written over it, and h over dh."""
    T, I = 129, 4864
    gu = randn((T, 2 * I), torch.bfloat16, 33)
    g, u = gu[:, :I], gu[:, I:]
    g0, u0 = g.cpu(), u.cpu()
    dh = randn((T, I), torch.bfloat16, 34)
    dh0 = dh.cpu()
    h_fwd = ftk.swiglu_fwd(g, u)
    ftk.swiglu_bwd_h(dh, g, u, dg=g, du=u, h=dh)
    torch.cuda.synchronize()
    assert torch.equal(dh, h_fwd)
    dgr, dur, dgs = oracle.swiglu_bwd(dh0, g0, u0, scales=True)
    assert_close("dg in place", g, dgr, dgs)
    assert_close("du in place", u, dur)


def test_swiglu_extremes():
    # +-89: e^89 overflows fp32, so sigmoid must not be formed as 1/(1+e^-g)
    g = torch.tensor([[0.0, 40.0, -40.0, 100.0, -100.0, 1e-30, -1e-30, 3.0,
                       -87.0, -89.0, 89.0, 20.0]], dtype=torch.float32, device=DEV)
    u = torch.full_like(g, 2.0)
    h = ftk.swiglu_fwd(g, u)
    assert_close("h extremes", h, oracle.swiglu_fwd(g.cpu(), u.cpu()), dtype="f32")
    dg, du = ftk.swiglu_bwd(torch.ones_like(g), g, u)
    dgr, dur, dgs = oracle.swiglu_bwd(np.ones(12)[None], g.cpu(), u.cpu(), scales=True)
    assert_close("dg extremes", dg, dgr, dgs, dtype="f32")
    assert_close("du extremes", du, dur, dtype="f32")
    assert torch.isfinite(dg).all() and torch.isfinite(h).all()


# ------------------------------------------------------------------ QK-RoPE

def rope_case(lens, Hq, Hkv, D, theta, dtype, seed=40):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    q, k = randn((T, Hq, D), dtype, seed), randn((T, Hkv, D), dtype, seed + 1)
    return cu, T, q, k


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("lens,Hq,Hkv,D", [
    ((1,), 4, 2, 16),                     # one token
    ((5, 17, 0, 32, 0, 10), 4, 2, 16),     # zero-length sequences
    ((300,), 14, 2, 64),                   # B = 1
    ((7, 1, 60, 3), 32, 8, 128),
    ((33, 12), 3, 1, 18),                  # D/2 = 9: element-wise path
    ((40,), 8, 0, 64),                     # no K heads
    ((20, 20), 5, 3, 512),                 # widest head
    ((20011,), 6, 2, 64),                  # many passes per warp, ragged last pass
    (tuple((i * 7) % 9 for i in range(2100)), 4, 2, 64),  # > 2,047 sequences: bounds via L1
    ((0, 0, 5, 0, 30000, 0, 7, 0), 14, 2, 64),  # empty sequences at both ends
    ((100, 0, 211), 8, 4, 32),             # half a head over two lanes (bf16)
    ((77, 50), 4, 2, 256),                 # half a head over sixteen lanes (bf16)
])
def test_rope_shapes(dtype, lens, Hq, Hkv, D):
    theta = 1e4
    cu, T, q, k = rope_case(lens, Hq, Hkv, D, theta, dtype)
    qg = Guarded((T, Hq, D), dtype, fill=q)
    kg = Guarded((T, Hkv, D), dtype, fill=k) if Hkv else None
    ftk.qk_rope_fwd(qg.t, kg.t if kg else None, torch.as_tensor(cu, device=DEV), theta)
    torch.cuda.synchronize()
    qg.check()
    if kg:
        kg.check()
    qr, kr, qs, ks = oracle.qk_rope(q.cpu(), k.cpu(), cu, theta, +1, scales=True)
    assert_close("q", qg.t, qr, qs, dtype=code(dtype))
    if kg:
        assert_close("k", kg.t, kr, ks, dtype=code(dtype))


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("lens,Hq,Hkv,D", [
    ((5, 17, 0, 32, 10), 4, 2, 16),
    ((300, 1, 77), 14, 2, 64),
    ((33, 12), 3, 1, 18),                  # element-wise path
    ((7000,), 8, 2, 128),                  # staged path
])
def test_rope_freq_table(dtype, lens, Hq, Hkv, D):
    """An arbitrary table in [0, 1] (both ends included) against the oracle;
    an all-zero table leaves q and k bit for bit."""
    rng = np.random.default_rng(D + Hq)
    f = rng.random(D // 2)
    f[0], f[-1] = 1.0, 0.0
    cu, T, q, k = rope_case(lens, Hq, Hkv, D, 1e4, dtype, seed=50)
    cu_d = torch.as_tensor(cu, device=DEV)
    qg, kg = Guarded((T, Hq, D), dtype, fill=q), Guarded((T, Hkv, D), dtype, fill=k)
    ftk.qk_rope_freq_fwd(qg.t, kg.t, cu_d, f)
    torch.cuda.synchronize()
    qg.check()
    kg.check()
    qr, kr, qs, ks = oracle.qk_rope_freq(q.cpu(), k.cpu(), cu, f, +1, scales=True)
    assert_close("q", qg.t, qr, qs, dtype=code(dtype))
    assert_close("k", kg.t, kr, ks, dtype=code(dtype))
    # the backward on the forward's output, against the oracle's backward
    q1, k1 = qg.t.cpu(), kg.t.cpu()
    ftk.qk_rope_freq_bwd(qg.t, kg.t, cu_d, f)
    q2, k2 = q.clone(), k.clone()
    ftk.qk_rope_freq_fwd(q2, k2, cu_d, np.zeros(D // 2))
    torch.cuda.synchronize()
    dqr, dkr, dqs, dks = oracle.qk_rope_freq(q1, k1, cu, f, -1, scales=True)
    assert_close("dq", qg.t, dqr, dqs, dtype=code(dtype))
    assert_close("dk", kg.t, dkr, dks, dtype=code(dtype))
    assert torch.equal(q2, q) and torch.equal(k2, k)


def test_rope_fused_qkv_buffer():
    lens, Hq, Hkv, D, theta = (50, 13, 61), 16, 4, 128, 5e5
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    T = int(cu[-1])
    qkv = randn((T, (Hq + 2 * Hkv) * D), torch.bfloat16, 50)
    v0 = qkv[:, (Hq + Hkv) * D:].clone()
    q = qkv[:, : Hq * D].view(T, Hq, D)
    k = qkv[:, Hq * D:(Hq + Hkv) * D].view(T, Hkv, D)
    q0, k0 = q.cpu(), k.cpu()
    ftk.qk_rope_fwd(q, k, torch.as_tensor(cu, device=DEV), theta)
    torch.cuda.synchronize()
    qr, kr, qs, ks = oracle.qk_rope(q0, k0, cu, theta, +1, scales=True)
    assert_close("q in qkv", q, qr, qs)
    assert_close("k in qkv", k, kr, ks)
    assert torch.equal(qkv[:, (Hq + Hkv) * D:], v0)  # V untouched


def test_rope_packing_invariance_bitwise():
    lens, Hq, Hkv, D, theta = (100, 3, 257, 40), 14, 2, 64, 1e6
    cu, T, q, k = rope_case(lens, Hq, Hkv, D, theta, torch.bfloat16, seed=60)
    qp, kp = q.clone(), k.clone()
    ftk.qk_rope_fwd(qp, kp, torch.as_tensor(cu, device=DEV), theta)
    for b in range(len(lens)):
        s, e = int(cu[b]), int(cu[b + 1])
        qs, ks = q[s:e].clone(), k[s:e].clone()
        ftk.qk_rope_fwd(qs, ks, torch.tensor([0, e - s], dtype=torch.int32, device=DEV), theta)
        assert torch.equal(qs, qp[s:e]) and torch.equal(ks, kp[s:e])


def test_rope_fwd_then_bwd_is_identity_and_deterministic():
    lens, Hq, Hkv, D, theta = (1000, 24), 8, 2, 128, 1e6
    cu, T, q, k = rope_case(lens, Hq, Hkv, D, theta, torch.float32, seed=70)
    cud = torch.as_tensor(cu, device=DEV)
    q1, k1 = q.clone(), k.clone()
    ftk.qk_rope_fwd(q1, k1, cud, theta)
    q2, k2 = q.clone(), k.clone()
    ftk.qk_rope_fwd(q2, k2, cud, theta)
    assert torch.equal(q1, q2) and torch.equal(k1, k2)
    ftk.qk_rope_bwd(q1, k1, cud, theta)
    torch.cuda.synchronize()
    assert (q1 - q).abs().max().item() < 1e-5 and (k1 - k).abs().max().item() < 1e-5


def test_rope_wide_index_matches_narrow():
    T, Hq, D = 3, 4, 64
    ld = ((1 << 31) // (T - 1) + 64) // 8 * 8
    big = torch.zeros(((T - 1) * ld + Hq * D,), dtype=torch.bfloat16, device=DEV)
    q = torch.as_strided(big, (T, Hq, D), (ld, D, 1))
    qs = randn((T, Hq, D), torch.bfloat16, 80)
    q.copy_(qs)
    cu = torch.tensor([0, T], dtype=torch.int32, device=DEV)
    ftk.qk_rope_fwd(q, None, cu, 1e6)
    ftk.qk_rope_fwd(qs, None, cu, 1e6)
    torch.cuda.synchronize()
    assert torch.equal(q, qs)


# --------------------------------------------------------- failure detection

def test_bounded_wait_times_out_and_reports():
    """A kernel whose barrier is never completed gives up after its cycle
    limit, sets the status bit and returns: the GPU stays usable."""
    ftk.device_status(clear=True)
    ftk.selftest_wait_timeout(2_000_000)
    torch.cuda.synchronize()
    assert ftk.device_status(clear=True) & ftk.WAIT_TIMEOUT
    assert ftk.device_status(clear=False) == 0
    # ordinary work afterwards runs and leaves the word clean
    x = randn((64, 896), torch.bfloat16, 90)
    w = torch.ones(896, dtype=torch.bfloat16, device=DEV)
    y, _ = ftk.rmsnorm_fwd(x, w, 1e-6)
    dx, dw = ftk.rmsnorm_bwd(x, x, w, None, 1e-6)
    torch.cuda.synchronize()
    assert torch.isfinite(y.float()).all() and ftk.device_status() == 0


@pytest.mark.parametrize("T,H", [
    (8000, 2304),   # three warps' plan, three packets per lane
    (8000, 3072),   # three warps, four packets
    (8000, 4096),   # four warps (Qwen3-8B rows)
    (4000, 5120),   # five warps (Qwen3-32B rows)
    (4000, 6144),   # six warps
    (4000, 7680),   # eight warps
])
def test_rmsnorm_multi_warp_rows_large_batch(T, H):
    # bf16 rows of three or more warps in batches large enough for the
    # TMA-staged kernels in both directions: the saved r must equal the one
    # the backward recomputes bit for bit (the same summation plan), and both
    # directions must match the oracle.
    eps = 1e-6
    x, dy = randn((T, H), torch.bfloat16, 91), randn((T, H), torch.bfloat16, 92)
    w = (1 + 0.1 * randn((H,), torch.float32, 93)).to(torch.bfloat16)
    yg, rg = Guarded((T, H), torch.bfloat16), Guarded((T,), torch.float32)
    ftk.rmsnorm_fwd(x, w, eps, y=yg.t, rstd=rg.t)
    dx1, dw1 = ftk.rmsnorm_bwd(dy, x, w, rg.t, eps)
    dx2, dw2 = ftk.rmsnorm_bwd(dy, x, w, None, eps)
    torch.cuda.synchronize()
    yg.check()
    rg.check()
    assert torch.equal(dx1, dx2) and torch.equal(dw1, dw2)
    rows = np.unique(np.concatenate([np.arange(3), np.arange(T - 3, T),
                                     np.random.default_rng(H).choice(T, 58, replace=False)]))
    ri = torch.as_tensor(rows, device=DEV)
    yr, rr = oracle.rmsnorm_fwd(x[ri].cpu(), w.cpu(), eps)
    assert_close("y", yg.t[ri], yr, dtype="bf16")
    assert_close("rstd", rg.t[ri], rr, dtype="f32")
    dxr, _, dxs, _ = oracle.rmsnorm_bwd(dy[ri].cpu(), x[ri].cpu(), w.cpu(), eps, scales=True)
    assert_close("dx", dx1[ri], dxr, dxs, dtype="bf16")
