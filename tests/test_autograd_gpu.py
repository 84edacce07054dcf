"""The optional autograd wrappers give exactly what the direct ftk calls
give (the calls themselves are checked against the oracle elsewhere)."""
import numpy as np
import pytest
import torch

from fine_tuning_gb300 import autograd as A
from fine_tuning_gb300 import build, ftk
from fine_tuning_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ftk.library()


def randn(shape, seed, dtype=torch.bfloat16, scale=1.0):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return (scale * torch.randn(shape, generator=g, device=DEV)).to(dtype)


def leaf(t):
    return t.clone().requires_grad_(True)


def test_rmsnorm_and_add_rmsnorm():
    x, res, dy = randn((300, 896), 1), randn((300, 896), 2), randn((300, 896), 3)
    w = (1 + 0.1 * randn((896,), 4, torch.float32)).to(torch.bfloat16)
    xl, wl = leaf(x), leaf(w)
    A.rmsnorm(xl, wl, 1e-6).backward(dy)
    y, rstd = ftk.rmsnorm_fwd(x, w, 1e-6)
    dx, dw = ftk.rmsnorm_bwd(dy, x, w, rstd, 1e-6)
    assert torch.equal(xl.grad, dx) and torch.equal(wl.grad, dw.to(torch.bfloat16))
    xl, rl, wl = leaf(x), leaf(res), leaf(w)
    dh_up = randn((300, 896), 5)
    h, y = A.add_rmsnorm(xl, rl, wl, 1e-6)
    torch.autograd.backward([h, y], [dh_up, dy])
    h2, y2, r2 = ftk.rmsnorm_add_fwd(x, res, w, 1e-6)
    dx2, dw2 = ftk.rmsnorm_add_bwd(dy, dh_up, h2, w, r2, 1e-6)
    assert torch.equal(h, h2) and torch.equal(y, y2)
    assert torch.equal(xl.grad, dx2) and torch.equal(rl.grad, dx2)
    assert torch.equal(wl.grad, dw2.to(torch.bfloat16))


def test_swiglu():
    g, u, dh = randn((77, 4864), 6), randn((77, 4864), 7), randn((77, 4864), 8)
    gl, ul = leaf(g), leaf(u)
    A.swiglu(gl, ul).backward(dh)
    dg, du = ftk.swiglu_bwd(dh, g, u)
    assert torch.equal(gl.grad, dg) and torch.equal(ul.grad, du)


def test_qk_rope_and_qk_norm_rope():
    lens = (40, 1, 23)
    cu = torch.as_tensor(np.concatenate([[0], np.cumsum(lens)]).astype(np.int32), device=DEV)
    T = sum(lens)
    q, k = randn((T, 8, 64), 9), randn((T, 2, 64), 10)
    dq, dk = randn((T, 8, 64), 11), randn((T, 2, 64), 12)
    ql, kl = leaf(q), leaf(k)
    qo, ko = A.qk_rope(ql, kl, cu, 1e6)
    torch.autograd.backward([qo, ko], [dq, dk])
    q2, k2 = q.clone(), k.clone()
    ftk.qk_rope_fwd(q2, k2, cu, 1e6)
    g1, g2 = dq.clone(), dk.clone()
    ftk.qk_rope_bwd(g1, g2, cu, 1e6)
    assert torch.equal(qo, q2) and torch.equal(ko, k2)
    assert torch.equal(ql.grad, g1) and torch.equal(kl.grad, g2)
    assert not torch.equal(q, q2)  # the input was not rotated in place
    wq = (1 + 0.1 * randn((64,), 13, torch.float32)).to(torch.bfloat16)
    wk = (1 + 0.1 * randn((64,), 14, torch.float32)).to(torch.bfloat16)
    ql, kl, wql, wkl = leaf(q), leaf(k), leaf(wq), leaf(wk)
    qo, ko = A.qk_norm_rope(ql, kl, wql, wkl, cu, 1e-6, 1e6)
    torch.autograd.backward([qo, ko], [dq, dk])
    qo2, ko2, rq, rk = ftk.qk_norm_rope_fwd(q, k, wq, wk, cu, 1e-6, theta=1e6)
    gq, gk, dwq, dwk = ftk.qk_norm_rope_bwd(dq, dk, q, k, wq, wk, rq, rk, cu, 1e-6, theta=1e6)
    assert torch.equal(qo, qo2) and torch.equal(ko, ko2)
    assert torch.equal(ql.grad, gq) and torch.equal(kl.grad, gk)
    assert torch.equal(wql.grad, dwq.to(torch.bfloat16)) and torch.equal(wkl.grad, dwk.to(torch.bfloat16))


def test_cross_entropy_head():
    d = W.head_inputs(W.HEAD_WORKLOADS["tiny-head"], DEV)
    hl, Wl = leaf(d["h"]), leaf(d["W"])
    loss = A.cross_entropy_head(hl, Wl, d["y"])
    (3.0 * loss).backward()
    loss2, lse = ftk.cce_fwd(d["h"], d["W"], d["y"])
    dh, dW = ftk.cce_bwd(d["h"], d["W"], d["y"], lse, torch.full((1,), 3.0, device=DEV))
    assert torch.equal(loss.reshape(1), loss2)
    assert torch.equal(hl.grad, dh) and torch.equal(Wl.grad, dW.to(torch.bfloat16))
