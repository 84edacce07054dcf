"""The LM-head cross-entropy (Cut Cross-Entropy) on the tensor cores against
the double-precision oracle (oracle/cce.py).

Tolerances come from the arithmetic:
  * logits: bf16 products are exact in fp32, so |dz| <= H 2^-24 sum|h||W|
    <= H 2^-24 |h_t| max_v |W_v| (Cauchy-Schwarz);
  * lse is 1-Lipschitz in the logits, plus the fp32 sums of e^z (half a
    tile, 128 columns, per partial, then 2 partials per tile:
    (128 + #partials + 8) 2^-24 relative), the hardware 2^x (about 2^-22
    relative per term and per rescaling, at most 10 of them on a path) and
    the fp32 log (1e-6 relative);
  * loss: the mean of the row losses, each within the lse and target-logit
    bounds, summed in fp32 in a fixed order (T 2^-24 of the mean);
  * dh, dW: dz is rounded to bf16 (2^-9 relative) before two fp32-
    accumulated contractions: |err| <= 2^-8 sum |dz||W| (resp. |dz||h|),
    plus 2 bf16 ulps for the bf16 dh.
"""
import numpy as np
import pytest
import torch

from oracle import cce
from fine_tuning_gb300 import build, ftk
from fine_tuning_gb300 import workloads as W

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ftk.library()
    ftk.device_status(clear=True)
    yield
    torch.cuda.empty_cache()


def f64(t):
    return t.detach().double().cpu().numpy()


def ulp_bf16(x):
    e = np.floor(np.log2(np.maximum(np.abs(x), 2.0 ** -126)))
    return 2.0 ** (e - 7)


def lse_bound(h64, W64, lse_ref, V):
    H = h64.shape[1]
    nparts = 2 * ((V + 255) // 256)
    zmax = H * 2.0 ** -24 * np.linalg.norm(h64, axis=1) * np.linalg.norm(W64, axis=1).max()
    return zmax, (zmax + (128 + nparts + 8) * 2.0 ** -24 + 10 * 2.0 ** -22
                  + 1e-6 * np.abs(lse_ref))


def check_forward(h, Wt, y, loss, lse, tok=None, full_loss=True):
    h64, W64, y64 = f64(h), f64(Wt), y.cpu().numpy()
    V = W64.shape[0]
    rows = np.arange(h64.shape[0]) if tok is None else np.asarray(tok)
    lse_ref, _ = cce.lse_and_target(h64, W64, y64, tok=rows)
    zmax, b = lse_bound(h64[rows], W64, lse_ref, V)
    err = np.abs(f64(lse)[rows] - lse_ref)
    assert np.all(err <= b), (err.max(), b[err.argmax()], rows[err.argmax()])
    if full_loss:
        loss_ref, lse_all, n, zy = cce.cce_fwd(h64, W64, y64, with_target=True)
        zmax_all, b_all = lse_bound(h64, W64, lse_all, V)
        valid = (y64 >= 0) & (y64 < V)
        rl = np.abs(lse_all - zy)
        lb = ((b_all + zmax_all)[valid].sum() / max(n, 1)
              + h64.shape[0] * 2.0 ** -24 * (rl[valid].mean() if n else 0.0))
        assert abs(float(loss.item()) - loss_ref) <= lb, (float(loss.item()), loss_ref, lb)


def check_backward(h, Wt, y, dh, dW, g=1.0, tok=None, vocab=None):
    h64, W64, y64 = f64(h), f64(Wt), y.cpu().numpy()
    rows = np.arange(h64.shape[0]) if tok is None else np.asarray(tok)
    vv = np.arange(W64.shape[0]) if vocab is None else np.asarray(vocab)
    dh_ref, dW_ref, dhs, dWs = cce.cce_bwd(h64, W64, y64, g, tok=rows, vocab=vv, scales=True)
    got_dh, got_dW = f64(dh)[rows], f64(dW)[vv]
    bh = 2 * ulp_bf16(dh_ref) + 2.0 ** -8 * dhs + 1e-30
    bw = 2.0 ** -8 * dWs + 1e-30
    eh, ew = np.abs(got_dh - dh_ref), np.abs(got_dW - dW_ref)
    assert np.all(eh <= bh), ("dh", int((eh > bh).sum()), np.argwhere(eh > bh)[:3])
    assert np.all(ew <= bw), ("dW", int((ew > bw).sum()), np.argwhere(ew > bw)[:3])


def run(hw, g=1.0):
    d = W.head_inputs(hw, DEV)
    h, Wt, y = d["h"], d["W"], d["y"]
    loss, lse = ftk.cce_fwd(h, Wt, y)
    dloss = torch.full((1,), g, dtype=torch.float32, device=DEV)
    dh, dW = ftk.cce_bwd(h, Wt, y, lse, dloss)
    torch.cuda.synchronize()
    assert ftk.device_status(clear=True) == 0
    return h, Wt, y, loss, lse, dh, dW


def test_tiny_full():
    h, Wt, y, loss, lse, dh, dW = run(W.HEAD_WORKLOADS["tiny-head"], g=0.5)
    check_forward(h, Wt, y, loss, lse)
    check_backward(h, Wt, y, dh, dW, g=0.5)


@pytest.mark.parametrize("T,H,V", [(1, 64, 300), (129, 128, 8192), (130, 96, 8193),
                                   (64, 200, 17000), (200, 448, 20000), (300, 576, 17001)])
def test_shapes(T, H, V):
    # one token; an exact chunk; one column past a chunk; ragged H; the
    # grouped dh + dW launches at tile widths 224 (H = 448) and 192 (H = 576),
    # over two vocabulary chunks
    hw = W.HeadWorkload("case", T=T, H=H, V=V, seed=T + V, w_std=H ** -0.5)
    h, Wt, y, loss, lse, dh, dW = run(hw)
    check_forward(h, Wt, y, loss, lse)
    check_backward(h, Wt, y, dh, dW)


def test_all_ignored_and_deterministic():
    hw = W.HeadWorkload("case", T=64, H=64, V=500, seed=3, w_std=0.1)
    d = W.head_inputs(hw, DEV)
    y = torch.full((64,), -100, dtype=torch.int32, device=DEV)
    loss, lse = ftk.cce_fwd(d["h"], d["W"], y)
    dh, dW = ftk.cce_bwd(d["h"], d["W"], y, lse, torch.ones(1, device=DEV))
    torch.cuda.synchronize()
    assert loss.item() == 0.0 and not dh.any() and not dW.any()
    a = ftk.cce_fwd(d["h"], d["W"], d["y"])
    b = ftk.cce_fwd(d["h"], d["W"], d["y"])
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.slow
def test_qwen_head_sampled():
    hw = W.HEAD_WORKLOADS["qwen2.5-0.5b-head"]
    h, Wt, y, loss, lse, dh, dW = run(hw)
    rng = np.random.default_rng(5)
    tok = np.unique(np.concatenate([[0, hw.T - 1], rng.choice(hw.T, 62, replace=False)]))
    ys = y.cpu().numpy()
    hot = ys[ys >= 0][:24]  # vocabulary rows some token targets
    vocab = np.unique(np.concatenate([[0, hw.V - 1], hot, rng.choice(hw.V, 38, replace=False)]))
    check_forward(h, Wt, y, loss, lse, tok=tok)
    check_backward(h, Wt, y, dh, dW, tok=tok, vocab=vocab)
