"""Cross-entropy of a linear LM head, written out plainly, in double.

TEST INFRASTRUCTURE ONLY (like the rest of oracle/): imported by tests/,
``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs, never by the
``fine_tuning_gb300`` package; it shares no code with the CUDA path.

"Chronicals" (arXiv 2601.02609), abstract, optimisation (2): Cut
Cross-Entropy computes the loss of the LM head with an online softmax, so
the [T, V] logits never sit in memory at once (5 GB down to 135 MB).  An
online softmax reaches the plain log-sum-exp up to rounding order, so this
oracle is that plain definition:

  z[t, v] = sum_j h[t, j] W[v, j]                      (logits)
  lse[t]  = log sum_v exp(z[t, v])
  loss    = (1/N) sum_{t valid} (lse[t] - z[t, y_t])   N = #valid tokens
  a token is valid unless y_t == ignore_index; N = 0 gives loss 0.

Backward for an upstream gradient g of the loss:

  dz[t, v] = (g / N) (softmax(z[t])_v - [v == y_t])     valid t, else 0
  dh = dz W,   dW = dz^T h

The logits are formed a chunk of tokens at a time (a library matmul per
chunk) only to bound the oracle's own memory; nothing else is blocked.
"""
from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):
        import torch
        a = a.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ints(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.asarray(a, dtype=np.int64)


def _rows(h, W, rows):
    """Logits of the given token rows: z = h[rows] W^T (double)."""
    return h[rows] @ W.T


def lse_and_target(h, W, y, ignore_index=-100, tok=None, chunk=256):
    """(lse[r], z[r, y_r]) for the rows r of ``tok`` (default: every token).
    z[r, y_r] is 0 for an ignored row."""
    h, W, y = _f64(h), _f64(W), _ints(y)
    rows = np.arange(h.shape[0]) if tok is None else _ints(tok)
    lse = np.empty(rows.size)
    zy = np.zeros(rows.size)
    for a in range(0, rows.size, chunk):
        r = rows[a:a + chunk]
        z = _rows(h, W, r)
        m = z.max(axis=1)
        lse[a:a + chunk] = m + np.log(np.exp(z - m[:, None]).sum(axis=1))
        yr = y[r]
        ok = yr != ignore_index
        zy[a:a + chunk][ok] = z[np.arange(r.size)[ok], yr[ok]]
    return lse, zy


def cce_fwd(h, W, y, ignore_index=-100, with_target=False):
    """Returns (loss, lse [T], n_valid), and z[t, y_t] [T] with_target."""
    y = _ints(y)
    lse, zy = lse_and_target(h, W, y, ignore_index)
    valid = y != ignore_index
    n = int(valid.sum())
    loss = float((lse[valid] - zy[valid]).sum() / n) if n else 0.0
    return (loss, lse, n, zy) if with_target else (loss, lse, n)


def dz_rows(h, W, y, g, n_valid, ignore_index=-100, tok=None, chunk=256):
    """dz for the token rows ``tok``: (g/N)(softmax - onehot), 0 if ignored."""
    h, W, y = _f64(h), _f64(W), _ints(y)
    rows = np.arange(h.shape[0]) if tok is None else _ints(tok)
    out = np.zeros((rows.size, W.shape[0]))
    if n_valid == 0:
        return out
    for a in range(0, rows.size, chunk):
        r = rows[a:a + chunk]
        z = _rows(h, W, r)
        m = z.max(axis=1)
        p = np.exp(z - m[:, None])
        p /= p.sum(axis=1)[:, None]
        yr = y[r]
        ok = yr != ignore_index
        p[np.arange(r.size)[ok], yr[ok]] -= 1.0
        p[~ok] = 0.0
        out[a:a + chunk] = p * (g / n_valid)
    return out


def cce_bwd(h, W, y, g=1.0, ignore_index=-100, tok=None, vocab=None, scales=False,
            chunk=256):
    """Gradients of g * loss.  dh for the token rows ``tok`` (default all)
    and dW for the vocabulary rows ``vocab`` (default all; every token's dz
    contributes, formed a chunk of tokens at a time).  With scales=True also
    their condition scales, sum |dz||W| and sum |dz||h|.
    Returns (dh, dW[, dh_scale, dW_scale])."""
    h, W, y = _f64(h), _f64(W), _ints(y)
    n = int((y != ignore_index).sum())
    rows = np.arange(h.shape[0]) if tok is None else _ints(tok)
    dz = dz_rows(h, W, y, g, n, ignore_index, rows, chunk)
    dh = dz @ W
    vv = np.arange(W.shape[0]) if vocab is None else _ints(vocab)
    dW = np.zeros((vv.size, h.shape[1]))
    dWs = np.zeros((vv.size, h.shape[1]))
    for a in range(0, h.shape[0], chunk):
        r = np.arange(a, min(h.shape[0], a + chunk))
        d = dz_rows(h, W, y, g, n, ignore_index, r, chunk)[:, vv]
        dW += d.T @ h[r]
        if scales:
            dWs += np.abs(d).T @ np.abs(h[r])
    if not scales:
        return dh, dW
    return dh, dW, np.abs(dz) @ np.abs(W), dWs
