"""Double-precision CPU oracle for RMSNorm, SwiGLU and varlen QK-RoPE.

TEST INFRASTRUCTURE ONLY: imported by tests/, by ``__graft_entry__.smoke()``
and by ``bench.py``'s CPU-baseline / reference leg, never by the
``fine_tuning_gb300`` package.  It shares no code with the CUDA library.

Every function takes array-likes (numpy or CPU torch tensors of any float
dtype), upcasts them exactly to float64 and returns float64 numpy arrays.
"""
from __future__ import annotations

import ctypes

import numpy as np

from .build import LIB, build_oracle

_lib = None


def _load():
    global _lib
    if _lib is None:
        build_oracle()
        lib = ctypes.CDLL(LIB)
        D = ctypes.POINTER(ctypes.c_double)
        I64 = ctypes.POINTER(ctypes.c_int64)
        I32 = ctypes.POINTER(ctypes.c_int32)
        i64, i32, f64 = ctypes.c_int64, ctypes.c_int32, ctypes.c_double
        lib.oracle_rmsnorm_fwd.argtypes = [D, D, D, D, i64, i64, f64]
        lib.oracle_rmsnorm_fwd.restype = None
        lib.oracle_rmsnorm_bwd.argtypes = [D, D, D, D, D, D, D, i64, i64, f64]
        lib.oracle_rmsnorm_bwd.restype = None
        lib.oracle_swiglu_fwd.argtypes = [D, D, D, i64]
        lib.oracle_swiglu_fwd.restype = None
        lib.oracle_swiglu_bwd.argtypes = [D, D, D, D, D, D, i64]
        lib.oracle_swiglu_bwd.restype = None
        lib.oracle_qk_rope.argtypes = [D, D, D, D, D, D, I64, i64, I32, i32,
                                       i32, i32, i32, f64, ctypes.c_int]
        lib.oracle_qk_rope.restype = ctypes.c_int
        lib.oracle_qk_rope_freq.argtypes = [D, D, D, D, D, D, I64, i64, I32, i32,
                                            i32, i32, i32, D, ctypes.c_int]
        lib.oracle_qk_rope_freq.restype = ctypes.c_int
        lib.oracle_rope_inv_freq.argtypes = [i32, f64, D]
        lib.oracle_rope_inv_freq.restype = None
        lib.oracle_rope_llama3_inv_freq.argtypes = [i32, f64, f64, f64, f64, f64, D]
        lib.oracle_rope_llama3_inv_freq.restype = ctypes.c_int
        lib.oracle_positions.argtypes = [I64, I64, i64, I32, i32]
        lib.oracle_positions.restype = ctypes.c_int
        lib.oracle_rmsnorm_add_fwd.argtypes = [D, D, D, D, D, D, i64, i64, f64, ctypes.c_int]
        lib.oracle_rmsnorm_add_fwd.restype = None
        lib.oracle_rmsnorm_add_bwd.argtypes = [D, D, D, D, D, D, D, D, i64, i64, f64]
        lib.oracle_rmsnorm_add_bwd.restype = None
        lib.oracle_threads.argtypes = []
        lib.oracle_threads.restype = ctypes.c_int
        lib.oracle_set_threads.argtypes = [ctypes.c_int]
        lib.oracle_set_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # torch tensor: exact upcast on the CPU
        import torch
        a = a.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a, ctype=ctypes.c_double):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def rmsnorm_fwd(x, w, eps):
    """Returns (y [T,H], rstd [T])."""
    x, w = _f64(x), _f64(w)
    T, H = x.shape
    y = np.empty_like(x)
    rstd = np.empty(T)
    _load().oracle_rmsnorm_fwd(_p(x), _p(w), _p(y), _p(rstd), T, H, float(eps))
    return y, rstd


def rmsnorm_bwd(dy, x, w, eps, scales=False):
    """Returns (dx, dw) or, with scales=True, (dx, dw, dx_scale, dw_scale)."""
    dy, x, w = _f64(dy), _f64(x), _f64(w)
    T, H = x.shape
    dx = np.empty_like(x)
    dw = np.empty(H)
    dxs = np.empty_like(x) if scales else None
    dws = np.empty(H) if scales else None
    _load().oracle_rmsnorm_bwd(_p(dy), _p(x), _p(w), _p(dx), _p(dw), _p(dxs),
                               _p(dws), T, H, float(eps))
    return (dx, dw, dxs, dws) if scales else (dx, dw)


STORAGE = {"f32": 0, "bf16": 1, "exact": 2}


def rmsnorm_add_fwd(x, res, w, eps, storage="bf16"):
    """Returns (h, y, rstd): h = x + res added in fp32 and rounded to the
    storage type ("f32", "bf16", or "exact" = no rounding), y = rmsnorm(h)*w."""
    x, res, w = _f64(x), _f64(res), _f64(w)
    T, H = x.shape
    h, y, rstd = np.empty_like(x), np.empty_like(x), np.empty(T)
    _load().oracle_rmsnorm_add_fwd(_p(x), _p(res), _p(w), _p(h), _p(y), _p(rstd), T, H,
                                   float(eps), STORAGE[storage])
    return h, y, rstd


def rmsnorm_add_bwd(dy, dh, h, w, eps, scales=False):
    """Returns (dx, dw) or (dx, dw, dx_scale, dw_scale); dx is the gradient
    of both x and res."""
    dy, dh, h, w = _f64(dy), _f64(dh), _f64(h), _f64(w)
    T, H = h.shape
    dx, dw = np.empty_like(h), np.empty(H)
    dxs = np.empty_like(h) if scales else None
    dws = np.empty(H) if scales else None
    _load().oracle_rmsnorm_add_bwd(_p(dy), _p(dh), _p(h), _p(w), _p(dx), _p(dw), _p(dxs),
                                   _p(dws), T, H, float(eps))
    return (dx, dw, dxs, dws) if scales else (dx, dw)


def swiglu_fwd(g, u):
    g, u = _f64(g), _f64(u)
    h = np.empty_like(g)
    _load().oracle_swiglu_fwd(_p(g), _p(u), _p(h), g.size)
    return h


def swiglu_bwd(dh, g, u, scales=False):
    """Returns (dg, du) or (dg, du, dg_scale)."""
    dh, g, u = _f64(dh), _f64(g), _f64(u)
    dg, du = np.empty_like(g), np.empty_like(g)
    dgs = np.empty_like(g) if scales else None
    _load().oracle_swiglu_bwd(_p(dh), _p(g), _p(u), _p(dg), _p(du), _p(dgs), g.size)
    return (dg, du, dgs) if scales else (dg, du)


def qk_rope(q, k, cu_seqlens, theta, sign=+1, tok=None, scales=False):
    """Rotate q [n,Hq,D] and k [n,Hkv,D] (row r = global token tok[r]).

    sign=+1 is the forward rotation, -1 the backward (transposed) one.
    Returns (q_out, k_out) or (q_out, k_out, q_scale, k_scale).
    """
    q, k = _f64(q), _f64(k)
    n, Hq, D = q.shape
    Hkv = k.shape[1]
    assert k.shape[0] == n and k.shape[2] == D
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    B = cu.size - 1
    tk = None if tok is None else np.ascontiguousarray(np.asarray(tok, dtype=np.int64))
    qo, ko = np.empty_like(q), np.empty_like(k)
    qs = np.empty_like(q) if scales else None
    ks = np.empty_like(k) if scales else None
    rc = _load().oracle_qk_rope(_p(q), _p(k), _p(qo), _p(ko), _p(qs), _p(ks),
                                _p(tk, ctypes.c_int64), n, _p(cu, ctypes.c_int32),
                                B, Hq, Hkv, D, float(theta), int(sign))
    if rc != 0:
        raise ValueError("oracle_qk_rope: token outside the packed batch or odd D")
    return (qo, ko, qs, ks) if scales else (qo, ko)


def qk_rope_freq(q, k, cu_seqlens, inv_freq, sign=+1, tok=None, scales=False):
    """qk_rope with an explicit inverse-frequency table inv_freq[D/2]
    (phi_i = p * inv_freq[i]) instead of theta."""
    q, k = _f64(q), _f64(k)
    n, Hq, D = q.shape
    Hkv = k.shape[1]
    assert k.shape[0] == n and k.shape[2] == D
    f = _f64(inv_freq)
    assert f.shape == (D // 2,)
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    B = cu.size - 1
    tk = None if tok is None else np.ascontiguousarray(np.asarray(tok, dtype=np.int64))
    qo, ko = np.empty_like(q), np.empty_like(k)
    qs = np.empty_like(q) if scales else None
    ks = np.empty_like(k) if scales else None
    rc = _load().oracle_qk_rope_freq(_p(q), _p(k), _p(qo), _p(ko), _p(qs), _p(ks),
                                     _p(tk, ctypes.c_int64), n, _p(cu, ctypes.c_int32),
                                     B, Hq, Hkv, D, _p(f), int(sign))
    if rc != 0:
        raise ValueError("oracle_qk_rope_freq: token outside the packed batch or odd D")
    return (qo, ko, qs, ks) if scales else (qo, ko)


def qk_norm_rope_fwd(q, k, wq, wk, eps, cu_seqlens, inv_freq, tok=None, scales=False):
    """Per-head RMSNorm of q [n,Hq,D] and k [n,Hkv,D] (weights wq, wk [D]),
    then the rotation with inv_freq [D/2]: the two pinned steps above run
    one after the other, in double, with no rounding between them.
    Returns (q_out, k_out, rstd_q [n,Hq], rstd_k [n,Hkv]) and, with
    scales=True, the rotation's condition scales of q_out and k_out."""
    q, k = _f64(q), _f64(k)
    n, Hq, D = q.shape
    Hkv = k.shape[1]
    nq, rq = rmsnorm_fwd(q.reshape(n * Hq, D), wq, eps)
    nk, rk = rmsnorm_fwd(k.reshape(n * Hkv, D), wk, eps)
    out = qk_rope_freq(nq.reshape(n, Hq, D), nk.reshape(n, Hkv, D), cu_seqlens, inv_freq, +1,
                       tok=tok, scales=scales)
    rq, rk = rq.reshape(n, Hq), rk.reshape(n, Hkv)
    if scales:
        return out[0], out[1], rq, rk, out[2], out[3]
    return out[0], out[1], rq, rk


def qk_norm_rope_bwd(dq, dk, q, k, wq, wk, eps, cu_seqlens, inv_freq, tok=None, scales=False):
    """Gradient of qk_norm_rope_fwd: the rotation's transpose takes dq, dk
    back to the normalised vectors, then the RMSNorm backward (per head
    vector, rows of D) gives the gradients of the pre-norm q, k and of wq,
    wk.  Returns (dq_in, dk_in, dwq, dwk) and, with scales=True, their
    condition scales: the rotation's scale of the intermediate gradient
    carried through the (linear in |dy|) RMSNorm scale."""
    q, k = _f64(q), _f64(k)
    n, Hq, D = q.shape
    Hkv = k.shape[1]
    dnq, dnk, sq, sk = qk_rope_freq(dq, dk, cu_seqlens, inv_freq, -1, tok=tok, scales=True)
    dvq, dwq = rmsnorm_bwd(dnq.reshape(n * Hq, D), q.reshape(n * Hq, D), wq, eps)
    dvk, dwk = rmsnorm_bwd(dnk.reshape(n * Hkv, D), k.reshape(n * Hkv, D), wk, eps)
    dvq, dvk = dvq.reshape(n, Hq, D), dvk.reshape(n, Hkv, D)
    if not scales:
        return dvq, dvk, dwq, dwk
    _, _, svq, swq = rmsnorm_bwd(sq.reshape(n * Hq, D), q.reshape(n * Hq, D), wq, eps, scales=True)
    _, _, svk, swk = rmsnorm_bwd(sk.reshape(n * Hkv, D), k.reshape(n * Hkv, D), wk, eps,
                                 scales=True)
    return dvq, dvk, dwq, dwk, svq.reshape(n, Hq, D), svk.reshape(n, Hkv, D), swq, swk


def rope_inv_freq(D, theta):
    """theta^(-2i/D), i < D/2."""
    out = np.empty(D // 2)
    _load().oracle_rope_inv_freq(int(D), float(theta), _p(out))
    return out


def rope_llama3_inv_freq(D, theta, factor, low_freq_factor, high_freq_factor,
                         original_max_position):
    """The "llama3"-scaled inverse frequencies (see oracle.c)."""
    out = np.empty(D // 2)
    rc = _load().oracle_rope_llama3_inv_freq(int(D), float(theta), float(factor),
                                             float(low_freq_factor), float(high_freq_factor),
                                             float(original_max_position), _p(out))
    if rc != 0:
        raise ValueError("llama3 scaling needs D even and high_freq_factor > low_freq_factor")
    return out


def positions(cu_seqlens, tok=None, n=None):
    cu = np.ascontiguousarray(np.asarray(cu_seqlens, dtype=np.int32))
    if tok is None:
        n = int(cu[-1]) if n is None else n
        tk = None
    else:
        tk = np.ascontiguousarray(np.asarray(tok, dtype=np.int64))
        n = tk.size
    pos = np.empty(n, dtype=np.int64)
    rc = _load().oracle_positions(_p(pos, ctypes.c_int64), _p(tk, ctypes.c_int64),
                                  n, _p(cu, ctypes.c_int32), cu.size - 1)
    if rc != 0:
        raise ValueError("oracle_positions: token outside the packed batch")
    return pos


def threads() -> int:
    """Threads the oracle's parallel loops run on."""
    return int(_load().oracle_threads())


def set_threads(n: int) -> int:
    """Runs the oracle's parallel loops on n threads from now on; returns the
    previous count.  For timing only: no result depends on it."""
    return int(_load().oracle_set_threads(int(n)))
