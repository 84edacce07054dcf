"""Python binding of libftk.so (the C ABI in include/ftk.h).

Argument marshalling only: each function checks that its tensors are CUDA
tensors with unit inner stride, allocates missing outputs with torch, and
calls the C entry point of the same name on the current torch stream.  Every
step of every op runs in the library's CUDA kernels; there is no other path.
If libftk.so is missing this module raises ImportError on first use.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import numpy as np
import torch

from .build import LIB as _LIB_PATH

F32, BF16 = 0, 1
_DTYPES = {torch.float32: F32, torch.bfloat16: BF16}

STATUS = {0: "FTK_OK", 1: "FTK_ERR_NULL", 2: "FTK_ERR_SHAPE", 3: "FTK_ERR_ALIGN",
          4: "FTK_ERR_DTYPE", 5: "FTK_ERR_WORKSPACE", 6: "FTK_ERR_CUDA", 7: "FTK_ERR_ALIAS"}


class FtkError(RuntimeError):
    def __init__(self, fn: str, status: int, lib):
        self.status = status
        msg = f"{fn}: {STATUS.get(status, status)} ({lib.ftk_status_str(status).decode()})"
        if status == 6:
            msg += f": {lib.ftk_last_cuda_error().decode()}"
        super().__init__(msg)


_lib = None


def library() -> ctypes.CDLL:
    """The loaded libftk.so (raises ImportError if it was never built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"{_LIB_PATH} is missing: build it with fine_tuning_gb300.build.build() "
            "(nvcc, sm_103a); the ftk ops have no other implementation")
    lib = ctypes.CDLL(_LIB_PATH)
    vp, i64, i32, f32, f64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                              ctypes.c_float, ctypes.c_double)
    st, dt, sz = ctypes.c_int, ctypes.c_int, ctypes.c_size_t
    sig = {
        "ftk_rmsnorm_fwd": (st, [vp, i64, vp, vp, i64, vp, i64, i64, f32, dt, vp]),
        "ftk_rmsnorm_bwd_workspace_bytes": (sz, [i64, i64, dt]),
        "ftk_rmsnorm_bwd": (st, [vp, i64, vp, i64, vp, vp, vp, i64, vp, vp, sz, i64, i64,
                                 f32, dt, vp]),
        "ftk_rmsnorm_add_fwd": (st, [vp, i64, vp, i64, vp, vp, i64, vp, i64, vp, i64, i64, f32,
                                     dt, vp]),
        "ftk_rmsnorm_add_bwd": (st, [vp, i64, vp, i64, vp, i64, vp, vp, vp, i64, vp, vp, sz,
                                     i64, i64, f32, dt, vp]),
        "ftk_swiglu_fwd": (st, [vp, vp, i64, vp, i64, i64, i64, dt, vp]),
        "ftk_swiglu_bwd": (st, [vp, i64, vp, vp, i64, vp, vp, i64, i64, i64, dt, vp]),
        "ftk_swiglu_bwd_h": (st, [vp, i64, vp, vp, i64, vp, vp, i64, vp, i64, i64, i64, dt,
                                  vp]),
        "ftk_qk_rope_fwd": (st, [vp, i64, vp, i64, vp, i32, i64, i32, i32, i32, f64, dt, vp]),
        "ftk_qk_rope_bwd": (st, [vp, i64, vp, i64, vp, i32, i64, i32, i32, i32, f64, dt, vp]),
        "ftk_qk_rope_freq_fwd": (st, [vp, i64, vp, i64, vp, i32, i64, i32, i32, i32, vp, dt,
                                      vp]),
        "ftk_qk_rope_freq_bwd": (st, [vp, i64, vp, i64, vp, i32, i64, i32, i32, i32, vp, dt,
                                      vp]),
        "ftk_rope_llama3_inv_freq": (st, [i32, f64, f64, f64, f64, f64, vp]),
        "ftk_qk_norm_rope_fwd": (st, [vp, i64, vp, i64, vp, vp, vp, i64, vp, i64, vp, vp, vp,
                                      i32, i64, i32, i32, i32, f64, vp, f32, dt, vp]),
        "ftk_qk_norm_rope_bwd_workspace_bytes": (sz, [i64, i32, dt]),
        "ftk_qk_norm_rope_bwd": (st, [vp, i64, vp, i64, vp, i64, vp, i64, vp, vp, vp, vp, vp,
                                      i64, vp, i64, vp, vp, vp, sz, vp, i32, i64, i32, i32, i32,
                                      f64, vp, f32, dt, vp]),
        "ftk_qk_norm_rope_fwd_checked": (st, [vp, i64, vp, i64, vp, vp, vp, i64, vp, i64, vp, vp,
                                              vp, i32, i64, i32, i32, i32, f64, vp, f32, vp, dt,
                                              vp]),
        "ftk_qk_norm_rope_bwd_checked": (st, [vp, i64, vp, i64, vp, i64, vp, i64, vp, vp, vp, vp,
                                              vp, i64, vp, i64, vp, vp, vp, sz, vp, i32, i64, i32,
                                              i32, i32, f64, vp, f32, vp, dt, vp]),
        "ftk_gemm_bf16": (st, [vp, i64, vp, i64, vp, i64, i64, i64, i64, vp]),
        "ftk_gemm_bf16_ex": (st, [vp, i64, i32, vp, i64, i32, vp, i64, i64, i64, i64, vp]),
        "ftk_cce_fwd_workspace_bytes": (sz, [i64, i64]),
        "ftk_cce_bwd_workspace_bytes": (sz, [i64, i64, i64]),
        "ftk_cce_bwd_chunk": (i64, [i64, i64, i64, i32]),
        "ftk_cce_fwd": (st, [vp, i64, vp, i64, vp, i64, i64, i64, vp, vp, vp, sz, dt, vp]),
        "ftk_cce_bwd": (st, [vp, i64, vp, i64, vp, vp, vp, i64, i64, i64, vp, i64, vp, i64, vp,
                             sz, dt, vp]),
        "ftk_check_seqlens": (st, [vp, i32, i64, vp, vp]),
        "ftk_qk_rope_fwd_checked": (st, [vp, i64, vp, i64, vp, i32, i64, i32, i32, i32, f64, vp,
                                         vp, dt, vp]),
        "ftk_qk_rope_bwd_checked": (st, [vp, i64, vp, i64, vp, i32, i64, i32, i32, i32, f64, vp,
                                         vp, dt, vp]),
        "ftk_bfd_pack": (st, [vp, i64, i32, vp, vp, vp, vp]),
        "ftk_device_status": (st, [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]),
        "ftk_selftest_wait_timeout": (st, [i64, vp]),
        "ftk_status_str": (ctypes.c_char_p, [st]),
        "ftk_last_cuda_error": (ctypes.c_char_p, []),
        "ftk_version": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype, fn.argtypes = res, args
    _lib = lib
    return lib


def _call(name: str, *args) -> None:
    lib = library()
    status = getattr(lib, name)(*args)
    if status != 0:
        raise FtkError(name, status, lib)


def _code(t: torch.Tensor) -> int:
    try:
        return _DTYPES[t.dtype]
    except KeyError:
        raise TypeError(f"ftk supports float32 and bfloat16 storage, got {t.dtype}") from None


def _cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("ftk ops take CUDA tensors (move inputs with .cuda())")


def _rows(t: torch.Tensor, name: str) -> int:
    """Row stride (elements) of a [rows, n] view with unit inner stride."""
    if t.dim() != 2:
        raise ValueError(f"{name} must be 2-D [tokens, features], got {tuple(t.shape)}")
    if t.stride(1) != 1 and t.shape[1] > 1:
        raise ValueError(f"{name} needs unit stride along features")
    return t.stride(0) if t.shape[0] > 1 else max(t.shape[1], t.stride(0))


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else t.data_ptr()


# ---------------------------------------------------------------- RMSNorm

def rmsnorm_fwd(x: torch.Tensor, w: torch.Tensor, eps: float, y: Optional[torch.Tensor] = None,
                rstd: Optional[torch.Tensor] = None, save_rstd: bool = True
                ) -> Tuple[torch.Tensor, Optional[torch.Tensor]]:
    """y = x * rsqrt(mean(x^2) + eps) * w over rows of x [T, H]; returns (y, rstd)."""
    _cuda(x, w, y, rstd)
    T, H = x.shape
    if y is None:
        y = torch.empty((T, H), dtype=x.dtype, device=x.device)
    if rstd is None and save_rstd:
        rstd = torch.empty((T,), dtype=torch.float32, device=x.device)
    if w.dtype != x.dtype or y.dtype != x.dtype or w.numel() != H or not w.is_contiguous():
        raise ValueError("w must be a contiguous [H] tensor and y must match x's dtype")
    if rstd is not None and (rstd.dtype != torch.float32 or rstd.numel() != T or not rstd.is_contiguous()):
        raise ValueError("rstd must be a contiguous fp32 [T] tensor")
    _call("ftk_rmsnorm_fwd", _ptr(x), _rows(x, "x"), _ptr(w), _ptr(y), _rows(y, "y"),
          _ptr(rstd), T, H, float(eps), _code(x), _stream(x))
    return y, rstd


def rmsnorm_bwd_workspace_bytes(T: int, H: int, dtype: torch.dtype) -> int:
    return int(library().ftk_rmsnorm_bwd_workspace_bytes(T, H, _DTYPES[dtype]))


def rmsnorm_bwd(dy: torch.Tensor, x: torch.Tensor, w: torch.Tensor, rstd: Optional[torch.Tensor],
                eps: float, dx: Optional[torch.Tensor] = None, dw: Optional[torch.Tensor] = None,
                workspace: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Returns (dx [T, H] in x's dtype, dw [H] fp32).  rstd=None recomputes it."""
    _cuda(dy, x, w, rstd, dx, dw, workspace)
    T, H = x.shape
    if dx is None:
        dx = torch.empty((T, H), dtype=x.dtype, device=x.device)
    if dw is None:
        dw = torch.empty((H,), dtype=torch.float32, device=x.device)
    if workspace is None:
        workspace = _workspace(T, H, x)
    if dy.shape != x.shape or dy.dtype != x.dtype or dx.dtype != x.dtype:
        raise ValueError("dy and dx must match x in shape and dtype")
    if dw.dtype != torch.float32 or dw.numel() != H or not dw.is_contiguous():
        raise ValueError("dw must be a contiguous fp32 [H] tensor")
    _call("ftk_rmsnorm_bwd", _ptr(dy), _rows(dy, "dy"), _ptr(x), _rows(x, "x"), _ptr(w),
          _ptr(rstd), _ptr(dx), _rows(dx, "dx"), _ptr(dw), _ptr(workspace),
          workspace.numel() * workspace.element_size(), T, H, float(eps), _code(x), _stream(x))
    return dx, dw


def _workspace(T: int, H: int, like: torch.Tensor) -> torch.Tensor:
    nbytes = max(16, rmsnorm_bwd_workspace_bytes(T, H, like.dtype))
    return torch.empty((nbytes + 3) // 4, dtype=torch.float32, device=like.device)


def rmsnorm_add_fwd(x: torch.Tensor, res: torch.Tensor, w: torch.Tensor, eps: float,
                    h: Optional[torch.Tensor] = None, y: Optional[torch.Tensor] = None,
                    rstd: Optional[torch.Tensor] = None, save_rstd: bool = True
                    ) -> Tuple[torch.Tensor, torch.Tensor, Optional[torch.Tensor]]:
    """h = x + res (stored, x's dtype), y = rmsnorm(h) * w; returns (h, y, rstd).
    Pass h=res (or h=x) to update the residual stream in place."""
    _cuda(x, res, w, h, y, rstd)
    T, H = x.shape
    if h is None:
        h = torch.empty((T, H), dtype=x.dtype, device=x.device)
    if y is None:
        y = torch.empty((T, H), dtype=x.dtype, device=x.device)
    if rstd is None and save_rstd:
        rstd = torch.empty((T,), dtype=torch.float32, device=x.device)
    for t in (res, h, y):
        if t.shape != x.shape or t.dtype != x.dtype:
            raise ValueError("res, h and y must match x in shape and dtype")
    if w.dtype != x.dtype or w.numel() != H or not w.is_contiguous():
        raise ValueError("w must be a contiguous [H] tensor of x's dtype")
    if rstd is not None and (rstd.dtype != torch.float32 or rstd.numel() != T or not rstd.is_contiguous()):
        raise ValueError("rstd must be a contiguous fp32 [T] tensor")
    _call("ftk_rmsnorm_add_fwd", _ptr(x), _rows(x, "x"), _ptr(res), _rows(res, "res"), _ptr(w),
          _ptr(h), _rows(h, "h"), _ptr(y), _rows(y, "y"), _ptr(rstd), T, H, float(eps),
          _code(x), _stream(x))
    return h, y, rstd


def rmsnorm_add_bwd(dy: torch.Tensor, dh: torch.Tensor, h: torch.Tensor, w: torch.Tensor,
                    rstd: Optional[torch.Tensor], eps: float, dx: Optional[torch.Tensor] = None,
                    dw: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None
                    ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Backward of rmsnorm_add_fwd: dx = dh + the norm's gradient at h (the
    gradient of both x and res), dw [H] fp32.  rstd=None recomputes it."""
    _cuda(dy, dh, h, w, rstd, dx, dw, workspace)
    T, H = h.shape
    if dx is None:
        dx = torch.empty((T, H), dtype=h.dtype, device=h.device)
    if dw is None:
        dw = torch.empty((H,), dtype=torch.float32, device=h.device)
    if workspace is None:
        workspace = _workspace(T, H, h)
    for t in (dy, dh, dx):
        if t.shape != h.shape or t.dtype != h.dtype:
            raise ValueError("dy, dh and dx must match h in shape and dtype")
    if dw.dtype != torch.float32 or dw.numel() != H or not dw.is_contiguous():
        raise ValueError("dw must be a contiguous fp32 [H] tensor")
    _call("ftk_rmsnorm_add_bwd", _ptr(dy), _rows(dy, "dy"), _ptr(dh), _rows(dh, "dh"), _ptr(h),
          _rows(h, "h"), _ptr(w), _ptr(rstd), _ptr(dx), _rows(dx, "dx"), _ptr(dw),
          _ptr(workspace), workspace.numel() * workspace.element_size(), T, H, float(eps),
          _code(h), _stream(h))
    return dx, dw


# ----------------------------------------------------------------- SwiGLU

def swiglu_fwd(g: torch.Tensor, u: torch.Tensor, h: Optional[torch.Tensor] = None) -> torch.Tensor:
    """h = silu(g) * u for g, u [T, I] (equal row strides, e.g. two halves of gate_up)."""
    _cuda(g, u, h)
    T, I = g.shape
    if u.shape != g.shape or u.dtype != g.dtype:
        raise ValueError("g and u must have the same shape and dtype")
    ld = _rows(g, "g")
    if _rows(u, "u") != ld:
        raise ValueError("g and u must share one row stride")
    if h is None:
        h = torch.empty((T, I), dtype=g.dtype, device=g.device)
    _call("ftk_swiglu_fwd", _ptr(g), _ptr(u), ld, _ptr(h), _rows(h, "h"), T, I, _code(g),
          _stream(g))
    return h


def swiglu_bwd(dh: torch.Tensor, g: torch.Tensor, u: torch.Tensor,
               dg: Optional[torch.Tensor] = None, du: Optional[torch.Tensor] = None
               ) -> Tuple[torch.Tensor, torch.Tensor]:
    """(dg, du) of h = silu(g) * u; dg/du may be g/u themselves (in place)."""
    _cuda(dh, g, u, dg, du)
    T, I = g.shape
    ld = _rows(g, "g")
    if _rows(u, "u") != ld or u.shape != g.shape or dh.shape != g.shape:
        raise ValueError("dh, g and u must have one shape; g and u one row stride")
    if dg is None and du is None:
        dg = torch.empty((T, I), dtype=g.dtype, device=g.device)
        du = torch.empty((T, I), dtype=g.dtype, device=g.device)
    elif dg is None or du is None:
        raise ValueError("pass both dg and du, or neither")
    ldo = _rows(dg, "dg")
    if _rows(du, "du") != ldo:
        raise ValueError("dg and du must share one row stride")
    _call("ftk_swiglu_bwd", _ptr(dh), _rows(dh, "dh"), _ptr(g), _ptr(u), ld, _ptr(dg), _ptr(du),
          ldo, T, I, _code(g), _stream(g))
    return dg, du


def swiglu_bwd_h(dh: torch.Tensor, g: torch.Tensor, u: torch.Tensor,
                 dg: Optional[torch.Tensor] = None, du: Optional[torch.Tensor] = None,
                 h: Optional[torch.Tensor] = None
                 ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """(dg, du, h): swiglu_bwd plus the forward's h, recomputed bit-identically
    (h may be dh, g or u themselves; not dg or du)."""
    _cuda(dh, g, u, dg, du, h)
    T, I = g.shape
    ld = _rows(g, "g")
    if _rows(u, "u") != ld or u.shape != g.shape or dh.shape != g.shape:
        raise ValueError("dh, g and u must have one shape; g and u one row stride")
    if dg is None and du is None:
        dg = torch.empty((T, I), dtype=g.dtype, device=g.device)
        du = torch.empty((T, I), dtype=g.dtype, device=g.device)
    elif dg is None or du is None:
        raise ValueError("pass both dg and du, or neither")
    if h is None:
        h = torch.empty((T, I), dtype=g.dtype, device=g.device)
    if h.shape != g.shape or h.dtype != g.dtype:
        raise ValueError("h must match g in shape and dtype")
    ldo = _rows(dg, "dg")
    if _rows(du, "du") != ldo:
        raise ValueError("dg and du must share one row stride")
    _call("ftk_swiglu_bwd_h", _ptr(dh), _rows(dh, "dh"), _ptr(g), _ptr(u), ld, _ptr(dg),
          _ptr(du), ldo, _ptr(h), _rows(h, "h"), T, I, _code(g), _stream(g))
    return dg, du, h


# ---------------------------------------------------------------- QK-RoPE

def _heads(t: Optional[torch.Tensor], name: str):
    """(row stride, heads, head_dim) of a [T, heads, D] view with contiguous heads."""
    if t is None:
        return 0, 0, 0
    if t.dim() != 3:
        raise ValueError(f"{name} must be [T, heads, head_dim], got {tuple(t.shape)}")
    T, nh, D = t.shape
    if (D > 1 and t.stride(2) != 1) or (nh > 1 and t.stride(1) != D):
        raise ValueError(f"{name} needs contiguous heads of contiguous head_dim values")
    return (t.stride(0) if T > 1 else nh * D), nh, D


def _rope(name, q, k, cu_seqlens, theta, inv_freq=None, checked=False, status=None):
    _cuda(q, k, cu_seqlens)
    ldq, Hq, Dq = _heads(q, "q")
    ldk, Hkv, Dk = _heads(k, "k")
    D = Dq or Dk
    if q is not None and k is not None and (q.shape[0] != k.shape[0] or Dq != Dk or q.dtype != k.dtype):
        raise ValueError("q and k must agree in tokens, head_dim and dtype")
    ref = q if q is not None else k
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or not cu_seqlens.is_contiguous():
        raise ValueError("cu_seqlens must be a contiguous int32 [B+1] device tensor")
    table, table_p = _table(inv_freq, D)
    if checked:
        _status_check(status)
        freq_args = (float(theta or 0.0), table_p, _ptr(status))
    else:
        freq_args = (float(theta),) if inv_freq is None else (table_p,)
    _call(name, _ptr(q), ldq, _ptr(k), ldk, _ptr(cu_seqlens), cu_seqlens.numel() - 1,
          ref.shape[0], Hq, Hkv, D, *freq_args, _code(ref), _stream(ref))
    del table
    return q, k


def qk_rope_fwd(q, k, cu_seqlens, theta):
    """Rotate q [T, Hq, D] and k [T, Hkv, D] IN PLACE at packed positions; returns (q, k)."""
    return _rope("ftk_qk_rope_fwd", q, k, cu_seqlens, theta)


def qk_rope_bwd(dq, dk, cu_seqlens, theta):
    """Backward of qk_rope_fwd: rotate dq, dk by -phi IN PLACE; returns (dq, dk)."""
    return _rope("ftk_qk_rope_bwd", dq, dk, cu_seqlens, theta)


def qk_rope_freq_fwd(q, k, cu_seqlens, inv_freq):
    """qk_rope_fwd with a host table of D/2 inverse frequencies (a scaled RoPE)."""
    return _rope("ftk_qk_rope_freq_fwd", q, k, cu_seqlens, None, inv_freq)


def qk_rope_freq_bwd(dq, dk, cu_seqlens, inv_freq):
    """Backward of qk_rope_freq_fwd, in place."""
    return _rope("ftk_qk_rope_freq_bwd", dq, dk, cu_seqlens, None, inv_freq)


def check_seqlens(cu_seqlens, T: int, status: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Validate a packed batch's boundaries on the device, without a host
    synchronisation: the returned int32 [1] device tensor (`status`, if
    given, is overwritten) receives the SEQLENS_* bits found (0: valid).
    Pass it to the *_checked rotations of every layer of the batch."""
    _cuda(cu_seqlens, status)
    _cu_check(cu_seqlens)
    if status is None:
        status = torch.empty(1, dtype=torch.int32, device=cu_seqlens.device)
    _status_check(status)
    _call("ftk_check_seqlens", _ptr(cu_seqlens), cu_seqlens.numel() - 1, int(T), _ptr(status),
          _stream(cu_seqlens))
    return status


SEQLENS_BAD_START, SEQLENS_DECREASING, SEQLENS_BAD_END = 1, 2, 4


def _status_check(status):
    if status is None or not status.is_cuda or status.dtype not in (torch.int32, torch.uint32) \
            or status.numel() < 1:
        raise ValueError("the seqlens status must be a 32-bit integer device tensor")


def qk_rope_fwd_checked(q, k, cu_seqlens, seqlens_status, theta: float = 0.0, inv_freq=None):
    """qk_rope_fwd (or, with inv_freq, qk_rope_freq_fwd) that leaves q and k
    untouched when the word check_seqlens wrote is non-zero."""
    return _rope("ftk_qk_rope_fwd_checked", q, k, cu_seqlens, theta, inv_freq, True,
                 seqlens_status)


def qk_rope_bwd_checked(dq, dk, cu_seqlens, seqlens_status, theta: float = 0.0, inv_freq=None):
    """Backward of qk_rope_fwd_checked, in place, under the same guard."""
    return _rope("ftk_qk_rope_bwd_checked", dq, dk, cu_seqlens, theta, inv_freq, True,
                 seqlens_status)


def _table(inv_freq, D):
    if inv_freq is None:
        return None, None
    table = np.ascontiguousarray(np.asarray(inv_freq, dtype=np.float64))
    if table.shape != (D // 2,):
        raise ValueError("inv_freq must hold D/2 values")
    return table, table.ctypes.data_as(ctypes.c_void_p)


def _cu_check(cu_seqlens):
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or not cu_seqlens.is_contiguous():
        raise ValueError("cu_seqlens must be a contiguous int32 [B+1] device tensor")


def qk_norm_rope_fwd(q, k, wq, wk, cu_seqlens, eps: float, theta: float = 0.0, inv_freq=None,
                     q_out=None, k_out=None, save_rstd: bool = True, rstd_q=None, rstd_k=None,
                     seqlens_status=None):
    """Per-head RMSNorm (weights wq, wk [D]) then RoPE of q [T, Hq, D] and
    k [T, Hkv, D]; returns (q_out, k_out, rstd_q [T, Hq], rstd_k [T, Hkv]).
    q_out=q / k_out=k update in place.  inv_freq (host, D/2) replaces theta.
    rstd_q / rstd_k: fp32 buffers to write r into (else allocated when
    save_rstd).  seqlens_status: the word check_seqlens wrote; when given,
    a non-zero word leaves every output untouched (the checked call)."""
    _cuda(q, k, wq, wk, cu_seqlens, q_out, k_out, rstd_q, rstd_k)
    if seqlens_status is not None:
        _status_check(seqlens_status)
    _cu_check(cu_seqlens)
    ldq, Hq, Dq = _heads(q, "q")
    ldk, Hkv, Dk = _heads(k, "k")
    D = Dq or Dk
    ref = q if q is not None else k
    T = ref.shape[0]
    if q is not None and q_out is None:
        q_out = torch.empty_like(q)
    if k is not None and k_out is None:
        k_out = torch.empty_like(k)
    ldqo, _, _ = _heads(q_out, "q_out")
    ldko, _, _ = _heads(k_out, "k_out")
    rq, rk = rstd_q, rstd_k
    if rq is None and save_rstd and Hq:
        rq = torch.empty((T, Hq), dtype=torch.float32, device=ref.device)
    if rk is None and save_rstd and Hkv:
        rk = torch.empty((T, Hkv), dtype=torch.float32, device=ref.device)
    for r, n in ((rq, Hq), (rk, Hkv)):
        if r is not None and (r.dtype != torch.float32 or r.numel() != T * n
                              or not r.is_contiguous()):
            raise ValueError("rstd buffers must be contiguous fp32 [T, heads]")
    table, tp = _table(inv_freq, D)
    args = [_ptr(q), ldq, _ptr(k), ldk, _ptr(wq), _ptr(wk), _ptr(q_out), ldqo, _ptr(k_out), ldko,
            _ptr(rq), _ptr(rk), _ptr(cu_seqlens), cu_seqlens.numel() - 1, T, Hq, Hkv, D,
            float(theta), tp, float(eps)]
    if seqlens_status is None:
        _call("ftk_qk_norm_rope_fwd", *args, _code(ref), _stream(ref))
    else:
        _call("ftk_qk_norm_rope_fwd_checked", *args, _ptr(seqlens_status), _code(ref),
              _stream(ref))
    del table
    return q_out, k_out, rq, rk


def qk_norm_rope_bwd_workspace_bytes(T: int, D: int, dtype: torch.dtype) -> int:
    return int(library().ftk_qk_norm_rope_bwd_workspace_bytes(T, D, _DTYPES[dtype]))


def qk_norm_rope_bwd(dq_out, dk_out, q, k, wq, wk, rstd_q, rstd_k, cu_seqlens, eps: float,
                     theta: float = 0.0, inv_freq=None, dq=None, dk=None, workspace=None,
                     dwq=None, dwk=None, seqlens_status=None):
    """Backward of qk_norm_rope_fwd from the output gradients and the
    PRE-norm q, k; returns (dq, dk, dwq [D] fp32, dwk [D] fp32).  dq=dq_out
    (dk=dk_out) writes in place.  rstd_q/rstd_k None: recomputed.  dwq, dwk:
    fp32 [D] buffers to write into (else allocated).  seqlens_status: the
    word check_seqlens wrote; when given, a non-zero word leaves every output
    untouched (the checked call)."""
    _cuda(dq_out, dk_out, q, k, wq, wk, rstd_q, rstd_k, cu_seqlens, dq, dk, workspace, dwq, dwk)
    if seqlens_status is not None:
        _status_check(seqlens_status)
    _cu_check(cu_seqlens)
    ldq, Hq, Dq = _heads(q, "q")
    ldk, Hkv, Dk = _heads(k, "k")
    D = Dq or Dk
    ref = q if q is not None else k
    T = ref.shape[0]
    if q is not None and dq is None:
        dq = torch.empty_like(q)
    if k is not None and dk is None:
        dk = torch.empty_like(k)
    ldgq, _, _ = _heads(dq_out, "dq_out")
    ldgk, _, _ = _heads(dk_out, "dk_out")
    lddq, _, _ = _heads(dq, "dq")
    lddk, _, _ = _heads(dk, "dk")
    for w_, n in ((dwq, "dwq"), (dwk, "dwk")):
        if w_ is not None and (w_.dtype != torch.float32 or w_.numel() != D
                               or not w_.is_contiguous()):
            raise ValueError(f"{n} must be a contiguous fp32 [D] tensor")
    if dwq is None and Hq:
        dwq = torch.empty(D, dtype=torch.float32, device=ref.device)
    if dwk is None and Hkv:
        dwk = torch.empty(D, dtype=torch.float32, device=ref.device)
    if workspace is None:
        nbytes = max(16, qk_norm_rope_bwd_workspace_bytes(T, D, ref.dtype))
        workspace = torch.empty((nbytes + 3) // 4, dtype=torch.float32, device=ref.device)
    table, tp = _table(inv_freq, D)
    args = [_ptr(dq_out), ldgq, _ptr(dk_out), ldgk, _ptr(q), ldq, _ptr(k), ldk, _ptr(wq),
            _ptr(wk), _ptr(rstd_q), _ptr(rstd_k), _ptr(dq), lddq, _ptr(dk), lddk, _ptr(dwq),
            _ptr(dwk), _ptr(workspace), workspace.numel() * workspace.element_size(),
            _ptr(cu_seqlens), cu_seqlens.numel() - 1, T, Hq, Hkv, D, float(theta), tp, float(eps)]
    if seqlens_status is None:
        _call("ftk_qk_norm_rope_bwd", *args, _code(ref), _stream(ref))
    else:
        _call("ftk_qk_norm_rope_bwd_checked", *args, _ptr(seqlens_status), _code(ref),
              _stream(ref))
    del table
    return dq, dk, dwq, dwk


def rope_llama3_inv_freq(D: int, theta: float, factor: float, low_freq_factor: float,
                         high_freq_factor: float, original_max_position: float) -> np.ndarray:
    """The llama3-scaled inverse frequencies (host; float64 [D/2])."""
    out = np.empty(D // 2, dtype=np.float64)
    _call("ftk_rope_llama3_inv_freq", int(D), float(theta), float(factor), float(low_freq_factor),
          float(high_freq_factor), float(original_max_position),
          out.ctypes.data_as(ctypes.c_void_p))
    return out


# ------------------------------------------------------ Cut Cross-Entropy

def gemm_bf16(a: torch.Tensor, b: torch.Tensor, c: Optional[torch.Tensor] = None,
              a_mn: bool = False, b_mn: bool = False) -> torch.Tensor:
    """C fp32 [M, N] = A @ B^T on the tensor cores (bf16 in).  A is a [M, K]
    or, with a_mn, a [K, M] (then A = a^T); B is b [N, K] or, with b_mn,
    b [K, N] (then B = b^T).  No transposed copy is made."""
    _cuda(a, b, c)
    if a.dtype != torch.bfloat16 or b.dtype != torch.bfloat16 or a.dim() != 2 or b.dim() != 2:
        raise ValueError("a and b must be 2-D bf16")
    K, M = a.shape if a_mn else a.shape[::-1]
    Kb, N = b.shape if b_mn else b.shape[::-1]
    if Kb != K:
        raise ValueError(f"contraction sizes differ: {K} vs {Kb}")
    c = torch.empty((M, N), dtype=torch.float32, device=a.device) if c is None else c
    _call("ftk_gemm_bf16_ex", _ptr(a), _rows(a, "a"), int(a_mn), _ptr(b), _rows(b, "b"),
          int(b_mn), _ptr(c), _rows(c, "c"), M, N, K, _stream(a))
    return c


def _ws(nbytes: int, like: torch.Tensor) -> torch.Tensor:
    return torch.empty(max(256, nbytes), dtype=torch.uint8, device=like.device)


def cce_fwd(h: torch.Tensor, W: torch.Tensor, y: torch.Tensor, loss=None, lse=None,
            workspace=None):
    """Mean cross-entropy of logits h W^T against y (int32; y outside [0, V)
    is ignored), without materialising the logits.  Returns (loss [1] fp32,
    lse [T] fp32), both on the device."""
    _cuda(h, W, y, loss, lse, workspace)
    T, H = h.shape
    V = W.shape[0]
    if W.shape[1] != H or h.dtype != torch.bfloat16 or W.dtype != torch.bfloat16:
        raise ValueError("h [T, H] and W [V, H] must be bf16")
    if y.dtype != torch.int32 or y.numel() != T or not y.is_contiguous():
        raise ValueError("y must be a contiguous int32 [T] tensor")
    loss = torch.empty(1, dtype=torch.float32, device=h.device) if loss is None else loss
    lse = torch.empty(T, dtype=torch.float32, device=h.device) if lse is None else lse
    if workspace is None:
        workspace = _ws(int(library().ftk_cce_fwd_workspace_bytes(T, V)), h)
    _call("ftk_cce_fwd", _ptr(h), _rows(h, "h"), _ptr(W), _rows(W, "W"), _ptr(y), T, H, V,
          _ptr(loss), _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(),
          _code(h), _stream(h))
    return loss, lse


def cce_bwd_chunk(T: int, H: int, V: int, sms: Optional[int] = None) -> int:
    """The vocabulary chunk width cce_bwd uses for these sizes on a device
    with `sms` SMs (default: the current CUDA device's count)."""
    if sms is None:
        sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return int(library().ftk_cce_bwd_chunk(T, H, V, sms))


def cce_bwd(h: torch.Tensor, W: torch.Tensor, y: torch.Tensor, lse: torch.Tensor,
            dloss: torch.Tensor, dh=None, dW=None, workspace=None):
    """Gradients of dloss * cce_fwd(h, W, y): (dh bf16 [T, H], dW fp32 [V, H])."""
    _cuda(h, W, y, lse, dloss, dh, dW, workspace)
    T, H = h.shape
    V = W.shape[0]
    dh = torch.empty_like(h) if dh is None else dh
    dW = torch.empty((V, H), dtype=torch.float32, device=h.device) if dW is None else dW
    if dloss.dtype != torch.float32 or dloss.numel() != 1:
        raise ValueError("dloss must be one fp32 value on the device")
    if workspace is None:
        workspace = _ws(int(library().ftk_cce_bwd_workspace_bytes(T, H, V)), h)
    _call("ftk_cce_bwd", _ptr(h), _rows(h, "h"), _ptr(W), _rows(W, "W"), _ptr(y), _ptr(lse),
          _ptr(dloss), T, H, V, _ptr(dh), _rows(dh, "dh"), _ptr(dW), _rows(dW, "dW"),
          _ptr(workspace), workspace.numel() * workspace.element_size(), _code(h), _stream(h))
    return dh, dW


# ---------------------------------------------------------------- packing

def bfd_pack(lengths, capacity: int):
    """Best-Fit-Decreasing packing (host).  Returns (bin_of, order, bin_start):
    numpy arrays; bin b holds sequences order[bin_start[b]:bin_start[b+1]]."""
    import numpy as np
    raw = np.asarray(lengths)
    if raw.size and not np.issubdtype(raw.dtype, np.integer):
        raise ValueError("lengths must be integers")
    if not 1 <= int(capacity) < 2**31:
        raise ValueError("capacity must lie in [1, 2^31)")
    if raw.size and (int(raw.min()) < 0 or int(raw.max()) > int(capacity)):
        # checked before the int32 cast, so a wide length cannot wrap into range
        raise ValueError("every length must lie in [0, capacity]")
    lens = np.ascontiguousarray(raw.astype(np.int32))
    n = lens.size
    bin_of = np.empty(n, dtype=np.int32)
    order = np.empty(n, dtype=np.int64)
    bin_start = np.empty(n + 1, dtype=np.int64)
    nb = ctypes.c_int64(0)
    _call("ftk_bfd_pack", lens.ctypes.data, n, int(capacity), bin_of.ctypes.data,
          order.ctypes.data, bin_start.ctypes.data, ctypes.byref(nb))
    return bin_of, order, bin_start[: nb.value + 1].copy()


def packed_cu_seqlens(lengths, order, bin_start, b: int):
    """int32 cu_seqlens of packed bin b (its sequences in placement order)."""
    import numpy as np
    members = np.asarray(order)[bin_start[b]:bin_start[b + 1]]
    cu = np.zeros(members.size + 1, dtype=np.int64)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64)[members])
    return cu.astype(np.int32)


WAIT_TIMEOUT = 1  # FTK_DEVSTAT_WAIT_TIMEOUT


def device_status(clear: bool = True) -> int:
    """Status word of the current device (bit WAIT_TIMEOUT: a kernel's
    bounded pipeline wait ran out, so some launch's results are invalid)."""
    v = ctypes.c_uint32(0)
    _call("ftk_device_status", ctypes.byref(v), 1 if clear else 0)
    return int(v.value)


def selftest_wait_timeout(limit_cycles: int = 1_000_000) -> None:
    """Run the bounded-wait timeout path on purpose (one CTA waits on a
    barrier nothing completes); afterwards device_status() has WAIT_TIMEOUT."""
    _call("ftk_selftest_wait_timeout", int(limit_cycles),
          torch.cuda.current_stream().cuda_stream)


def version() -> str:
    return library().ftk_version().decode()
