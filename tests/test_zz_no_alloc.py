"""ftk_rmsnorm_bwd_noalloc: the RMSNorm backward for callers that cannot
allocate device memory (code inside a fixed memory pool, a runtime that
forbids cudaMalloc after start-up, a plugin given only input and output
pointers).  It uses a scratch array built into the library instead of a
caller workspace.

Each GPU case makes two calls in a row through the C ABI (the second one
finds the first one's leftovers in the shared scratch) and compares both
against ftk_rmsnorm_bwd with a workspace and against the double-precision
oracle, within the parity tolerance of the other tests.  This file is named to be collected last, so a run that
stops at its first failure has already run every other test; it also
passes on its own in a fresh process.
"""
import ctypes

import pytest
import torch

import oracle
from oracle.tolerance import assert_close
from fine_tuning_gb300 import build, ftk

OK, WORKSPACE = 0, 5
CODES = {torch.float32: 0, torch.bfloat16: 1}


@pytest.fixture(scope="module")
def lib():
    build.build()
    lib = ftk.library()
    fn = lib.ftk_rmsnorm_bwd_noalloc
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    fn.restype = ctypes.c_int
    fn.argtypes = [vp, i64, vp, i64, vp, vp, vp, i64, vp, i64, i64, ctypes.c_float,
                   ctypes.c_int, vp]
    return lib


def test_rejects_rows_too_long_for_the_scratch(lib):
    # checked on the host before any CUDA call; the pointers are never used
    a, H = 1 << 20, (1 << 20) + 1
    assert lib.ftk_rmsnorm_bwd_noalloc(a, H, a, H, a, None, a, H, a, 4, H, 1e-6, 1,
                                       None) == WORKSPACE


def noalloc(lib, dy, x, w, rstd, eps):
    T, H = x.shape
    dx = torch.empty_like(x)
    dw = torch.empty(H, dtype=torch.float32, device=x.device)
    st = lib.ftk_rmsnorm_bwd_noalloc(
        dy.data_ptr(), dy.stride(0), x.data_ptr(), x.stride(0), w.data_ptr(),
        None if rstd is None else rstd.data_ptr(), dx.data_ptr(), dx.stride(0), dw.data_ptr(),
        T, H, eps, CODES[x.dtype], torch.cuda.current_stream().cuda_stream)
    assert st == OK, st
    return dx, dw


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,T,H,with_rstd", [
    (torch.bfloat16, 16384, 896, True),   # Qwen2.5-0.5B rows
    (torch.bfloat16, 3000, 5120, False),  # rstd recomputed, multi-warp rows
    (torch.float32, 64, 64, True),
    (torch.bfloat16, 7, 20000, True),     # rows too long for registers
])
def test_matches_workspace_version_two_calls_in_a_row(lib, dtype, T, H, with_rstd):
    code = "f32" if dtype == torch.float32 else "bf16"
    eps = 1e-6
    for call in range(2):
        g = torch.Generator(device="cuda")
        g.manual_seed(100 * call + H)
        x = torch.randn((T, H), generator=g, device="cuda").to(dtype)
        dy = torch.randn((T, H), generator=g, device="cuda").to(dtype)
        w = (1 + 0.1 * torch.randn(H, generator=g, device="cuda")).to(dtype)
        _, rstd = ftk.rmsnorm_fwd(x, w, eps)
        r = rstd if with_rstd else None
        dx_new, dw_new = noalloc(lib, dy, x, w, r, eps)
        dx_ref, dw_ref = ftk.rmsnorm_bwd(dy, x, w, r, eps)
        torch.cuda.synchronize()
        dxo, dwo, dxs, dws = oracle.rmsnorm_bwd(dy.cpu(), x.cpu(), w.cpu(), eps, scales=True)
        # against the entry point that takes a workspace ...
        assert_close(f"dx call {call}", dx_new, dx_ref.double().cpu().numpy(), dxs, dtype=code)
        assert_close(f"dw call {call}", dw_new, dw_ref.double().cpu().numpy(), dws, dtype=code,
                     kind="dw")
        # ... and against the double-precision oracle's own values
        assert_close(f"dx call {call} vs oracle", dx_new, dxo, dxs, dtype=code)
        assert_close(f"dw call {call} vs oracle", dw_new, dwo, dws, dtype=code, kind="dw")
