"""Host-side checks of the C ABI, no GPU needed.

The library must build, load and export every function include/ftk.h
declares; argument errors must come back as the documented status before
any CUDA call is made (the pointers below are never dereferenced).
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ftk.h")

OK, NULL, SHAPE, ALIGN, DTYPE, WORKSPACE, CUDA, ALIAS = range(8)
F32, BF16 = 0, 1


@pytest.fixture(scope="module")
def lib():
    from fine_tuning_gb300 import build
    build.build()
    from fine_tuning_gb300 import ftk
    return ftk.library()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"FTK_API\s+[\w\s\*]+?\b(ftk_\w+)\s*\(", text)))


def test_header_declares_the_hot_path():
    names = declared_functions()
    for n in ("ftk_rmsnorm_fwd", "ftk_rmsnorm_bwd", "ftk_rmsnorm_bwd_workspace_bytes",
              "ftk_swiglu_fwd", "ftk_swiglu_bwd", "ftk_qk_rope_fwd", "ftk_qk_rope_bwd"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_exports_nothing_undeclared(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True,
                         text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l and "ftk_" in l}
    assert exported == set(declared_functions())


def test_status_strings(lib):
    for s in range(8):
        assert lib.ftk_status_str(s)
    assert lib.ftk_version().decode().count(".") == 2


A = 1 << 20  # a 1 MiB-aligned fake device address, never dereferenced


def test_rmsnorm_fwd_argument_errors(lib):
    f = lib.ftk_rmsnorm_fwd
    assert f(A, 64, A + 4096, A + 8192, 64, None, 0, 64, 1e-6, BF16, None) == OK  # T = 0
    assert f(A, 64, A + 4096, A + 8192, 64, None, 4, 64, 1e-6, 7, None) == DTYPE
    assert f(A, 64, A + 4096, A + 8192, 64, None, -1, 64, 1e-6, BF16, None) == SHAPE
    assert f(A, 63, A + 4096, A + 8192, 64, None, 4, 64, 1e-6, BF16, None) == SHAPE  # ld < H
    assert f(A, 64, A + 4096, A + 8192, 64, None, 4, 0, 1e-6, BF16, None) == SHAPE
    assert f(None, 64, A + 4096, A + 8192, 64, None, 4, 64, 1e-6, BF16, None) == NULL
    assert f(A + 1, 64, A + 4096, A + 8192, 64, None, 4, 64, 1e-6, BF16, None) == ALIGN
    assert f(A, 64, A + 4096, A + 8192, 64, A + 2, 4, 64, 1e-6, F32, None) == ALIGN
    # y overlapping x without being x
    assert f(A, 64, A + 4096, A + 2, 64, None, 4, 64, 1e-6, BF16, None) == ALIAS
    # rstd inside y
    assert f(A, 64, A + 4096, A + 8192, 64, A + 8192 + 16, 4, 64, 1e-6, BF16, None) == ALIAS


def test_rmsnorm_bwd_argument_errors(lib):
    f = lib.ftk_rmsnorm_bwd
    dy, x, w, dx, dw, ws = A, A + 65536, A + 2 * 65536, A + 3 * 65536, A + 4 * 65536, A + 5 * 65536
    args = lambda **k: [k.get("dy", dy), 64, k.get("x", x), 64, w, None, k.get("dx", dx), 64,
                        k.get("dw", dw), k.get("ws", ws), k.get("wsb", 1 << 16),
                        k.get("T", 4), 64, 1e-6, k.get("dt", BF16), None]
    assert f(*args(T=0)) == OK
    assert f(*args(dt=3)) == DTYPE
    assert f(*args(ws=None)) == WORKSPACE
    assert f(*args(wsb=64)) == WORKSPACE  # less than one row of partials
    assert f(*args(dw=None)) == NULL
    assert f(*args(ws=A + 5 * 65536 + 8)) == ALIGN
    assert f(*args(dw=x + 16)) == ALIAS       # dw inside x
    assert f(*args(ws=dx + 64)) == ALIAS      # workspace overlapping dx
    assert f(*args(dx=dy + 2)) == ALIAS       # dx partially over dy


def test_rmsnorm_add_fwd_argument_errors(lib):
    f = lib.ftk_rmsnorm_add_fwd
    x, res, w, h, y, r = (A + i * 65536 for i in range(6))
    names = ["x", "ldx", "res", "ldr", "w", "h", "ldh", "y", "ldy", "rstd", "T", "H", "eps",
             "dt", "s"]
    ok = [x, 64, res, 64, w, h, 64, y, 64, r, 4, 64, 1e-6, BF16, None]

    def call(**kw):
        a = list(ok)
        for n, v in kw.items():
            a[names.index(n)] = v
        return f(*a)

    assert call(T=0) == OK
    assert call(res=None, T=0) == OK
    assert call(dt=4) == DTYPE
    assert call(ldr=63) == SHAPE
    assert call(ldh=32) == SHAPE
    assert call(res=None) == NULL
    assert call(h=None) == NULL
    assert call(res=res + 1) == ALIGN
    assert call(h=h + 2, dt=F32) == ALIGN
    assert call(h=x + 2) == ALIAS               # h partly over x
    assert call(h=res + 64) == ALIAS            # h partly over res
    assert call(y=x) == ALIAS                   # y over an input
    assert call(y=h) == ALIAS                   # y over h
    assert call(rstd=h + 16) == ALIAS           # rstd inside h
    assert call(rstd=res + 16) == ALIAS         # rstd inside res
    assert call(h=x, T=0) == OK and call(h=res, T=0) == OK


def test_rmsnorm_add_bwd_argument_errors(lib):
    f = lib.ftk_rmsnorm_add_bwd
    dy, dh, h, w, dx, dw, ws = (A + i * 65536 for i in range(7))
    names = ["dy", "lddy", "dh", "lddh", "h", "ldh", "w", "rstd", "dx", "lddx", "dw", "ws",
             "wsb", "T", "H", "eps", "dt", "s"]
    ok = [dy, 64, dh, 64, h, 64, w, None, dx, 64, dw, ws, 1 << 16, 4, 64, 1e-6, BF16, None]

    def call(**kw):
        a = list(ok)
        for n, v in kw.items():
            a[names.index(n)] = v
        return f(*a)

    assert call(T=0) == OK
    assert call(dt=2) == DTYPE
    assert call(lddh=60) == SHAPE
    assert call(dh=None) == NULL
    assert call(h=None) == NULL
    assert call(ws=None) == WORKSPACE
    assert call(dh=dh + 1) == ALIGN
    assert call(dx=dh + 2) == ALIAS             # dx partly over dh
    assert call(dx=h) == ALIAS                  # dx over h
    assert call(dw=dh + 16) == ALIAS            # dw inside dh
    assert call(ws=dh) == ALIAS                 # workspace over dh


def test_swiglu_argument_errors(lib):
    f, b = lib.ftk_swiglu_fwd, lib.ftk_swiglu_bwd
    g, u, h = A, A + 65536, A + 2 * 65536
    assert f(g, u, 64, h, 64, 0, 64, BF16, None) == OK
    assert f(g, u, 64, h, 64, 4, 0, BF16, None) == OK
    assert f(g, u, 32, h, 64, 4, 64, BF16, None) == SHAPE
    assert f(g, None, 64, h, 64, 4, 64, BF16, None) == NULL
    assert f(g, u, 64, g + 2, 64, 4, 64, BF16, None) == ALIAS
    # fused gate_up view: g and u interleave in one [T, 2I] buffer, h separate
    assert f(g, g + 128, 128, h, 64, 0, 64, BF16, None) == OK
    dh, dg, du = A + 3 * 65536, A + 4 * 65536, A + 5 * 65536
    assert b(dh, 64, g, u, 64, dg, dg + 16, 64, 4, 64, BF16, None) == ALIAS  # dg/du overlap
    assert b(dh, 64, g, u, 64, dg, du, 64, 4, 64, 9, None) == DTYPE
    bh, h2 = lib.ftk_swiglu_bwd_h, A + 6 * 65536
    assert bh(dh, 64, g, u, 64, dg, du, 64, h2, 64, 0, 64, BF16, None) == OK
    assert bh(dh, 64, g, u, 64, dg, du, 64, None, 64, 4, 64, BF16, None) == NULL
    assert bh(dh, 64, g, u, 64, dg, du, 64, h2, 32, 4, 64, BF16, None) == SHAPE
    assert bh(dh, 64, g, u, 64, dg, du, 64, h2 + 1, 64, 4, 64, BF16, None) == ALIGN
    assert bh(dh, 64, g, u, 64, dg, du, 64, dg, 64, 4, 64, BF16, None) == ALIAS   # h over dg
    assert bh(dh, 64, g, u, 64, dg, du, 64, du + 8, 64, 4, 64, BF16, None) == ALIAS
    assert bh(dh, 64, g, u, 64, dg, du, 64, g + 2, 64, 4, 64, BF16, None) == ALIAS  # partly over g


def test_qk_rope_argument_errors(lib):
    f = lib.ftk_qk_rope_fwd
    q, k, cu = A, A + (1 << 22), A + (1 << 23)
    ok = [q, 4 * 16, k, 2 * 16, cu, 4, 64, 4, 2, 16, 1e4, F32, None]

    def call(**kw):
        a = list(ok)
        names = ["q", "ldq", "k", "ldk", "cu", "B", "T", "Hq", "Hkv", "D", "theta", "dt", "s"]
        for n, v in kw.items():
            a[names.index(n)] = v
        return f(*a)

    assert call(T=0) == OK
    assert call(D=15) == SHAPE
    assert call(D=0) == SHAPE
    assert call(D=1026) == SHAPE
    assert call(Hq=0, Hkv=0) == SHAPE
    assert call(ldq=60) == SHAPE
    assert call(theta=0.0) == SHAPE
    assert call(B=0) == SHAPE
    assert call(cu=None) == NULL
    assert call(k=None) == NULL
    assert call(q=q + 2) == ALIGN
    assert call(k=q + 64) == ALIAS            # k inside q
    # fused QKV layout: q and k interleaved with the same row stride
    assert call(ldq=8 * 16, k=q + 4 * 16 * 4, ldk=8 * 16, T=0) == OK
    assert call(dt=5) == DTYPE


def test_qk_rope_freq_argument_errors(lib):
    import numpy as np
    f = lib.ftk_qk_rope_freq_fwd
    q, k, cu = A, A + (1 << 22), A + (1 << 23)
    good = np.full(8, 0.5)
    bad_hi, bad_nan = np.full(8, 0.5), np.full(8, 0.5)
    bad_hi[3], bad_nan[5] = 1.5, np.nan
    ptr = lambda a: a.ctypes.data
    base = [q, 4 * 16, k, 2 * 16, cu, 4, 64, 4, 2, 16]
    assert f(*(base[:6] + [0] + base[7:]), ptr(good), F32, None) == OK       # T = 0
    assert f(*base, None, F32, None) == NULL
    assert f(*base, ptr(bad_hi), F32, None) == SHAPE
    assert f(*base, ptr(bad_nan), F32, None) == SHAPE
    assert lib.ftk_qk_rope_freq_bwd(*base, ptr(good), 7, None) == DTYPE


def test_llama3_table_host(lib):
    # host code: runs here, against the oracle's table
    import numpy as np
    import oracle
    from fine_tuning_gb300 import ftk
    for D, theta, fac, lo, hi, L in ((64, 5e5, 32.0, 1.0, 4.0, 8192.0),
                                     (128, 5e5, 8.0, 1.0, 4.0, 8192.0),
                                     (128, 1e6, 16.0, 2.0, 5.0, 4096.0),
                                     (32, 1e4, 1.0, 1.0, 4.0, 2048.0)):
        got = ftk.rope_llama3_inv_freq(D, theta, fac, lo, hi, L)
        ref = oracle.rope_llama3_inv_freq(D, theta, fac, lo, hi, L)
        np.testing.assert_allclose(got, ref, rtol=1e-14, atol=0)
    out = np.empty(32)
    p = out.ctypes.data
    assert lib.ftk_rope_llama3_inv_freq(63, 5e5, 32.0, 1.0, 4.0, 8192.0, p) == SHAPE
    assert lib.ftk_rope_llama3_inv_freq(64, 5e5, 32.0, 4.0, 4.0, 8192.0, p) == SHAPE
    assert lib.ftk_rope_llama3_inv_freq(64, 5e5, 0.5, 1.0, 4.0, 8192.0, p) == SHAPE
    assert lib.ftk_rope_llama3_inv_freq(64, 5e5, 32.0, 1.0, 4.0, 8192.0, None) == NULL


def test_workspace_query_rejects_bad_arguments(lib):
    assert lib.ftk_rmsnorm_bwd_workspace_bytes(0, 64, BF16) == 0
    assert lib.ftk_rmsnorm_bwd_workspace_bytes(16, 0, BF16) == 0
    assert lib.ftk_rmsnorm_bwd_workspace_bytes(16, 64, 9) == 0


def test_cce_backward_chunk_choice(lib):
    """The backward's vocabulary chunk: all of V (rounded up to 64) when V
    fits one chunk, else a multiple of 256 in [4096, 16384] whose workspace
    the query covers; pure host logic, the same answer every time."""
    lib.ftk_cce_bwd_chunk.restype = ctypes.c_int64
    lib.ftk_cce_bwd_chunk.argtypes = [ctypes.c_int64] * 3 + [ctypes.c_int32]
    lib.ftk_cce_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.ftk_cce_bwd_workspace_bytes.argtypes = [ctypes.c_int64] * 3
    assert lib.ftk_cce_bwd_chunk(300, 64, 1000, 152) == 1024
    assert lib.ftk_cce_bwd_chunk(8192, 896, 16384, 152) == 16384
    for T, H, V, sms in [(8192, 896, 151936, 152), (8192, 2048, 128256, 152),
                         (4096, 4096, 151936, 148), (1, 64, 100000, 2)]:
        C = lib.ftk_cce_bwd_chunk(T, H, V, sms)
        assert C % 256 == 0 and 4096 <= C <= 16384, (T, H, V, C)
        assert C == lib.ftk_cce_bwd_chunk(T, H, V, sms)
        assert lib.ftk_cce_bwd_workspace_bytes(T, H, V) >= T * C * 2 + T * H * 4
    for bad in [(0, 896, 151936, 152), (8192, 0, 151936, 152), (8192, 896, 0, 152),
                (8192, 896, 151936, 0)]:
        assert lib.ftk_cce_bwd_chunk(*bad) == 0


def test_check_seqlens_argument_errors(lib):
    f = lib.ftk_check_seqlens
    cu, st = A, A + (1 << 20)
    assert f(cu, -1, 10, st, None) == SHAPE
    assert f(cu, 2, -1, st, None) == SHAPE
    assert f(None, 2, 10, st, None) == NULL
    assert f(cu, 2, 10, None, None) == NULL
    assert f(cu + 2, 2, 10, st, None) == ALIGN
    assert f(cu, 2, 10, st + 2, None) == ALIGN
    assert f(cu, 2, 10, cu + 8, None) == ALIAS  # the word inside cu[0..2]


def test_checked_rope_argument_errors(lib):
    for f in (lib.ftk_qk_rope_fwd_checked, lib.ftk_qk_rope_bwd_checked):
        q, k, cu, st = A, A + (1 << 22), A + (1 << 23), A + (1 << 24)
        ok = [q, 4 * 16, k, 2 * 16, cu, 4, 64, 4, 2, 16, 1e4, None, st, F32, None]
        names = ["q", "ldq", "k", "ldk", "cu", "B", "T", "Hq", "Hkv", "D", "theta", "inv", "st",
                 "dt", "s"]

        def call(**kw):
            a = list(ok)
            for n, v in kw.items():
                a[names.index(n)] = v
            return f(*a)

        assert call(T=0) == OK
        assert call(T=0, st=None) == OK
        assert call(st=None) == NULL
        assert call(st=st + 2) == ALIGN
        assert call(st=q + 64) == ALIAS   # the word inside q
        assert call(D=15) == SHAPE
        assert call(theta=0.0) == SHAPE   # no table and no theta
        bad = (ctypes.c_double * 8)(*([0.5] * 7 + [1.5]))
        assert call(inv=ctypes.cast(bad, ctypes.c_void_p)) == SHAPE
        assert call(cu=None) == NULL


def test_checked_qk_norm_rope_argument_errors(lib):
    M = 1 << 22
    q, k, wq, wk, qo, ko, rq, rk, cu, st = (A + i * M for i in range(10))
    ok = [q, 4 * 16, k, 2 * 16, wq, wk, qo, 4 * 16, ko, 2 * 16, rq, rk, cu, 4, 64, 4, 2, 16,
          1e4, None, 1e-6, st, F32, None]
    names = ["q", "ldq", "k", "ldk", "wq", "wk", "qo", "ldqo", "ko", "ldko", "rq", "rk", "cu",
             "B", "T", "Hq", "Hkv", "D", "theta", "inv", "eps", "st", "dt", "s"]
    f = lib.ftk_qk_norm_rope_fwd_checked

    def call(**kw):
        a = list(ok)
        for n, v in kw.items():
            a[names.index(n)] = v
        return f(*a)

    assert call(T=0) == OK
    assert call(T=0, st=None) == OK
    assert call(st=None) == NULL
    assert call(st=st + 2) == ALIGN
    assert call(st=qo + 64) == ALIAS   # the word inside an output
    assert call(st=rk + 4) == ALIAS
    assert call(D=15) == SHAPE
    assert call(cu=None) == NULL

    # the backward: the word must not overlap dq, dk, dwq, dwk or the workspace
    gq, gk, dq, dk, dwq, dwk, ws = (A + (10 + i) * M for i in range(7))
    okb = [gq, 4 * 16, gk, 2 * 16, q, 4 * 16, k, 2 * 16, wq, wk, None, None, dq, 4 * 16, dk,
           2 * 16, dwq, dwk, ws, 1 << 20, cu, 4, 64, 4, 2, 16, 1e4, None, 1e-6, st, F32, None]
    nb = ["gq", "ldgq", "gk", "ldgk", "q", "ldq", "k", "ldk", "wq", "wk", "rq", "rk", "dq", "lddq",
          "dk", "lddk", "dwq", "dwk", "ws", "wsb", "cu", "B", "T", "Hq", "Hkv", "D", "theta", "inv",
          "eps", "st", "dt", "s"]
    g = lib.ftk_qk_norm_rope_bwd_checked

    def callb(**kw):
        a = list(okb)
        for n, v in kw.items():
            a[nb.index(n)] = v
        return g(*a)

    assert callb(T=0) == OK
    assert callb(st=None) == NULL
    assert callb(st=st + 2) == ALIGN
    assert callb(st=dwq + 8) == ALIAS
    assert callb(st=ws + 256) == ALIAS
    assert callb(st=dq + 64) == ALIAS
