"""The tensor-core GEMM (tcgen05) against a double-precision matmul.

C = A B^T with bf16 A, B and fp32 accumulation: every product of two bf16
values is exact in fp32, so the only error is the fp32 summation, at most
K * 2^-24 * sum_k |a_k b_k| whatever the order (the recursive-summation
bound).  Shapes cover one tile, ragged M / N / K, every tile width the
launcher picks (256, 224, 192), strided rows, and enough tiles to wrap the
persistent grid, with each operand read K-major or MN-major.
"""
import numpy as np
import pytest
import torch

from fine_tuning_gb300 import build, ftk

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ftk.library()
    ftk.device_status(clear=True)


def randn(shape, seed, scale=1.0):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    return (scale * torch.randn(shape, generator=g, device=DEV)).to(torch.bfloat16)


def check(c, a, b):
    a64, b64 = a.double().cpu().numpy(), b.double().cpu().numpy()
    ref = a64 @ b64.T
    s = np.abs(a64) @ np.abs(b64).T
    K = a.shape[1]
    got = c.double().cpu().numpy()
    bound = K * 2.0 ** -24 * s + 1e-30
    bad = np.abs(got - ref) > bound
    assert not bad.any(), (int(bad.sum()), np.argwhere(bad)[:3], got[bad][:3], ref[bad][:3])


@pytest.mark.parametrize("M,N,K", [
    (128, 256, 64),      # one tile, one k-step
    (128, 256, 896),
    (300, 500, 200),     # ragged M, N and K
    (257, 896, 72),      # N = 4 x 224
    (64, 576, 64),       # N = 3 x 192
    (1, 1, 8),
    (1000, 1000, 1024),
    (2048, 4096, 256),   # more tiles than SMs: the persistent loop wraps
])
def test_gemm(M, N, K):
    a, b = randn((M, K), M + 1), randn((N, K), N + 2)
    c = ftk.gemm_bf16(a, b)
    torch.cuda.synchronize()
    assert ftk.device_status(clear=True) == 0
    check(c, a, b)


def test_gemm_strided_rows():
    M, N, K = 200, 300, 128
    abuf, bbuf = randn((M, K + 64), 5), randn((N, K + 32), 6)
    a, b = abuf[:, :K], bbuf[:, :K]
    cbuf = torch.full((M, N + 8), 7.0, device=DEV)
    ftk.gemm_bf16(a, b, c=cbuf[:, :N])
    torch.cuda.synchronize()
    assert ftk.device_status(clear=True) == 0
    check(cbuf[:, :N], a, b)
    assert torch.all(cbuf[:, N:] == 7.0)


def test_gemm_rejects_bad_layout():
    a = randn((16, 64), 1)
    with pytest.raises(ftk.FtkError):
        ftk.gemm_bf16(a[:, 1:], randn((16, 63), 2))  # misaligned base


def mn_major(x, pad, seed):
    """x [R, K] stored the other way round: a [K, ld] buffer (ld = R rounded
    up to 8, plus pad) whose first R columns hold x^T; returns the view."""
    R, K = x.shape
    ld = (R + 7) // 8 * 8 + pad
    buf = randn((K, ld), seed)  # the padding columns hold unrelated values
    buf[:, :R] = x.t()
    return buf[:, :R]


@pytest.mark.parametrize("a_mn,b_mn", [(True, False), (False, True), (True, True)])
@pytest.mark.parametrize("M,N,K,pad", [
    (128, 256, 64, 0),     # one tile, one k-step
    (300, 500, 200, 8),    # ragged M, N and K; padded rows
    (257, 896, 72, 0),     # N = 4 x 224: the last 64-column block is half used
    (64, 576, 136, 0),     # N = 3 x 192; M = one 64-column block of A
    (65, 200, 64, 16),     # A's second block holds a single row
    (1, 1, 8, 0),
    (1000, 1000, 1024, 0),
    (2048, 4096, 256, 0),  # more tiles than SMs
])
def test_gemm_mn_major(a_mn, b_mn, M, N, K, pad):
    a, b = randn((M, K), M + 11), randn((N, K), N + 12)
    aa = mn_major(a, pad, 3) if a_mn else a
    bb = mn_major(b, pad, 4) if b_mn else b
    c = ftk.gemm_bf16(aa, bb, a_mn=a_mn, b_mn=b_mn)
    torch.cuda.synchronize()
    assert ftk.device_status(clear=True) == 0
    check(c, a, b)


def test_gemm_mn_major_rejects_bad_layout():
    b = randn((32, 64), 2)
    with pytest.raises(ftk.FtkError):  # MN-major A [K 64, M 12] with a row stride of 12
        ftk.gemm_bf16(randn((64, 12), 1), b, a_mn=True)
    with pytest.raises(ValueError):    # K of a (its rows) differs from b's
        ftk.gemm_bf16(randn((48, 16), 1), b, a_mn=True)
