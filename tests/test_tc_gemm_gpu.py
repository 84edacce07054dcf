"""The tensor-core GEMM (tcgen05) against a double-precision matmul.

C = A B^T with bf16 A, B and fp32 accumulation: every product of two bf16
values is exact in fp32, so the only error is the fp32 summation, at most
K * 2^-24 * sum_k |a_k b_k| whatever the order (the recursive-summation
bound).  Shapes cover one tile, ragged M / N / K, every tile width the
launcher picks (256, 224, 192), strided rows, and enough tiles to wrap the
persistent grid.
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
