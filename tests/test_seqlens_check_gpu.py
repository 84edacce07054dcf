"""Device-side validation of a packed batch's boundaries (the checked-seqlens
mode) and the RoPE calls it guards.

Bad metadata is made on the host and copied in: nothing faults, traps or
hangs.  The check kernel's word must equal the oracle's bits for every case
(integer work: exact), a guarded rotation must leave q and k bit for bit as
they were whenever the word is non-zero, and equal the unguarded rotation
when it is zero.
"""
import numpy as np
import pytest
import torch

from oracle.seqlens import check_seqlens as oracle_check
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
    assert ftk.device_status(clear=True) == 0


def word(cu, T, garbage=0x5A5A5A5A):
    cu_d = torch.as_tensor(np.asarray(cu, dtype=np.int32), device=DEV)
    status = torch.full((1,), garbage, dtype=torch.int32, device=DEV)
    ftk.check_seqlens(cu_d, T, status)
    return int(status.item()) & 0xFFFFFFFF


CASES = [
    ([0, 5, 22, 54, 64], 64), ([0, 0, 0, 7], 7), ([0], 0), ([0], 3), ([1, 5, 9], 9),
    ([0, 5, 4, 9], 9), ([0, 5, 9], 10), ([0, 5, 11], 10), ([-2, 5, 3, 4], 9),
    ([0, 2**31 - 1], 2**31 - 1), ([0, 7], 2**31 + 7),
]


@pytest.mark.parametrize("cu,T", CASES)
def test_word_equals_the_oracle(cu, T):
    assert word(cu, T) == oracle_check(cu, T)


@pytest.mark.parametrize("seed", range(6))
def test_many_sequences_one_decrease_anywhere(seed):
    # more boundaries than the check's 1024 threads, one decrease at a random place
    rng = np.random.default_rng(seed)
    lens = rng.integers(0, 40, size=int(rng.integers(1025, 5000)))
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T = int(cu[-1])
    assert word(cu, T) == 0
    i = int(rng.integers(1, cu.size - 1))
    bad = cu.copy()
    bad[i] = bad[i - 1] - 1
    assert word(bad, T) == oracle_check(bad.tolist(), T) != 0


@pytest.mark.parametrize("name", W.WORKLOAD_ORDER)
def test_workload_boundaries_pass(name):
    wl = W.WORKLOADS[name]
    assert word(W.cu_seqlens_from_lengths(W.draw_lengths(wl)), wl.T) == 0


def rope_case(T=300, Hq=4, Hkv=2, D=64, dtype=torch.bfloat16, seed=3):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    q = torch.randn((T, Hq, D), generator=g, device=DEV).to(dtype)
    k = torch.randn((T, Hkv, D), generator=g, device=DEV).to(dtype)
    return q, k


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("backward", [False, True])
def test_guarded_rope_equals_the_plain_one_on_valid_metadata(dtype, backward):
    T, theta = 300, 1e4
    cu = torch.tensor([0, 17, 17, 160, 300], dtype=torch.int32, device=DEV)
    status = ftk.check_seqlens(cu, T)
    q, k = rope_case(T, dtype=dtype)
    q2, k2 = q.clone(), k.clone()
    if backward:
        ftk.qk_rope_bwd(q, k, cu, theta)
        ftk.qk_rope_bwd_checked(q2, k2, cu, status, theta=theta)
    else:
        ftk.qk_rope_fwd(q, k, cu, theta)
        ftk.qk_rope_fwd_checked(q2, k2, cu, status, theta=theta)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(q, q2) and torch.equal(k, k2)


def test_guarded_rope_with_a_frequency_table():
    T = 300
    cu = torch.tensor([0, 100, 300], dtype=torch.int32, device=DEV)
    status = ftk.check_seqlens(cu, T)
    table = ftk.rope_llama3_inv_freq(64, 5e5, 32.0, 1.0, 4.0, 8192.0)
    q, k = rope_case(T)
    q2, k2 = q.clone(), k.clone()
    ftk.qk_rope_freq_fwd(q, k, cu, table)
    ftk.qk_rope_fwd_checked(q2, k2, cu, status, inv_freq=table)
    torch.cuda.synchronize()
    assert torch.equal(q, q2) and torch.equal(k, k2)


# shapes that reach each RoPE kernel form: the per-warp pipeline (D 64, 128),
# one warp per token (D/2 not a power-of-two multiple of the packet), the
# element-wise forms (D 6; D 130, whose half exceeds a warp) and a TMA-staged
# batch (many tokens of a non-power-of-two head)
SHAPES = [
    dict(T=300, Hq=4, Hkv=2, D=64, dtype=torch.bfloat16),
    dict(T=5000, Hq=8, Hkv=8, D=128, dtype=torch.bfloat16),
    dict(T=300, Hq=3, Hkv=1, D=96, dtype=torch.float32),
    dict(T=200, Hq=2, Hkv=1, D=6, dtype=torch.float32),
    dict(T=100, Hq=2, Hkv=1, D=130, dtype=torch.float32),
    dict(T=100000, Hq=6, Hkv=2, D=96, dtype=torch.bfloat16),
]


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"T{s['T']}D{s['D']}")
@pytest.mark.parametrize("bad", ["start", "decrease", "end_short", "end_long"])
def test_bad_metadata_leaves_q_and_k_untouched(shape, bad):
    T = shape["T"]
    good = [0, T // 3, T // 3, (2 * T) // 3, T]
    cu_h = {"start": [1] + good[1:], "decrease": [0, T // 3, T // 4, (2 * T) // 3, T],
            "end_short": good[:-1] + [T - 1], "end_long": good[:-1] + [T + 5]}[bad]
    cu = torch.tensor(cu_h, dtype=torch.int32, device=DEV)
    status = ftk.check_seqlens(cu, T)
    q, k = rope_case(T, shape["Hq"], shape["Hkv"], shape["D"], shape["dtype"])
    q0, k0 = q.clone(), k.clone()
    ftk.qk_rope_fwd_checked(q, k, cu, status, theta=1e4)
    ftk.qk_rope_bwd_checked(q, k, cu, status, theta=1e4)
    torch.cuda.synchronize()
    assert int(status.item()) == oracle_check(cu_h, T) != 0
    assert torch.equal(q, q0) and torch.equal(k, k0)


def test_a_word_set_by_the_caller_also_skips():
    T = 64
    cu = torch.tensor([0, 64], dtype=torch.int32, device=DEV)
    status = torch.tensor([8], dtype=torch.int32, device=DEV)  # not a check bit, still non-zero
    q, k = rope_case(T)
    q0 = q.clone()
    ftk.qk_rope_fwd_checked(q, k, cu, status, theta=1e4)
    torch.cuda.synchronize()
    assert torch.equal(q, q0)


def test_check_then_rope_in_one_graph():
    # the check and the guarded rotation replay together; a later batch's bad
    # metadata, copied into the same cu buffer, stops the rotation
    T = 256
    cu = torch.tensor([0, 100, 256], dtype=torch.int32, device=DEV)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    q, k = rope_case(T)
    ref_q, ref_k = q.clone(), k.clone()
    ftk.qk_rope_fwd(ref_q, ref_k, cu, 1e4)
    q1, k1 = q.clone(), k.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):  # first (non-captured) calls outside the capture
        ftk.check_seqlens(cu, T, status)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        ftk.check_seqlens(cu, T, status)
        ftk.qk_rope_fwd_checked(q1, k1, cu, status, theta=1e4)
    q1.copy_(q)
    k1.copy_(k)
    g.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and torch.equal(q1, ref_q) and torch.equal(k1, ref_k)
    cu.copy_(torch.tensor([0, 300, 256], dtype=torch.int32, device=DEV))
    q1.copy_(q)
    k1.copy_(k)
    g.replay()
    torch.cuda.synchronize()
    assert int(status.item()) == oracle_check([0, 300, 256], T) != 0
    assert torch.equal(q1, q) and torch.equal(k1, k)


# ------------------------------------------------ the fused QK-norm rotation

# shapes that reach each QK-norm RoPE kernel form: the lean bf16 kernels (D 64,
# 128), the fp32 pipelined forward / warp backward, and the element-wise
# forms (D 96 in fp32: half a head is not a power-of-two number of lanes)
NORM_SHAPES = [
    dict(T=300, Hq=4, Hkv=2, D=64, dtype=torch.bfloat16),
    dict(T=5000, Hq=8, Hkv=4, D=128, dtype=torch.bfloat16),
    dict(T=300, Hq=3, Hkv=1, D=64, dtype=torch.float32),
    dict(T=200, Hq=3, Hkv=1, D=96, dtype=torch.float32),
]


def norm_case(shape, seed=7):
    T, D, dt = shape["T"], shape["D"], shape["dtype"]
    q, k = rope_case(T, shape["Hq"], shape["Hkv"], D, dt, seed)
    gq, gk = rope_case(T, shape["Hq"], shape["Hkv"], D, dt, seed + 1)
    g = torch.Generator(device=DEV)
    g.manual_seed(seed + 2)
    wq = (1 + 0.1 * torch.randn(D, generator=g, device=DEV)).to(dt)
    wk = (1 + 0.1 * torch.randn(D, generator=g, device=DEV)).to(dt)
    return q, k, gq, gk, wq, wk


def filled(like, value):
    return torch.full_like(like, value)


@pytest.mark.parametrize("shape", NORM_SHAPES, ids=lambda s: f"T{s['T']}D{s['D']}{s['dtype']}")
@pytest.mark.parametrize("bad", ["start", "decrease", "end_short", "end_long"])
def test_bad_metadata_leaves_every_qk_norm_output_untouched(shape, bad):
    T, Hq, Hkv, D = shape["T"], shape["Hq"], shape["Hkv"], shape["D"]
    good = [0, T // 3, T // 3, (2 * T) // 3, T]
    cu_h = {"start": [1] + good[1:], "decrease": [0, T // 3, T // 4, (2 * T) // 3, T],
            "end_short": good[:-1] + [T - 1], "end_long": good[:-1] + [T + 5]}[bad]
    cu = torch.tensor(cu_h, dtype=torch.int32, device=DEV)
    status = ftk.check_seqlens(cu, T)
    q, k, gq, gk, wq, wk = norm_case(shape)
    q0, k0, gq0, gk0 = q.clone(), k.clone(), gq.clone(), gk.clone()
    qo, ko = filled(q, 3.0), filled(k, -3.0)
    rq = torch.full((T, Hq), 7.0, device=DEV)
    rk = torch.full((T, Hkv), 7.0, device=DEV)
    ftk.qk_norm_rope_fwd(q, k, wq, wk, cu, 1e-6, theta=1e4, q_out=qo, k_out=ko, rstd_q=rq,
                         rstd_k=rk, seqlens_status=status)
    dq, dk = filled(q, 5.0), filled(k, -5.0)
    dwq = torch.full((D,), 9.0, device=DEV)
    dwk = torch.full((D,), 9.0, device=DEV)
    ftk.qk_norm_rope_bwd(gq, gk, q, k, wq, wk, None, None, cu, 1e-6, theta=1e4, dq=dq, dk=dk,
                         dwq=dwq, dwk=dwk, seqlens_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == oracle_check(cu_h, T) != 0
    assert torch.equal(q, q0) and torch.equal(k, k0) and torch.equal(gq, gq0) and \
        torch.equal(gk, gk0)
    assert torch.equal(qo, filled(q, 3.0)) and torch.equal(ko, filled(k, -3.0))
    assert bool((rq == 7.0).all()) and bool((rk == 7.0).all())
    assert torch.equal(dq, filled(q, 5.0)) and torch.equal(dk, filled(k, -5.0))
    assert bool((dwq == 9.0).all()) and bool((dwk == 9.0).all())


@pytest.mark.parametrize("shape", NORM_SHAPES, ids=lambda s: f"T{s['T']}D{s['D']}{s['dtype']}")
def test_guarded_qk_norm_rope_equals_the_plain_one_on_valid_metadata(shape):
    T = shape["T"]
    cu = torch.tensor([0, T // 7, T // 7, T // 2, T], dtype=torch.int32, device=DEV)
    status = ftk.check_seqlens(cu, T)
    q, k, gq, gk, wq, wk = norm_case(shape)
    a = ftk.qk_norm_rope_fwd(q, k, wq, wk, cu, 1e-6, theta=1e4)
    b = ftk.qk_norm_rope_fwd(q, k, wq, wk, cu, 1e-6, theta=1e4, seqlens_status=status)
    ga = ftk.qk_norm_rope_bwd(gq, gk, q, k, wq, wk, a[2], a[3], cu, 1e-6, theta=1e4)
    gb = ftk.qk_norm_rope_bwd(gq, gk, q, k, wq, wk, b[2], b[3], cu, 1e-6, theta=1e4,
                              seqlens_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for x, y in zip(list(a) + list(ga), list(b) + list(gb)):
        assert torch.equal(x, y)
