"""The library's Best-Fit-Decreasing packing (host C++) against the oracle:
the same bins, members and order, exactly (integer work is bit-exact)."""
import numpy as np
import pytest

from oracle.packing import bfd_pack as oracle_bfd, cu_seqlens_of_bin
from fine_tuning_gb300 import build, workloads as W


@pytest.fixture(scope="module")
def ftk():
    build.build()
    from fine_tuning_gb300 import ftk
    ftk.library()
    return ftk


def check(ftk, lens, cap):
    bin_of, order, bin_start = ftk.bfd_pack(lens, cap)
    ob, obins = oracle_bfd(list(lens), cap)
    assert bin_of.tolist() == ob
    assert len(bin_start) - 1 == len(obins)
    for b, members in enumerate(obins):
        assert order[bin_start[b]:bin_start[b + 1]].tolist() == members
        assert ftk.packed_cu_seqlens(lens, order, bin_start, b).tolist() == \
            cu_seqlens_of_bin(lens, members)


@pytest.mark.parametrize("seed", range(20))
def test_random_small(ftk, seed):
    rng = np.random.default_rng(seed)
    cap = int(rng.integers(1, 200))
    lens = rng.integers(0, cap + 1, size=int(rng.integers(0, 300))).tolist()
    check(ftk, lens, cap)


@pytest.mark.parametrize("name", ["qwen2.5-0.5b", "llama-3.2-1b", "qwen3-8b"])
def test_workload_length_mixes(ftk, name):
    # a corpus of sequences with the workload's length mix, packed into bins
    # of the workload's token budget
    wl = W.WORKLOADS[name]
    lens = np.concatenate([W.draw_lengths(wl)] * 3)[:400]
    check(ftk, lens.tolist(), wl.T)


@pytest.mark.parametrize("n,cap", [(300, 2223), (300, 2224), (300, 2225), (300, 50_000_000),
                                   (5000, 20_000), (0, 1 << 30)])
def test_capacities_around_the_counting_sort_limit(ftk, n, cap):
    # capacities up to 4 n + 1024 take the counting sort, larger ones a
    # stable sort: the same packing either way
    rng = np.random.default_rng(cap % 1000)
    lens = rng.integers(0, cap + 1, size=n)
    if n:
        lens[::7] = lens[3]  # ties in length, ordered by index
        lens[::11] = cap     # full bins
        lens[::13] = 0
    check(ftk, lens.tolist(), cap)


def test_wide_lengths_are_rejected_not_wrapped(ftk):
    # 2^32 + 3 would wrap to 3 in an int32 cast: the binding refuses it
    with pytest.raises(ValueError):
        ftk.bfd_pack(np.array([5, (1 << 32) + 3], dtype=np.int64), 10)
    with pytest.raises(ValueError):
        ftk.bfd_pack(np.array([-1], dtype=np.int64), 10)
    with pytest.raises(ValueError):
        ftk.bfd_pack([1, 2], 1 << 31)


def test_edges(ftk):
    check(ftk, [], 5)
    check(ftk, [5], 5)
    check(ftk, [0, 0, 0], 1)
    check(ftk, [3] * 50, 6)
    check(ftk, [1] * 100 + [99] * 10, 100)
    lib = ftk.library()
    import ctypes
    a = (ctypes.c_int32 * 1)(6)
    out32 = (ctypes.c_int32 * 1)()
    out64 = (ctypes.c_int64 * 2)()
    nb = ctypes.c_int64()
    assert lib.ftk_bfd_pack(a, 1, 5, out32, out64, out64, ctypes.byref(nb)) == 2  # too long
    assert lib.ftk_bfd_pack(a, 1, 0, out32, out64, out64, ctypes.byref(nb)) == 2  # no capacity
