"""Pins of the Best-Fit-Decreasing packing oracle (oracle/packing.py).

A hand-worked example, the exhaustive optimum on tiny inputs together with
the known worst-case bound of first/best-fit decreasing (at most
11/9 OPT + 6/9 bins), and invariants every any-fit packing obeys.
"""
import random

import pytest

from oracle.packing import bfd_pack, cu_seqlens_of_bin, optimal_bins


def test_hand_example():
    # capacity 10, lengths 7 5 4 3 1 (indices 0..4):
    # 7 -> new bin 0 (room 3); 5 -> new bin 1 (room 5); 4 -> bin 1 (room 1);
    # 3 -> bin 0 (room 0); 1 -> bin 1 (room 0)
    bin_of, bins = bfd_pack([7, 5, 4, 3, 1], 10)
    assert bins == [[0, 3], [1, 2, 4]]
    assert bin_of == [0, 1, 1, 0, 1]
    assert cu_seqlens_of_bin([7, 5, 4, 3, 1], bins[1]) == [0, 5, 9, 10]


def test_best_fit_not_first_fit():
    # capacity 10, lengths 7 4 4 1: 7 -> bin 0 (room 3); 4 -> bin 1 (room 6);
    # 4 -> bin 1 (room 2; bin 0's 3 is too small); 1 -> rooms are 3 (bin 0)
    # and 2 (bin 1): best fit takes the tighter bin 1 (first fit would take 0)
    _, bins = bfd_pack([7, 4, 4, 1], 10)
    assert bins == [[0], [1, 2, 3]]


def test_ties_take_lower_index():
    bin_of, bins = bfd_pack([3, 3, 3, 3], 6)
    assert bins == [[0, 1], [2, 3]]


def test_edge_cases():
    assert bfd_pack([], 5) == ([], [])
    assert bfd_pack([5], 5) == ([0], [[0]])
    assert bfd_pack([0, 0, 2], 2)[1] == [[2, 0, 1]]
    with pytest.raises(ValueError):
        bfd_pack([6], 5)


@pytest.mark.parametrize("seed", range(40))
def test_invariants_and_bound_vs_exhaustive_optimum(seed):
    rng = random.Random(seed)
    cap = rng.randint(8, 30)
    n = rng.randint(1, 9)
    lens = [rng.randint(1, cap) for _ in range(n)]
    bin_of, bins = bfd_pack(lens, cap)
    # every sequence placed exactly once, no bin over capacity
    assert sorted(i for b in bins for i in b) == list(range(n))
    assert all(sum(lens[i] for i in b) <= cap for b in bins)
    assert all(bin_of[i] == k for k, b in enumerate(bins) for i in b)
    # any-fit: a new bin opens only when nothing fits, so no two bins could
    # have been one
    loads = [sum(lens[i] for i in b) for b in bins]
    assert all(loads[a] + loads[b] > cap for a in range(len(bins)) for b in range(a))
    opt = optimal_bins(lens, cap)
    assert opt <= len(bins) <= (11 * opt + 6) / 9


def test_exhaustive_optimum_itself():
    # 4 items of 5 in bins of 10 -> 2; 3 items of 6 -> 3; 4+6, 3+7, 5+5 -> 3
    assert optimal_bins([5, 5, 5, 5], 10) == 2
    assert optimal_bins([6, 6, 6], 10) == 3
    assert optimal_bins([4, 6, 3, 7, 5, 5], 10) == 3
