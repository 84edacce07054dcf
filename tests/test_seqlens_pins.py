"""Pins of the boundary-validity oracle: hand cases whose answer follows from
the definition of packed metadata (start at 0, never decrease, end at T),
and the boundaries the workloads draw, which are valid by construction."""
import pytest

from oracle.seqlens import BAD_END, BAD_START, DECREASING, check_seqlens
from fine_tuning_gb300 import workloads as W


@pytest.mark.parametrize("cu,T,bits", [
    ([0, 5, 22, 54, 64], 64, 0),             # the tiny workload's four sequences
    ([0, 0, 0, 7], 7, 0),                    # empty sequences are legal
    ([0], 0, 0),                             # no sequence, no token
    ([0], 3, BAD_END),                       # no sequence but three tokens
    ([1, 5, 9], 9, BAD_START),
    ([0, 5, 4, 9], 9, DECREASING),
    ([0, 5, 9], 10, BAD_END),                # one token left over
    ([0, 5, 11], 10, BAD_END),               # runs past the batch
    ([-2, 5, 3, 4], 9, BAD_START | DECREASING | BAD_END),
])
def test_hand_cases(cu, T, bits):
    assert check_seqlens(cu, T) == bits


@pytest.mark.parametrize("name", W.WORKLOAD_ORDER)
def test_workload_boundaries_are_valid(name):
    wl = W.WORKLOADS[name]
    assert check_seqlens(W.cu_seqlens_from_lengths(W.draw_lengths(wl)), wl.T) == 0


def test_each_violation_is_seen_alone():
    good = [0, 3, 3, 8, 20]
    assert check_seqlens(good, 20) == 0
    for i in range(len(good) - 1):  # lowering one inner boundary below its left neighbour
        bad = list(good)
        bad[i + 1] = bad[i] - 1
        want = DECREASING | (BAD_END if i + 1 == len(good) - 1 else 0)
        assert check_seqlens(bad, 20) == want
