"""Validity of a packed batch's sequence boundaries, written out plainly.

TEST INFRASTRUCTURE ONLY (like the rest of oracle/).

A packed batch of T tokens holds B sequences back to back; cu_seqlens[b] is
where sequence b starts and cu_seqlens[B] where the last one ends (the
auto-packing paragraph of the Unsloth item on seventnews.com: one 1-D token
tensor plus the sequence-length metadata).  The metadata is well formed when
it starts at 0, never decreases and ends at T.  The result is a bit set:
1 for a bad start, 2 for a decrease anywhere, 4 for a bad end; 0 means valid.
"""
from typing import Sequence

BAD_START, DECREASING, BAD_END = 1, 2, 4


def check_seqlens(cu: Sequence[int], T: int) -> int:
    cu = [int(c) for c in cu]
    if not cu:
        raise ValueError("cu_seqlens holds B + 1 >= 1 entries")
    bits = 0
    if cu[0] != 0:
        bits |= BAD_START
    for b in range(len(cu) - 1):
        if cu[b + 1] < cu[b]:
            bits |= DECREASING
    if cu[-1] != T:
        bits |= BAD_END
    return bits
