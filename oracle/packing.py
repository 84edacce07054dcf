"""Best-Fit-Decreasing sequence packing, written out plainly.

TEST INFRASTRUCTURE ONLY (like the rest of oracle/).

Chronicals (arXiv 2601.02609), abstract, optimisation (4): Best-Fit
Decreasing packing of variable-length sequences into fixed-size token
bins, to recover the compute that padding wastes.  The page names the
algorithm; its steps are the textbook ones:

  1. take the sequences longest first (equal lengths: lower index first);
  2. put each into the open bin with the least room left that still holds
     it (equal room: lower bin index);
  3. if no open bin holds it, open a new bin for it.

This is O(n * bins): every bin is scanned for every sequence.
"""
from typing import List, Sequence, Tuple


def bfd_pack(lengths: Sequence[int], capacity: int) -> Tuple[List[int], List[List[int]]]:
    """Returns (bin_of, bins): bin_of[i] = bin of sequence i; bins[b] = the
    sequence indices of bin b in the order they were placed."""
    if capacity < 1:
        raise ValueError("capacity must be positive")
    for n in lengths:
        if n < 0 or n > capacity:
            raise ValueError("every length must lie in [0, capacity]")
    order = sorted(range(len(lengths)), key=lambda i: (-lengths[i], i))
    room: List[int] = []
    bins: List[List[int]] = []
    bin_of = [-1] * len(lengths)
    for i in order:
        best = -1
        for b in range(len(room)):
            if room[b] >= lengths[i] and (best < 0 or room[b] < room[best]):
                best = b
        if best < 0:
            room.append(capacity)
            bins.append([])
            best = len(room) - 1
        room[best] -= lengths[i]
        bins[best].append(i)
        bin_of[i] = best
    return bin_of, bins


def cu_seqlens_of_bin(lengths: Sequence[int], members: Sequence[int]) -> List[int]:
    """Sequence boundaries of one packed bin, members in placement order."""
    cu = [0]
    for i in members:
        cu.append(cu[-1] + lengths[i])
    return cu


def optimal_bins(lengths: Sequence[int], capacity: int) -> int:
    """Fewest bins for a tiny instance, by exhaustive search (n <= ~10)."""
    items = sorted(lengths, reverse=True)
    best = [len(items)]

    def place(k: int, rooms: List[int]) -> None:
        if len(rooms) >= best[0]:
            return
        if k == len(items):
            best[0] = len(rooms)
            return
        seen = set()
        for b in range(len(rooms)):
            if rooms[b] >= items[k] and rooms[b] not in seen:
                seen.add(rooms[b])
                rooms[b] -= items[k]
                place(k + 1, rooms)
                rooms[b] += items[k]
        rooms.append(capacity - items[k])
        place(k + 1, rooms)
        rooms.pop()

    place(0, [])
    return best[0]
