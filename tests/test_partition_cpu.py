"""The split-K partition the library documents, checked as plain integer
arithmetic on the host (no GPU): every visible block of every (request, KV
head) lands in exactly one piece, pieces of a segment take consecutive
slots from 0, and the slot counts stay within the workspace the library
sizes (S of paged_decode_splitk_plan)."""
import numpy as np
import pytest

from tests.splitk_partition import split_ranges, visible_blocks


def plan(max_seq_len, window, bs=16):
    """paged_decode_splitk_plan restated: C = max(4, ceil(T / 32)), S = ceil(T / C) + 1."""
    T = -(-max_seq_len // bs)
    if window > 0:
        T = min(T, (window - 1) // bs + 2)
    if T <= 0:
        return 1, 1
    C = max(4, -(-T // 32))
    return -(-T // C) + 1, C


CASES = [
    ([int(x) for x in np.random.default_rng(0).integers(512, 4097, 32)], 0, 2, 304),
    ([int(x) for x in np.random.default_rng(0).integers(512, 4097, 32)], 512, 2, 304),
    ([int(x) for x in np.random.default_rng(1).integers(32768, 131073, 4)], 0, 4, 304),
    ([int(x) for x in np.random.default_rng(2).integers(1, 257, 4)], 0, 2, 304),
    ([0, 40, 0, 0, 700, 1, 0], 0, 2, 304),
    ([0, 0, 0], 0, 2, 304),
    ([int(x) for x in np.random.default_rng(3).integers(1024, 16385, 64)], 1024, 2, 176),
    ([5000, 17, 33], 0, 1, 3),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_partitions_cover_each_block_once(case):
    L, window, hkv, grid = CASES[case]
    S, C = plan(max(L), window)
    pieces = [[[(s, j0, j1) for s, (j0, j1) in enumerate(per)] for per in head]
              for head in split_ranges(L, window, 16, hkv, grid, C)]
    for b, per_head in enumerate(pieces):
        jlo, jhi = visible_blocks(L[b], window, 16)
        for pcs in per_head:
            covered = sorted(j for (_, j0, j1) in pcs for j in range(j0, j1))
            assert covered == list(range(jlo, jhi)), b
            slots = [s for (s, _, _) in pcs]
            assert slots == list(range(len(pcs))), (b, slots)
            assert len(pcs) <= S, (b, len(pcs), S)
