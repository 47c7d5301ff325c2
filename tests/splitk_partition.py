"""The split-K work partition the library documents for ``paged_decode_splitk``.

The partition is a scheduling choice of the library, not part of the
attention arithmetic (the combined result is the same for any partition), so
it lives with the tests rather than in the oracle.  This module restates the
contract written beside ``paged_decode_splitk`` in ``include/paged_attn.h``
as plain integer arithmetic, so that a test can ask the oracle for the
partial each slot must hold (``oracle.splitk_partials(ranges=...)``).
"""
from __future__ import annotations

PIECE_UNITS = 4  # work units a segment takes for its partial, before its tiles


def visible_blocks(seq_len: int, window: int, block_size: int):
    """[jlo, jhi): the blocks holding the keys a decode query sees."""
    if seq_len <= 0:
        return 0, 0
    pos = seq_len - 1
    first = 0 if window <= 0 else max(0, pos - window + 1)
    return first // block_size, pos // block_size + 1


def split_ranges(seq_lens, window, block_size, num_kv_heads, grid, min_chunk,
                 piece_units=PIECE_UNITS):
    """ranges[b][kvh] = the (j0, j1) block range of each slot, in slot order.

    Segments (request, KV head) in that order on a line of units: a segment
    of n > 0 tiles takes ``piece_units`` units, then one unit per tile.  The
    T units are cut into chunks of q = max(min_chunk, ceil(T / grid)); the
    tiles of a segment whose first tile is at unit A that fall in chunk c
    form the piece of slot c - floor(A / q).
    """
    span = [visible_blocks(int(L), window, block_size) for L in seq_lens]
    units = [(j1 - j0) + piece_units if j1 > j0 else 0 for j0, j1 in span]
    total = num_kv_heads * sum(units)
    q = max(min_chunk, -(-total // grid), 1)
    ranges = []
    start = 0  # unit where the current segment begins
    for (j0, j1), u in zip(span, units):
        per_head = []
        for _ in range(num_kv_heads):
            n = j1 - j0
            slots = []
            if n > 0:
                A = start + piece_units
                for c in range(A // q, (A + n - 1) // q + 1):
                    lo, hi = max(A, c * q), min(A + n, (c + 1) * q)
                    slots.append((j0 + lo - A, j0 + hi - A))
            per_head.append(slots)
            start += u
        ranges.append(per_head)
    return ranges



DIRECT_SLACK = 24  # units beyond the chunk within which a fused launch streams whole


def streams_whole(seq_lens, window, block_size, num_kv_heads, pipelines, min_chunk,
                  piece_units=PIECE_UNITS, slack=DIRECT_SLACK):
    """True when a fused launch (``paged_decode_attn_ws``, and the decode rows
    of ``paged_prefill_attn_ws``) streams every segment whole instead of
    splitting it: the B * Hkv segments fit one per pipeline and none is
    longer than the chunk q plus ``slack`` units (the header's rule)."""
    span = [visible_blocks(int(L), window, block_size) for L in seq_lens]
    units = [(j1 - j0) + piece_units if j1 > j0 else 0 for j0, j1 in span]
    total = num_kv_heads * sum(units)
    q = max(min_chunk, -(-total // pipelines), 1)
    return (len(seq_lens) * num_kv_heads <= pipelines and
            max(units, default=0) <= q + slack)
