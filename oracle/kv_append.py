"""Oracle of the KV-cache append (TEST INFRASTRUCTURE; see the package doc).

The cache write before attention on every tick: "Block-paged per-layer KV
with refcounted blocks, lazy allocation, and SDPA gather -- vLLM/PagedAttention
layout" (github README, "What's inside", Paged KV cache row).  The pages do
not spell out how a new token names its place; the reading taken here is the
vLLM one: a slot number s = block * block_size + offset per token, s < 0 for
a padding token that is not written.
"""
from __future__ import annotations

import numpy as np


def kv_append(k_pool: np.ndarray, v_pool: np.ndarray, k_new: np.ndarray, v_new: np.ndarray,
              slot_mapping: np.ndarray, block_size: int):
    """New pools with token t's rows written at slot ``slot_mapping[t]``.

    Pools ``[num_blocks][Hkv][block_size][D]``, new rows ``[T][Hkv][D]``.
    Token t with slot s >= 0 goes to block s // block_size, offset
    s % block_size, for every KV head; s < 0 is skipped, as is a slot past the
    pool (the library reports that one).  Returns copies, the inputs are left
    as they are.
    """
    k_out = k_pool.copy()
    v_out = v_pool.copy()
    num_blocks = k_pool.shape[0]
    for t, s in enumerate(np.asarray(slot_mapping).tolist()):
        if s < 0:
            continue
        blk, off = divmod(int(s), block_size)
        if blk >= num_blocks:
            continue
        k_out[blk, :, off, :] = k_new[t]
        v_out[blk, :, off, :] = v_new[t]
    return k_out, v_out
