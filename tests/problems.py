"""Small fp64 problems for pinning the oracle (host only, numpy).

Builds pools, block tables and queries directly as numpy arrays so the oracle
pins need neither torch nor the product package.
"""
from __future__ import annotations

import numpy as np


def tables_for(rng, seq_lens, block_size, num_blocks=None, shuffle=True):
    need = sum(-(-L // block_size) for L in seq_lens)
    if num_blocks is None:
        num_blocks = need + 3
    ids = rng.permutation(num_blocks) if shuffle else np.arange(num_blocks)
    width = max([-(-L // block_size) for L in seq_lens] + [1])
    bt = np.full((len(seq_lens), width), -1, dtype=np.int64)
    cur = 0
    for b, L in enumerate(seq_lens):
        nb = -(-L // block_size)
        bt[b, :nb] = ids[cur:cur + nb]
        cur += nb
    return bt, num_blocks


def problem(rng, seq_lens, q_lens, Hq=4, Hkv=2, D=8, bs=4, num_blocks=None,
            shuffle=True, dv=None):
    dv = D if dv is None else dv
    bt, nblk = tables_for(rng, seq_lens, bs, num_blocks, shuffle)
    total_q = int(sum(q_lens))
    qsl = np.zeros(len(q_lens) + 1, dtype=np.int64)
    qsl[1:] = np.cumsum(q_lens)
    return dict(
        q=rng.standard_normal((total_q, Hq, D)),
        k_pool=rng.standard_normal((nblk, Hkv, bs, D)),
        v_pool=rng.standard_normal((nblk, Hkv, bs, dv)),
        block_tables=bt,
        seq_lens=np.array(seq_lens, dtype=np.int64),
        query_start_loc=qsl,
    )


def contiguous_kv(p, b):
    """Request b's K and V as [L][Hkv][D] by walking its table (test helper)."""
    bs = p["k_pool"].shape[2]
    L = int(p["seq_lens"][b])
    K = np.stack([p["k_pool"][p["block_tables"][b][t // bs], :, t % bs, :] for t in range(L)]) \
        if L else np.zeros((0,) + p["k_pool"].shape[1:2] + p["k_pool"].shape[3:])
    V = np.stack([p["v_pool"][p["block_tables"][b][t // bs], :, t % bs, :] for t in range(L)]) \
        if L else np.zeros((0,) + p["v_pool"].shape[1:2] + p["v_pool"].shape[3:])
    return K, V
