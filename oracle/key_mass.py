"""Oracle of the H2O attention mass (TEST INFRASTRUCTURE; see the package doc).

The engine's cache offers an H2O eviction policy ("Eviction policies --
Pluggable per-session: LRU, AttentionSink, H2O", github README, "What's
inside"), which keeps the keys that drew the most attention.  What one
decode step contributes: for each request b and KV head kvh, each key t the
step's query sees gets the attention probability it received, summed over
the G query heads that read that KV head.  (The pages do not say how the
mass is kept; this reading accumulates the softmax probabilities per
(request, KV head, key), the H2O paper's per-head score summed over a
group's heads.)
"""
from __future__ import annotations

import numpy as np

from .paged_attention import gather_request_kv, visible_keys


def key_mass(q, k_pool, block_tables, seq_lens, scale, softcap=0.0, window=0,
             block_size=16, num_keys=None):
    """Mass ``[B][Hkv][num_keys]`` (fp64) added by one decode step.

    ``q`` [B][Hq][D] (one query per request at position ``seq_len - 1``),
    ``k_pool`` [num_blocks][Hkv][bs][D].  Logits ``s = scale * q.k``, capped
    as in attention; probabilities by the max-subtracted softmax over the
    visible keys.  Keys not visible get 0.
    """
    q = np.asarray(q, dtype=np.float64)
    k_pool = np.asarray(k_pool, dtype=np.float64)
    B, Hq, _ = q.shape
    Hkv = k_pool.shape[1]
    G = Hq // Hkv
    if num_keys is None:
        num_keys = max([int(L) for L in seq_lens] + [1])
    mass = np.zeros((B, Hkv, num_keys))
    for b in range(B):
        L = int(seq_lens[b])
        if L <= 0:
            continue
        keys = visible_keys(L - 1, L, window)
        kc = gather_request_kv(k_pool, np.asarray(block_tables[b]), L, block_size)
        for kvh in range(Hkv):
            kk = kc[keys, kvh, :]
            for g in range(G):
                s = scale * (kk @ q[b, kvh * G + g])
                if softcap > 0:
                    s = softcap * np.tanh(s / softcap)
                p = np.exp(s - s.max())
                mass[b, kvh, keys] += p / p.sum()
    return mass
