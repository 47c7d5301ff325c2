"""Pure-Python brute force for tiny paged-attention cases.

TEST INFRASTRUCTURE.  Used only to pin the fp64 oracle: it reaches the same
result by a different route, so a slip in one of them shows up as a
disagreement.

* K/V are read token by token through the block table (no gathered copy):
  block ``table[t // bs]``, slot ``t % bs``.
* Masks are tested one key at a time against the query's absolute position.
* The softmax is the ratio ``exp(s_t) / sum_u exp(s_u)`` with no max shift
  (safe for the small logits of tiny cases), every sum taken with
  ``math.fsum``.

Inputs are nested Python lists (or anything indexable the same way).
"""
from __future__ import annotations

import math


def brute_force_attention(q, k_pool, v_pool, block_tables, seq_lens, query_start_loc,
                          scale, softcap=0.0, window=0):
    """Returns (out[total_q][Hq][D], lse[total_q][Hq]) as Python floats."""
    total_q = len(q)
    Hq = len(q[0]) if total_q else 0
    Hkv = len(k_pool[0])
    bs = len(k_pool[0][0])
    Dv = len(v_pool[0][0][0])
    group = Hq // Hkv
    out = [[[0.0] * Dv for _ in range(Hq)] for _ in range(total_q)]
    lse = [[-math.inf] * Hq for _ in range(total_q)]
    for b in range(len(seq_lens)):
        L = int(seq_lens[b])
        q0, q1 = int(query_start_loc[b]), int(query_start_loc[b + 1])
        n = q1 - q0
        for i in range(n):
            pos = L - n + i
            for h in range(Hq):
                kvh = h // group
                weights = []
                rows = []
                for t in range(L):
                    if t > pos:
                        continue
                    if window > 0 and pos - t >= window:
                        continue
                    blk = int(block_tables[b][t // bs])
                    slot = t % bs
                    krow = k_pool[blk][kvh][slot]
                    s = scale * math.fsum(float(a) * float(c) for a, c in zip(q[q0 + i][h], krow))
                    if softcap > 0:
                        s = softcap * math.tanh(s / softcap)
                    weights.append(math.exp(s))
                    rows.append(v_pool[blk][kvh][slot])
                if not weights:
                    continue
                z = math.fsum(weights)
                for d in range(Dv):
                    out[q0 + i][h][d] = math.fsum(w * float(r[d]) for w, r in zip(weights, rows)) / z
                lse[q0 + i][h] = math.log(z)
    return out, lse
