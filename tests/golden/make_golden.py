"""Writes decode_small.json: a seeded small case and the oracle's output.

Calls only the oracle (no CUDA path).  Re-run after a deliberate change to
the oracle's arithmetic, and say in the commit which reading of the pages
justified the change.
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import paged_attention  # noqa: E402


def case():
    rng = np.random.default_rng(2024)
    bs, Hkv, G, D = 4, 2, 2, 8
    seq_lens = [5, 19, 11]
    q_lens = [1, 4, 1]
    nblk = 12
    perm = rng.permutation(nblk)
    tables, cur = [], 0
    for L in seq_lens:
        nb = -(-L // bs)
        tables.append([int(x) for x in perm[cur:cur + nb]] + [-1] * (5 - nb))
        cur += nb
    # values on a 1/8 grid so the inputs are exact in any float format
    k = np.round(rng.standard_normal((nblk, Hkv, bs, D)) * 8) / 8
    v = np.round(rng.standard_normal((nblk, Hkv, bs, D)) * 8) / 8
    q = np.round(rng.standard_normal((sum(q_lens), Hkv * G, D)) * 8) / 8
    qsl = [0]
    for n in q_lens:
        qsl.append(qsl[-1] + n)
    return dict(q=q, k_pool=k, v_pool=v, block_tables=np.array(tables),
                seq_lens=np.array(seq_lens), query_start_loc=np.array(qsl),
                scale=0.35, softcap=2.5, window=6)


def main():
    c = case()
    out, lse = paged_attention(c["q"], c["k_pool"], c["v_pool"], c["block_tables"],
                               c["seq_lens"], c["query_start_loc"], c["scale"], c["softcap"],
                               c["window"])
    doc = {k: (v.tolist() if hasattr(v, "tolist") else v) for k, v in c.items()}
    doc["out"] = out.tolist()
    doc["lse"] = lse.tolist()
    with open(os.path.join(HERE, "decode_small.json"), "w") as f:
        json.dump(doc, f)


if __name__ == "__main__":
    main()
