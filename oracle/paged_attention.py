"""fp64 CPU oracle for attention read through a block-paged KV cache.

TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
CPU-baseline leg may import this module.  It shares no code with the CUDA
path and imports nothing from it.

What it computes is the plain definition of the operation the inference-server
pages describe: "Block-paged per-layer KV with refcounted blocks, lazy
allocation, and SDPA gather" (github README, "What's inside", Paged KV cache
row).  The oracle takes that "SDPA gather" reading literally:

1. materialise each request's contiguous K and V from its block table
   (token ``t`` of request ``b`` lives in block ``table[b][t // bs]``,
   slot ``t % bs``);
2. run textbook masked softmax attention over the visible keys, in fp64.

Conventions where the pages are silent (each is one reading, stated once):

* GQA ("GQA with QK/V-norm + KV sharing", github README, "Custom Gemma 4
  forward" row): query head ``h`` reads KV head ``h // (Hq / Hkv)``.
* Positions: query ``i`` of a request with ``n`` new tokens and context
  length ``L`` sits at absolute position ``p = L - n + i``; it sees key ``t``
  iff ``t <= p`` (causal) and, with a sliding window ``W > 0`` ("window-aware
  sliding layers", inference-server README feature list), ``t > p - W``
  (W keys including itself).
* Softcap ("softcapping", same Gemma row): logits are scaled first, then
  ``cap * tanh(s / cap)`` when ``cap > 0``.
* LSE is the natural-log log-sum-exp of the (capped) logits; an empty
  visible set gives output 0 and LSE ``-inf``.
* Split-K ("split-K decode variant", inference-server README feature list):
  the pages give no partition, and the combined result does not depend on
  it, so the partition is an input: each split covers a contiguous range of
  the request's visible blocks; its partial is the (softmax-normalised
  output, LSE) over that range and the combine is the log-sum-exp merge of
  the partials.  Which partition a GPU launch uses is the library's
  scheduling choice and is not restated here.
"""
from __future__ import annotations

import math

import numpy as np


def gather_request_kv(pool: np.ndarray, table_row: np.ndarray, seq_len: int,
                      block_size: int) -> np.ndarray:
    """Contiguous ``[seq_len][Hkv][D]`` cache of one request.

    Row ``t`` is ``pool[table_row[t // block_size], :, t % block_size, :]``
    (the block-table lookup of a vLLM/PagedAttention-layout cache).
    """
    t = np.arange(seq_len)
    return pool[table_row[t // block_size], :, t % block_size, :]


def visible_keys(pos: int, seq_len: int, window: int) -> np.ndarray:
    """Key positions a query at absolute position ``pos`` attends to."""
    t = np.arange(seq_len)
    keep = t <= pos
    if window > 0:
        keep &= t > pos - window
    return t[keep]


def softmax_attention(q_rows: np.ndarray, keys: np.ndarray, values: np.ndarray,
                      scale: float, softcap: float):
    """Textbook attention of ``G`` query rows over one key set.

    ``q_rows`` [G][D], ``keys``/``values`` [T][D].  Returns (out [G][D],
    lse [G]).  Logits: ``s = scale * k.q``, then the optional tanh cap; the
    softmax uses the usual max subtraction.
    """
    G, D = q_rows.shape
    if keys.shape[0] == 0:
        return np.zeros((G, values.shape[1])), np.full(G, -np.inf)
    s = scale * (keys @ q_rows.T)                  # [T][G]
    if softcap > 0:
        s = softcap * np.tanh(s / softcap)
    m = s.max(axis=0)                               # [G]
    e = np.exp(s - m)                               # [T][G]
    l = e.sum(axis=0)                               # [G]
    out = (e.T @ values) / l[:, None]               # [G][D]
    lse = m + np.log(l)
    return out, lse


def paged_attention(q, k_pool, v_pool, block_tables, seq_lens, query_start_loc,
                    scale, softcap=0.0, window=0):
    """Varlen paged attention (decode rows and prefill chunks alike).

    q [total_q][Hq][D]; pools [num_blocks][Hkv][bs][D]; block_tables
    [B][max_blocks]; seq_lens [B]; query_start_loc [B+1].
    Returns (out [total_q][Hq][D], lse [total_q][Hq]) in fp64.
    """
    q = np.asarray(q, dtype=np.float64)
    total_q, Hq, D = q.shape
    num_blocks, Hkv, bs, _ = k_pool.shape
    G = Hq // Hkv
    out = np.zeros((total_q, Hq, v_pool.shape[3]))
    lse = np.full((total_q, Hq), -np.inf)
    for b in range(len(seq_lens)):
        L = int(seq_lens[b])
        q0, q1 = int(query_start_loc[b]), int(query_start_loc[b + 1])
        n = q1 - q0
        if L == 0 or n == 0:
            continue
        # Only keys the request's queries can see are gathered (blocks wholly
        # outside a sliding window may already be freed).
        lo = 0 if window <= 0 else max(0, L - n - window + 1)
        Kb = np.zeros((L, Hkv, D))
        Vb = np.zeros((L, Hkv, v_pool.shape[3]))
        Kb[lo:] = gather_request_kv(k_pool, block_tables[b], L, bs)[lo:]
        Vb[lo:] = gather_request_kv(v_pool, block_tables[b], L, bs)[lo:]
        for i in range(n):
            pos = L - n + i
            T = visible_keys(pos, L, window)
            for kvh in range(Hkv):
                heads = slice(kvh * G, (kvh + 1) * G)
                o, s = softmax_attention(q[q0 + i, heads, :], Kb[T, kvh, :],
                                         Vb[T, kvh, :], scale, softcap)
                out[q0 + i, heads, :] = o
                lse[q0 + i, heads] = s
    return out, lse


def paged_decode(q, k_pool, v_pool, block_tables, seq_lens, scale, softcap=0.0,
                 window=0):
    """Decode: one query token per request at position ``seq_len - 1``."""
    B = len(seq_lens)
    return paged_attention(q, k_pool, v_pool, block_tables, seq_lens,
                           np.arange(B + 1), scale, softcap, window)


def visible_block_range(seq_len: int, window: int, block_size: int):
    """[jlo, jhi) logical blocks holding the keys a decode query sees."""
    if seq_len <= 0:
        return 0, 0
    pos = seq_len - 1
    first = 0 if window <= 0 else max(0, pos - window + 1)
    return first // block_size, pos // block_size + 1


def splitk_partials(q, k_pool, v_pool, block_tables, seq_lens, scale, softcap,
                    window, num_splits, split_blocks=None, ranges=None):
    """Per-split (output, LSE) of decode attention.

    The split of each request's visible keys is an input.  Either
    ``ranges[b][s] = (j0, j1)`` (logical blocks of split ``s``, or ``None``
    for an unused split) or, when only ``split_blocks`` C is given, the fixed
    partition: split ``s`` covers blocks ``[jlo + s*C, jlo + (s+1)*C)``.
    The same ranges apply to every KV head of a request unless ``ranges``
    is indexed ``ranges[b][kvh][s]`` (a list per head).
    Returns partial_o [B][Hq][S][D] and partial_lse [B][Hq][S]; an empty
    split has output 0 and LSE ``-inf``.
    """
    q = np.asarray(q, dtype=np.float64)
    B = len(seq_lens)
    _, Hq, D = q.shape
    _, Hkv, bs, _ = k_pool.shape
    G = Hq // Hkv
    po = np.zeros((B, Hq, num_splits, v_pool.shape[3]))
    pl = np.full((B, Hq, num_splits), -np.inf)
    for b in range(B):
        L = int(seq_lens[b])
        if L == 0:
            continue
        pos = L - 1
        jlo, jhi = visible_block_range(L, window, bs)
        T_all = visible_keys(pos, L, window)
        Kb = np.zeros((L, Hkv, D))
        Vb = np.zeros((L, Hkv, v_pool.shape[3]))
        Kb[T_all] = gather_request_kv(k_pool, block_tables[b], L, bs)[T_all]
        Vb[T_all] = gather_request_kv(v_pool, block_tables[b], L, bs)[T_all]
        for kvh in range(Hkv):
            heads = slice(kvh * G, (kvh + 1) * G)
            for s in range(num_splits):
                if ranges is None:
                    j0 = jlo + s * split_blocks
                    rng = (j0, min(jhi, j0 + split_blocks))
                else:
                    per = ranges[b][kvh] if isinstance(ranges[b][0], list) else ranges[b]
                    rng = per[s] if s < len(per) else None
                if rng is None:
                    continue
                j0, j1 = rng
                T = T_all[(T_all >= j0 * bs) & (T_all < j1 * bs)]
                o, l = softmax_attention(q[b, heads, :], Kb[T, kvh, :], Vb[T, kvh, :],
                                         scale, softcap)
                po[b, heads, s, :] = o
                pl[b, heads, s] = l
    return po, pl


def lse_combine(partial_o, partial_lse):
    """Log-sum-exp merge of split partials over the split axis.

    With ``M = max_s LSE_s`` and ``w_s = exp(LSE_s - M)``:
    ``out = sum_s w_s O_s / sum_s w_s`` and ``LSE = M + ln sum_s w_s``.
    All-empty rows give output 0 and LSE ``-inf``.
    """
    partial_o = np.asarray(partial_o, dtype=np.float64)
    partial_lse = np.asarray(partial_lse, dtype=np.float64)
    M = partial_lse.max(axis=-1)
    finite = np.isfinite(M)
    Ms = np.where(finite, M, 0.0)
    w = np.where(np.isfinite(partial_lse), np.exp(partial_lse - Ms[..., None]), 0.0)
    den = w.sum(axis=-1)
    num = (w[..., None] * partial_o).sum(axis=-2)
    out = np.where(finite[..., None], num / np.where(den > 0, den, 1.0)[..., None], 0.0)
    lse = np.where(finite, Ms + np.log(np.where(den > 0, den, 1.0)), -np.inf)
    return out, lse


def run_batch(arrays):
    """Oracle output for a dict made by the workload module's numpy export."""
    return paged_attention(arrays["q"], arrays["k_pool"], arrays["v_pool"],
                           arrays["block_tables"], arrays["seq_lens"],
                           arrays["query_start_loc"], arrays["scale"],
                           arrays["softcap"], arrays["window"])


__all__ = [
    "gather_request_kv", "visible_keys", "softmax_attention", "paged_attention",
    "paged_decode", "visible_block_range", "splitk_partials", "lse_combine",
    "run_batch",
]
