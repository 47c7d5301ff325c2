"""Pins for the fp64 oracle: brute force, closed forms, invariants, a library routine.

None of these retypes the oracle's formula.  Each pin is chosen so that a
plausible slip in the oracle (a dropped scale, cap before scale, the wrong
GQA grouping, a window off by one, a wrong slot in the table walk, a causal
offset in prefill, a wrong LSE merge) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch
from scipy.special import logsumexp

from oracle import (brute_force_attention, lse_combine, paged_attention,
                    paged_decode, splitk_partials, visible_block_range)
from tests.problems import contiguous_kv, problem


def run(p, scale=0.5, softcap=0.0, window=0):
    return paged_attention(p["q"], p["k_pool"], p["v_pool"], p["block_tables"],
                           p["seq_lens"], p["query_start_loc"], scale, softcap, window)


# --------------------------------------------------------------------------
# brute force on tiny inputs (different route: per-token table walk, no max
# shift, fsum everywhere)
# --------------------------------------------------------------------------
@pytest.mark.parametrize("case", range(24))
def test_brute_force_agrees(case):
    rng = np.random.default_rng(100 + case)
    B = int(rng.integers(1, 4))
    bs = int(rng.choice([1, 2, 4, 16]))
    Hkv = int(rng.choice([1, 2]))
    G = int(rng.choice([1, 2, 4]))
    D = int(rng.choice([4, 8]))
    L = [int(rng.integers(1, 41)) for _ in range(B)]
    n = [int(rng.integers(1, l + 1)) if rng.random() < 0.5 else 1 for l in L]
    window = int(rng.choice([0, 0, 1, 3, 7, 64]))
    softcap = float(rng.choice([0.0, 0.0, 0.7, 5.0]))
    scale = float(rng.choice([0.3, 1.0 / math.sqrt(D)]))
    p = problem(rng, L, n, Hq=G * Hkv, Hkv=Hkv, D=D, bs=bs)
    out, lse = run(p, scale, softcap, window)
    bo, bl = brute_force_attention(p["q"].tolist(), p["k_pool"].tolist(), p["v_pool"].tolist(),
                                   p["block_tables"].tolist(), p["seq_lens"].tolist(),
                                   p["query_start_loc"].tolist(), scale, softcap, window)
    np.testing.assert_allclose(out, np.array(bo), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse, np.array(bl), rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------
# special cases with exact answers
# --------------------------------------------------------------------------
def test_seq_len_one_returns_v0():
    rng = np.random.default_rng(1)
    p = problem(rng, [1, 1, 1], [1, 1, 1], Hq=8, Hkv=2, D=16, bs=16)
    out, lse = run(p, 0.25, 50.0, 0)
    for b in range(3):
        _, V = contiguous_kv(p, b)
        for h in range(8):
            assert np.array_equal(out[b, h], V[0, h // 4])
        s = 0.25 * p["q"][b] @ np.repeat(contiguous_kv(p, b)[0][0], 4, axis=0).T
        np.testing.assert_allclose(lse[b], 50.0 * np.tanh(np.diag(s) / 50.0), rtol=1e-14)


def test_identical_keys_give_mean_of_v():
    rng = np.random.default_rng(2)
    L = [13, 29]
    p = problem(rng, L, [1, 1], Hq=4, Hkv=2, D=8, bs=4)
    p["k_pool"][:] = rng.standard_normal(8)  # every key row identical
    out, lse = run(p, 0.7, 0.0, 0)
    for b in range(2):
        K, V = contiguous_kv(p, b)
        for h in range(4):
            np.testing.assert_allclose(out[b, h], V[:, h // 2].mean(axis=0), rtol=1e-12)
            s = 0.7 * float(p["q"][b, h] @ K[0, 0])
            assert lse[b, h] == pytest.approx(s + math.log(L[b]), rel=1e-13)


@pytest.mark.parametrize("softcap,window", [(0.0, 0), (30.0, 0), (0.0, 5)])
def test_zero_scale_gives_mean_of_visible_values(softcap, window):
    """scale = 0 makes every visible logit 0 (capped or not): each query row
    returns the plain mean of the V rows it sees, whatever q and K are."""
    rng = np.random.default_rng(6)
    L = [13, 29, 1]
    n = [1, 6, 1]
    p = problem(rng, L, n, Hq=4, Hkv=2, D=8, bs=4)
    out, lse = run(p, 0.0, softcap, window)
    qs = p["query_start_loc"]
    for b in range(3):
        _, V = contiguous_kv(p, b)
        for i in range(n[b]):
            pos = L[b] - n[b] + i
            lo = 0 if window <= 0 else max(0, pos - window + 1)
            for h in range(4):
                np.testing.assert_allclose(out[qs[b] + i, h], V[lo:pos + 1, h // 2].mean(axis=0),
                                           rtol=1e-12, atol=1e-14)
                assert lse[qs[b] + i, h] == pytest.approx(math.log(pos + 1 - lo), rel=1e-13)


@pytest.mark.parametrize("softcap", [0.0, 4.0])
def test_negative_scale_equals_negated_queries(softcap):
    """s = scale * q.k and the tanh cap is odd, so a negative scale is the
    positive one applied to -q (the keys that were least aligned win)."""
    rng = np.random.default_rng(7)
    p = problem(rng, [21, 40], [3, 1], Hq=4, Hkv=2, D=8, bs=4)
    out, lse = run(p, -0.4, softcap, 0)
    neg = dict(p, q=-p["q"])
    out2, lse2 = run(neg, 0.4, softcap, 0)
    np.testing.assert_allclose(out, out2, rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse, lse2, rtol=1e-13, atol=1e-14)


def test_gqa_grouping_with_constant_values():
    """V of KV head j is the constant j+1: query head h must read h // G."""
    rng = np.random.default_rng(3)
    p = problem(rng, [9, 20], [1, 3], Hq=8, Hkv=2, D=4, bs=4)
    for j in range(2):
        p["v_pool"][:, j] = j + 1.0
    out, _ = run(p, 0.5, 0.0, 0)
    for r in range(out.shape[0]):
        for h in range(8):
            np.testing.assert_allclose(out[r, h], np.full(4, h // 4 + 1.0), rtol=1e-14)


def test_window_one_returns_own_value():
    rng = np.random.default_rng(4)
    L = [7, 19]
    p = problem(rng, L, [3, 5], Hq=2, Hkv=1, D=8, bs=4)
    out, _ = run(p, 0.3, 0.0, 1)
    qs = p["query_start_loc"]
    for b in range(2):
        _, V = contiguous_kv(p, b)
        n = qs[b + 1] - qs[b]
        for i in range(n):
            pos = L[b] - n + i
            for h in range(2):
                assert np.array_equal(out[qs[b] + i, h], V[pos, 0])


def test_window_at_least_length_is_full():
    rng = np.random.default_rng(5)
    L = [17, 33]
    p = problem(rng, L, [4, 1], Hq=4, Hkv=2, D=8, bs=4)
    full, lf = run(p, 0.4, 0.0, 0)
    for W in (33, 34, 1000):
        o, l = run(p, 0.4, 0.0, W)
        np.testing.assert_array_equal(o, full)
        np.testing.assert_array_equal(l, lf)
    # W=17 still keeps every key of the shorter request but not of the longer one
    o, _ = run(p, 0.4, 0.0, 17)
    assert np.allclose(o[:4], full[:4])
    assert not np.allclose(o[4:], full[4:])


def _sigmoid(x):
    return 1.0 / (1.0 + math.exp(-x))


@pytest.mark.parametrize("softcap", [0.0, 0.9, 3.0])
@pytest.mark.parametrize("window", [0, 2])
def test_two_key_closed_form(softcap, window):
    """Two visible keys: out = sig(D)*v1 + (1-sig(D))*v0, D = f(s1) - f(s0)."""
    rng = np.random.default_rng(6)
    for trial in range(5):
        p = problem(rng, [2], [1], Hq=1, Hkv=1, D=6, bs=1, num_blocks=5)
        scale = 0.8
        out, lse = run(p, scale, softcap, window)
        K, V = contiguous_kv(p, 0)
        s = [scale * float(p["q"][0, 0] @ K[t, 0]) for t in range(2)]
        f = [softcap * math.tanh(x / softcap) if softcap > 0 else x for x in s]
        w1 = _sigmoid(f[1] - f[0])
        np.testing.assert_allclose(out[0, 0], w1 * V[1, 0] + (1 - w1) * V[0, 0], rtol=1e-12)
        assert lse[0, 0] == pytest.approx(math.log(math.exp(f[0]) + math.exp(f[1])), rel=1e-12)


def test_huge_cap_equals_no_cap():
    rng = np.random.default_rng(7)
    p = problem(rng, [30, 11], [5, 1], Hq=4, Hkv=1, D=8, bs=2)
    a, la = run(p, 0.35, 0.0, 0)
    b, lb = run(p, 0.35, 1e6, 0)
    np.testing.assert_allclose(a, b, rtol=1e-9, atol=1e-9)
    np.testing.assert_allclose(la, lb, rtol=1e-9, atol=1e-9)


def test_cap_bounds_logits():
    """With the cap, |s| < cap for every key, so LSE <= cap + ln(#keys)."""
    rng = np.random.default_rng(8)
    p = problem(rng, [40], [1], Hq=1, Hkv=1, D=8, bs=4)
    p["q"] *= 50.0
    _, lse = run(p, 1.0, 2.0, 0)
    assert lse[0, 0] <= 2.0 + math.log(40) + 1e-12


# --------------------------------------------------------------------------
# paging invariants
# --------------------------------------------------------------------------
def test_paged_equals_contiguous_and_permutation_invariant():
    rng = np.random.default_rng(9)
    L = [25, 3, 40]
    p = problem(rng, L, [1, 1, 1], Hq=4, Hkv=2, D=8, bs=4, shuffle=False)
    base, lb = run(p, 0.5, 0.0, 0)
    perm = rng.permutation(p["k_pool"].shape[0])
    inv = np.argsort(perm)
    q = dict(p)
    q["k_pool"] = p["k_pool"][perm]
    q["v_pool"] = p["v_pool"][perm]
    q["block_tables"] = np.where(p["block_tables"] >= 0, inv[np.maximum(p["block_tables"], 0)], -1)
    out, lo = run(q, 0.5, 0.0, 0)
    np.testing.assert_array_equal(out, base)
    np.testing.assert_array_equal(lo, lb)
    # block size 1 with the same token order gives the same answer
    r = dict(p)
    tok_k = np.concatenate([contiguous_kv(p, b)[0] for b in range(3)])
    tok_v = np.concatenate([contiguous_kv(p, b)[1] for b in range(3)])
    r["k_pool"] = tok_k[:, :, None, :]
    r["v_pool"] = tok_v[:, :, None, :]
    starts = np.cumsum([0] + L[:-1])
    bt = np.full((3, max(L)), -1)
    for b in range(3):
        bt[b, :L[b]] = starts[b] + np.arange(L[b])
    r["block_tables"] = bt
    out1, _ = run(r, 0.5, 0.0, 0)
    np.testing.assert_allclose(out1, base, rtol=1e-13, atol=1e-15)


def test_shared_prefix_blocks_equal_private_copies():
    rng = np.random.default_rng(10)
    bs, Hkv, D = 4, 2, 8
    shared = rng.standard_normal((3, Hkv, bs, D)), rng.standard_normal((3, Hkv, bs, D))
    own = rng.standard_normal((4, Hkv, bs, D)), rng.standard_normal((4, Hkv, bs, D))
    # shared pool: blocks 0-2 shared; request 0 owns 3-4, request 1 owns 5-6
    kp = np.concatenate([shared[0], own[0]])
    vp = np.concatenate([shared[1], own[1]])
    bt = np.array([[0, 1, 2, 3, 4], [0, 1, 2, 5, 6]])
    q = rng.standard_normal((2, 4, D))
    sl = np.array([19, 20])
    a, _ = paged_decode(q, kp, vp, bt, sl, 0.5)
    # private copies: each request has its own copy of the prefix blocks
    kp2 = np.concatenate([shared[0], own[0][:2], shared[0], own[0][2:]])
    vp2 = np.concatenate([shared[1], own[1][:2], shared[1], own[1][2:]])
    bt2 = np.array([[0, 1, 2, 3, 4], [5, 6, 7, 8, 9]])
    b, _ = paged_decode(q, kp2, vp2, bt2, sl, 0.5)
    np.testing.assert_array_equal(a, b)


def test_one_hot_position_through_table():
    """V[t] = t and a key equal to a large multiple of q at t*: output is t*."""
    rng = np.random.default_rng(11)
    L = [37]
    p = problem(rng, L, [1], Hq=1, Hkv=1, D=8, bs=4)
    bs = 4
    for t in range(L[0]):
        blk = p["block_tables"][0][t // bs]
        p["v_pool"][blk, 0, t % bs, :] = float(t)
        p["k_pool"][blk, 0, t % bs, :] = 0.0
    qv = p["q"][0, 0]
    for tstar in (0, 5, 16, 36):
        k = p["k_pool"].copy()
        blk = p["block_tables"][0][tstar // bs]
        k[blk, 0, tstar % bs, :] = 200.0 * qv / float(qv @ qv)
        out, _ = paged_decode(p["q"], k, p["v_pool"], p["block_tables"], p["seq_lens"], 1.0)
        np.testing.assert_allclose(out[0, 0], float(tstar), rtol=1e-12, atol=1e-60)


# --------------------------------------------------------------------------
# algebraic invariants
# --------------------------------------------------------------------------
def test_shift_of_all_keys_leaves_output_unchanged():
    rng = np.random.default_rng(12)
    p = problem(rng, [21, 8], [3, 1], Hq=2, Hkv=1, D=8, bs=4)
    a, la = run(p, 0.5, 0.0, 0)
    c = rng.standard_normal(8)
    q = dict(p)
    q["k_pool"] = p["k_pool"] + c
    b, lb = run(q, 0.5, 0.0, 0)
    np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12)
    shift = 0.5 * p["q"] @ c  # [total_q][Hq]
    np.testing.assert_allclose(lb - la, shift, rtol=1e-10, atol=1e-12)


def test_linear_in_values():
    rng = np.random.default_rng(13)
    p = problem(rng, [18, 6], [2, 1], Hq=4, Hkv=2, D=8, bs=4)
    v2 = rng.standard_normal(p["v_pool"].shape)
    a, _ = run(p, 0.5, 3.0, 5)
    q = dict(p)
    q["v_pool"] = v2
    b, _ = run(q, 0.5, 3.0, 5)
    q["v_pool"] = p["v_pool"] + 2.5 * v2
    c, _ = run(q, 0.5, 3.0, 5)
    np.testing.assert_allclose(c, a + 2.5 * b, rtol=1e-11, atol=1e-12)


def test_matches_torch_sdpa_fp64():
    """A library routine: torch SDPA on the gathered cache with an explicit mask."""
    rng = np.random.default_rng(14)
    L = [30, 45]
    n = [6, 1]
    Hq, Hkv, D = 8, 2, 16
    p = problem(rng, L, n, Hq=Hq, Hkv=Hkv, D=D, bs=4)
    for window in (0, 9):
        out, _ = run(p, 0.3, 0.0, window)
        qs = p["query_start_loc"]
        for b in range(2):
            K, V = contiguous_kv(p, b)
            Kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)
            Vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)
            Qt = torch.from_numpy(p["q"][qs[b]:qs[b + 1]]).permute(1, 0, 2)
            pos = torch.arange(L[b] - n[b], L[b])[:, None]
            t = torch.arange(L[b])[None, :]
            mask = t <= pos
            if window:
                mask &= t > pos - window
            ref = torch.nn.functional.scaled_dot_product_attention(
                Qt, Kt, Vt, attn_mask=mask, scale=0.3)
            np.testing.assert_allclose(out[qs[b]:qs[b + 1]], ref.permute(1, 0, 2).numpy(),
                                       rtol=1e-10, atol=1e-12)


def test_lse_is_logsumexp_of_logits():
    rng = np.random.default_rng(15)
    p = problem(rng, [33], [1], Hq=2, Hkv=2, D=8, bs=4)
    _, lse = run(p, 0.6, 4.0, 0)
    K, _ = contiguous_kv(p, 0)
    for h in range(2):
        s = 0.6 * K[:, h] @ p["q"][0, h]
        s = 4.0 * np.tanh(s / 4.0)
        assert lse[0, h] == pytest.approx(logsumexp(s), rel=1e-13)


def test_prefill_row_equals_decode_at_that_length():
    rng = np.random.default_rng(16)
    P, n = 23, 9
    p = problem(rng, [P + n], [n], Hq=4, Hkv=2, D=8, bs=4)
    for window in (0, 6):
        out, _ = run(p, 0.5, 2.0, window)
        for i in range(n):
            d, _ = paged_decode(p["q"][i:i + 1], p["k_pool"], p["v_pool"],
                                p["block_tables"], np.array([P + i + 1]), 0.5, 2.0, window)
            np.testing.assert_array_equal(out[i], d[0])


def test_mixed_batch_equals_separate_calls():
    rng = np.random.default_rng(17)
    L = [20, 31, 12]
    n = [1, 7, 1]
    p = problem(rng, L, n, Hq=4, Hkv=2, D=8, bs=4)
    out, _ = run(p, 0.5, 0.0, 8)
    qs = p["query_start_loc"]
    for b in range(3):
        o, _ = paged_attention(p["q"][qs[b]:qs[b + 1]], p["k_pool"], p["v_pool"],
                               p["block_tables"][b:b + 1], p["seq_lens"][b:b + 1],
                               np.array([0, n[b]]), 0.5, 0.0, 8)
        np.testing.assert_array_equal(out[qs[b]:qs[b + 1]], o)


def test_empty_visible_set():
    rng = np.random.default_rng(18)
    p = problem(rng, [5, 0], [1, 0], Hq=2, Hkv=1, D=4, bs=4)
    out, lse = run(p, 0.5)
    assert np.all(np.isfinite(out))
    o, l = paged_decode(p["q"][:1], p["k_pool"], p["v_pool"], p["block_tables"][1:],
                        np.array([0]), 0.5)
    assert np.all(o == 0) and np.all(np.isneginf(l))


# --------------------------------------------------------------------------
# split-K and the LSE combine
# --------------------------------------------------------------------------
def test_lse_combine_closed_forms():
    o = np.array([[[1.0, 2.0], [3.0, 6.0]]])          # [1][S=2][D=2]
    l = np.array([[0.3, 0.3]])
    out, lse = lse_combine(o, l)
    np.testing.assert_allclose(out, [[2.0, 4.0]])
    assert lse[0] == pytest.approx(0.3 + math.log(2.0))
    l2 = np.array([[0.0, math.log(3.0)]])              # weights 1 : 3
    out2, _ = lse_combine(o, l2)
    np.testing.assert_allclose(out2, [[(1 + 9) / 4.0, (2 + 18) / 4.0]])
    out3, lse3 = lse_combine(o, np.array([[-np.inf, 1.0]]))  # empty split ignored
    np.testing.assert_allclose(out3, [[3.0, 6.0]])
    out4, lse4 = lse_combine(o, np.array([[-np.inf, -np.inf]]))
    assert np.all(out4 == 0) and np.isneginf(lse4[0])


@pytest.mark.parametrize("window", [0, 11])
def test_splitk_combine_equals_full(window):
    rng = np.random.default_rng(19)
    L = [57, 3, 100, 16]
    p = problem(rng, L, [1] * 4, Hq=4, Hkv=2, D=8, bs=4)
    full, lf = paged_decode(p["q"], p["k_pool"], p["v_pool"], p["block_tables"],
                            p["seq_lens"], 0.5, 1.5, window)
    maxvis = max(visible_block_range(x, window, 4)[1] - visible_block_range(x, window, 4)[0]
                 for x in L)
    for S in (1, 2, 3, 7, maxvis):
        C = -(-maxvis // S)
        po, pl = splitk_partials(p["q"], p["k_pool"], p["v_pool"], p["block_tables"],
                                 p["seq_lens"], 0.5, 1.5, window, S, C)
        out, lse = lse_combine(po, pl)
        np.testing.assert_allclose(out, full, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, lf, rtol=1e-12, atol=1e-13)
        if S == 1:
            np.testing.assert_allclose(po[:, :, 0], full, rtol=1e-13)
    # each split covers its own keys only: split s of a request with one
    # visible block beyond the first split is empty
    po, pl = splitk_partials(p["q"], p["k_pool"], p["v_pool"], p["block_tables"],
                             p["seq_lens"], 0.5, 1.5, window, 4, 1)
    assert np.isneginf(pl[1, :, 1:]).all()  # L=3 -> one block


@pytest.mark.parametrize("piece_units", [0, 2, 4, 5])
@pytest.mark.parametrize("grid,min_chunk", [(1, 1), (3, 2), (7, 4), (64, 1)])
def test_documented_partition_covers_and_combines(grid, min_chunk, piece_units):
    """The split partition the library documents (restated in the tests'
    helper): ranges of each (request, head) are disjoint, contiguous and
    cover exactly the visible blocks; combining the oracle's partials over
    them gives full attention."""
    from tests.splitk_partition import split_ranges
    rng = np.random.default_rng(20 + grid)
    L = [57, 0, 3, 100, 16, 1]
    p = problem(rng, L, [1 if x else 0 for x in L], Hq=4, Hkv=2, D=8, bs=4)
    q = rng.standard_normal((len(L), 4, 8))
    for window in (0, 9):
        ranges = split_ranges(L, window, 4, 2, grid, min_chunk, piece_units)
        S = max(len(r) for per in ranges for r in per) or 1
        # a segment's splits never outnumber ceil(n / min_chunk) + 1
        for b, per in enumerate(ranges):
            jlo, jhi = visible_block_range(L[b], window, 4)
            for splits in per:
                assert len(splits) <= -(-(jhi - jlo) // min_chunk) + 1
        for b, per in enumerate(ranges):
            jlo, jhi = visible_block_range(L[b], window, 4)
            for splits in per:
                covered = [j for (j0, j1) in splits for j in range(j0, j1)]
                assert covered == list(range(jlo, jhi))
        full, lf = paged_decode(q, p["k_pool"], p["v_pool"], p["block_tables"],
                                np.array(L), 0.5, 0.0, window)
        po, pl = splitk_partials(q, p["k_pool"], p["v_pool"], p["block_tables"], np.array(L),
                                 0.5, 0.0, window, S, ranges=ranges)
        out, lse = lse_combine(po, pl)
        np.testing.assert_allclose(out, full, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, lf, rtol=1e-12, atol=1e-13)


def test_golden_regression_anchor():
    """The oracle still reproduces the stored small case (tests/golden)."""
    import json
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "decode_small.json")
    d = json.load(open(path))
    out, lse = paged_attention(np.array(d["q"]), np.array(d["k_pool"]), np.array(d["v_pool"]),
                               np.array(d["block_tables"]), np.array(d["seq_lens"]),
                               np.array(d["query_start_loc"]), d["scale"], d["softcap"],
                               d["window"])
    np.testing.assert_allclose(out, np.array(d["out"]), rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(lse, np.array(d["lse"]), rtol=1e-13, atol=1e-15)
