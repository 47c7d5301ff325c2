"""Pins of the H2O key-mass oracle: per (request, KV head) the step adds G
(each head's probabilities sum to one) over exactly the visible keys;
identical keys share the mass equally; a dominant key takes it all; and
each head's share matches the attention oracle's weights recovered from
one-hot values."""
import numpy as np

import oracle


def _case(seed=0, B=3, Hq=8, Hkv=2, D=16, L=(37, 5, 80), window=0, softcap=0.0):
    rng = np.random.default_rng(seed)
    nblk = sum(-(-x // 16) for x in L) + 2
    k_pool = rng.standard_normal((nblk, Hkv, 16, D))
    perm = rng.permutation(nblk)
    tables, o = [], 0
    for x in L:
        n = -(-x // 16)
        tables.append(list(perm[o:o + n]))
        o += n
    q = rng.standard_normal((B, Hq, D))
    return q, k_pool, tables, np.array(L)


def test_mass_sums_to_group_size_over_visible_keys():
    q, k, t, L = _case()
    for window in (0, 9):
        m = oracle.key_mass(q, k, t, L, 0.25, window=window, num_keys=96)
        for b in range(3):
            vis = oracle.visible_keys(L[b] - 1, L[b], window)
            for kvh in range(2):
                assert abs(m[b, kvh].sum() - 4.0) < 1e-12
                outside = np.setdiff1d(np.arange(96), vis)
                assert not m[b, kvh, outside].any()


def test_identical_keys_share_equally():
    q, k, t, L = _case(seed=1)
    k[:] = k[0, 0, 0]
    m = oracle.key_mass(q, k, t, L, 0.3, num_keys=80)
    for b in range(3):
        assert np.allclose(m[b, :, :L[b]], 4.0 / L[b], atol=1e-12)


def test_dominant_key_takes_the_mass():
    q, k, t, L = _case(seed=2, L=(40, 40, 40))
    b, tstar = 1, 17
    blk, off = t[b][tstar // 16], tstar % 16
    for kvh in range(2):
        q[b, kvh * 4:(kvh + 1) * 4] = q[b, kvh * 4]  # the group's heads agree
        k[blk, kvh, off] = 50.0 * q[b, kvh * 4]
    m = oracle.key_mass(q, k, t, L, 1.0, num_keys=40)
    assert np.allclose(m[b, :, tstar], 4.0, atol=1e-9)


def test_matches_attention_weights_read_through_one_hot_values():
    """With V = one-hot rows of key positions, attention's output row h is
    head h's probability vector; summing a group's rows gives the mass."""
    q, k, t, L = _case(seed=3, L=(20, 33, 7), softcap=0.0)
    nblk, Hkv, bs, _ = k.shape
    num_keys = 48
    v = np.zeros((nblk, Hkv, bs, num_keys))
    for b in range(3):
        for tok in range(L[b]):
            v[t[b][tok // 16], :, tok % 16, tok] = 1.0
    width = max(len(r) for r in t)
    bt = np.full((3, width), -1)
    for b, r in enumerate(t):
        bt[b, :len(r)] = r
    for window, cap in ((0, 0.0), (11, 3.0)):
        out, _ = oracle.paged_decode(q, k, v, bt, L, 0.4, softcap=cap, window=window)
        m = oracle.key_mass(q, k, t, L, 0.4, softcap=cap, window=window, num_keys=num_keys)
        for b in range(3):
            for kvh in range(2):
                assert np.allclose(out[b, kvh * 4:(kvh + 1) * 4].sum(0), m[b, kvh], atol=1e-12)
