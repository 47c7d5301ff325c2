"""Pins of the KV-append oracle: what it writes is exactly what the
attention oracle's block-table gather reads back, nothing else moves,
padding tokens are skipped, and a hand-worked case."""
import numpy as np

import oracle


def _pools(num_blocks=6, hkv=2, bs=4, d=3, seed=0):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((num_blocks, hkv, bs, d)), rng.standard_normal((num_blocks, hkv, bs, d))


def test_hand_worked_case():
    k = np.zeros((2, 1, 2, 1))
    v = np.zeros((2, 1, 2, 1))
    k_new = np.array([[[1.0]], [[2.0]], [[3.0]]])
    v_new = -k_new
    # slots: token 0 -> block 1 offset 1, token 1 skipped, token 2 -> block 0 offset 0
    k2, v2 = oracle.kv_append(k, v, k_new, v_new, np.array([3, -1, 0]), block_size=2)
    assert k2[:, 0, :, 0].tolist() == [[3.0, 0.0], [0.0, 1.0]]
    assert v2[:, 0, :, 0].tolist() == [[-3.0, 0.0], [0.0, -1.0]]
    assert not k.any()  # inputs untouched


def test_appended_tokens_read_back_through_the_block_table():
    """Request with blocks [4, 1, 5]: its tokens 5..9 appended by slot; the
    attention oracle's gather must return exactly the appended rows."""
    bs = 4
    k, v = _pools(bs=bs)
    table = np.array([4, 1, 5])
    pos = np.arange(5, 10)
    slots = table[pos // bs] * bs + pos % bs
    rng = np.random.default_rng(1)
    k_new = rng.standard_normal((5, 2, 3))
    v_new = rng.standard_normal((5, 2, 3))
    k2, v2 = oracle.kv_append(k, v, k_new, v_new, slots, bs)
    kc = oracle.gather_request_kv(k2, table, 10, bs)
    vc = oracle.gather_request_kv(v2, table, 10, bs)
    assert np.array_equal(kc[5:10], k_new) and np.array_equal(vc[5:10], v_new)
    # the request's older tokens are where they were
    assert np.array_equal(kc[:5], oracle.gather_request_kv(k, table, 10, bs)[:5])


def test_only_the_named_slots_change():
    bs = 4
    k, v = _pools(bs=bs)
    slots = np.array([7, -1, 21, 2])
    rng = np.random.default_rng(2)
    k_new = rng.standard_normal((4, 2, 3))
    v_new = rng.standard_normal((4, 2, 3))
    k2, v2 = oracle.kv_append(k, v, k_new, v_new, slots, bs)
    changed = {(b, o) for b in range(6) for o in range(bs) if not np.array_equal(k2[b, :, o], k[b, :, o])}
    assert changed == {(1, 3), (5, 1), (0, 2)}
    assert {(b, o) for b in range(6) for o in range(bs)
            if not np.array_equal(v2[b, :, o], v[b, :, o])} == changed


def test_slot_past_the_pool_is_skipped():
    k, v = _pools(num_blocks=2, bs=4)
    k2, v2 = oracle.kv_append(k, v, np.ones((1, 2, 3)), np.ones((1, 2, 3)), np.array([8]), 4)
    assert np.array_equal(k2, k) and np.array_equal(v2, v)
