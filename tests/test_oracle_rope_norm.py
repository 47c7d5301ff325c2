"""Pins of the RMS-norm / RoPE oracle against what the mathematics fixes:
a rotation keeps norms and is the identity at position 0, attention logits
of rotated q and k depend only on the position difference, a hand-worked
rotation, unit RMS after the norm, and the fused append's placement."""
import numpy as np

import oracle


def test_rotation_keeps_norm_and_is_identity_at_zero():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((5, 64))
    for r in (64, 32, 16):
        y = oracle.rope(x, np.arange(5) * 97, 10000.0, r)
        assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), atol=1e-12)
        assert np.array_equal(y[:, r:], x[:, r:])
        assert np.allclose(oracle.rope(x, np.zeros(5), 10000.0, r), x, atol=0)


def test_logits_depend_only_on_relative_position():
    rng = np.random.default_rng(1)
    a, b = rng.standard_normal(128), rng.standard_normal(128)
    for theta in (10000.0, 1e6):
        for r in (128, 64):
            ref = oracle.rope(a, 700, theta, r) @ oracle.rope(b, 500, theta, r)
            for shift in (1, 37, 100000):
                got = oracle.rope(a, 700 + shift, theta, r) @ oracle.rope(b, 500 + shift, theta, r)
                assert abs(got - ref) < 1e-8


def test_hand_worked_rotation():
    # D = r = 4, base 100: pairs (0, 2) turn by p, (1, 3) by p / 10
    x = np.array([1.0, 2.0, 3.0, 4.0])
    p = 0.5
    y = oracle.rope(x, p, 100.0, 4)
    c0, s0, c1, s1 = np.cos(p), np.sin(p), np.cos(p / 10), np.sin(p / 10)
    want = [1 * c0 - 3 * s0, 2 * c1 - 4 * s1, 3 * c0 + 1 * s0, 4 * c1 + 2 * s1]
    assert np.allclose(y, want, atol=1e-15)


def test_rms_norm_unit_rms_and_weight():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 4, 128)) * 7.0
    y = oracle.rms_norm(x, None, 0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 1.0, atol=1e-12)
    w = rng.standard_normal(128)
    assert np.allclose(oracle.rms_norm(x, w, 0.0), y * w, atol=1e-12)
    assert np.allclose(oracle.rms_norm(3.0 * x, None, 0.0), y, atol=1e-12)  # scale-free


def test_fused_append_places_normed_rotated_rows():
    rng = np.random.default_rng(3)
    T, Hq, Hkv, D, bs = 3, 4, 2, 32, 4
    q = rng.standard_normal((T, Hq, D))
    k_new, v_new = rng.standard_normal((T, Hkv, D)), rng.standard_normal((T, Hkv, D))
    k_pool, v_pool = np.zeros((4, Hkv, bs, D)), np.zeros((4, Hkv, bs, D))
    wq, wk = rng.standard_normal(D), rng.standard_normal(D)
    slots, pos = np.array([5, -1, 14]), np.array([9, 10, 11])
    qo, kp, vp = oracle.kv_append_rope(q, k_pool, v_pool, k_new, v_new, slots, pos, wq, wk, True,
                                       1e-6, 10000.0, 16, bs)
    for t, s in ((0, 5), (2, 14)):
        blk, off = divmod(s, bs)
        want_k = oracle.rope(oracle.rms_norm(k_new[t], wk, 1e-6), pos[t], 10000.0, 16)
        assert np.allclose(kp[blk, :, off], want_k, atol=1e-12)
        assert np.allclose(vp[blk, :, off], oracle.rms_norm(v_new[t], None, 1e-6), atol=1e-12)
    assert np.count_nonzero(kp.any(axis=(1, 3))) == 2  # token 1 (slot -1) not written
    assert np.allclose(qo[1], oracle.rope(oracle.rms_norm(q[1], wq, 1e-6), 10, 10000.0, 16))
