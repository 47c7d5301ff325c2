"""Oracle of the per-head math before attention (TEST INFRASTRUCTURE; see the
package doc): RMS norm of q, k (learned weight) and v (unit weight), rotary
position embedding of q and k, then the KV append.

"Custom Gemma 4 forward -- Dual-RoPE, GQA with QK/V-norm + KV sharing"
(github README, "What's inside").  The pages give no formulas; the readings:
RMS norm x / sqrt(mean(x^2) + eps) * w per head over the D channels; RoPE in
the rotate-half form (channel i pairs with i + r/2, angle pos * base^(-2i/r)
for i < r/2, channels >= r untouched); "dual" = two such rotations with their
own base and width (one call each).
"""
from __future__ import annotations

import numpy as np

from .kv_append import kv_append


def rms_norm(x: np.ndarray, weight, eps: float) -> np.ndarray:
    """Over the last axis: x / sqrt(mean(x^2) + eps) * weight (None = 1)."""
    x = np.asarray(x, dtype=np.float64)
    y = x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps)
    return y if weight is None else y * np.asarray(weight, dtype=np.float64)


def rope(x: np.ndarray, pos, theta: float, rotary_dim: int) -> np.ndarray:
    """Rotate-half RoPE of the last axis of ``x`` ([..., D]) at positions
    ``pos`` (broadcast against the leading axes)."""
    x = np.asarray(x, dtype=np.float64)
    if rotary_dim == 0:
        return x.copy()
    half = rotary_dim // 2
    i = np.arange(half)
    ang = np.asarray(pos, dtype=np.float64)[..., None] * theta ** (-2.0 * i / rotary_dim)
    c, s = np.cos(ang), np.sin(ang)
    out = x.copy()
    x1, x2 = x[..., :half], x[..., half:rotary_dim]
    out[..., :half] = x1 * c - x2 * s
    out[..., half:rotary_dim] = x2 * c + x1 * s
    return out


def kv_append_rope(q, k_pool, v_pool, k_new, v_new, slot_mapping, positions, q_norm_w,
                   k_norm_w, v_norm, eps, theta, rotary_dim, block_size):
    """(q', k_pool', v_pool'): q [T][Hq][D] normalised and rotated; k/v rows
    normalised (k rotated) and appended at their slots."""
    pos = np.asarray(positions)
    qo = None
    if q is not None:
        qo = np.asarray(q, dtype=np.float64)
        if q_norm_w is not None:
            qo = rms_norm(qo, q_norm_w, eps)
        qo = rope(qo, pos[:, None], theta, rotary_dim)
    k = np.asarray(k_new, dtype=np.float64)
    if k_norm_w is not None:
        k = rms_norm(k, k_norm_w, eps)
    k = rope(k, pos[:, None], theta, rotary_dim)
    v = np.asarray(v_new, dtype=np.float64)
    if v_norm:
        v = rms_norm(v, None, eps)
    kp, vp = kv_append(np.asarray(k_pool, dtype=np.float64), np.asarray(v_pool, dtype=np.float64),
                       k, v, slot_mapping, block_size)
    return qo, kp, vp
