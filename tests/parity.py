"""Parity helpers: compare CUDA outputs with the fp64 oracle.

Tolerances (bf16 inputs, fp32 accumulation, bf16 output): max-abs error
<= 2e-2 and relative L2 error <= 5e-3 against the fp64 oracle.
"""
from __future__ import annotations

import numpy as np

MAX_ABS = 2e-2
REL_L2 = 5e-3


def errors(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    diff = got - ref
    max_abs = float(np.max(np.abs(diff))) if diff.size else 0.0
    den = float(np.linalg.norm(ref.ravel()))
    rel = float(np.linalg.norm(diff.ravel()) / den) if den > 0 else float(np.linalg.norm(diff.ravel()))
    return max_abs, rel


def assert_close(got, ref, what="", max_abs=MAX_ABS, rel_l2=REL_L2):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output (stray read of a poisoned slot?)"
    ma, rl = errors(got, ref)
    assert ma <= max_abs and rl <= rel_l2, f"{what}: max_abs={ma:.3e} rel_l2={rl:.3e}"
    return ma, rl


def to_f64(t):
    return t.float().cpu().numpy().astype(np.float64)
