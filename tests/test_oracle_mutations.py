"""Plant one mistake at a time in a copy of the oracle; the pins must catch each.

Runs on the CPU only.  Every mutation is a plausible slip (window off by one,
wrong GQA grouping, cap applied to the unscaled logit, dropped scale, wrong
slot in the table walk, causal offset, wrong LSE, wrong combine weights, split
ranges not anchored at the visible start) and must make the pin suite fail.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = [
    ("window off by one", "keep &= t > pos - window", "keep &= t >= pos - window"),
    ("GQA as h % Hkv", "heads = slice(kvh * G, (kvh + 1) * G)", "heads = slice(kvh, Hq, Hkv)"),
    ("cap on unscaled ratio", "s = softcap * np.tanh(s / softcap)", "s = softcap * np.tanh(s)"),
    ("dropped scale", "s = scale * (keys @ q_rows.T)", "s = (keys @ q_rows.T)"),
    ("wrong slot", "t % block_size, :]", "(t + 1) % block_size, :]"),
    ("causal offset", "pos = L - n + i", "pos = L - n + i - 1"),
    ("half LSE", "lse = m + np.log(l)", "lse = m + 0.5 * np.log(l)"),
    ("combine weights squared", "np.exp(partial_lse - Ms[..., None])",
     "np.exp(2.0 * (partial_lse - Ms[..., None]))"),
    ("splits not anchored", "j0 = jlo + s * split_blocks", "j0 = s * split_blocks"),
]


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_planted_mistake(tmp_path, name, old, new):
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle",
                    ignore=shutil.ignore_patterns("__pycache__", "*.so", "*.o"))
    (tmp_path / "tests").mkdir()
    for f in ("conftest.py", "problems.py", "test_oracle_pins.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), tmp_path / "tests" / f)
    src = (tmp_path / "oracle" / "paged_attention.py").read_text()
    assert src.count(old) >= 1, f"mutation site for {name!r} not found"
    (tmp_path / "oracle" / "paged_attention.py").write_text(src.replace(old, new))
    env = dict(os.environ, PYTHONPATH=str(tmp_path), PYTHONDONTWRITEBYTECODE="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_oracle_pins.py"], cwd=tmp_path, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"pins did not catch {name!r}:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout


APPEND_MUTATIONS = [
    ("block and offset swapped", "blk, off = divmod(int(s), block_size)",
     "off, blk = divmod(int(s), block_size)"),
    ("padding not skipped", "if s < 0:\n            continue", "if s < -1:\n            continue"),
    ("K and V crossed", "v_out[blk, :, off, :] = v_new[t]", "v_out[blk, :, off, :] = k_new[t]"),
    ("head axis dropped", "k_out[blk, :, off, :] = k_new[t]", "k_out[blk, 0, off, :] = k_new[t][0]"),
]


@pytest.mark.parametrize("name,old,new", APPEND_MUTATIONS, ids=[m[0] for m in APPEND_MUTATIONS])
def test_append_pins_catch_planted_mistake(tmp_path, name, old, new):
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle",
                    ignore=shutil.ignore_patterns("__pycache__", "*.so", "*.o"))
    (tmp_path / "tests").mkdir()
    for f in ("conftest.py", "test_oracle_kv_append.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), tmp_path / "tests" / f)
    src = (tmp_path / "oracle" / "kv_append.py").read_text()
    assert src.count(old) >= 1, f"mutation site for {name!r} not found"
    (tmp_path / "oracle" / "kv_append.py").write_text(src.replace(old, new))
    env = dict(os.environ, PYTHONPATH=str(tmp_path), PYTHONDONTWRITEBYTECODE="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_oracle_kv_append.py"], cwd=tmp_path, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"pins did not catch {name!r}:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout


MASS_MUTATIONS = [
    ("unnormalised probabilities", "mass[b, kvh, keys] += p / p.sum()", "mass[b, kvh, keys] += p"),
    ("cap ignored", "s = softcap * np.tanh(s / softcap)", "s = s"),
    ("window ignored", "keys = visible_keys(L - 1, L, window)", "keys = visible_keys(L - 1, L, 0)"),
    ("heads grouped by stride", "q[b, kvh * G + g]", "q[b, kvh + g * Hkv]"),
]


@pytest.mark.parametrize("name,old,new", MASS_MUTATIONS, ids=[m[0] for m in MASS_MUTATIONS])
def test_key_mass_pins_catch_planted_mistake(tmp_path, name, old, new):
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle",
                    ignore=shutil.ignore_patterns("__pycache__", "*.so", "*.o"))
    (tmp_path / "tests").mkdir()
    for f in ("conftest.py", "test_oracle_key_mass.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), tmp_path / "tests" / f)
    src = (tmp_path / "oracle" / "key_mass.py").read_text()
    assert src.count(old) >= 1, f"mutation site for {name!r} not found"
    (tmp_path / "oracle" / "key_mass.py").write_text(src.replace(old, new))
    env = dict(os.environ, PYTHONPATH=str(tmp_path), PYTHONDONTWRITEBYTECODE="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_oracle_key_mass.py"], cwd=tmp_path, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"pins did not catch {name!r}:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout


ROPE_MUTATIONS = [
    ("pairs adjacent instead of halves", "x1, x2 = x[..., :half], x[..., half:rotary_dim]",
     "x1, x2 = x[..., 0:rotary_dim:2], x[..., 1:rotary_dim:2]"),
    ("sine sign flipped", "out[..., :half] = x1 * c - x2 * s", "out[..., :half] = x1 * c + x2 * s"),
    ("frequency exponent over D/2", "theta ** (-2.0 * i / rotary_dim)", "theta ** (-1.0 * i / rotary_dim)"),
    ("norm by mean absolute value", "np.mean(x * x, axis=-1, keepdims=True)",
     "np.mean(np.abs(x), axis=-1, keepdims=True) ** 2"),
]


@pytest.mark.parametrize("name,old,new", ROPE_MUTATIONS, ids=[m[0] for m in ROPE_MUTATIONS])
def test_rope_norm_pins_catch_planted_mistake(tmp_path, name, old, new):
    shutil.copytree(os.path.join(ROOT, "oracle"), tmp_path / "oracle",
                    ignore=shutil.ignore_patterns("__pycache__", "*.so", "*.o"))
    (tmp_path / "tests").mkdir()
    for f in ("conftest.py", "test_oracle_rope_norm.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), tmp_path / "tests" / f)
    src = (tmp_path / "oracle" / "rope_norm.py").read_text()
    assert src.count(old) >= 1, f"mutation site for {name!r} not found"
    (tmp_path / "oracle" / "rope_norm.py").write_text(src.replace(old, new))
    env = dict(os.environ, PYTHONPATH=str(tmp_path), PYTHONDONTWRITEBYTECODE="1")
    r = subprocess.run([sys.executable, "-m", "pytest", "-q", "-x", "-p", "no:cacheprovider",
                        "tests/test_oracle_rope_norm.py"], cwd=tmp_path, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 1, f"pins did not catch {name!r}:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout
