"""The benchmark's reference arm (the fp64 oracle on the host) runs without a
GPU: check its JSON line against the harness contract, and the pure helpers
the GPU arm uses to count bytes and FLOPs against hand counts."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from paged_kv_attention_12_gb300 import workload  # noqa: E402


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [x for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "config", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["metric"] == bench.METRIC and d["unit"] == "GB/s" and d["higher_is_better"] is True
    assert d["value"] > 0 and d["steps"] == 1 and d["warmup"] == 1
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_step_bytes_count_each_visible_key_once():
    b = workload.make_batch(seq_lens=[40, 17], q_lens=[1, 1], num_q_heads=4, num_kv_heads=2,
                            head_dim=128, num_blocks=8, window=16, cfg_id=31)
    # window 16: the decode query at position L-1 sees keys L-16 .. L-1
    kv_row = 2 * 2 * 128 * 2  # K and V, Hkv heads, bf16
    want = (16 + 16) * kv_row + b.q.numel() * 2
    assert bench.batch_kv_bytes(b) == want


def test_attention_pairs_of_a_causal_chunk():
    b = workload.make_batch(seq_lens=[10], q_lens=[4], num_q_heads=1, num_kv_heads=1,
                            head_dim=128, num_blocks=2, cfg_id=32)
    # queries at positions 6..9 see 7, 8, 9, 10 keys
    assert bench.attention_pairs(b) == 7 + 8 + 9 + 10


def test_profile_traffic_is_read_only_for_the_current_kernel_source(tmp_path, monkeypatch):
    """bench.py takes roofline.traffic from the committed ncu summary only if
    the summary names the hash of the decode kernel's current source."""
    import bench
    h = bench.decode_source_hash()
    assert len(h) == 16
    p = tmp_path / "summary.md"
    monkeypatch.setattr(bench, "PROFILE_SUMMARY", str(p))
    p.write_text(f"# x\n\n- decode kernel source sha256[:16]: {h} (files)\n"
                 "- dram bytes per launch (avg): 93396736\n")
    assert bench.traffic_from_profile() == 93396736.0
    p.write_text("- decode kernel source sha256[:16]: 0123456789abcdef\n"
                 "- dram bytes per launch (avg): 93396736\n")
    assert bench.traffic_from_profile() is None
