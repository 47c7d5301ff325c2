"""GPU parity of the H2O key mass (split-K logits + LSE -> per-key attention
probability summed over each KV head's query heads) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_12_gb300 import _build, binding, workload
from tests.parity import assert_close, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    binding.lib()


def run_mass(b, prior=None):
    r = binding.DecodeSplitK(b)
    B, Hq = b.num_requests, b.num_q_heads
    nk = b.block_tables.shape[1] * 16
    logits = torch.full((B, Hq, nk), float("nan"), device=DEV)
    lse = torch.empty((B, Hq), device=DEV)
    mass = prior.clone() if prior is not None else torch.zeros((B, b.num_kv_heads, nk), device=DEV)
    binding.paged_decode_splitk_logits(b.q, r.partial_o, r.partial_lse, logits, b.k_pool,
                                       b.v_pool, b.block_tables, b.seq_lens, b.max_seq_len,
                                       r.num_splits, r.split_blocks, scale=b.scale,
                                       softcap=b.softcap, window=b.window)
    binding.paged_decode_splitk_combine(r.partial_o, r.partial_lse, r.out, lse)
    binding.paged_decode_key_mass(logits, lse, b.seq_lens, b.num_kv_heads, mass, window=b.window)
    torch.cuda.synchronize()
    return r.out, mass


def oracle_mass(b):
    arr = workload.to_numpy_f64(b)
    return oracle.key_mass(arr["q"], arr["k_pool"], arr["block_tables"], arr["seq_lens"],
                           b.scale, b.softcap, b.window, 16, b.block_tables.shape[1] * 16)


@pytest.mark.parametrize("cfg", [1, 2, 3])
def test_key_mass_matches_oracle(cfg):
    for b in workload.workload(cfg, seed=0, device=DEV, poison=True, scale_down=True):
        out, mass = run_mass(b)
        ref = oracle_mass(b)
        got = mass.double().cpu().numpy()
        assert np.isfinite(got).all()
        assert np.abs(got - ref).max() < 2e-3, (b.name, np.abs(got - ref).max())
        G = b.num_q_heads // b.num_kv_heads
        sums = got.sum(-1)
        live = np.array(b.seq_lens_host) > 0
        assert np.allclose(sums[live], G, atol=5e-3)
        # the decode output is untouched by storing the logits
        arr = workload.to_numpy_f64(b)
        want, _ = oracle.run_batch(arr)
        assert_close(to_f64(out), want, f"{b.name} output with logits")


def test_key_mass_accumulates():
    b = workload.decode_tiny(1, DEV)
    _, m1 = run_mass(b)
    _, m2 = run_mass(b, prior=m1)
    assert torch.allclose(m2, 2 * m1, rtol=1e-6, atol=1e-7)
