"""The allocation-free decode entry point (collected last on purpose).

``paged_decode_attn_noalloc`` serves callers that cannot allocate device
memory: it keeps the split-K partials in an array compiled into the library.
These tests call it through the C ABI and compare it with the fp64 oracle and
with the regular split-K path (caller-owned workspace) on two calls in a
row, so a stale array from the first call would show up in the second.
"""
import ctypes

import pytest
import torch

import oracle
from paged_kv_attention_12_gb300 import _build, binding, workload
from tests.parity import assert_close, to_f64

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    binding.lib()


def _noalloc(batch, err=None):
    out = torch.full_like(batch.q, float("nan"))
    binding.paged_decode_attn_noalloc(batch.q, out, batch.k_pool, batch.v_pool,
                                      batch.block_tables, batch.seq_lens, batch.max_seq_len,
                                      scale=batch.scale, softcap=batch.softcap,
                                      window=batch.window, err=err)
    return out


@pytest.mark.gpu
def test_noalloc_matches_split_k_on_two_calls_in_a_row():
    batches = workload.decode_serving(0, DEV, poison=True) + \
        [workload.decode_long(1, DEV, poison=True, scale_down=True)]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for batch in batches:
        want = to_f64(binding.DecodeSplitK(batch).run())
        for call in range(2):
            got = _noalloc(batch, err)
            torch.cuda.synchronize()
            assert err.item() == 0, f"{batch.name} call {call}: device error word {err.item()}"
            assert_close(to_f64(got), want, f"{batch.name} call {call}")


@pytest.mark.gpu
def test_noalloc_matches_oracle_on_two_calls_in_a_row():
    batches = workload.decode_serving(2, DEV, poison=True, scale_down=True) + \
        [workload.decode_long(2, DEV, poison=True, scale_down=True),
         workload.decode_tiny(2, DEV, poison=True)]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    for batch in batches:
        want, _ = oracle.run_batch(workload.to_numpy_f64(batch))
        for call in range(2):
            got = _noalloc(batch, err)
            torch.cuda.synchronize()
            assert err.item() == 0, f"{batch.name} call {call}: device error word {err.item()}"
            assert_close(to_f64(got), want, f"{batch.name} call {call} vs oracle")


def test_noalloc_rejects_partials_beyond_its_array():
    # 256 requests x 32 heads x 33 slots x 257 floats > 16 MiB: refused before any launch
    L = binding.lib()
    pool = binding.PkaKvPool(16, 16, 1 << 20, 4, 16, 256)
    par = binding.PkaAttnParams(0.1, 0.0, 0, None)
    st = L.paged_decode_attn_noalloc(16, 16, ctypes.byref(pool), 16, 256, 16, 256, 32, 4096,
                                     ctypes.byref(par), None)
    assert st == -5  # PKA_ERR_WORKSPACE
