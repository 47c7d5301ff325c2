"""GPU checks of paged_kv_append: bit-exact against the oracle, padding and
out-of-pool slots, and a decode over a cache the library appended to."""
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


def _bf16(shape, g):
    return torch.randn(shape, generator=g, device=DEV).to(torch.bfloat16)


@pytest.mark.parametrize("D,hkv,T", [(128, 1, 1), (128, 4, 33), (256, 2, 4096), (256, 8, 257)])
def test_append_bit_exact(D, hkv, T):
    g = torch.Generator(device=DEV).manual_seed(D + hkv + T)
    nb, bs = max(8, (T + 15) // 16 + 5), 16
    k_pool, v_pool = _bf16((nb, hkv, bs, D), g), _bf16((nb, hkv, bs, D), g)
    k_new, v_new = _bf16((T, hkv, D), g), _bf16((T, hkv, D), g)
    perm = torch.randperm(nb * bs, generator=torch.Generator().manual_seed(T))[:T]
    slots = perm.to(torch.int32)
    if T > 2:
        slots[1] = -1                                  # a padding token
    slots = slots.to(DEV)
    k_ref, v_ref = oracle.kv_append(k_pool.cpu().view(torch.int16).numpy(),
                                    v_pool.cpu().view(torch.int16).numpy(),
                                    k_new.cpu().view(torch.int16).numpy(),
                                    v_new.cpu().view(torch.int16).numpy(),
                                    slots.cpu().numpy(), bs)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.paged_kv_append(k_new, v_new, k_pool, v_pool, slots, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert np.array_equal(k_pool.cpu().view(torch.int16).numpy(), k_ref)
    assert np.array_equal(v_pool.cpu().view(torch.int16).numpy(), v_ref)


def test_slot_past_the_pool_is_reported_and_skipped():
    g = torch.Generator(device=DEV).manual_seed(7)
    k_pool, v_pool = _bf16((4, 2, 16, 128), g), _bf16((4, 2, 16, 128), g)
    k0, v0 = k_pool.clone(), v_pool.clone()
    k_new, v_new = _bf16((2, 2, 128), g), _bf16((2, 2, 128), g)
    slots = torch.tensor([64, 5], dtype=torch.int32, device=DEV)  # 64 = block 4: past the pool
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.paged_kv_append(k_new, v_new, k_pool, v_pool, slots, err)
    torch.cuda.synchronize()
    assert err.item() & binding.DEVERR_BAD_TABLE
    k0[0, :, 5], v0[0, :, 5] = k_new[1], v_new[1]
    assert torch.equal(k_pool, k0) and torch.equal(v_pool, v0)


def test_decode_over_appended_cache():
    """Append each request's newest token through the library, then decode:
    the result matches the oracle on the oracle-appended cache."""
    b = workload.make_batch(seq_lens=[37, 300, 16, 129], q_lens=[1, 1, 1, 1], num_q_heads=8,
                            num_kv_heads=2, head_dim=256, num_blocks=48, device=DEV, cfg_id=33,
                            seed=1)
    g = torch.Generator(device=DEV).manual_seed(3)
    k_new, v_new = _bf16((4, 2, 256), g), _bf16((4, 2, 256), g)
    tbl = b.tables_host
    pos = [L - 1 for L in b.seq_lens_host]
    slots = torch.tensor([int(tbl[i][p // 16]) * 16 + p % 16 for i, p in enumerate(pos)],
                         dtype=torch.int32, device=DEV)
    k_ref, v_ref = oracle.kv_append(b.k_pool.cpu().float().numpy(), b.v_pool.cpu().float().numpy(),
                                    k_new.cpu().float().numpy(), v_new.cpu().float().numpy(),
                                    slots.cpu().numpy(), 16)
    binding.paged_kv_append(k_new, v_new, b.k_pool, b.v_pool, slots)
    out = torch.empty_like(b.q)
    binding.paged_decode_attn(b.q, out, b.k_pool, b.v_pool, b.block_tables, b.seq_lens,
                              b.max_seq_len, scale=b.scale, softcap=b.softcap, window=b.window)
    # the oracle's view: the same batch over the oracle-appended pools (bf16
    # values, so the round trip through bf16 is exact)
    b_ref = workload.PagedBatch(**{**b.__dict__,
                                   "k_pool": torch.from_numpy(k_ref).to(torch.bfloat16),
                                   "v_pool": torch.from_numpy(v_ref).to(torch.bfloat16)})
    ref, _ = oracle.run_batch(workload.to_numpy_f64(b_ref))
    assert_close(to_f64(out), ref, "decode after append")
