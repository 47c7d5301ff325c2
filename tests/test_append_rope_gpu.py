"""GPU parity of the fused RMS-norm + RoPE append against the oracle.  The
outputs are bf16 roundings (to nearest even) of fp32 math, so each must lie
within one bf16 unit in the last place (2^-8 relative) of the fp64 value,
plus a small floor for values near zero; rows not named by a slot stay
bit-identical."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_12_gb300 import _build, binding


def assert_bf16_close(got, ref, what):
    err = np.abs(got - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-4
    assert np.isfinite(got).all(), what
    worst = np.max(err / bound)
    assert worst <= 1.0, f"{what}: error {worst:.3f} x the one-ulp bound"

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    binding.lib()


def _f64(x):
    return x.detach().float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("D,Hq,Hkv,rd,theta,norms", [
    (256, 8, 2, 256, 10000.0, True),      # local-layer style: full rotation, base 1e4
    (256, 8, 2, 64, 1e6, True),           # global-layer style: partial rotation, base 1e6
    (128, 16, 4, 128, 10000.0, False),    # no norms
    (128, 8, 8, 0, 10000.0, True),        # norms only
])
def test_append_rope_matches_oracle(D, Hq, Hkv, rd, theta, norms):
    T, nb, bs = 300, 64, 16
    g = torch.Generator(device=DEV).manual_seed(D + Hq + rd)
    bf = lambda *s: (torch.randn(s, generator=g, device=DEV) * 3.0).to(torch.bfloat16)
    q, k_new, v_new = bf(T, Hq, D), bf(T, Hkv, D), bf(T, Hkv, D)
    k_pool, v_pool = bf(nb, Hkv, bs, D), bf(nb, Hkv, bs, D)
    slots = torch.randperm(nb * bs, generator=torch.Generator().manual_seed(rd))[:T].to(torch.int32)
    slots[7] = -1
    positions = torch.randint(0, 131072, (T,), generator=torch.Generator().manual_seed(3),
                              dtype=torch.int32)
    wq = (torch.randn(D, generator=g, device=DEV) * 0.5 + 1.0) if norms else None
    wk = (torch.randn(D, generator=g, device=DEV) * 0.5 + 1.0) if norms else None
    ref_q, ref_k, ref_v = oracle.kv_append_rope(
        _f64(q), _f64(k_pool), _f64(v_pool), _f64(k_new), _f64(v_new), slots.numpy(),
        positions.numpy(), None if wq is None else _f64(wq), None if wk is None else _f64(wk),
        norms, 1e-6, theta, rd, bs)
    k0, v0 = k_pool.clone(), v_pool.clone()
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    binding.paged_kv_append_rope(q, k_new, v_new, k_pool, v_pool, slots.to(DEV),
                                 positions.to(DEV), q_norm_weight=wq, k_norm_weight=wk,
                                 v_norm=norms, eps=1e-6, rope_theta=theta, rotary_dim=rd, err=err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert_bf16_close(_f64(q), ref_q, "q")
    written = np.zeros((nb, bs), dtype=bool)
    s = slots.numpy()
    written[s[s >= 0] // bs, s[s >= 0] % bs] = True
    for name, got, ref, before in (("k", k_pool, ref_k, k0), ("v", v_pool, ref_v, v0)):
        g64 = _f64(got)
        assert_bf16_close(g64.transpose(0, 2, 1, 3)[written], ref.transpose(0, 2, 1, 3)[written],
                          name)
        untouched = ~torch.from_numpy(written).to(DEV)
        assert torch.equal(got.permute(0, 2, 1, 3)[untouched], before.permute(0, 2, 1, 3)[untouched])
