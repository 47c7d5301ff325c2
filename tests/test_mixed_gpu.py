"""GPU parity of the mixed-batch launch with a workspace
(``paged_prefill_attn_ws``): decode rows on the decode pipelines, chunks on
the tensor-core prefill pipeline, one launch, against the oracle."""
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


def counters(runner):
    """Arrival counters of the workspace (the fused decode's layout)."""
    b = runner.batch
    S, _ = binding.paged_decode_splitk_plan(b.num_requests, b.num_kv_heads, b.max_seq_len, 16,
                                            b.window)
    B, Hq, D, Hkv = b.num_requests, b.num_q_heads, b.head_dim, b.num_kv_heads
    off = B * Hq * S * D * 4 + (B * Hq * S * 4 + 15) // 16 * 16
    assert runner.workspace.numel() == off + (B * Hkv * 4 + 15) // 16 * 16
    return runner.workspace[off:off + B * Hkv * 4].view(torch.int32)


def check(batch, what, reqs=None, calls=2):
    runner = binding.MixedBatch(batch)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    runner.out.fill_(float("nan"))
    outs = []
    for _ in range(calls):
        outs.append(runner.run(err).clone())
    arr = workload.to_numpy_f64(batch, reqs)
    ref, _ = oracle.run_batch(arr)
    got = outs[0][arr["q_rows"]] if reqs is not None else outs[0]
    assert_close(to_f64(got), ref, what)
    torch.cuda.synchronize()
    assert err.item() == 0, f"{what}: device error word {err.item()}"
    for o in outs[1:]:
        assert torch.equal(o, outs[0]), f"{what}: repeated call differs"
    assert torch.all(counters(runner) == 0), "arrival counters must be left zero"
    return outs[0]


def small(seq_lens, q_lens, D=256, G=4, Hkv=2, **kw):
    return workload.make_batch(seq_lens=seq_lens, q_lens=q_lens, num_q_heads=G * Hkv,
                               num_kv_heads=Hkv, head_dim=D,
                               num_blocks=kw.pop("num_blocks", sum(-(-L // 16) for L in seq_lens) + 8),
                               device=DEV, poison=True, cfg_id=kw.pop("cfg_id", 31), **kw)


@pytest.mark.parametrize("seed", range(3))
def test_mixed_batch_small(seed):
    b = workload.mixed_batch(seed, DEV, poison=True, scale_down=True, drop_out_of_window=True)
    check(b, f"cfg5 small {seed}")


@pytest.mark.parametrize("D,G", [(128, 1), (128, 4), (128, 8), (256, 1), (256, 2), (256, 4),
                                 (256, 8)])
def test_shapes(D, G):
    L = [900, 33, 1, 300, 16, 17, 250]
    n = [1, 1, 1, 120, 16, 1, 40]
    check(small(L, n, D=D, G=G, Hkv=2 if G < 8 else 1, seed=D + G), f"D={D} G={G}")


@pytest.mark.parametrize("window,softcap", [(0, 0.0), (0, 50.0), (64, 0.0), (300, 30.0)])
def test_window_and_softcap(window, softcap):
    L = [1200, 700, 90, 2, 333, 64]
    n = [1, 1, 1, 1, 100, 64]
    check(small(L, n, window=window, softcap=softcap, seed=window + int(softcap)),
          f"W={window} cap={softcap}")


@pytest.mark.parametrize("scale", [0.0, -0.0625])
@pytest.mark.parametrize("softcap", [0.0, 50.0])
def test_zero_and_negative_scale(scale, softcap):
    """Both pipelines of the launch take any finite scale (at 0 each row is
    the mean of the V rows it sees)."""
    L = [1200, 700, 90, 333, 64]
    n = [1, 1, 1, 100, 64]
    check(small(L, n, softcap=softcap, scale=scale, seed=8), f"scale={scale} cap={softcap}")


def test_only_decode_rows():
    L = [int(x) for x in np.random.default_rng(3).integers(1, 2000, 40)]
    check(small(L, [1] * len(L), softcap=50.0, window=256, seed=3), "decode rows only")


def test_only_prefill_chunks():
    check(small([500, 200, 64], [200, 200, 64], seed=4), "prefill chunks only")


def test_empty_requests_between_rows():
    """Requests with no query rows (q_len 0) sit between decode rows and
    chunks: nothing is written for them and the others are unaffected."""
    L = [100, 40, 300, 50, 17]
    n = [1, 0, 60, 0, 1]
    check(small(L, n, seed=6), "empty requests")


def test_matches_single_pipeline_launch():
    """Same batch through paged_prefill_attn (every row on the tensor-core
    pipeline): both agree with the oracle, hence with each other."""
    b = workload.mixed_batch(1, DEV, poison=True, scale_down=True, drop_out_of_window=True)
    a = check(b, "ws path")
    c = binding.run_batch(b)
    ref, _ = oracle.run_batch(workload.to_numpy_f64(b))
    assert_close(to_f64(c), ref, "single-pipeline path")
    assert_close(to_f64(a), to_f64(c), "ws vs single-pipeline")


def test_full_size_mixed_sampled_requests():
    """The mixed workload at full size in the benchmark's launch, checked on
    decode requests (shared prefix and not) and on every prefill chunk."""
    batch = workload.workload(5, seed=0, device=DEV, poison=True)[0]
    B = batch.num_requests
    reqs = [0, 17, 31, 32, 50, 63, 64, 65, 66, B - 1]
    check(batch, "cfg5 full size", reqs=reqs)
