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


SPLIT_SLOTS = 160  # prefill pieces the workspace holds (include/paged_attn.h)


def counters(runner):
    """Arrival counters of the workspace: the decode segments' (the fused
    decode's layout), then the prefill pieces' after their rows and LSEs."""
    b = runner.batch
    S, _ = binding.paged_decode_splitk_plan(b.num_requests, b.num_kv_heads, b.max_seq_len, 16,
                                            b.window)
    B, Hq, D, Hkv = b.num_requests, b.num_q_heads, b.head_dim, b.num_kv_heads
    off = B * Hq * S * D * 4 + (B * Hq * S * 4 + 15) // 16 * 16
    dec_end = off + (B * Hkv * 4 + 15) // 16 * 16
    poff = dec_end + SPLIT_SLOTS * 128 * (D + 1) * 4
    assert runner.workspace.numel() == poff + (SPLIT_SLOTS * 4 + 15) // 16 * 16
    ws = runner.workspace
    return torch.cat([ws[off:off + B * Hkv * 4].view(torch.int32),
                      ws[poff:poff + SPLIT_SLOTS * 4].view(torch.int32)])


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


def expected_pieces(batch):
    """Pieces per prefill item the header's rule gives for this batch on
    this GPU (every item's key tiles, the wave of SMs the decode CTAs leave),
    restated from the paged_prefill_attn_ws comment."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    L = batch.seq_lens.tolist()
    qsl = batch.query_start_loc.tolist()
    B, Hkv, D = batch.num_requests, batch.num_kv_heads, batch.head_dim
    G = batch.num_q_heads // Hkv
    pair = D == 256  # CTA pairs: two query tiles per item, 128-key tiles
    TQ = 128 // G * (2 if pair else 1)
    BN = 128
    W = batch.window
    tiles = []
    for r in range(B):
        n = qsl[r + 1] - qsl[r]
        if n <= 1 or n > L[r]:
            continue
        for qt in range(-(-n // TQ)):
            p_first = L[r] - n + qt * TQ
            p_last = L[r] - n + min(n, (qt + 1) * TQ) - 1
            t_lo = max(0, p_first - W + 1) if W > 0 else 0
            tiles.append(-(-(p_last + 1 - (t_lo // 16) * 16) // BN))
    # the SMs left to the prefill items (the host's split of the SMs)
    extra = qsl[-1] - B
    tq = 128 // G  # the host's estimate: one-CTA tiles, 64 keys at D = 256
    bn = 64 if D == 256 else 128
    est = -(-extra // tq) * Hkv if extra > 0 else 0
    mql, msl = batch.max_query_len, batch.max_seq_len
    keys = min(msl, W + tq) if W > 0 else msl
    prefill_us = est * (-(-keys // bn) + 1) * 2.0
    chunks = -(-extra // (mql - 1)) if extra > 0 and mql > 1 else 0
    dec_rows = max(0, B - chunks)
    dec_keys = min(msl, W) if W > 0 else msl
    decode_us = dec_rows * Hkv * (-(-dec_keys // 16)) * (64.0 * D) / 70.0e3
    wave = 0
    if est > 0:
        share = int(sms * prefill_us / (prefill_us + decode_us) + 0.5)
        wave = share if share >= 2 * est else est
        wave = min(max(wave, 1), sms - sms // 4)
    slots, piece_slots = wave, SPLIT_SLOTS
    if pair and est > 0:
        dec = max(1, sms - wave)
        dec -= dec % 2  # an even number of decode CTAs before the pairs
        slots, piece_slots = (sms - dec) // 2, SPLIT_SLOTS // 2
    items = len(tiles) * Hkv
    if not (0 < items < slots and items <= piece_slots):
        return [1] * len(tiles)
    if pair:
        # the host launches the pair kernel that cuts items only when the
        # items the sizes suggest are fewer than the pair slots
        est_pairs = -(-extra // (2 * tq)) * Hkv
        if not (est_pairs < slots and est_pairs <= piece_slots):
            return [1] * len(tiles)
    budget = min(slots, piece_slots)

    def pieces(t, th):
        return min(8, max(1, -(-t // th)))
    lo, hi = 4, max(4, max(tiles))
    while lo < hi:
        mid = (lo + hi) // 2
        if sum(pieces(t, mid) for t in tiles) * Hkv <= budget:
            hi = mid
        else:
            lo = mid + 1
    return [pieces(t, hi) for t in tiles]


@pytest.mark.parametrize("D,G,window,softcap", [(256, 4, 0, 0.0), (256, 4, 1024, 50.0),
                                                (128, 4, 0, 30.0), (256, 8, 0, 0.0),
                                                (128, 1, 2000, 0.0), (256, 1, 0, 0.0),
                                                (256, 2, 512, 30.0)])
def test_prefill_tiles_split_along_keys(D, G, window, softcap):
    """A few long-context chunk tiles next to decode rows: the items fill far
    less than the wave of SMs left to them, so each is cut along its keys
    into pieces on separate CTAs, merged by the piece that finishes last;
    the result matches the oracle, repeats bit for bit, and every counter is
    left zero."""
    Hkv = 2 if G < 8 else 1
    L = [3000, 40, 2500, 1, 700, 4100]
    n = [1, 1, 40, 1, 1, 16]
    b = small(L, n, D=D, G=G, Hkv=Hkv, window=window, softcap=softcap, seed=D + G + window)
    assert max(expected_pieces(b)) > 1, "the case must force pieces"
    check(b, f"split D={D} G={G} W={window} cap={softcap}")


def test_split_pieces_short_and_ragged_tiles():
    """Pieces of 4-8 key tiles, a chunk whose last query tile is ragged, and
    a chunk short enough to stay whole, in one launch."""
    L = [1, 900, 33, 2100, 520]
    n = [1, 37, 1, 200, 3]
    b = small(L, n, seed=77, softcap=50.0)
    assert max(expected_pieces(b)) > 1
    check(b, "split ragged")


def lse_region(runner):
    """The decode rows' partial LSEs in the workspace ([B][Hq][S] fp32 after
    the partial outputs, as paged_decode_attn_ws lays them out)."""
    b = runner.batch
    S, _ = binding.paged_decode_splitk_plan(b.num_requests, b.num_kv_heads, b.max_seq_len, 16,
                                            b.window)
    B, Hq, D = b.num_requests, b.num_q_heads, b.head_dim
    off = B * Hq * S * D * 4
    return runner.workspace[off:off + B * Hq * S * 4].view(torch.float32)


@pytest.mark.parametrize("kind", ["short rows", "long rows"])
def test_decode_rows_stream_whole_or_split(kind):
    """Decode rows that fit one per pipeline and are short of the split's
    chunk plus 24 units stream whole, writing no partial; long rows without
    a window are split and merged.  The partial LSEs are filled with NaN
    first: untouched in the first case, written in the second; the output
    matches the oracle either way."""
    if kind == "short rows":
        L, n, W = [300, 900, 1, 60, 700, 1500], [1, 1, 1, 1, 60, 1], 256
    else:
        L, n, W = [3000, 4000, 1, 2500, 700, 1500], [1, 1, 1, 1, 60, 1], 0
    b = small(L, n, window=W, softcap=50.0, seed=91)
    runner = binding.MixedBatch(b)
    lse_region(runner).fill_(float("nan"))
    out = runner.run(torch.zeros(1, dtype=torch.int32, device=DEV)).clone()
    torch.cuda.synchronize()
    written = int((~torch.isnan(lse_region(runner))).sum())
    if kind == "short rows":
        assert written == 0, "short decode rows must not go through partials"
    else:
        assert written > 0, "long decode rows must be split"
    ref, _ = oracle.run_batch(workload.to_numpy_f64(b))
    assert_close(to_f64(out), ref, kind)
    assert torch.all(counters(runner) == 0)
