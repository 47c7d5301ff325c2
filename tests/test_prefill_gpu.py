"""GPU parity of the tcgen05 prefill / mixed-batch kernel against the oracle.

Ordered from the smallest case up, so that a layout or descriptor slip shows
on a one-tile problem first.
"""
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


def run(batch, err=None):
    out = torch.full_like(batch.q, float("nan"))
    binding.run_batch(batch, out, err)
    return out


def check(batch, what, reqs=None):
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run(batch, err)
    arr = workload.to_numpy_f64(batch, reqs)
    ref, _ = oracle.run_batch(arr)
    got = out[arr["q_rows"]] if reqs is not None else out
    ma, rl = assert_close(to_f64(got), ref, what)
    torch.cuda.synchronize()
    assert err.item() == 0, f"{what}: device error word {err.item()}"
    return ma, rl


def small(seq_lens, q_lens, D=128, G=4, Hkv=1, **kw):
    return workload.make_batch(seq_lens=seq_lens, q_lens=q_lens, num_q_heads=G * Hkv,
                               num_kv_heads=Hkv, head_dim=D,
                               num_blocks=kw.pop("num_blocks", sum(-(-L // 16) for L in seq_lens) + 8),
                               device=DEV, poison=True, cfg_id=kw.pop("cfg_id", 21), **kw)


def test_one_tile_no_prefix():
    check(small([32], [32]), "L=32 n=32")


def test_one_tile_ragged():
    check(small([23], [23]), "L=23 n=23")


@pytest.mark.parametrize("D", [128, 256])
def test_prefix_plus_chunk(D):
    check(small([100, 300, 77], [40, 64, 77], D=D, Hkv=2, seed=1), f"D={D}")


@pytest.mark.parametrize("D,G", [(128, 1), (128, 2), (128, 8), (256, 1), (256, 2), (256, 8)])
def test_group_sizes(D, G):
    check(small([150, 61], [90, 61], D=D, G=G, Hkv=2 if G < 8 else 1, seed=G), f"D={D} G={G}")


@pytest.mark.parametrize("window,softcap", [(0, 30.0), (37, 0.0), (100, 50.0), (0, 2.0),
                                            (64, 8.0)])
def test_window_and_softcap(window, softcap):
    check(small([400, 130, 57], [130, 1, 57], D=256, Hkv=2, window=window, softcap=softcap,
                seed=window), f"W={window} cap={softcap}")


@pytest.mark.parametrize("scale,softcap", [(1e-3, 1e4), (0.0625, 1e6), (2.0, 0.5)])
def test_softcap_scale_extremes(scale, softcap):
    """Ratios scale / softcap at which the capped logit's Taylor terms
    underflow (tiny ratio) or the exp2 form is needed (large ratio): every
    path of the capped softmax against the oracle, on causal and ragged
    tiles."""
    check(small([400, 130, 57, 20], [130, 1, 57, 1], D=256, Hkv=2, softcap=softcap,
                scale=scale, seed=19), f"scale={scale} cap={softcap}")
    check(small([300, 75], [75, 75], D=128, Hkv=2, softcap=softcap, scale=scale, seed=20),
          f"D=128 scale={scale} cap={softcap}")


@pytest.mark.parametrize("scale", [0.0, -0.0625, -0.25])
@pytest.mark.parametrize("softcap", [0.0, 30.0])
def test_zero_and_negative_scale(scale, softcap):
    """scale may be any finite number: at 0 each row is the mean of the V rows
    it sees, below 0 the least aligned keys win; causal diagonals, a decode
    row and a ragged chunk are in the batch."""
    check(small([400, 130, 57, 20], [130, 1, 57, 1], D=256, Hkv=2, softcap=softcap,
                scale=scale, seed=17), f"scale={scale} cap={softcap}")


def test_decode_rows_in_varlen_batch():
    check(small([33, 700, 1, 16, 17], [1, 1, 1, 16, 1], D=128, Hkv=2, seed=5), "decode rows")


@pytest.mark.parametrize("seed", range(3))
def test_chunked_prefill_small(seed):
    check(workload.chunked_prefill(seed, DEV, poison=True, scale_down=True), f"cfg4 small {seed}")


@pytest.mark.parametrize("seed", range(3))
def test_mixed_batch_small(seed):
    b = workload.mixed_batch(seed, DEV, poison=True, scale_down=True, drop_out_of_window=True)
    check(b, f"cfg5 small {seed}")


@pytest.mark.parametrize("D", [128, 256])
def test_one_hot_prefill_exact(D):
    """Each query row's own key is c*q (every other weight underflows): the
    output row is exactly that key's V row (D = 256 runs on CTA pairs)."""
    G, Hkv = 4, 1
    L, n = 50, 20
    batch = small([L], [n], D=D, G=G, Hkv=Hkv, seed=9)
    q = batch.q.view(n, Hkv, G, D)
    q[:] = q[:, :, :1, :]
    k = batch.k_pool.mul(0.01)
    blocks = batch.tables_host[0]
    for i in range(n):
        t = L - n + i
        qv = q[i, 0, 0].float()
        k[blocks[t // 16], 0, t % 16] = (qv * (300.0 / qv.pow(2).sum()) * 16.0).to(torch.bfloat16)
    # with window 1 each query sees only its own key
    b2 = workload.PagedBatch(**{**batch.__dict__, "k_pool": k, "window": 1, "scale": 1.0 / 16})
    out = run(b2)
    for i in range(n):
        t = L - n + i
        want = batch.v_pool[blocks[t // 16], 0, t % 16]
        for g in range(G):
            assert torch.equal(out[i, g], want), (i, g)
    # full causal attention: the own key still dominates every earlier key
    b3 = workload.PagedBatch(**{**batch.__dict__, "k_pool": k, "scale": 1.0 / 16})
    out = run(b3)
    for i in range(n):
        t = L - n + i
        want = batch.v_pool[blocks[t // 16], 0, t % 16]
        assert torch.equal(out[i, 0], want), i


@pytest.mark.parametrize("D", [128, 256])
def test_rising_logits_rescale_every_tile(D):
    """Keys along one direction with growing length and every query along
    it: each key's logit is 1/16 above the previous key's, so every 128-key
    tile lifts the running maximum by far more than the lazy rescale's
    threshold and O is rescaled at every tile -- through the pair kernel's
    single S buffer and alternating P buffers at D = 256, the one-CTA
    kernel at D = 128 -- against the oracle."""
    G, Hkv = 4, 2
    L, n = [1500, 900, 333], [300, 130, 333]
    batch = small(L, n, D=D, G=G, Hkv=Hkv, seed=33)
    gen = torch.Generator(device="cpu").manual_seed(5)
    u = torch.randn(D, generator=gen)
    u = (u / u.norm()).to(DEV)
    q = u.to(torch.bfloat16).expand_as(batch.q).contiguous()
    k = batch.k_pool.clone()
    for b, Lb in enumerate(L):
        blocks = batch.tables_host[b]
        for t0 in range(0, Lb, 16):
            rows = torch.arange(t0, min(Lb, t0 + 16), device=DEV, dtype=torch.float32)
            vals = (rows[:, None] * u[None, :]).to(torch.bfloat16)
            for h in range(Hkv):
                k[blocks[t0 // 16], h, : rows.numel()] = vals
    b2 = workload.PagedBatch(**{**batch.__dict__, "q": q, "k_pool": k, "scale": 1.0})
    check(b2, f"rising logits D={D}")


@pytest.mark.parametrize("cfg", [4, 5])
def test_full_size_sampled_requests(cfg):
    batch = workload.workload(cfg, seed=0, device=DEV, poison=True)[0]
    B = batch.num_requests
    if cfg == 4:
        reqs = sorted({0, 3, 4, B - 1, int(np.argmax(batch.seq_lens_host))})
    else:
        reqs = [0, 31, 32, 63, 64, B - 1]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run(batch, err)
    arr = workload.to_numpy_f64(batch, reqs)
    ref, _ = oracle.run_batch(arr)
    assert_close(to_f64(out[arr["q_rows"]]), ref, f"cfg{cfg} full size")
    torch.cuda.synchronize()
    assert err.item() == 0


def test_repeated_launches_are_deterministic_and_never_time_out():
    batch = workload.mixed_batch(1, DEV, scale_down=True)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ref = run(batch, err).clone()
    out = torch.empty_like(batch.q)
    for it in range(100):
        binding.run_batch(batch, out, err)
    torch.cuda.synchronize()
    assert err.item() == 0
    assert torch.equal(out, ref)


@pytest.mark.parametrize("cfg", [4, 5])
def test_full_size_repeated_launches_identical(cfg):
    """A pipeline hazard (a stage or TMEM buffer reused while still being
    read) shows up as run-to-run differences or non-finite values at full
    size, where timing varies most: every launch must give the same bits."""
    batch = workload.workload(cfg, seed=1, device=DEV, poison=True)[0]
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    ref = run(batch, err).clone()
    assert torch.isfinite(ref.float()).all()
    out = torch.empty_like(batch.q)
    for _ in range(8):
        out.fill_(float("nan"))
        binding.run_batch(batch, out, err)
        assert torch.equal(out, ref)
    torch.cuda.synchronize()
    assert err.item() == 0


# ---- long chunks: several query tiles (128 / G tokens each) per request,
# odd tile counts, a one-token request and a request with no query mixed in.

def long_chunk_batch(D, G, Hkv=1, window=0, softcap=0.0, extra_q=(), extra_L=(), seed=0):
    tq = 128 // G
    q = [int(tq * 3.3), int(tq * 2.5) + 1, int(tq * 1.7)] + list(extra_q)
    L = [q[0] + 2 * tq + 37, q[1] + 300, q[2] + 5] + list(extra_L)
    return small(L, q, D=D, G=G, Hkv=Hkv, window=window, softcap=softcap, seed=seed, cfg_id=23)


@pytest.mark.parametrize("D,G", [(128, 1), (128, 4), (128, 8), (256, 1), (256, 2), (256, 4),
                                 (256, 8)])
def test_long_chunks_shapes(D, G):
    check(long_chunk_batch(D, G, Hkv=2 if G < 8 else 1, seed=G), f"long chunks D={D} G={G}")


@pytest.mark.parametrize("window,softcap", [(57, 0.0), (0, 30.0), (200, 50.0)])
def test_long_chunks_window_softcap(window, softcap):
    check(long_chunk_batch(256, 4, Hkv=2, window=window, softcap=softcap, seed=window),
          f"long chunks W={window} cap={softcap}")


def test_long_chunks_with_decode_rows_and_empty_requests():
    """A one-token request, a request with no query at all and long chunks
    in the same launch."""
    check(long_chunk_batch(256, 4, Hkv=2, extra_q=(1, 0, 300), extra_L=(900, 40, 333), seed=3),
          "long chunks + decode rows")


def test_long_chunk_max_sizes():
    """One 8192-token chunk on an 8192-token prefix (G = 1: 64 query tiles of
    128 rows, 128 key tiles each at the end) next to a one-token request and a
    short chunk; rows sampled across the long chunk are checked."""
    batch = small([16384, 300, 5000], [8192, 1, 333], D=128, G=1, Hkv=4, seed=11, cfg_id=42)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run(batch, err)
    arr = workload.to_numpy_f64(batch, [0])
    rows = [0, 1, 127, 128, 4095, 8190, 8191]
    q_rows = arr["q_rows"]
    # reference on the sampled rows only: their keys gathered through the
    # request's table, textbook softmax attention per row and head
    Lr, n = 16384, 8192
    keys = np.asarray(arr["block_tables"][0])
    kc = oracle.gather_request_kv(arr["k_pool"], keys, Lr, 16)
    vc = oracle.gather_request_kv(arr["v_pool"], keys, Lr, 16)
    got = to_f64(out[[q_rows[r] for r in rows]])
    for i, r in enumerate(rows):
        pos = Lr - n + r
        vis = oracle.visible_keys(pos, Lr, 0)
        for h in range(4):
            o, _ = oracle.softmax_attention(arr["q"][r, h:h + 1], kc[vis, h], vc[vis, h],
                                            batch.scale, 0.0)
            assert_close(got[i, h:h + 1], o, f"long chunk row {r} head {h}")
    torch.cuda.synchronize()
    assert err.item() == 0


def test_many_requests_rank_from_global_memory():
    """More requests than the ranking keeps in shared memory (4096): the
    ranking reads (rows, length) from global memory; decode rows, short
    chunks and empty requests mixed, checked on sampled requests through both
    the single-pipeline and the mixed launch."""
    rng = np.random.default_rng(12)
    B = 4500
    L = rng.integers(1, 40, size=B)
    n = np.ones(B, dtype=np.int64)
    chunks = [5, 1000, 2222, 4499]
    n[chunks] = [33, 20, 40, 7]
    L[chunks] = np.maximum(L[chunks], n[chunks]) + 50
    n[[7, 3000]] = 0
    batch = workload.make_batch(seq_lens=L.tolist(), q_lens=n.tolist(), num_q_heads=8,
                                num_kv_heads=2, head_dim=128,
                                num_blocks=int(sum(-(-x // 16) for x in L)) + 8, cfg_id=43,
                                seed=12, device=DEV, poison=True)
    reqs = [0, 5, 6, 1000, 2222, 3001, 4498, 4499]
    arr = workload.to_numpy_f64(batch, reqs)
    ref, _ = oracle.run_batch(arr)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = run(batch, err)
    assert_close(to_f64(out[arr["q_rows"]]), ref, "single pipeline, 4500 requests")
    mixed = binding.MixedBatch(batch).run(err)
    assert_close(to_f64(mixed[arr["q_rows"]]), ref, "mixed launch, 4500 requests")
    torch.cuda.synchronize()
    assert err.item() == 0


@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("window", [0, 45])
def test_pair_items_odd_tiles_and_stale_slots(G, window):
    """D = 256 runs two query tiles per CTA pair: a chunk with an odd number
    of tiles (the last pair's second CTA has no rows), a chunk one row past a
    pair, an exact pair, a one-token request and ragged sequence ends (the
    last block's stale slots hold NaN and must be zeroed in both CTAs'
    halves of V)."""
    tq = 128 // G
    Hkv = 2 if G < 8 else 1
    n = [3 * tq, 2 * tq + 1, 2 * tq, 1, tq - 3]
    L = [x + 131 for x in n[:3]] + [77, tq + 500]
    check(small(L, n, D=256, G=G, Hkv=Hkv, window=window, softcap=30.0 if window else 0.0,
                seed=G + window, cfg_id=24), f"pairs G={G} W={window}")
