"""Failure handling on the GPU without a GPU fault: a wait that can never
complete must end with an error status and leave the context usable, and
every call must write only inside its output and workspace (canary words
around them stay intact)."""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_attention_12_gb300 import _build, binding, workload
from tests.parity import assert_close, to_f64

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
PAD = 4096  # bytes of canary on each side (a multiple of 16)


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    binding.lib()


def test_bounded_wait_ends_with_timeout_and_context_stays_usable():
    for budget in (1, 200_000, 20_000_000):
        err = torch.zeros(1, dtype=torch.int32, device=DEV)
        binding.selftest_bounded_wait(err, budget)
        torch.cuda.synchronize()
        assert err.item() == binding.DEVERR_TIMEOUT, (budget, err.item())
    # the context still runs the library's kernels correctly
    batch = workload.decode_tiny(1, DEV, poison=True)
    ref, _ = oracle.run_batch(workload.to_numpy_f64(batch))
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = binding.DecodeSplitK(batch).run(err=err)
    assert_close(to_f64(out), ref, "decode after a timed-out wait")
    torch.cuda.synchronize()
    assert err.item() == 0


class Guarded:
    """A device buffer of ``nbytes`` with PAD canary bytes on each side; the
    body starts on a 16-byte boundary."""

    def __init__(self, nbytes, fill=0):
        g = torch.Generator(device="cpu").manual_seed(nbytes % 1009)
        self.canary = torch.randint(0, 256, (2, PAD), generator=g, dtype=torch.uint8).to(DEV)
        self.raw = torch.empty(nbytes + 2 * PAD, dtype=torch.uint8, device=DEV)
        self.raw[:PAD] = self.canary[0]
        self.raw[PAD + nbytes:] = self.canary[1]
        self.raw[PAD:PAD + nbytes].fill_(fill)
        self.nbytes = nbytes

    def view(self, dtype, shape):
        return self.raw[PAD:PAD + self.nbytes].view(dtype).view(shape)

    def intact(self):
        torch.cuda.synchronize()
        return (torch.equal(self.raw[:PAD], self.canary[0]) and
                torch.equal(self.raw[PAD + self.nbytes:], self.canary[1]))


def nbytes_of(t):
    return t.numel() * t.element_size()


@pytest.mark.parametrize("maker", ["tiny", "serving_w", "long"])
def test_decode_paths_write_only_their_buffers(maker):
    if maker == "tiny":
        batch = workload.decode_tiny(2, DEV, poison=True)
    elif maker == "serving_w":
        batch = workload.decode_serving(2, DEV, poison=True, scale_down=True)[1]
    else:
        batch = workload.decode_long(2, DEV, poison=True, scale_down=True)
    ref, _ = oracle.run_batch(workload.to_numpy_f64(batch))
    B, Hq, D = batch.q.shape
    # direct
    g_out = Guarded(nbytes_of(batch.q))
    out = g_out.view(torch.bfloat16, batch.q.shape)
    binding.paged_decode_attn(batch.q, out, batch.k_pool, batch.v_pool, batch.block_tables,
                              batch.seq_lens, batch.max_seq_len, scale=batch.scale,
                              softcap=batch.softcap, window=batch.window)
    assert g_out.intact(), "direct decode wrote outside out"
    assert_close(to_f64(out), ref, "direct")
    # split-K partials + combine
    S, C = binding.paged_decode_splitk_plan(B, batch.num_kv_heads, batch.max_seq_len, 16,
                                            batch.window)
    g_po = Guarded(B * Hq * S * D * 4)
    g_pl = Guarded(B * Hq * S * 4)
    g_o2 = Guarded(nbytes_of(batch.q))
    po = g_po.view(torch.float32, (B, Hq, S, D))
    pl = g_pl.view(torch.float32, (B, Hq, S))
    o2 = g_o2.view(torch.bfloat16, batch.q.shape)
    binding.paged_decode_splitk(batch.q, po, pl, batch.k_pool, batch.v_pool, batch.block_tables,
                                batch.seq_lens, batch.max_seq_len, S, C, scale=batch.scale,
                                softcap=batch.softcap, window=batch.window)
    binding.paged_decode_splitk_combine(po, pl, o2)
    assert g_po.intact() and g_pl.intact() and g_o2.intact(), "split-K wrote outside its buffers"
    assert_close(to_f64(o2), ref, "split-K")
    # fused combine with a workspace
    nws = binding.paged_decode_attn_ws_bytes(B, Hq, batch.num_kv_heads, D, batch.max_seq_len,
                                             batch.window)
    g_ws = Guarded(nws, fill=0)
    g_o3 = Guarded(nbytes_of(batch.q))
    o3 = g_o3.view(torch.bfloat16, batch.q.shape)
    for _ in range(2):
        binding.paged_decode_attn_ws(batch.q, o3, batch.k_pool, batch.v_pool, batch.block_tables,
                                     batch.seq_lens, batch.max_seq_len, g_ws.view(torch.uint8, (nws,)),
                                     scale=batch.scale, softcap=batch.softcap, window=batch.window)
    assert g_ws.intact() and g_o3.intact(), "fused decode wrote outside its buffers"
    assert_close(to_f64(o3), ref, "fused")


def test_prefill_and_mixed_paths_write_only_their_buffers():
    batch = workload.mixed_batch(2, DEV, poison=True, scale_down=True, drop_out_of_window=True)
    ref, _ = oracle.run_batch(workload.to_numpy_f64(batch))
    g_out = Guarded(nbytes_of(batch.q))
    out = g_out.view(torch.bfloat16, batch.q.shape)
    binding.run_batch(batch, out)
    assert g_out.intact(), "prefill wrote outside out"
    assert_close(to_f64(out), ref, "prefill")
    B, Hq, D = batch.num_requests, batch.num_q_heads, batch.head_dim
    nws = binding.paged_prefill_attn_ws_bytes(B, Hq, batch.num_kv_heads, D, batch.max_seq_len,
                                              batch.window)
    g_ws = Guarded(nws, fill=0)
    g_o2 = Guarded(nbytes_of(batch.q))
    o2 = g_o2.view(torch.bfloat16, batch.q.shape)
    binding.paged_prefill_attn_ws(batch.q, o2, batch.k_pool, batch.v_pool, batch.block_tables,
                                  batch.query_start_loc, batch.seq_lens, batch.max_query_len,
                                  batch.max_seq_len, g_ws.view(torch.uint8, (nws,)),
                                  scale=batch.scale, softcap=batch.softcap, window=batch.window)
    assert g_ws.intact() and g_o2.intact(), "mixed launch wrote outside its buffers"
    assert_close(to_f64(o2), ref, "mixed")


def _bad_offsets_cases():
    """(name, query_start_loc, max_query_len, requests whose spans are valid)
    for a batch of rows [0, 40), [40, 104), [104, 161), [161, 162): each case
    breaks one or two offsets; the rest must still be served."""
    return [
        ("span past total_q", [0, 40, 170, 161, 162], 64, [0, 3]),
        ("negative start", [0, -5, 104, 161, 162], 64, [2, 3]),
        ("span longer than max_query_len", [0, 40, 104, 161, 162], 60, [0, 2, 3]),
        ("decode row past total_q", [0, 40, 104, 170, 171], 64, [0, 1]),
    ]


@pytest.mark.parametrize("case", range(4))
@pytest.mark.parametrize("path", ["single", "mixed"])
def test_bad_query_start_loc_is_skipped_and_reported(case, path):
    """A malformed query_start_loc (device data the host cannot check) never
    makes a kernel write outside out: the requests with bad spans are
    skipped, PKA_DEVERR_QUERY_LOC is reported, and every other request's rows
    are still right."""
    name, qsl, mql, good = _bad_offsets_cases()[case]
    L, n = [100, 300, 57, 20], [40, 64, 57, 1]
    batch = workload.make_batch(seq_lens=L, q_lens=n, num_q_heads=8, num_kv_heads=2,
                                head_dim=256, num_blocks=40, cfg_id=51, seed=case,
                                device=DEV, poison=True)
    arr = workload.to_numpy_f64(batch, good)
    ref, _ = oracle.run_batch(arr)
    bad = torch.tensor(qsl, dtype=torch.int32, device=DEV)
    g_out = Guarded(nbytes_of(batch.q), fill=0xFF)
    out = g_out.view(torch.bfloat16, batch.q.shape)
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    if path == "single":
        binding.paged_prefill_attn(batch.q, out, batch.k_pool, batch.v_pool, batch.block_tables,
                                   bad, batch.seq_lens, mql, batch.max_seq_len,
                                   scale=batch.scale, err=err)
    else:
        nws = binding.paged_prefill_attn_ws_bytes(4, 8, 2, 256, batch.max_seq_len)
        g_ws = Guarded(nws, fill=0)
        binding.paged_prefill_attn_ws(batch.q, out, batch.k_pool, batch.v_pool,
                                      batch.block_tables, bad, batch.seq_lens, mql,
                                      batch.max_seq_len, g_ws.view(torch.uint8, (nws,)),
                                      scale=batch.scale, err=err)
        assert g_ws.intact(), f"{name}: workspace canary"
    torch.cuda.synchronize()
    assert g_out.intact(), f"{name}: a kernel wrote outside out"
    assert err.item() & binding.DEVERR_QUERY_LOC, f"{name}: not reported ({err.item()})"
    assert_close(to_f64(out[arr["q_rows"]]), ref, f"{name}: valid requests")
    # rows that belong to no valid request keep their fill
    untouched = torch.ones(batch.q.shape[0], dtype=torch.bool)
    untouched[list(arr["q_rows"])] = False
    rows = out.view(torch.int16)[untouched.to(DEV)]
    assert bool((rows == -1).all()), f"{name}: rows of a skipped request were written"
