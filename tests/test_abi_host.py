"""Host-side checks of the C ABI that need no GPU.

The library must load and export every function ``include/paged_attn.h``
declares, and argument errors must be rejected on the host before any CUDA
call (so these run on a machine without a GPU).
"""
import ctypes
import os
import re

import pytest

from paged_kv_attention_12_gb300 import _build, binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    _build.build()
    return binding.lib()


def declared_functions():
    names = []
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(",
                                text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_function(L):
    names = declared_functions()
    assert "paged_decode_attn" in names and "paged_prefill_attn" in names
    for n in names:
        assert hasattr(L, n), f"{n} declared in include/ but not exported"
    assert set(binding.EXPORTS) <= set(names)


def test_version_and_status_strings(L):
    assert L.pka_version() >= 100
    for code in binding.STATUS:
        assert L.pka_status_string(code)
    assert L.pka_status_string(12345) == b"unknown status"


def _pool(**kw):
    d = dict(k=16, v=16, num_blocks=8, num_kv_heads=2, block_size=16, head_dim=128)
    d.update(kw)
    return binding.PkaKvPool(d["k"], d["v"], d["num_blocks"], d["num_kv_heads"],
                             d["block_size"], d["head_dim"])


def _decode(L, q=32, out=32, pool=None, tables=64, max_blocks=4, seq=64, B=2, Hq=8,
            max_seq_len=64, params=True, scale=0.1, softcap=0.0):
    pool = pool or _pool()
    par = binding.PkaAttnParams(scale, softcap, 0, None)
    return L.paged_decode_attn(q, out, ctypes.byref(pool), tables, max_blocks, seq, B, Hq,
                               max_seq_len, ctypes.byref(par) if params else None, None)


def test_decode_argument_errors_are_host_side(L):
    assert _decode(L, q=None) == -1
    assert _decode(L, out=None) == -1
    assert _decode(L, tables=None) == -1
    assert _decode(L, params=False) == -1
    assert _decode(L, pool=_pool(k=None)) == -1
    assert _decode(L, Hq=7) == -2                       # Hq % Hkv
    assert _decode(L, Hq=6) == -4                       # G = 3
    assert _decode(L, pool=_pool(head_dim=96)) == -4
    assert _decode(L, pool=_pool(block_size=32)) == -4
    assert _decode(L, Hq=32) == -4                      # G = 16
    assert _decode(L, q=40) == -3                       # misaligned q
    assert _decode(L, pool=_pool(v=24)) == -3
    assert _decode(L, max_seq_len=65) == -2             # beyond max_blocks * bs
    assert _decode(L, B=-1) == -2


def test_splitk_plan_and_workspace(L):
    # slots S = ceil(T / C) + 1 for T visible blocks and minimum chunk C >= 4
    for (B, Hkv, L_max, W) in [(32, 2, 4096, 0), (4, 4, 131072, 0), (32, 2, 4096, 512),
                              (4, 2, 256, 0), (1, 1, 1, 0)]:
        S, C = binding.paged_decode_splitk_plan(B, Hkv, L_max, 16, W, sm_count=152)
        T = -(-L_max // 16) if W <= 0 else min(-(-L_max // 16), (W - 1) // 16 + 2)
        assert C >= 4 and S == -(-T // C) + 1 and S <= 33, (B, Hkv, L_max, W, S, C)
    S, C = binding.paged_decode_splitk_plan(32, 2, 4096, 16, 512, sm_count=0)  # no CUDA call
    assert (S, C) == (10, 4)
    assert binding.paged_decode_splitk_workspace_bytes(4, 16, 128, 10) == 4 * 16 * 10 * 129 * 4
    assert binding.paged_decode_splitk_workspace_bytes(0, 16, 128, 10) == 0


def test_splitk_rejects_uncovering_partition(L):
    pool = _pool()
    par = binding.PkaAttnParams(0.1, 0.0, 0, None)
    # 64 tokens = 4 blocks; chunks of 3 blocks need ceil(4/3) + 1 = 3 slots
    st = L.paged_decode_splitk(32, 64, 96, ctypes.byref(pool), 64, 4, 64, 2, 8, 64, 2, 3,
                               ctypes.byref(par), None)
    assert st == -5
    st = L.paged_decode_splitk(32, None, 96, ctypes.byref(pool), 64, 4, 64, 2, 8, 64, 1, 4,
                               ctypes.byref(par), None)
    assert st == -1


def test_combine_and_prefill_and_check_argument_errors(L):
    assert L.paged_decode_splitk_combine(None, 16, 1, 8, 128, 2, 32, None, None) == -1
    assert L.paged_decode_splitk_combine(16, 16, 1, 8, 96, 2, 32, None, None) == -4
    assert L.paged_decode_splitk_combine(16, 16, 1, 8, 128, 0, 32, None, None) == -2
    pool = _pool()
    par = binding.PkaAttnParams(0.1, 0.0, 0, None)
    assert L.paged_prefill_attn(32, 32, ctypes.byref(pool), 64, 4, None, 64, 2, 8, 10, 5, 64,
                                ctypes.byref(par), None) == -1
    assert L.paged_prefill_attn(32, 32, ctypes.byref(pool), 64, 4, 80, 64, 2, 8, 10, 65, 64,
                                ctypes.byref(par), None) == -2
    assert L.paged_attn_check_tables(64, 4, 64, 2, 8, 16, None, None) == -1
    assert L.paged_attn_check_tables(64, 0, 64, 2, 8, 16, 32, None) == -2


def test_selftest_argument_errors(L):
    assert L.pka_selftest_bounded_wait(None, 1000, None) == -1
    assert L.pka_selftest_bounded_wait(16, 0, None) == -2
    assert L.pka_selftest_bounded_wait(16, 2000000001, None) == -2


def test_mixed_workspace_argument_errors(L):
    """paged_prefill_attn_ws: the prefill checks, then the workspace's
    presence, alignment and size, all before any launch."""
    pool = _pool()
    par = binding.PkaAttnParams(0.1, 0.0, 0, None)
    need = L.paged_prefill_attn_ws_bytes(2, 8, 2, 128, 64, 0)
    # the decode workspace, then 160 prefill piece slots of 128 rows x D fp32,
    # their LSEs and their counters (the header's layout)
    dec = L.paged_decode_attn_ws_bytes(2, 8, 2, 128, 64, 0)
    assert dec > 0
    assert need == dec + 160 * 128 * 128 * 4 + 160 * 128 * 4 + 160 * 4

    def call(qsl=80, ws=256, nbytes=None, max_query_len=5):
        return L.paged_prefill_attn_ws(32, 32, ctypes.byref(pool), 64, 4, qsl, 64, 2, 8, 10,
                                       max_query_len, 64, ctypes.byref(par), ws,
                                       need if nbytes is None else nbytes, None)

    assert call(qsl=None) == -1
    assert call(max_query_len=65) == -2
    assert call(ws=None) == -1
    assert call(ws=264) == -3
    assert call(nbytes=need - 1) == -5
    assert L.paged_prefill_attn_ws_bytes(0, 8, 2, 128, 64, 0) == 0


def test_zero_batch_is_a_no_op(L):
    assert _decode(L, B=0) == 0


def test_scale_and_softcap_values(L):
    """scale: any finite value (zero and negative included); softcap: NaN is
    refused, +inf means no cap.  Checked with B = 0, so nothing launches."""
    inf, nan = float("inf"), float("nan")
    for sc in (0.0, -0.5, 1e-30, 3e38):
        assert _decode(L, B=0, scale=sc) == 0, sc
    for sc in (inf, -inf, nan):
        assert _decode(L, B=0, scale=sc) == -2, sc
    assert _decode(L, B=0, softcap=inf) == 0
    assert _decode(L, B=0, softcap=-inf) == 0
    assert _decode(L, B=0, softcap=nan) == -2
    pool = _pool()
    par = binding.PkaAttnParams(inf, 0.0, 0, None)
    assert L.paged_prefill_attn(32, 32, ctypes.byref(pool), 64, 4, 80, 64, 0, 8, 0, 5, 64,
                                ctypes.byref(par), None) == -2


def test_noalloc_checks_arguments_before_the_empty_batch(L):
    """The allocation-free decode validates like every other entry point, even
    when B = 0 makes the call a no-op."""
    pool = _pool()
    par = binding.PkaAttnParams(0.1, 0.0, 0, None)

    def call(q=32, B=0, Hq=8, max_seq_len=64):
        return L.paged_decode_attn_noalloc(q, 32, ctypes.byref(pool), 64, 4, 64, B, Hq,
                                           max_seq_len, ctypes.byref(par), None)

    assert call() == 0
    assert call(q=None) == -1
    assert call(q=40) == -3
    assert call(Hq=6) == -4
    assert call(max_seq_len=65) == -2
    assert L.pka_status_string(-5).startswith(b"split-K workspace too small")


def _append(L, k_new=32, v_new=32, k_pool=64, v_pool=64, nb=8, hkv=2, bs=16, d=128,
            slots=128, T=4):
    return L.paged_kv_append(k_new, v_new, k_pool, v_pool, nb, hkv, bs, d, slots, T, None, None)


def test_kv_append_host_errors(L):
    assert _append(L, T=0) == 0                      # nothing to do, nothing launched
    assert _append(L, T=-1) == -2
    assert _append(L, nb=0) == -2
    assert _append(L, hkv=0) == -2
    assert _append(L, bs=32) == -4
    assert _append(L, d=64) == -4
    assert _append(L, k_new=0) == -1
    assert _append(L, slots=0) == -1
    assert _append(L, v_pool=72) == -3              # not 16-byte aligned
    assert _append(L, k_new=40) == -3


def test_kv_append_rope_host_errors(L):
    def call(q=32, T=4, rd=128, theta=10000.0, eps=1e-6, d=128, bs=16, hq=8, hkv=2, pos=256):
        return L.paged_kv_append_rope(q, 64, 96, 128, 160, 8, hq, hkv, bs, d, 192, pos, T, None,
                                      None, 0, eps, theta, rd, None, None)
    assert call(T=0) == 0
    assert call(rd=24) == -2        # not a multiple of 16
    assert call(rd=256) == -2       # wider than D
    assert call(theta=1.0) == -2
    assert call(eps=-1.0) == -2
    assert call(bs=8) == -4
    assert call(d=96) == -4
    assert call(hq=7) == -2         # not a multiple of Hkv
    assert call(pos=0) == -1        # RoPE needs positions
    assert call(q=40) == -3
