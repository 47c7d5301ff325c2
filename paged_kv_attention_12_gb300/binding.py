"""ctypes binding of the C ABI in ``include/paged_attn.h``.

Argument marshalling only: every function here forwards device pointers,
sizes and the current CUDA stream to the library, where all of the work runs
in CUDA kernels.  There is no CPU fallback: if the library is missing or was
built for another machine, loading it raises.

The raw C functions are available under their C names on :func:`lib`; the
helpers below take torch tensors for convenience (the tensors are only used
for their device pointers, shapes and the current stream).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "lib", "libpaged_attn.so")

PKA_OK = 0
STATUS = {
    0: "PKA_OK", -1: "PKA_ERR_NULL", -2: "PKA_ERR_SHAPE", -3: "PKA_ERR_ALIGN",
    -4: "PKA_ERR_UNSUPPORTED", -5: "PKA_ERR_WORKSPACE", -6: "PKA_ERR_BAD_TABLE",
    -7: "PKA_ERR_TIMEOUT", -8: "PKA_ERR_CUDA",
}
DEVERR_BAD_TABLE = 1
DEVERR_TIMEOUT = 2
DEVERR_SEQ_LEN = 4
DEVERR_QUERY_LOC = 8

EXPORTS = [
    "pka_version", "pka_status_string", "paged_decode_attn", "paged_decode_splitk_plan",
    "paged_decode_splitk_workspace_bytes", "paged_decode_splitk",
    "paged_decode_splitk_combine", "paged_prefill_attn", "paged_attn_check_tables",
    "paged_decode_attn_noalloc", "paged_decode_attn_ws_bytes", "paged_decode_attn_ws",
    "paged_kv_append", "paged_decode_splitk_logits", "paged_decode_key_mass",
    "paged_kv_append_rope", "paged_prefill_attn_ws_bytes", "paged_prefill_attn_ws",
    "pka_selftest_bounded_wait",
]


class PkaKvPool(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("num_blocks", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("head_dim", ctypes.c_int32)]


class PkaAttnParams(ctypes.Structure):
    _fields_ = [("scale", ctypes.c_float), ("softcap", ctypes.c_float),
                ("window", ctypes.c_int32), ("err", ctypes.c_void_p)]


class PagedAttnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {STATUS.get(status, status)}")
        self.status = status


_lib = None


def use_library(path: str) -> None:
    """Load ``path`` (an instrumented build of the same library) instead of
    the default one; only before the first call into the library."""
    global LIB_PATH
    if _lib is not None and os.path.abspath(path) != os.path.abspath(LIB_PATH):
        raise RuntimeError("the library is already loaded")
    LIB_PATH = path


def lib() -> ctypes.CDLL:
    """Load the CUDA library (raises if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    L = ctypes.CDLL(LIB_PATH)
    P, I32, VP = ctypes.POINTER, ctypes.c_int32, ctypes.c_void_p
    L.pka_version.restype = ctypes.c_int
    L.pka_version.argtypes = []
    L.pka_status_string.restype = ctypes.c_char_p
    L.pka_status_string.argtypes = [ctypes.c_int]
    L.paged_decode_attn.restype = ctypes.c_int
    L.paged_decode_attn.argtypes = [VP, VP, P(PkaKvPool), VP, I32, VP, I32, I32, I32,
                                    P(PkaAttnParams), VP]
    L.paged_decode_splitk_plan.restype = ctypes.c_int
    L.paged_decode_splitk_plan.argtypes = [I32, I32, I32, I32, I32, I32, P(I32), P(I32)]
    L.paged_decode_splitk_workspace_bytes.restype = ctypes.c_size_t
    L.paged_decode_splitk_workspace_bytes.argtypes = [I32, I32, I32, I32]
    L.paged_decode_splitk.restype = ctypes.c_int
    L.paged_decode_splitk.argtypes = [VP, VP, VP, P(PkaKvPool), VP, I32, VP, I32, I32, I32,
                                      I32, I32, P(PkaAttnParams), VP]
    L.paged_decode_splitk_combine.restype = ctypes.c_int
    L.paged_decode_splitk_combine.argtypes = [VP, VP, I32, I32, I32, I32, VP, VP, VP]
    L.paged_prefill_attn.restype = ctypes.c_int
    L.paged_prefill_attn.argtypes = [VP, VP, P(PkaKvPool), VP, I32, VP, VP, I32, I32, I32,
                                     I32, I32, P(PkaAttnParams), VP]
    L.paged_attn_check_tables.restype = ctypes.c_int
    L.paged_attn_check_tables.argtypes = [VP, I32, VP, I32, I32, I32, VP, VP]
    L.paged_decode_attn_ws_bytes.restype = ctypes.c_size_t
    L.paged_decode_attn_ws_bytes.argtypes = [I32, I32, I32, I32, I32, I32]
    L.paged_decode_attn_ws.restype = ctypes.c_int
    L.paged_decode_attn_ws.argtypes = [VP, VP, P(PkaKvPool), VP, I32, VP, I32, I32, I32,
                                       P(PkaAttnParams), VP, ctypes.c_size_t, VP]
    L.paged_decode_attn_noalloc.restype = ctypes.c_int
    L.paged_decode_attn_noalloc.argtypes = [VP, VP, P(PkaKvPool), VP, I32, VP, I32, I32, I32,
                                            P(PkaAttnParams), VP]
    L.paged_decode_splitk_logits.restype = ctypes.c_int
    L.paged_decode_splitk_logits.argtypes = [VP, VP, VP, VP, P(PkaKvPool), VP, I32, VP, I32, I32,
                                             I32, I32, I32, P(PkaAttnParams), VP]
    L.paged_decode_key_mass.restype = ctypes.c_int
    L.paged_decode_key_mass.argtypes = [VP, VP, VP, I32, I32, I32, I32, I32, I32, VP, VP]
    L.paged_kv_append_rope.restype = ctypes.c_int
    L.paged_kv_append_rope.argtypes = [VP, VP, VP, VP, VP, I32, I32, I32, I32, I32, VP, VP, I32,
                                       VP, VP, I32, ctypes.c_float, ctypes.c_float, I32, VP, VP]
    L.paged_prefill_attn_ws_bytes.restype = ctypes.c_size_t
    L.paged_prefill_attn_ws_bytes.argtypes = [I32, I32, I32, I32, I32, I32]
    L.paged_prefill_attn_ws.restype = ctypes.c_int
    L.paged_prefill_attn_ws.argtypes = [VP, VP, P(PkaKvPool), VP, I32, VP, VP, I32, I32, I32, I32,
                                        I32, P(PkaAttnParams), VP, ctypes.c_size_t, VP]
    L.pka_selftest_bounded_wait.restype = ctypes.c_int
    L.pka_selftest_bounded_wait.argtypes = [VP, ctypes.c_int64, VP]
    L.paged_kv_append.restype = ctypes.c_int
    L.paged_kv_append.argtypes = [VP, VP, VP, VP, I32, I32, I32, I32, VP, I32, VP, VP]
    _lib = L
    return L


def _check(fn: str, status: int) -> None:
    if status != PKA_OK:
        raise PagedAttnError(fn, status)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def kv_pool(k_pool, v_pool) -> PkaKvPool:
    nb, hkv, bs, d = k_pool.shape
    return PkaKvPool(k_pool.data_ptr(), v_pool.data_ptr(), nb, hkv, bs, d)


def attn_params(scale: float, softcap: float = 0.0, window: int = 0, err=None) -> PkaAttnParams:
    return PkaAttnParams(float(scale), float(softcap), int(window), _ptr(err))


# ------------------------------------------------------------------ helpers
def paged_decode_attn(q, out, k_pool, v_pool, block_tables, seq_lens, max_seq_len, *,
                      scale, softcap=0.0, window=0, err=None, stream=None):
    pool = kv_pool(k_pool, v_pool)
    par = attn_params(scale, softcap, window, err)
    st = lib().paged_decode_attn(q.data_ptr(), out.data_ptr(), ctypes.byref(pool),
                                 block_tables.data_ptr(), block_tables.shape[1],
                                 seq_lens.data_ptr(), q.shape[0], q.shape[1], int(max_seq_len),
                                 ctypes.byref(par), _stream(stream))
    _check("paged_decode_attn", st)


def paged_decode_attn_noalloc(q, out, k_pool, v_pool, block_tables, seq_lens, max_seq_len, *,
                              scale, softcap=0.0, window=0, err=None, stream=None):
    """Split-K decode with the partials in the library's own fixed array (no
    device allocation by anyone); raises PagedAttnError(PKA_ERR_WORKSPACE)
    when the partials would not fit its 16 MiB."""
    pool = kv_pool(k_pool, v_pool)
    par = attn_params(scale, softcap, window, err)
    st = lib().paged_decode_attn_noalloc(q.data_ptr(), out.data_ptr(), ctypes.byref(pool),
                                         block_tables.data_ptr(), block_tables.shape[1],
                                         seq_lens.data_ptr(), q.shape[0], q.shape[1],
                                         int(max_seq_len), ctypes.byref(par), _stream(stream))
    _check("paged_decode_attn_noalloc", st)


def paged_decode_attn_ws_bytes(B, Hq, Hkv, D, max_seq_len, window=0) -> int:
    return int(lib().paged_decode_attn_ws_bytes(B, Hq, Hkv, D, int(max_seq_len), int(window)))


def paged_decode_attn_ws(q, out, k_pool, v_pool, block_tables, seq_lens, max_seq_len, workspace,
                         *, scale, softcap=0.0, window=0, err=None, stream=None):
    pool = kv_pool(k_pool, v_pool)
    par = attn_params(scale, softcap, window, err)
    st = lib().paged_decode_attn_ws(q.data_ptr(), out.data_ptr(), ctypes.byref(pool),
                                    block_tables.data_ptr(), block_tables.shape[1],
                                    seq_lens.data_ptr(), q.shape[0], q.shape[1], int(max_seq_len),
                                    ctypes.byref(par), workspace.data_ptr(),
                                    workspace.numel() * workspace.element_size(), _stream(stream))
    _check("paged_decode_attn_ws", st)


def paged_decode_splitk_plan(B, Hkv, max_seq_len, block_size=16, window=0, sm_count=0):
    s, c = ctypes.c_int32(), ctypes.c_int32()
    st = lib().paged_decode_splitk_plan(B, Hkv, int(max_seq_len), block_size, int(window),
                                        int(sm_count), ctypes.byref(s), ctypes.byref(c))
    _check("paged_decode_splitk_plan", st)
    return s.value, c.value


def paged_decode_splitk_workspace_bytes(B, Hq, D, num_splits) -> int:
    return int(lib().paged_decode_splitk_workspace_bytes(B, Hq, D, num_splits))


def paged_decode_splitk(q, partial_o, partial_lse, k_pool, v_pool, block_tables, seq_lens,
                        max_seq_len, num_splits, split_blocks, *, scale, softcap=0.0, window=0,
                        err=None, stream=None):
    pool = kv_pool(k_pool, v_pool)
    par = attn_params(scale, softcap, window, err)
    st = lib().paged_decode_splitk(q.data_ptr(), partial_o.data_ptr(), partial_lse.data_ptr(),
                                   ctypes.byref(pool), block_tables.data_ptr(),
                                   block_tables.shape[1], seq_lens.data_ptr(), q.shape[0],
                                   q.shape[1], int(max_seq_len), int(num_splits),
                                   int(split_blocks), ctypes.byref(par), _stream(stream))
    _check("paged_decode_splitk", st)


def paged_decode_splitk_logits(q, partial_o, partial_lse, logits, k_pool, v_pool, block_tables,
                               seq_lens, max_seq_len, num_splits, split_blocks, *, scale,
                               softcap=0.0, window=0, err=None, stream=None):
    """paged_decode_splitk that also stores the visible keys' log2-domain
    logits in ``logits`` fp32 [B][Hq][max_blocks * 16]."""
    pool = kv_pool(k_pool, v_pool)
    par = attn_params(scale, softcap, window, err)
    st = lib().paged_decode_splitk_logits(q.data_ptr(), partial_o.data_ptr(),
                                          partial_lse.data_ptr(), logits.data_ptr(),
                                          ctypes.byref(pool), block_tables.data_ptr(),
                                          block_tables.shape[1], seq_lens.data_ptr(), q.shape[0],
                                          q.shape[1], int(max_seq_len), int(num_splits),
                                          int(split_blocks), ctypes.byref(par), _stream(stream))
    _check("paged_decode_splitk_logits", st)


def paged_decode_key_mass(logits, lse, seq_lens, num_kv_heads, key_mass, *, window=0,
                          block_size=16, stream=None):
    """key_mass fp32 [B][Hkv][max_blocks * 16] += each visible key's attention
    probability summed over its KV head's query heads (``lse``: [B][Hq]
    natural-log LSE from the combine)."""
    B, Hq, nk = logits.shape
    st = lib().paged_decode_key_mass(logits.data_ptr(), lse.data_ptr(), seq_lens.data_ptr(), B,
                                     Hq, int(num_kv_heads), nk // block_size, block_size,
                                     int(window), key_mass.data_ptr(), _stream(stream))
    _check("paged_decode_key_mass", st)


def paged_decode_splitk_combine(partial_o, partial_lse, out, lse_out=None, stream=None):
    B, Hq, S, D = partial_o.shape
    st = lib().paged_decode_splitk_combine(partial_o.data_ptr(), partial_lse.data_ptr(), B, Hq,
                                           D, S, out.data_ptr(), _ptr(lse_out), _stream(stream))
    _check("paged_decode_splitk_combine", st)


def paged_prefill_attn(q, out, k_pool, v_pool, block_tables, query_start_loc, seq_lens,
                       max_query_len, max_seq_len, *, scale, softcap=0.0, window=0, err=None,
                       stream=None):
    pool = kv_pool(k_pool, v_pool)
    par = attn_params(scale, softcap, window, err)
    st = lib().paged_prefill_attn(q.data_ptr(), out.data_ptr(), ctypes.byref(pool),
                                  block_tables.data_ptr(), block_tables.shape[1],
                                  query_start_loc.data_ptr(), seq_lens.data_ptr(),
                                  seq_lens.shape[0], q.shape[1], q.shape[0], int(max_query_len),
                                  int(max_seq_len), ctypes.byref(par), _stream(stream))
    _check("paged_prefill_attn", st)


def paged_prefill_attn_ws_bytes(B, Hq, Hkv, D, max_seq_len, window=0) -> int:
    return int(lib().paged_prefill_attn_ws_bytes(B, Hq, Hkv, D, int(max_seq_len), int(window)))


def paged_prefill_attn_ws(q, out, k_pool, v_pool, block_tables, query_start_loc, seq_lens,
                          max_query_len, max_seq_len, workspace, *, scale, softcap=0.0, window=0,
                          err=None, stream=None):
    """Mixed batch in one launch: decode rows on decode pipelines, chunks on
    the tensor-core prefill pipeline.  ``workspace``: zero-initialised device
    bytes, at least ``paged_prefill_attn_ws_bytes``; left zeroed."""
    pool = kv_pool(k_pool, v_pool)
    par = attn_params(scale, softcap, window, err)
    st = lib().paged_prefill_attn_ws(q.data_ptr(), out.data_ptr(), ctypes.byref(pool),
                                     block_tables.data_ptr(), block_tables.shape[1],
                                     query_start_loc.data_ptr(), seq_lens.data_ptr(),
                                     seq_lens.shape[0], q.shape[1], q.shape[0],
                                     int(max_query_len), int(max_seq_len), ctypes.byref(par),
                                     workspace.data_ptr(), workspace.numel(), _stream(stream))
    _check("paged_prefill_attn_ws", st)


def selftest_bounded_wait(err, budget_cycles, stream=None):
    """A wait that can never complete, with the library's wait routine and a
    budget of ``budget_cycles``: it must end with PKA_DEVERR_TIMEOUT in
    ``err`` (device int32)."""
    st = lib().pka_selftest_bounded_wait(err.data_ptr(), int(budget_cycles), _stream(stream))
    _check("pka_selftest_bounded_wait", st)


def paged_attn_check_tables(block_tables, seq_lens, num_blocks, err, block_size=16, stream=None):
    st = lib().paged_attn_check_tables(block_tables.data_ptr(), block_tables.shape[1],
                                       seq_lens.data_ptr(), seq_lens.shape[0], int(num_blocks),
                                       block_size, err.data_ptr(), _stream(stream))
    _check("paged_attn_check_tables", st)


def paged_kv_append(k_new, v_new, k_pool, v_pool, slot_mapping, err=None, stream=None):
    """Write token t's K/V rows (``k_new``/``v_new`` bf16 [T][Hkv][D]) into
    the pools at slot ``slot_mapping[t]`` (int32, block * bs + offset; < 0
    skips the token)."""
    nb, hkv, bs, d = k_pool.shape
    st = lib().paged_kv_append(k_new.data_ptr(), v_new.data_ptr(), k_pool.data_ptr(),
                               v_pool.data_ptr(), nb, hkv, bs, d, slot_mapping.data_ptr(),
                               slot_mapping.shape[0], err.data_ptr() if err is not None else None,
                               _stream(stream))
    _check("paged_kv_append", st)


def paged_kv_append_rope(q, k_new, v_new, k_pool, v_pool, slot_mapping, positions, *,
                         q_norm_weight=None, k_norm_weight=None, v_norm=False, eps=1e-6,
                         rope_theta=10000.0, rotary_dim=None, err=None, stream=None):
    """RMS-norm q / k / v, rotate q and k (rotate-half RoPE over the first
    ``rotary_dim`` channels, default all), append k / v at their slots and
    overwrite q (or skip it when ``q`` is None)."""
    nb, hkv, bs, d = k_pool.shape
    rd = d if rotary_dim is None else int(rotary_dim)
    st = lib().paged_kv_append_rope(
        _ptr(q), k_new.data_ptr(), v_new.data_ptr(), k_pool.data_ptr(), v_pool.data_ptr(), nb,
        q.shape[1] if q is not None else 0, hkv, bs, d, slot_mapping.data_ptr(),
        _ptr(positions), slot_mapping.shape[0], _ptr(q_norm_weight), _ptr(k_norm_weight),
        1 if v_norm else 0, float(eps), float(rope_theta), rd, _ptr(err), _stream(stream))
    _check("paged_kv_append_rope", st)


# ------------------------------------------------------------ batch runners
class DecodeSplitK:
    """Split-K decode of one batch: plan once, own the fp32 partials, run.

    ``run`` issues two launches (split-K partials, then the combine) on the
    current stream.
    """

    def __init__(self, batch, sm_count: int = 0):
        import torch
        self.batch = batch
        B, Hkv, D, Hq = batch.num_requests, batch.num_kv_heads, batch.head_dim, batch.num_q_heads
        self.num_splits, self.split_blocks = paged_decode_splitk_plan(
            B, Hkv, batch.max_seq_len, batch.block_size, batch.window, sm_count)
        dev = batch.q.device
        self.partial_o = torch.empty((B, Hq, self.num_splits, D), dtype=torch.float32, device=dev)
        self.partial_lse = torch.empty((B, Hq, self.num_splits), dtype=torch.float32, device=dev)
        self.out = torch.empty_like(batch.q)

    def run(self, err=None, lse_out=None):
        b = self.batch
        paged_decode_splitk(b.q, self.partial_o, self.partial_lse, b.k_pool, b.v_pool,
                            b.block_tables, b.seq_lens, b.max_seq_len, self.num_splits,
                            self.split_blocks, scale=b.scale, softcap=b.softcap,
                            window=b.window, err=err)
        paged_decode_splitk_combine(self.partial_o, self.partial_lse, self.out, lse_out)
        return self.out


class DecodeFused:
    """Split-K decode with the combine fused in: one launch per call.  Owns a
    zero-initialised workspace (its counters are left zero by each call)."""

    def __init__(self, batch):
        import torch
        self.batch = batch
        nbytes = paged_decode_attn_ws_bytes(batch.num_requests, batch.num_q_heads,
                                            batch.num_kv_heads, batch.head_dim, batch.max_seq_len,
                                            batch.window)
        self.workspace = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=batch.q.device)
        self.out = torch.empty_like(batch.q)

    def run(self, err=None):
        b = self.batch
        paged_decode_attn_ws(b.q, self.out, b.k_pool, b.v_pool, b.block_tables, b.seq_lens,
                             b.max_seq_len, self.workspace, scale=b.scale, softcap=b.softcap,
                             window=b.window, err=err)
        return self.out


class MixedBatch:
    """A varlen batch (decode rows and prefill chunks) in one launch through
    ``paged_prefill_attn_ws``.  Owns a zero-initialised workspace."""

    def __init__(self, batch):
        import torch
        self.batch = batch
        nbytes = paged_prefill_attn_ws_bytes(batch.num_requests, batch.num_q_heads,
                                             batch.num_kv_heads, batch.head_dim,
                                             batch.max_seq_len, batch.window)
        self.workspace = torch.zeros(max(nbytes, 16), dtype=torch.uint8, device=batch.q.device)
        self.out = torch.empty_like(batch.q)

    def run(self, err=None):
        b = self.batch
        paged_prefill_attn_ws(b.q, self.out, b.k_pool, b.v_pool, b.block_tables,
                              b.query_start_loc, b.seq_lens, b.max_query_len, b.max_seq_len,
                              self.workspace, scale=b.scale, softcap=b.softcap, window=b.window,
                              err=err)
        return self.out


def run_batch(batch, out=None, err=None):
    """Attention of one batch through the library (decode or varlen prefill)."""
    import torch
    if out is None:
        out = torch.empty_like(batch.q)
    paged_prefill_attn(batch.q, out, batch.k_pool, batch.v_pool, batch.block_tables,
                       batch.query_start_loc, batch.seq_lens, batch.max_query_len,
                       batch.max_seq_len, scale=batch.scale, softcap=batch.softcap,
                       window=batch.window, err=err)
    return out
