"""Seeded synthetic inputs for paged-KV attention.

This module builds the inputs only: block pools, block tables with shared
prefix blocks, sequence lengths and query layouts.  It holds none of the
attention arithmetic, so both the CUDA path and the CPU oracle can be fed
from it without sharing any of the method.

Structure follows the inference-server pages ("Block-paged KV cache with
refcounted blocks, window-aware sliding layers", inference-server README,
engine feature list; "Block-paged per-layer KV with refcounted blocks, lazy
allocation ... vLLM/PagedAttention layout", github README, "What's inside"):

* K and V pools per layer, layout ``[num_blocks][Hkv][block_size][D]`` bf16.
* ``block_tables[b][j]`` is the physical block holding tokens
  ``j*bs .. j*bs+bs-1`` of request ``b``; padded with -1.
* Refcount-shared prefix blocks are the same ids repeated in several tables.

Generation recipe (one CPU ``torch.Generator`` seeded ``1000*cfg + seed`` for
all structure; values come from a second generator with the same seed on the
target device):

1. Lengths / prefixes: ``randint`` with inclusive bounds.
2. Block ids: one ``randperm(num_blocks)``.  The shared prefix takes the first
   ids of the permutation, then each request takes its remaining
   ``ceil(L/bs)`` blocks in request order.
3. Q, K, V ~ N(0, 1) drawn directly in bf16.
4. Parity runs poison every unreferenced block and every tail slot at or
   beyond ``seq_len`` in a request's last block with NaN, and (sliding
   windows) may point blocks no query can see at a NaN block.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import List, Optional, Sequence

import torch

BLOCK_SIZE = 16


@dataclass
class PagedBatch:
    """One attention call over a paged KV cache.

    Device tensors: ``q`` bf16 [total_q][Hq][D]; ``k_pool``/``v_pool`` bf16
    [num_blocks][Hkv][bs][D]; ``block_tables`` int32 [B][max_blocks];
    ``seq_lens`` int32 [B] (context length including the new tokens);
    ``query_start_loc`` int32 [B+1].  Host copies of the integer arrays are
    kept in the ``*_host`` lists so that callers never need a device sync.
    """

    q: torch.Tensor
    k_pool: torch.Tensor
    v_pool: torch.Tensor
    block_tables: torch.Tensor
    seq_lens: torch.Tensor
    query_start_loc: torch.Tensor
    scale: float
    softcap: float
    window: int
    seq_lens_host: List[int]
    q_lens_host: List[int]
    tables_host: List[List[int]]
    name: str = ""
    # number of distinct physical blocks referenced (shared blocks once)
    unique_blocks: int = 0

    @property
    def num_requests(self) -> int:
        return len(self.seq_lens_host)

    @property
    def num_q_heads(self) -> int:
        return self.q.shape[1]

    @property
    def num_kv_heads(self) -> int:
        return self.k_pool.shape[1]

    @property
    def head_dim(self) -> int:
        return self.q.shape[2]

    @property
    def block_size(self) -> int:
        return self.k_pool.shape[2]

    @property
    def num_blocks(self) -> int:
        return self.k_pool.shape[0]

    @property
    def max_blocks(self) -> int:
        return self.block_tables.shape[1]

    @property
    def total_q(self) -> int:
        return self.q.shape[0]

    @property
    def max_seq_len(self) -> int:
        return max(self.seq_lens_host) if self.seq_lens_host else 0

    @property
    def max_query_len(self) -> int:
        return max(self.q_lens_host) if self.q_lens_host else 0

    @property
    def is_decode(self) -> bool:
        return all(n == 1 for n in self.q_lens_host)

    def query_start_host(self) -> List[int]:
        out = [0]
        for n in self.q_lens_host:
            out.append(out[-1] + n)
        return out


def _gen(cfg_id: int, seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(1000 * cfg_id + seed)
    return g


def _randint(g: torch.Generator, lo: int, hi: int, n: int) -> List[int]:
    """``n`` integers uniform in [lo, hi] (inclusive)."""
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


def assign_blocks(g: torch.Generator, num_blocks: int, seq_lens: Sequence[int],
                  block_size: int, shared_prefix_tokens: int = 0,
                  sharers: Sequence[int] = ()) -> List[List[int]]:
    """Block tables from one seeded permutation of the pool.

    The shared prefix (whole blocks only) takes the first ids of the
    permutation; every request then takes its own blocks in request order.
    Sharers' first ``shared_prefix_tokens/bs`` entries are the shared ids.
    """
    assert shared_prefix_tokens % block_size == 0
    perm = torch.randperm(num_blocks, generator=g).tolist()
    n_shared = shared_prefix_tokens // block_size if sharers else 0
    shared = perm[:n_shared]
    cursor = n_shared
    sharer_set = set(sharers)
    tables = []
    for b, L in enumerate(seq_lens):
        nb = -(-L // block_size)
        if b in sharer_set:
            assert nb > n_shared, "a sharer's own tokens must not land in shared blocks"
            own = nb - n_shared
            row = shared + perm[cursor:cursor + own]
        else:
            own = nb
            row = perm[cursor:cursor + own]
        cursor += own
        if cursor > num_blocks:
            raise ValueError(f"pool of {num_blocks} blocks too small")
        tables.append(row)
    return tables


def _pad_tables(tables: List[List[int]], max_blocks: Optional[int] = None) -> torch.Tensor:
    width = max([len(r) for r in tables] + [1])
    if max_blocks is not None:
        assert max_blocks >= width
        width = max_blocks
    t = torch.full((len(tables), width), -1, dtype=torch.int32)
    for b, row in enumerate(tables):
        if row:
            t[b, :len(row)] = torch.tensor(row, dtype=torch.int32)
    return t


def _randn_bf16(shape, g_dev: torch.Generator, device) -> torch.Tensor:
    return torch.randn(shape, generator=g_dev, device=device, dtype=torch.bfloat16)


def make_batch(*, seq_lens: Sequence[int], q_lens: Sequence[int], num_q_heads: int,
               num_kv_heads: int, head_dim: int, num_blocks: int,
               block_size: int = BLOCK_SIZE, scale: Optional[float] = None,
               softcap: float = 0.0, window: int = 0, shared_prefix_tokens: int = 0,
               sharers: Sequence[int] = (), cfg_id: int = 0, seed: int = 0,
               device="cpu", poison: bool = False, drop_out_of_window: bool = False,
               max_blocks: Optional[int] = None, name: str = "") -> PagedBatch:
    """Build one paged batch from explicit lengths (all structure is seeded)."""
    g = _gen(cfg_id, seed)
    seq_lens = [int(x) for x in seq_lens]
    q_lens = [int(x) for x in q_lens]
    assert len(seq_lens) == len(q_lens)
    for L, n in zip(seq_lens, q_lens):
        assert 0 <= n <= L
    tables = assign_blocks(g, num_blocks, seq_lens, block_size,
                           shared_prefix_tokens, sharers)
    return _materialise(tables=tables, seq_lens=seq_lens, q_lens=q_lens,
                        num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                        head_dim=head_dim, num_blocks=num_blocks,
                        block_size=block_size, scale=scale, softcap=softcap,
                        window=window, cfg_id=cfg_id, seed=seed, device=device,
                        poison=poison, drop_out_of_window=drop_out_of_window,
                        max_blocks=max_blocks, name=name)


def _materialise(*, tables, seq_lens, q_lens, num_q_heads, num_kv_heads, head_dim,
                 num_blocks, block_size, scale, softcap, window, cfg_id, seed,
                 device, poison, drop_out_of_window, max_blocks, name,
                 pools=None) -> PagedBatch:
    device = torch.device(device)
    g_dev = torch.Generator(device=device)
    g_dev.manual_seed(1000 * cfg_id + seed + 7919)
    total_q = sum(q_lens)
    if pools is None:
        k_pool = _randn_bf16((num_blocks, num_kv_heads, block_size, head_dim), g_dev, device)
        v_pool = _randn_bf16((num_blocks, num_kv_heads, block_size, head_dim), g_dev, device)
    else:
        k_pool, v_pool = pools
    q = _randn_bf16((total_q, num_q_heads, head_dim), g_dev, device)
    referenced = sorted({i for row in tables for i in row})
    tables_used = [list(r) for r in tables]
    if poison:
        nan = float("nan")
        mask = torch.ones(num_blocks, dtype=torch.bool)
        if referenced:
            mask[torch.tensor(referenced)] = False
        free_ids = mask.nonzero().flatten()
        if free_ids.numel():
            fi = free_ids.to(device)
            k_pool[fi] = nan
            v_pool[fi] = nan
        for b, L in enumerate(seq_lens):
            if L % block_size and tables[b]:
                last = tables[b][(L - 1) // block_size]
                k_pool[last, :, L % block_size:, :] = nan
                v_pool[last, :, L % block_size:, :] = nan
        if drop_out_of_window and window > 0 and free_ids.numel():
            nan_block = int(free_ids[0])
            for b, L in enumerate(seq_lens):
                first_pos = L - q_lens[b]
                lo = max(0, first_pos - window + 1)  # earliest key any query sees
                for j in range(len(tables_used[b])):
                    if (j + 1) * block_size - 1 < lo:
                        tables_used[b][j] = nan_block
    bt = _pad_tables(tables_used, max_blocks).to(device)
    qsl = [0]
    for n in q_lens:
        qsl.append(qsl[-1] + n)
    if scale is None:
        scale = 1.0 / math.sqrt(head_dim)
    return PagedBatch(
        q=q, k_pool=k_pool, v_pool=v_pool, block_tables=bt,
        seq_lens=torch.tensor(seq_lens, dtype=torch.int32, device=device),
        query_start_loc=torch.tensor(qsl, dtype=torch.int32, device=device),
        scale=float(scale), softcap=float(softcap), window=int(window),
        seq_lens_host=list(seq_lens), q_lens_host=list(q_lens),
        tables_host=tables_used, name=name, unique_blocks=len(referenced))


# ---------------------------------------------------------------------------
# The five workloads.  ``scale_down`` shrinks lengths and pool for parity
# cases the oracle finishes in seconds while keeping the structure (several
# tiles, ragged tails, sharing, windows).
# ---------------------------------------------------------------------------

WORKLOADS = {
    1: "decode tiny: B=4, L~U[1,256], Hq=8, Hkv=2, D=128, bs=16, pool 128",
    2: "decode serving: B=32, L~U[512,4096], Hq=8, Hkv=2, D=256, bs=16, pool 16384, "
       "layers W=0 and W=512, softcap 50",
    3: "decode long-context split-K: B=4, L~U[32768,131072], Hq=16, Hkv=4, D=128, "
       "bs=16, pool 32768",
    4: "chunked prefill: 8 requests, prefix~U[0,8192] + chunk 512, requests 0-3 "
       "share 2048 prefix tokens, Hq=8, Hkv=2, D=256, bs=16",
    5: "mixed batch: 64 decode (L~U[1024,16384], 0-31 share a 2048-token prefix) + "
       "4 prefill chunks of 256 (prefix~U[0,4096]), Hq=8, Hkv=2, D=256, pool 65536, "
       "W=1024, softcap 50",
}


def decode_tiny(seed=0, device="cpu", poison=False) -> PagedBatch:
    g = _gen(1, seed)
    L = _randint(g, 1, 256, 4)
    return make_batch(seq_lens=L, q_lens=[1] * 4, num_q_heads=8, num_kv_heads=2,
                      head_dim=128, num_blocks=128, cfg_id=1, seed=seed,
                      device=device, poison=poison, name="decode_tiny")


def decode_serving(seed=0, device="cpu", poison=False, scale_down=False,
                   drop_out_of_window=False) -> List[PagedBatch]:
    """Two layers (separate pools, same lengths): W=0 then W=512; cap 50."""
    g = _gen(2, seed)
    if scale_down:
        B, lo, hi, nblk = 5, 40, 700, 512
    else:
        B, lo, hi, nblk = 32, 512, 4096, 16384
    L = _randint(g, lo, hi, B)
    tables = assign_blocks(g, nblk, L, BLOCK_SIZE)
    out = []
    for layer, window in enumerate((0, 512 if not scale_down else 96)):
        out.append(_materialise(
            tables=tables, seq_lens=L, q_lens=[1] * B, num_q_heads=8, num_kv_heads=2,
            head_dim=256, num_blocks=nblk, block_size=BLOCK_SIZE, scale=1.0 / 16.0,
            softcap=50.0, window=window, cfg_id=2, seed=seed * 10 + layer,
            device=device, poison=poison,
            drop_out_of_window=drop_out_of_window and window > 0, max_blocks=None,
            name=f"decode_serving_layer{layer}"))
    return out


def decode_long(seed=0, device="cpu", poison=False, scale_down=False) -> PagedBatch:
    g = _gen(3, seed)
    if scale_down:
        B, lo, hi = 3, 600, 2500
        nblk = 3 * (-(-hi // BLOCK_SIZE)) + 8
    else:
        B, lo, hi = 4, 32768, 131072
        nblk = 32768
    L = _randint(g, lo, hi, B)
    return make_batch(seq_lens=L, q_lens=[1] * B, num_q_heads=16, num_kv_heads=4,
                      head_dim=128, num_blocks=nblk, cfg_id=3, seed=seed,
                      device=device, poison=poison, name="decode_long")


def chunked_prefill(seed=0, device="cpu", poison=False, scale_down=False) -> PagedBatch:
    """8 requests (prefix + chunk), causal; requests 0-3 share a prefix."""
    g = _gen(4, seed)
    if scale_down:
        B, pmax, chunk, shared = 4, 300, 80, 64
    else:
        B, pmax, chunk, shared = 8, 8192, 512, 2048
    P = _randint(g, 0, pmax, B)
    sharers = list(range(min(4, B)))
    for b in sharers:
        P[b] = max(P[b], shared)
    L = [p + chunk for p in P]
    need = sum(-(-x // BLOCK_SIZE) for x in L) - (len(sharers) - 1) * (shared // BLOCK_SIZE)
    nblk = int(math.ceil(need * 1.1)) + 1
    tables = assign_blocks(g, nblk, L, BLOCK_SIZE, shared, sharers)
    return _materialise(tables=tables, seq_lens=L, q_lens=[chunk] * B, num_q_heads=8,
                        num_kv_heads=2, head_dim=256, num_blocks=nblk,
                        block_size=BLOCK_SIZE, scale=None, softcap=0.0, window=0,
                        cfg_id=4, seed=seed, device=device, poison=poison,
                        drop_out_of_window=False, max_blocks=None,
                        name="chunked_prefill")


def mixed_batch(seed=0, device="cpu", poison=False, scale_down=False,
                drop_out_of_window=False) -> PagedBatch:
    """Decode rows then prefill chunks in one varlen batch (W=1024, cap 50)."""
    g = _gen(5, seed)
    if scale_down:
        nd, dlo, dhi, npf, chunk, pmax, shared, window, nblk = 6, 80, 600, 2, 48, 200, 64, 160, 512
    else:
        nd, dlo, dhi, npf, chunk, pmax, shared, window, nblk = 64, 1024, 16384, 4, 256, 4096, 2048, 1024, 65536
    Ld = _randint(g, dlo, dhi, nd)
    sharers = list(range(nd // 2))
    for b in sharers:
        Ld[b] = max(Ld[b], shared + 1)
    P = _randint(g, 0, pmax, npf)
    L = Ld + [p + chunk for p in P]
    q_lens = [1] * nd + [chunk] * npf
    tables = assign_blocks(g, nblk, L, BLOCK_SIZE, shared, sharers)
    return _materialise(tables=tables, seq_lens=L, q_lens=q_lens, num_q_heads=8,
                        num_kv_heads=2, head_dim=256, num_blocks=nblk,
                        block_size=BLOCK_SIZE, scale=None, softcap=50.0, window=window,
                        cfg_id=5, seed=seed, device=device, poison=poison,
                        drop_out_of_window=drop_out_of_window, max_blocks=None,
                        name="mixed_batch")


def workload(cfg_id: int, seed=0, device="cpu", poison=False, scale_down=False):
    """Return the list of calls one step of workload ``cfg_id`` makes."""
    if cfg_id == 1:
        return [decode_tiny(seed, device, poison)]
    if cfg_id == 2:
        return decode_serving(seed, device, poison, scale_down)
    if cfg_id == 3:
        return [decode_long(seed, device, poison, scale_down)]
    if cfg_id == 4:
        return [chunked_prefill(seed, device, poison, scale_down)]
    if cfg_id == 5:
        return [mixed_batch(seed, device, poison, scale_down)]
    raise ValueError(cfg_id)


def to_numpy_f64(batch: PagedBatch, only_requests: Optional[Sequence[int]] = None):
    """Host fp64 copies (exact upcast of bf16) in the form the oracle takes.

    With ``only_requests`` the pools are cut down to the blocks those
    requests reference (tables renumbered), so that full-size workloads can
    be checked on sampled requests without copying a multi-GB pool.
    """
    import numpy as np
    reqs = list(range(batch.num_requests)) if only_requests is None else list(only_requests)
    qsl = batch.query_start_host()
    q_rows = [r for b in reqs for r in range(qsl[b], qsl[b + 1])]
    q = batch.q[torch.tensor(q_rows, dtype=torch.long, device=batch.q.device)] \
        if q_rows else batch.q[:0]
    tables = [batch.tables_host[b] for b in reqs]
    used = sorted({i for row in tables for i in row})
    remap = {old: new for new, old in enumerate(used)}
    if used:
        idx = torch.tensor(used, dtype=torch.long, device=batch.k_pool.device)
        kp = batch.k_pool[idx]
        vp = batch.v_pool[idx]
    else:
        kp = batch.k_pool[:1]
        vp = batch.v_pool[:1]
    width = max([len(r) for r in tables] + [1])
    bt = np.full((len(reqs), width), -1, dtype=np.int64)
    for i, row in enumerate(tables):
        bt[i, :len(row)] = [remap[x] for x in row]
    q_lens = [batch.q_lens_host[b] for b in reqs]
    qs = np.zeros(len(reqs) + 1, dtype=np.int64)
    qs[1:] = np.cumsum(q_lens)
    return dict(
        q=q.float().cpu().numpy().astype(np.float64),
        k_pool=kp.float().cpu().numpy().astype(np.float64),
        v_pool=vp.float().cpu().numpy().astype(np.float64),
        block_tables=bt,
        seq_lens=np.array([batch.seq_lens_host[b] for b in reqs], dtype=np.int64),
        query_start_loc=qs,
        scale=batch.scale, softcap=batch.softcap, window=batch.window,
        q_rows=q_rows,
    )
