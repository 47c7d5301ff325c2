#!/usr/bin/env python3
"""Benchmark of the paged-KV attention hot path on GB300.

Workload (one step): the serving-shaped decode batch -- B=32 requests,
seq_lens ~ U[512, 4096], Hq=8, Hkv=2, head_dim=256, block_size=16, a pool of
16384 blocks in shuffled order, bf16 N(0,1) K/V, tanh softcap 50 -- run
through two layers with separate pools: a global layer (window 0) and a
sliding layer (window 512).

Each layer is one split-K decode launch followed by one LSE-combine launch
(``--path fused`` puts the combine into the decode launch instead).

Metric: paged-decode KV GB/s, counting algorithmic bytes (K/V rows of every
visible key plus the query rows) per step over the device time of the step.
The L2 is flushed before every timed step by a 512 MiB write followed by a
256 MiB read of the written buffer: the write evicts every line the step
could reuse, and the read evicts the flush's own dirty lines, whose
write-back would otherwise land inside the next step (a decode step is
preceded in a real engine by kernels that leave a few MB dirty, not 100+ MB).
The step is also timed after the write alone (``dirty_l2``).  The flush is
outside the per-step CUDA-event window.

``--impl reference`` times the fp64 CPU oracle on a bounded sample of the
same workload on the host cores instead.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)
# The CPU baseline (fp64 oracle) runs on one host thread; keep BLAS at one too.
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

WORKLOAD_NAME = ("decode serving: B=32, seq_lens~U[512,4096], Hq=8, Hkv=2, head_dim=256, "
                 "block_size=16, pool 16384 shuffled blocks, bf16 N(0,1), softcap 50, "
                 "two layers per step (window 0 and window 512)")
METRIC = "paged-decode KV GB/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_splitk_serving.md")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-clocks", action="store_true", help="do not sample nvidia-smi clocks")
    p.add_argument("--path", choices=["fused", "split"], default="split",
                   help="fused: split-K decode with the combine in the same launch; "
                        "split: split-K decode launch + combine launch")
    p.add_argument("--no-other", action="store_true",
                   help="skip the per-workload measurements of the other configurations")
    p.add_argument("--cpu-seconds", type=float, default=6.0,
                   help="budget of each leg of the oracle samples (CPU baseline)")
    p.add_argument("--workload", type=int, choices=[1, 3, 4, 5], default=None,
                   help="time only this other configuration (--steps launches after "
                        "--warmup) and print its entry as the JSON line")
    return p.parse_args()


def step_bytes(calls) -> float:
    """Algorithmic bytes of one step: K and V rows of every visible key, plus q."""
    total = 0
    for b in calls:
        kv_row = 2 * b.num_kv_heads * b.head_dim * 2  # K and V, bf16
        for L in b.seq_lens_host:
            vis = L if b.window <= 0 else min(L, b.window)
            total += vis * kv_row
        total += b.q.numel() * 2
    return float(total)


def launch_bytes(batch) -> float:
    kv_row = 2 * batch.num_kv_heads * batch.head_dim * 2
    vis = sum(L if batch.window <= 0 else min(L, batch.window) for L in batch.seq_lens_host)
    return float(vis * kv_row + batch.q.numel() * 2)


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            for key in ("hbm_gbs", "hbm_GBps", "hbm"):
                if key in d and isinstance(d[key], (int, float)):
                    return float(d[key]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


DECODE_SOURCES = ("decode.cu", "decode_body.cuh", "common.cuh", "tmaps.cuh")


def decode_source_hash() -> str:
    """sha256[:16] over the decode kernel's source files, in a fixed order."""
    import hashlib
    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        h.update(open(os.path.join(ROOT, "paged_kv_attention_12_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def traffic_from_profile():
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current decode kernel source (else None)."""
    import hashlib
    if not os.path.exists(PROFILE_SUMMARY):
        return None
    h = decode_source_hash()
    vals = {}
    for line in open(PROFILE_SUMMARY):
        if ": " in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(": ", 1)
            vals[k.strip()] = (v.split() or [""])[0]
    if vals.get("decode kernel source sha256[:16]") != h:
        return None
    try:
        return float(vals["dram bytes per launch (avg)"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi SM clock / throttle-reason samples during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        import tempfile
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def _oracle_task(task):
    """One piece of the CPU baseline, run in a spawned host process: the
    oracle on a saved sub-batch (``path``, an .npz of oracle inputs),
    ``reps`` times.  The loaded inputs stay cached in the process."""
    import numpy as np
    import oracle
    path, reps = task
    cache = _oracle_task.__dict__.setdefault("cache", {})
    if path not in cache:
        with np.load(path) as z:
            arr = {k: z[k] for k in z.files}
        for k in ("scale", "softcap"):
            arr[k] = float(arr[k])
        arr["window"] = int(arr["window"])
        cache[path] = arr
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.run_batch(cache[path])
    return time.perf_counter() - t0


def _noop(_):
    return os.getpid()


def _save_sub_batch(arr, path, rows=None):
    """Writes the oracle inputs of one request (``arr`` from to_numpy_f64 with
    one request), optionally only query rows [r0, r1) of its chunk: the rows
    keep their positions (seq_len shortened by the rows dropped after r1)."""
    import numpy as np
    out = {k: v for k, v in arr.items() if k != "q_rows"}
    if rows is not None:
        r0, r1 = rows
        n = int(arr["query_start_loc"][1])
        out["q"] = arr["q"][r0:r1]
        out["query_start_loc"] = np.array([0, r1 - r0], dtype=np.int64)
        out["seq_lens"] = arr["seq_lens"] - (n - r1)
    np.savez(path, **out)


def _run_pool(tasks, procs):
    """Wall time of the tasks over ``procs`` spawned processes (already
    started and warmed up before the clock starts)."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")  # never fork a process that holds a CUDA context
    with ctx.Pool(procs) as pool:
        pool.map(_noop, range(4 * procs), chunksize=1)
        t0 = time.perf_counter()
        pool.map(_oracle_task, tasks, chunksize=1)
        return time.perf_counter() - t0


def cpu_baseline(calls, prefill_batch, budget_s: float):
    """The fp64 oracle, as it stands, on bounded samples of the workloads, on
    one host thread and on every host core (one spawned process per core,
    BLAS at one thread each); inputs are saved beforehand, so the timings
    cover the oracle alone.

    decode: every request of both layers, each repeated to fill the budget
    (GB/s of K/V + q, the metric's unit); prefill (the chunked-prefill
    workload): 16-row groups of query rows spread evenly over each request's
    chunk (TFLOP/s over the sampled rows' visible (query, key) pairs)."""
    import shutil
    import tempfile

    from paged_kv_attention_12_gb300 import workload
    procs = max(1, os.cpu_count() or 1)
    tmp = tempfile.mkdtemp(prefix="pka_oracle_")
    try:
        # ---- decode: one file per request of each layer
        files, nbytes, t_pass = [], 0.0, 0.0
        for li, batch in enumerate(calls):
            for b in range(batch.num_requests):
                arr = workload.to_numpy_f64(batch, [b])
                path = os.path.join(tmp, f"d{li}_{b}.npz")
                _save_sub_batch(arr, path)
                files.append(path)
                L = batch.seq_lens_host[b]
                vis = L if batch.window <= 0 else min(L, batch.window)
                nbytes += vis * 2 * batch.num_kv_heads * batch.head_dim * 2 + \
                    batch.num_q_heads * batch.head_dim * 2
                t_pass += _oracle_task((path, 1))  # calibration pass, in this process
        reps1 = max(1, int(round(budget_s / max(t_pass, 1e-6))))
        t1 = _run_pool([(f, reps1) for f in files], 1)
        repsn = reps1 * procs
        tn = _run_pool([(f, repsn) for f in files], procs)
        dec1 = nbytes * reps1 / t1 / 1e9
        decn = nbytes * repsn / tn / 1e9
        # ---- prefill: 16-row groups spread evenly over every chunk
        pre = {}
        if prefill_batch is not None:
            B = prefill_batch.num_requests
            qsl = prefill_batch.query_start_host()
            arrs = [workload.to_numpy_f64(prefill_batch, [b]) for b in range(B)]
            paths = []
            for b in range(B):
                p = os.path.join(tmp, f"p{b}.npz")
                _save_sub_batch(arrs[b], p)
                paths.append(p)

            def pairs(b, r0, r1):
                L, n = prefill_batch.seq_lens_host[b], qsl[b + 1] - qsl[b]
                return sum(L - n + i + 1 for i in range(r0, r1))  # causal, no window

            # calibration: the last group of the longest request
            bl = max(range(B), key=lambda x: prefill_batch.seq_lens_host[x])
            n_bl = qsl[bl + 1] - qsl[bl]
            cal = os.path.join(tmp, "pcal.npz")
            _save_sub_batch(arrs[bl], cal, (n_bl - 16, n_bl))
            t_pair = _oracle_task((cal, 1)) / pairs(bl, n_bl - 16, n_bl)
            total_pairs = sum(pairs(b, 0, qsl[b + 1] - qsl[b]) for b in range(B))

            def sample(frac):
                tasks, npairs = [], 0
                for b in range(B):
                    n = qsl[b + 1] - qsl[b]
                    groups = max(1, n // 16)
                    take = max(1, min(groups, int(round(groups * frac))))
                    for k in range(take):
                        g = (k * groups) // take
                        r0, r1 = g * 16, min(n, g * 16 + 16)
                        p = os.path.join(tmp, f"p{b}_{r0}.npz")
                        if not os.path.exists(p):
                            _save_sub_batch(arrs[b], p, (r0, r1))
                        tasks.append((p, 1))
                        npairs += pairs(b, r0, r1)
                return tasks, npairs

            fl = 4.0 * prefill_batch.head_dim * prefill_batch.num_q_heads
            frac1 = min(1.0, budget_s / max(total_pairs * t_pair, 1e-6))
            tasks1, np1 = sample(frac1)
            p1 = _run_pool(tasks1, 1)
            tasksn, npn = sample(min(1.0, frac1 * procs))
            pn = _run_pool(tasksn, procs)
            pre = {"unit": "TFLOP/s", "single_thread": fl * np1 / p1 / 1e12,
                   "all_cores": fl * npn / pn / 1e12, "cores": procs,
                   "sample": f"chunked-prefill workload: {np1} of {total_pairs} visible "
                             f"(query, key) pairs on one thread ({p1:.1f} s), {npn} on "
                             f"{procs} processes ({pn:.1f} s); 16-row groups spread over "
                             f"each chunk"}
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
    return {"value": decn, "unit": "GB/s", "cores": procs, "kind": "oracle",
            "cpu_model": cpu_model(),
            "single_thread": {"value": dec1, "unit": "GB/s", "cores": 1},
            "sample": f"decode serving workload, all {len(files)} requests of both layers: "
                      f"{reps1} passes on one thread ({t1:.1f} s), {repsn} passes over "
                      f"{procs} spawned processes ({tn:.1f} s); fp64 numpy oracle, BLAS at "
                      f"one thread per process",
            "prefill": pre}


def cpu_model() -> str:
    """The host CPU's model: /proc/cpuinfo's model name, or on Arm its
    implementer and part numbers (0x41/0xd4f is an Arm Neoverse V2 core, the
    core of NVIDIA Grace)."""
    import platform
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key, _, val = line.partition(":")
                fields.setdefault(key.strip(), val.strip())
    except OSError:
        pass
    if "model name" in fields:
        return fields["model name"]
    impl, part = fields.get("CPU implementer"), fields.get("CPU part")
    if impl and part:
        known = {("0x41", "0xd4f"): "Arm Neoverse V2"}
        name = known.get((impl.lower(), part.lower()), "Arm")
        return f"{name} (implementer {impl}, part {part}, {platform.machine()})"
    return platform.machine()


def bf16_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            d = json.load(open(path))
            for key in ("bf16_tflops", "bf16_TFLOPs", "bf16"):
                if key in d and isinstance(d[key], (int, float)):
                    return float(d[key]), "measured"
        except Exception:
            pass
    return FALLBACK_BF16_TFLOPS, "fallback"


def attention_pairs(batch) -> int:
    """Visible (query, key) pairs of a varlen batch."""
    pairs = 0
    for L, n in zip(batch.seq_lens_host, batch.q_lens_host):
        for i in range(n):
            pos = L - n + i
            lo = 0 if batch.window <= 0 else max(0, pos - batch.window + 1)
            pairs += pos - lo + 1
    return pairs


def batch_kv_bytes(batch) -> float:
    """K/V rows of every key some query of the request sees (each once)."""
    kv_row = 2 * batch.num_kv_heads * batch.head_dim * 2
    total = 0
    for L, n in zip(batch.seq_lens_host, batch.q_lens_host):
        if n == 0:
            continue
        lo = 0 if batch.window <= 0 else max(0, L - n - batch.window + 1)
        total += (L - lo) * kv_row
    return float(total + batch.q.numel() * 2)


class L2Flush:
    """Evicts the L2 before a timed region: a write of a 512 MiB buffer (four
    times the L2), then, unless ``dirty``, a read of its first 256 MiB, which
    evicts the dirty lines the write left so that their write-back does not
    fall into the timed region."""

    def __init__(self, dev):
        import torch
        self.buf = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
        self.acc = torch.empty((), dtype=torch.float32, device=dev)
        self.dirty = False

    def __call__(self, value: float = 1.0, dirty: bool = None):
        import torch
        self.buf.fill_(value)
        if not (self.dirty if dirty is None else dirty):
            torch.sum(self.buf[: self.buf.numel() // 2], dim=0, out=self.acc)


def time_launches(fn, flush, iters, warmup):
    """Median device time (ms) of fn() with the L2 flushed before it: CUDA
    events around the replay of a CUDA graph of (L2 flush, fn), minus the
    same around a graph of the flush alone -- as the serving step's launches
    are timed -- so that neither the flush nor a graph's own start-up latency
    counts as fn's time."""
    import torch
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        flush(1.0)
        fn()
    torch.cuda.synchronize()

    def graph_of(body):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            body()
        return g
    g_flush = graph_of(lambda: flush(1.0))
    g_both = graph_of(lambda: (flush(1.0), fn()))
    for g in (g_flush, g_both):
        g.replay()
    torch.cuda.synchronize()
    t_flush, t_both = [], []
    for _ in range(iters):
        for g, acc in ((g_flush, t_flush), (g_both, t_both)):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            acc.append((e0, e1))
    torch.cuda.synchronize()
    med = lambda ts: statistics.median(a.elapsed_time(b) for a, b in ts)
    return med(t_both) - med(t_flush)


def other_workloads(dev, flush, iters=10, warmup=3, cfgs=(1, 3, 4, 5)):
    """The tiny decode, long-context split-K, chunked-prefill and mixed-batch
    workloads, each timed alone (L2 flushed first)."""
    import torch
    from paged_kv_attention_12_gb300 import binding, workload
    hbm, hbm_kind = hbm_peak()
    tc, tc_kind = bf16_peak()
    res = {}
    for cfg in cfgs:
        batch = workload.workload(cfg, seed=0, device=dev)[0]
        nbytes = batch_kv_bytes(batch)
        flops = 4.0 * batch.head_dim * batch.num_q_heads * attention_pairs(batch)
        if cfg in (1, 3):
            r = binding.DecodeFused(batch)
            fn, path = r.run, ("paged_decode_attn_ws (split-K, combine fused; segments that "
                               "fit one per pipeline stream whole)")
        elif cfg == 5:
            r = binding.MixedBatch(batch)
            fn, path = r.run, ("paged_prefill_attn_ws (one launch: decode rows on decode "
                               "pipelines, chunks on the tcgen05 prefill pipeline -- CTA "
                               "pairs at D = 256)")
        else:
            out = torch.empty_like(batch.q)
            fn, path = (lambda b=batch, o=out: binding.run_batch(b, o)), "paged_prefill_attn"
        ms = time_launches(fn, flush, iters, warmup)
        gbs = nbytes / (ms * 1e-3) / 1e9
        tfs = flops / (ms * 1e-3) / 1e12
        entry = {"workload": workload.WORKLOADS[cfg], "path": path, "ms": ms,
                 "kv_gbs": gbs, "tflops": tfs, "bytes": nbytes, "flops": flops}
        if cfg == 4:
            entry["roofline"] = {"bound": "tensor", "achieved": tfs, "peak": tc,
                                 "peak_kind": tc_kind, "unit": "TFLOP/s", "frac": tfs / tc}
        else:
            entry["roofline"] = {"bound": "hbm", "achieved": gbs, "peak": hbm,
                                 "peak_kind": hbm_kind, "unit": "GB/s", "frac": gbs / hbm}
        if cfg == 3:
            entry["split_sweep"] = split_sweep(batch, flush, iters, warmup, hbm)
        res[str(cfg)] = entry
        del batch, fn
        torch.cuda.empty_cache()
    if cfgs == (1, 3, 4, 5):
        res["append"] = time_append(dev, flush, iters, warmup)
        res["long_chunk"] = time_long_chunk(dev, flush, iters, warmup, tc, tc_kind)
    return res


def split_sweep(batch, flush, iters, warmup, hbm):
    """The long-context decode through paged_decode_splitk + combine with
    the work line cut for fewer pipelines than the plan's (min chunk C =
    ceil(T / k) units for k pipelines, T the line's units): how many pieces a
    segment gets, against the time."""
    import torch
    from paged_kv_attention_12_gb300 import binding
    B, Hkv, Hq, D = batch.num_requests, batch.num_kv_heads, batch.num_q_heads, batch.head_dim
    nb = (batch.seq_lens.cpu() + 15) // 16
    T = int(((nb + 4) * Hkv).sum())
    tmax = (batch.max_seq_len + 15) // 16
    nbytes = batch_kv_bytes(batch)
    out = torch.empty_like(batch.q)
    res = []
    S0, C0 = binding.paged_decode_splitk_plan(B, Hkv, batch.max_seq_len, 16, batch.window)
    for k in (0, 152, 76, 38, 19):
        C = C0 if k == 0 else max(C0, -(-T // k))
        S = S0 if k == 0 else -(-tmax // C) + 1
        po = torch.empty((B, Hq, S, D), dtype=torch.float32, device=batch.q.device)
        pl = torch.empty((B, Hq, S), dtype=torch.float32, device=batch.q.device)

        def fn(C=C, S=S, po=po, pl=pl):
            binding.paged_decode_splitk(batch.q, po, pl, batch.k_pool, batch.v_pool,
                                        batch.block_tables, batch.seq_lens, batch.max_seq_len,
                                        S, C, scale=batch.scale, softcap=batch.softcap,
                                        window=batch.window)
            binding.paged_decode_splitk_combine(po, pl, out)
        ms = time_launches(fn, flush, iters, warmup)
        res.append({"pipelines_used": "plan" if k == 0 else k, "min_chunk_units": C,
                    "num_splits": S, "ms": ms, "kv_gbs": nbytes / (ms * 1e-3) / 1e9,
                    "frac": nbytes / (ms * 1e-3) / 1e9 / hbm})
        del po, pl
    return res


def time_long_chunk(dev, flush, iters, warmup, tc, tc_kind):
    """One 512-token chunk at a 16K-token prefix beside 32 decode rows of 2K
    tokens (Hq=8, Hkv=2, D=256, softcap 50): through paged_prefill_attn_ws,
    whose 16 CTA-pair items fill far less than their pair slots and are cut
    along their keys, and through paged_prefill_attn, whole pair items."""
    import torch
    from paged_kv_attention_12_gb300 import binding, workload
    L = [16896] + [2048] * 32
    n = [512] + [1] * 32
    batch = workload.make_batch(seq_lens=L, q_lens=n, num_q_heads=8, num_kv_heads=2,
                                head_dim=256, num_blocks=sum(-(-x // 16) for x in L) + 8,
                                device=dev, poison=False, cfg_id=42, seed=0, softcap=50.0)
    flops = 4.0 * batch.head_dim * batch.num_q_heads * attention_pairs(batch)
    mixed = binding.MixedBatch(batch)
    out = torch.empty_like(batch.q)
    res = {"workload": "one 512-token chunk at a 16384-token prefix + 32 decode rows of 2048 "
                       "tokens, Hq=8, Hkv=2, D=256, softcap 50", "flops": flops}
    for key, fn in (("ws_key_pieces", mixed.run),
                    ("whole_tiles", lambda: binding.run_batch(batch, out))):
        ms = time_launches(fn, flush, iters, warmup)
        res[key] = {"ms": ms, "tflops": flops / (ms * 1e-3) / 1e12,
                    "frac": flops / (ms * 1e-3) / 1e12 / tc, "peak_kind": tc_kind}
    del batch, mixed, out
    torch.cuda.empty_cache()
    return res


def time_append(dev, flush, iters, warmup):
    """paged_kv_append of the new tokens of a serving decode tick (B=32) and
    of a chunked-prefill tick (8 x 512 tokens): Hkv=2, D=256, pool 16384
    blocks, slots a random permutation; bytes = new rows read + written."""
    import torch
    from paged_kv_attention_12_gb300 import binding
    hbm, hbm_kind = hbm_peak()
    g = torch.Generator(device=dev).manual_seed(11)
    nb, hkv, bs, d = 16384, 2, 16, 256
    k_pool = torch.randn((nb, hkv, bs, d), generator=g, device=dev).to(torch.bfloat16)
    v_pool = torch.randn((nb, hkv, bs, d), generator=g, device=dev).to(torch.bfloat16)
    out = {}
    for name, T in (("decode tick, 32 tokens", 32), ("prefill tick, 4096 tokens", 4096)):
        k_new = torch.randn((T, hkv, d), generator=g, device=dev).to(torch.bfloat16)
        v_new = torch.randn((T, hkv, d), generator=g, device=dev).to(torch.bfloat16)
        slots = torch.randperm(nb * bs, generator=torch.Generator().manual_seed(T))[:T]
        slots = slots.to(torch.int32).to(dev)
        ms = time_launches(lambda: binding.paged_kv_append(k_new, v_new, k_pool, v_pool, slots),
                           flush, iters, warmup)
        nbytes = 2.0 * 2 * T * hkv * d * 2
        out[name] = {"ms": ms, "bytes": nbytes, "gbs": nbytes / (ms * 1e-3) / 1e9,
                     "roofline": {"bound": "hbm", "peak": hbm, "peak_kind": hbm_kind,
                                  "frac": nbytes / (ms * 1e-3) / 1e9 / hbm}}
    # the same prefill tick with RMS norm of q, k, v and RoPE of q, k fused in
    # (Hq = 8: q rows are read and written too)
    T, hq = 4096, 8
    q = torch.randn((T, hq, d), generator=g, device=dev).to(torch.bfloat16)
    k_new = torch.randn((T, hkv, d), generator=g, device=dev).to(torch.bfloat16)
    v_new = torch.randn((T, hkv, d), generator=g, device=dev).to(torch.bfloat16)
    slots = torch.randperm(nb * bs, generator=torch.Generator().manual_seed(T))[:T]
    slots = slots.to(torch.int32).to(dev)
    pos = torch.arange(T, dtype=torch.int32, device=dev) + 8000
    w = torch.ones(d, device=dev)
    ms = time_launches(lambda: binding.paged_kv_append_rope(
        q, k_new, v_new, k_pool, v_pool, slots, pos, q_norm_weight=w, k_norm_weight=w,
        v_norm=True, rope_theta=1e6), flush, iters, warmup)
    nbytes = 2.0 * T * (hq + 2 * hkv) * d * 2
    out["prefill tick, 4096 tokens, norms + RoPE"] = {
        "ms": ms, "bytes": nbytes, "gbs": nbytes / (ms * 1e-3) / 1e9,
        "roofline": {"bound": "hbm", "peak": hbm, "peak_kind": hbm_kind,
                     "frac": nbytes / (ms * 1e-3) / 1e9 / hbm}}
    return out


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device(f"cuda:{local}"))
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest value over the ranks (the slowest rank's time)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_seed(seed: int, rank: int) -> int:
    """Each replica draws its own workload (weak scaling, no data exchange)."""
    return seed + 1000 * rank


def run_reference(args):
    """Oracle arm: each step is a bounded sample of the workload on host cores."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from paged_kv_attention_12_gb300 import workload
    calls = workload.decode_serving(args.seed, "cpu")
    import oracle
    per_step = []
    step_budget = max(1.0, 60.0 / max(1, args.steps + args.warmup))
    vals = []
    for it in range(args.warmup + args.steps):
        done, t = 0.0, 0.0
        for batch in calls:
            b = it % batch.num_requests
            arr = workload.to_numpy_f64(batch, [b])
            t0 = time.perf_counter()
            oracle.run_batch(arr)
            t += time.perf_counter() - t0
            L = batch.seq_lens_host[b]
            vis = L if batch.window <= 0 else min(L, batch.window)
            done += vis * 2 * batch.num_kv_heads * batch.head_dim * 2 + \
                batch.num_q_heads * batch.head_dim * 2
            if t > step_budget:
                break
        if it >= args.warmup:
            vals.append(done / t / 1e9)
            per_step.append(t)
    value = statistics.median(vals)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * statistics.median(per_step), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME, "sample": "one request per layer per step"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "one decode request of each layer per step, fp64 numpy "
                                   "oracle, one thread"},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    import torch
    world, rank, local = dist_setup(args)
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    from paged_kv_attention_12_gb300 import _build, binding, workload
    if rank == 0 or world > 1:
        _build.build()
    binding.lib()

    if args.workload is not None:
        flush = L2Flush(dev)
        entry = other_workloads(dev, flush, iters=args.steps, warmup=max(args.warmup, 1),
                                cfgs=(args.workload,))[str(args.workload)]
        if rank == 0:
            print(json.dumps({"workload_only": args.workload, "n_gpus": world, "steps": args.steps,
                              "warmup": args.warmup, "data": "synthetic", **entry}))
        return 0

    calls = workload.decode_serving(replica_seed(args.seed, rank), dev)
    if args.path == "fused":
        runners = [binding.DecodeFused(b) for b in calls]
    else:
        runners = [binding.DecodeSplitK(b) for b in calls]
    bytes_step = step_bytes(calls)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()

    # A step's per-call inputs (q, block tables, seq_lens of both layers) live
    # in one device buffer and its outputs in another, so that the end-to-end
    # measurement moves them with one host->device and one device->host copy
    # per step, as a serving engine would batch its uploads.
    def packed(tensors):
        offs, n = [], 0
        for t in tensors:
            offs.append(n)
            n += (t.numel() * t.element_size() + 255) // 256 * 256
        buf = torch.zeros(n, dtype=torch.uint8, device=dev)
        views = []
        for t, o in zip(tensors, offs):
            v = buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
            v.copy_(t)
            views.append(v)
        return buf, views

    in_buf, in_views = packed([x for b in calls for x in (b.q, b.block_tables, b.seq_lens)])
    for i, b in enumerate(calls):
        b.q, b.block_tables, b.seq_lens = in_views[3 * i:3 * i + 3]
    out_buf, out_views = packed([r.out for r in runners])
    for r, v in zip(runners, out_views):
        r.out = v

    def launch(i):
        """The decode kernel of call i (the dominant kernel)."""
        b, r = calls[i], runners[i]
        if args.path == "fused":
            binding.paged_decode_attn_ws(b.q, r.out, b.k_pool, b.v_pool, b.block_tables,
                                         b.seq_lens, b.max_seq_len, r.workspace, scale=b.scale,
                                         softcap=b.softcap, window=b.window)
        else:
            binding.paged_decode_splitk(b.q, r.partial_o, r.partial_lse, b.k_pool, b.v_pool,
                                        b.block_tables, b.seq_lens, b.max_seq_len, r.num_splits,
                                        r.split_blocks, scale=b.scale, softcap=b.softcap,
                                        window=b.window)

    def step():
        for i, r in enumerate(runners):
            launch(i)
            if args.path == "split":
                binding.paged_decode_splitk_combine(r.partial_o, r.partial_lse, r.out)

    for _ in range(args.warmup):
        flush(1.0)
        step()
    torch.cuda.synchronize()
    # One step as a CUDA graph: the launches of a step run back to back on the
    # GPU, whatever the host-side cost of issuing them.
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(2):
        flush(1.0)
        graph.replay()
    torch.cuda.synchronize()

    sampler = ClockSampler(local) if (rank == 0 and not args.no_clocks) else None
    if sampler:
        sampler.start()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    for s_ in range(args.steps):
        flush(float(s_))
        ev[s_][0].record(stream)
        graph.replay()
        ev[s_][1].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t_wall
    clocks = sampler.stop() if sampler else None
    step_ms = [a.elapsed_time(b) for a, b in ev]
    print("step ms: " + " ".join(f"{x:.3f}" for x in step_ms), file=sys.stderr)
    total_ms = max_over_ranks(sum(step_ms), world)
    ms_per_step = total_ms / args.steps
    value = world * bytes_step / (ms_per_step * 1e-3) / 1e9

    # the same steps after the write alone: the flush's dirty lines are
    # written back while the step runs
    dev_ev = []
    barrier(world)
    for s_ in range(args.steps):
        flush(float(s_), dirty=True)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        graph.replay()
        e1.record(stream)
        dev_ev.append((e0, e1))
    torch.cuda.synchronize()
    dirty_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in dev_ev), world) / args.steps
    dirty_l2 = {"value": world * bytes_step / (dirty_ms * 1e-3) / 1e9, "unit": "GB/s",
                "ms_per_step": dirty_ms,
                "l2": "512 MiB write only before every step (its dirty lines are written "
                      "back during the step)"}

    # the dominant kernel alone: each decode launch timed by CUDA events on its
    # stream as the difference between a CUDA graph of (L2 flush, launch) and
    # a graph of the flush alone, so that neither the flush nor the graph's
    # own start-up latency counts as kernel time
    def graph_of(fn):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        return g
    fgraph = graph_of(lambda: flush(1.0))
    kgraphs = [graph_of(lambda i=i: (flush(1.0), launch(i))) for i in range(len(calls))]
    torch.cuda.synchronize()

    def timed(g):
        k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k0.record(stream)
        g.replay()
        k1.record(stream)
        return (k0, k1)
    t_flush, t_kern = [], [[] for _ in calls]
    for s_ in range(args.steps):
        t_flush.append(timed(fgraph))
        for i in range(len(calls)):
            t_kern[i].append(timed(kgraphs[i]))
    torch.cuda.synchronize()
    flush_med = statistics.median(a.elapsed_time(b) for a, b in t_flush)
    kern_ms = []  # per step, per call (flattened in call order within a step)
    kmed = [statistics.median(a.elapsed_time(b) for a, b in t_kern[i]) - flush_med
            for i in range(len(calls))]
    for s_ in range(args.steps):
        for i in range(len(calls)):
            kern_ms.append(kmed[i])

    # end to end through the public API with pinned host buffers
    e2e = None
    if not args.no_e2e:
        host_in = in_buf.cpu().pin_memory()
        host_out = torch.empty(out_buf.shape, dtype=out_buf.dtype).pin_memory()
        h2d = host_in.numel()
        d2h = host_out.numel()

        def e2e_step():
            in_buf.copy_(host_in, non_blocking=True)
            step()
            host_out.copy_(out_buf, non_blocking=True)

        # the copies are part of the step's graph (memcpy nodes before and
        # after the kernels): every replay moves the step's inputs from and its
        # outputs to pinned host memory
        e2e_step()
        torch.cuda.synchronize()
        e2e_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(e2e_graph):
            e2e_step()
        e_ms = []
        for s in range(args.warmup + args.steps):
            flush(float(s))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            e2e_graph.replay()
            e1.record(stream)
            e1.synchronize()
            if s >= args.warmup:
                e_ms.append(e0.elapsed_time(e1))
        e2e_ms = max_over_ranks(sum(e_ms) / len(e_ms), world)
        e2e = {"value": world * bytes_step / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return 0

    peak, peak_kind = hbm_peak()
    kern_avg_s = sum(kern_ms) / len(kern_ms) * 1e-3
    achieved = (bytes_step / len(calls)) / kern_avg_s / 1e9
    # each layer's decode launch on its own (median over the steps)
    per_launch = []
    for i, b in enumerate(calls):
        ms_i = kmed[i]
        gbs_i = launch_bytes(b) / (ms_i * 1e-3) / 1e9
        per_launch.append({"call": b.name or f"call {i}", "window": b.window,
                           "bytes": launch_bytes(b), "ms": ms_i, "achieved": gbs_i,
                           "frac": gbs_i / peak})
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": WORKLOAD_NAME,
                   "l2": "flushed before every step: 512 MiB write, then a 256 MiB read of "
                         "the written buffer (evicts the flush's dirty lines)",
                   "path": ("paged_decode_attn_ws (split-K, combine fused)" if args.path == "fused"
                            else "paged_decode_splitk + paged_decode_splitk_combine"),
                   "timing": "each step one CUDA-graph replay, CUDA events around it; a "
                             "launch alone: graph of (flush, launch) minus graph of the flush",
                   "bytes_per_step": bytes_step, "parallelism": f"replicas{world}"},
        "roofline": {"bound": "hbm", "kernel": "paged_decode_kernel" + (" (split-K, fused combine)" if args.path == "fused" else " (split-K)"),
                     "achieved": achieved, "peak": peak, "peak_kind": peak_kind,
                     "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic_from_profile(), "per_launch": per_launch},
        "gpu_launches": args.steps * len(calls) * (1 if args.path == "fused" else 2),
        "wall_s": wall,
    }
    line["dirty_l2"] = dirty_l2
    if e2e:
        line["e2e"] = e2e
    if clocks:
        line["clocks"] = clocks
    if not args.no_other and world == 1:
        line["other_workloads"] = other_workloads(dev, flush)
    if not args.no_cpu_baseline and world == 1:
        pre = workload.chunked_prefill(0, dev)
        line["cpu_baseline"] = cpu_baseline(calls, pre, args.cpu_seconds)
        del pre
    print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
