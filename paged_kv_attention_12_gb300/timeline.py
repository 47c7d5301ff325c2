"""Per-pipeline phase timeline of the split-K decode kernel.

Builds an instrumented copy of the library (``-DPKA_TIMELINE``, linked to
``lib_timeline/libpaged_attn_timeline.so``; the product library is not
touched), runs the serving decode step (both layers: split-K partials, then
the combine) with the L2 evicted before every step (a 512 MiB write, then a
256 MiB read of it, so that no dirty line is written back during the step),
and reads back the
global-timer stamps that every decode pipeline wrote:

  entry        the pipeline starts
  partition    the producer knows its share of the work line
  first_issue  the producer issued the copies of its first tile
  first_tile   consumer warp 0 saw the first tile land
  last_issue   the producer issued its last copies
  last_tile    the last consumer warp finished its last tile
  exit         the last consumer warp left (results stored)

Times are in microseconds from the earliest entry of the same launch;
printed as percentiles over pipelines, medians over the steps.  The stamps
cost a few stores per pipeline and one atomic per warp and piece, so the
instrumented kernel is a little slower than the product one.

    python -m paged_kv_attention_12_gb300.timeline --steps 20 [--out FILE]
"""
from __future__ import annotations

import argparse
import os
import statistics
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

TL_LIB = os.path.join(HERE, "lib_timeline", "libpaged_attn_timeline.so")
FIELDS = ["entry", "partition", "first_issue", "first_tile", "last_issue", "last_tile", "exit"]
PIPES, NF = 1024, 8
LAYERS = ["full attention", "sliding window"]


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--out", default=None, help="also write the summary to this file")
    args = ap.parse_args(argv)

    import ctypes
    import numpy as np
    import torch

    from paged_kv_attention_12_gb300 import _build, binding, workload
    _build.build(extra=("-DPKA_TIMELINE",), lib_path=TL_LIB, verbose=True)
    binding.use_library(TL_LIB)
    L = binding.lib()
    L.pka_timeline_copy.restype = ctypes.c_int
    L.pka_timeline_copy.argtypes = [ctypes.c_void_p]
    L.pka_timeline_clear.restype = ctypes.c_int
    L.pka_timeline_clear.argtypes = [ctypes.c_void_p]

    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream()
    calls = workload.decode_serving(args.seed, dev)
    runners = [binding.DecodeSplitK(b) for b in calls]
    flush_buf = torch.empty(128 << 20, dtype=torch.float32, device=dev)
    flush_acc = torch.empty((), dtype=torch.float32, device=dev)
    snap = torch.empty(2 * PIPES * NF, dtype=torch.int64, device=dev)

    per_step = []  # [step][layer] -> ndarray (pipes, NF) relative times in us
    for s in range(args.warmup + args.steps):
        flush_buf.fill_(float(s))
        torch.sum(flush_buf[: flush_buf.numel() // 2], dim=0, out=flush_acc)
        if L.pka_timeline_clear(ctypes.c_void_p(stream.cuda_stream)) != 0:
            raise RuntimeError("timeline clear failed")
        for r in runners:
            r.run()
        torch.cuda.synchronize()
        if L.pka_timeline_copy(ctypes.c_void_p(snap.data_ptr())) != 0:
            raise RuntimeError("timeline copy failed")
        if s < args.warmup:
            continue
        raw = snap.cpu().numpy().view(np.uint64).reshape(2, PIPES, NF)
        layers = []
        for li in range(2):
            rows = raw[li]
            live = rows[:, 0] > 0
            rows = rows[live].astype(np.float64)
            t0 = rows[:, 0].min()
            rel = (rows[:, :7] - t0) / 1000.0
            layers.append((rel, rows[:, 7], t0, rows[:, 6].max()))
        per_step.append(layers)

    lines = []
    dev_name = torch.cuda.get_device_name(dev)
    lines.append(f"decode serving step, {args.steps} steps after {args.warmup} warm-up, "
                 f"L2 evicted before each step (512 MiB write + 256 MiB read), "
                 f"device {dev_name}")
    for li in range(2):
        b = calls[li]
        lines.append("")
        lines.append(f"layer {li} ({LAYERS[1 if b.window > 0 else 0]}, B={b.num_requests}, "
                     f"Hkv={b.num_kv_heads}, D={b.head_dim}, window={b.window}): "
                     f"{per_step[0][li][0].shape[0]} pipelines")
        lines.append("| stamp | p10 us | median us | p90 us | max us |")
        lines.append("|---|---|---|---|---|")
        for fi, name in enumerate(FIELDS):
            q = [np.percentile(st[li][0][:, fi], [10, 50, 90, 100]) for st in per_step]
            med = [statistics.median(x[k] for x in q) for k in range(4)]
            lines.append(f"| {name} | {med[0]:.2f} | {med[1]:.2f} | {med[2]:.2f} | {med[3]:.2f} |")
        stream_us = [np.median(st[li][0][:, 5] - st[li][0][:, 3]) for st in per_step]
        tiles = [np.median(st[li][1]) for st in per_step]
        span = [st[li][0][:, 6].max() for st in per_step]
        lines.append(f"median per-pipeline streaming time (first_tile -> last_tile): "
                     f"{statistics.median(stream_us):.2f} us over {statistics.median(tiles):.0f} "
                     f"tiles; launch span entry -> last exit: median "
                     f"{statistics.median(span):.2f} us, min {min(span):.2f} us")
    between = [(st[1][2] - st[0][3]) / 1000.0 for st in per_step]
    lines.append("")
    lines.append(f"layer 0 last exit -> layer 1 first entry (layer 0's combine launch and the "
                 f"launch gaps): median {statistics.median(between):.2f} us")
    text = "\n".join(lines)
    print(text)
    if args.out:
        with open(args.out, "w") as f:
            f.write(text + "\n")
    return 0


if __name__ == "__main__":
    sys.exit(main())
