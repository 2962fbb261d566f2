"""Measure single-pass vs partitioned decode on this GPU across batch shapes.

For every (num_seqs, seq_len) of the grid below, with equal lengths in the
batch, times ``pa_decode`` (single pass), ``pa_decode_partitioned`` +
``pa_partition_reduce`` for each partition size, and ``pa_decode_auto`` with
the library's default heuristic (threshold, partition size and launch form
all chosen by the library), and prints one JSON line per point plus a
markdown table of the winner.  It is the data behind the launch heuristic
(``pa_default_single_pass_max_len``, ``pa_default_partition_size``,
``pa_auto_resolve``): the pages split sequences
longer than 8192 tokens (project_6 commit cd0d9e1, the forward_decode
heuristic) and report partition sizes of 512 and 256 (blame of
optimizations/prefix_prefill_patch.py, the _PARTITION_SIZE note); this
measures where the split pays off on GB300.

Usage: ``python -m paged_kv_decode_partitioned_gb300.sweep [--reps 60]``.
Timing: CUDA events on the launching stream, L2 flushed between reps (one
2x-L2 buffer written, another read).  The event times of a short call
cluster just below multiples of about 2.05 us, so a single rep of a 15 us
call reads one of a few values; the figure is the mean over reps after
dropping the top and bottom tenth, which resolves below that step.
"""
from __future__ import annotations

import argparse
import json
import statistics

import torch

from . import (auto_resolve, auto_workspace_bytes, decode, decode_auto, decode_partitioned,
               num_partitions, partition_buffers, partition_reduce)

SEQS = (1, 4, 16, 64, 256)
LENS = (1024, 2048, 4096, 8192, 16384, 32768, 65536)
PARTS = (256, 512, 1024)
MAX_TOKENS = 1 << 22   # points above 4M tokens (8 GiB of K+V) are skipped


def _timer(fn, reps, flush):
    times = []
    stream = torch.cuda.current_stream()
    for _ in range(3):
        fn()
    for _ in range(reps):
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    times.sort()
    cut = len(times) // 10
    kept = times[cut:len(times) - cut] if len(times) > 2 * cut else times
    return statistics.fmean(kept)


def run(reps: int = 60, seqs=SEQS, lens=LENS, parts=PARTS, hq=24, hkv=4, d=128, bs=16):
    import sys
    import os
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    from workloads import custom_workload, make_case

    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    fw = torch.empty(2 * l2, dtype=torch.uint8, device="cuda")
    fr = torch.ones(2 * l2 // 4, dtype=torch.float32, device="cuda")
    sink = torch.empty((), dtype=torch.float32, device="cuda")

    def flush():
        fw.fill_(1)
        torch.sum(fr, dim=0, out=sink)

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    w = custom_workload(num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                        dtype=torch.bfloat16)
    rows = []
    for S in seqs:
        for L in lens:
            if S * L > MAX_TOKENS:
                continue
            case = make_case(w, lengths=[L] * S, device="cuda", seed=S * 100003 + L)
            args = (case.query, case.key_cache, case.value_cache, case.block_tables,
                    case.seq_lens, w.scale)
            kvb = S * L * 2 * hkv * d * 2
            out = torch.empty_like(case.query)
            res = {"num_seqs": S, "seq_len": L}
            res["single"] = _timer(lambda: decode(*args, out=out), reps, flush)
            for P in parts:
                NP = num_partitions(L, P)
                tmp, es, ml = partition_buffers(S, hq, d, NP, "cuda")

                def part_step(P=P, NP=NP, tmp=tmp, es=es, ml=ml):
                    decode_partitioned(*args, P, NP, tmp, es, ml)
                    partition_reduce(tmp, es, ml, case.seq_lens, P, out=out, dtype=out.dtype)
                res[f"P{P}"] = _timer(part_step, reps, flush)
            thr, Pa, form = auto_resolve(S, hkv, d, bs, L, -1, 0, sms, max_total_tokens=S * L)
            ws = torch.empty(max(256, auto_workspace_bytes(S, hq, hkv, d, bs, L, S * L, -1, 0)),
                             dtype=torch.uint8, device="cuda")

            def auto_step():
                decode_auto(*args, L, -1, 0, workspace=ws, out=out, max_total_tokens=S * L)
            res["auto"] = _timer(auto_step, reps, flush)
            res["auto_threshold"] = thr
            res["auto_partition"] = Pa
            res["auto_form"] = ("single", "dense", "worklist")[form]
            modes = ["single"] + [f"P{P}" for P in parts]
            best = min(modes, key=lambda m: res[m])
            res["best"] = best
            res["best_gbs"] = round(kvb / (res[best] * 1e-3) / 1e9, 1)
            res["auto_gbs"] = round(kvb / (res["auto"] * 1e-3) / 1e9, 1)
            res["single_gbs"] = round(kvb / (res["single"] * 1e-3) / 1e9, 1)
            for m in modes + ["auto"]:
                res[m] = round(res[m], 4)
            print(json.dumps(res), flush=True)
            rows.append(res)
            del case, tmp, es, ml
            torch.cuda.empty_cache()
    return rows


def markdown(rows, parts=PARTS):
    head = "| seqs | seq_len | single ms | " + " | ".join(f"P={P} ms" for P in parts) + \
        " | best | best GB/s | auto ms (threshold, P, form) | auto GB/s | auto / best |"
    sep = "|" + "---|" * (8 + len(parts))
    lines = [head, sep]
    for r in rows:
        lines.append(f"| {r['num_seqs']} | {r['seq_len']} | {r['single']} | " +
                     " | ".join(str(r[f'P{P}']) for P in parts) +
                     f" | {r['best']} | {r['best_gbs']} | {r['auto']} ({r['auto_threshold']}, "
                     f"{r['auto_partition']}, {r['auto_form']}) | {r['auto_gbs']} | "
                     f"{r['auto'] / r[r['best']]:.3f} |")
    return "\n".join(lines)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--reps", type=int, default=60)
    a = ap.parse_args()
    from . import build
    build.build()
    rows = run(a.reps)
    print(markdown(rows))


if __name__ == "__main__":
    main()
