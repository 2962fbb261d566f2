"""Measure the prefix prefill (``pa_prefill``) on this GPU across shapes.

For every point of the grid below -- head_dim, (query heads, KV heads), block
size, and a batch of (sequences, chunk tokens, cached tokens before the
chunk) -- times one ``pa_prefill`` call and prints one JSON line per point
plus a markdown table.  The rate counts the algorithmic FLOPs, 4 * head_dim *
query heads per (chunk row, cache token it sees), the causal triangle of the
chunk included once (row i of a chunk of n over c cached tokens sees c + i + 1
tokens), against the call's CUDA-event time.

Usage: ``python -m paged_kv_decode_partitioned_gb300.prefill_sweep [--reps 10]``.
Inputs: seeded synthetic caches and queries (``workloads.make_prefill_case``),
bf16 unless ``--dtype f16``.  Timing: CUDA events on the launching stream, L2
flushed between reps (a 2x-L2 buffer written); the median over reps.
"""
from __future__ import annotations

import argparse
import json
import statistics

import torch

from . import prefill

HEAD_DIMS = (64, 128, 256)
HEADS = ((32, 32), (32, 8), (24, 4), (64, 8), (32, 2))   # GQA 1, 4, 6, 8, 16
BATCHES = (   # (sequences, chunk tokens, cached tokens before the chunk)
    (16, 512, 4096),
    (4, 2048, 16384),
    (2, 8192, 0),
    (8, 128, 32768),
)
BLOCK_SIZES = (16,)


def flops(seqs: int, n: int, ctx: int, hq: int, d: int) -> float:
    visible = n * ctx + n * (n + 1) // 2
    return 4.0 * d * hq * seqs * visible


def time_point(d, hq, hkv, bs, seqs, n, ctx, dtype, reps, flush):
    from workloads import custom_workload, make_prefill_case
    w = custom_workload(num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                        dtype=dtype)
    pc = make_prefill_case(w, ctx_lens=[ctx] * seqs, q_lens=[n] * seqs, device="cuda",
                           seed=11)
    c = pc.case
    out = torch.empty_like(pc.query)

    def call():
        prefill(pc.query, c.key_cache, c.value_cache, c.block_tables, c.seq_lens, pc.q_start,
                c.scale, n, out=out)

    for _ in range(3):
        call()
    stream = torch.cuda.current_stream()
    times = []
    for _ in range(reps):
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        call()
        e1.record(stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1))
    ms = statistics.median(times)
    del pc, c, out
    torch.cuda.empty_cache()
    return ms


def run(reps: int = 10, dtype=torch.bfloat16, head_dims=HEAD_DIMS, heads=HEADS,
        batches=BATCHES, block_sizes=BLOCK_SIZES):
    from . import load_library
    load_library()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    buf = torch.empty(2 * l2, dtype=torch.uint8, device="cuda")

    def flush():
        buf.fill_(1)

    rows = []
    for d in head_dims:
        for hq, hkv in heads:
            for bs in block_sizes:
                for seqs, n, ctx in batches:
                    ms = time_point(d, hq, hkv, bs, seqs, n, ctx, dtype, reps, flush)
                    tf = flops(seqs, n, ctx, hq, d) / (ms * 1e-3) / 1e12
                    r = {"head_dim": d, "num_q_heads": hq, "num_kv_heads": hkv,
                         "block_size": bs, "seqs": seqs, "chunk": n, "ctx": ctx,
                         "ms": round(ms, 4), "tflops": round(tf, 1)}
                    print(json.dumps(r), flush=True)
                    rows.append(r)
    return rows


def table(rows) -> str:
    batches = []
    for r in rows:
        k = (r["seqs"], r["chunk"], r["ctx"])
        if k not in batches:
            batches.append(k)
    head = "| head_dim | q / kv heads | block | " + " | ".join(
        f"{s} x {n} over {c}" for s, n, c in batches) + " |"
    lines = [head, "|" + "---|" * (3 + len(batches))]
    keys = []
    for r in rows:
        k = (r["head_dim"], r["num_q_heads"], r["num_kv_heads"], r["block_size"])
        if k not in keys:
            keys.append(k)
    for d, hq, hkv, bs in keys:
        vals = []
        for s, n, c in batches:
            v = [r["tflops"] for r in rows if (r["head_dim"], r["num_q_heads"], r["num_kv_heads"],
                                              r["block_size"], r["seqs"], r["chunk"],
                                              r["ctx"]) == (d, hq, hkv, bs, s, n, c)]
            vals.append(f"{v[0]:.0f}" if v else "-")
        lines.append(f"| {d} | {hq} / {hkv} | {bs} | " + " | ".join(vals) + " |")
    return "\n".join(lines)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--reps", type=int, default=10)
    ap.add_argument("--dtype", choices=("bf16", "f16"), default="bf16")
    ap.add_argument("--block-sizes", type=int, nargs="+", default=list(BLOCK_SIZES))
    args = ap.parse_args()
    dt = torch.bfloat16 if args.dtype == "bf16" else torch.float16
    rows = run(args.reps, dt, block_sizes=tuple(args.block_sizes))
    print()
    print(f"TFLOP/s ({args.dtype}, median of {args.reps} calls, L2 flushed)")
    print(table(rows))


if __name__ == "__main__":
    main()
