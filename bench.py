#!/usr/bin/env python3
"""Benchmark of the paged-attention decode step on GB300; prints one JSON line.

A step is one pass of the whole decode path over one batch: the work list /
V1-V2 choice, the paged K/V walk, QK^T, online softmax, PV, the partition
epilogue and the log-sum-exp reduce.  The default workload is the mixed
serving batch (256 sequences, lengths log-uniform in [128, 65536], 24 query /
4 KV heads, head_dim 128, block 16, bf16; sequences <= 8192 tokens single
pass, longer ones split into 512-token partitions), the one workload whose
step runs every stage of the path.  ``--workload N`` selects another.

Timing: W untimed warm-up steps, then exactly K steps bracketed by a barrier
and a device synchronise; every step is timed with two CUDA events on the
stream the kernels are launched on, with a 2x-L2 buffer write then read
between steps, outside the events (the KV inputs are also far larger than
L2).  Per-launch times, and the attention kernel's time for the roofline,
come from a second pass of K steps with an event after every launch (an
event between two launches would add ~1 us to a timed step).  ``e2e`` repeats the step through ``pa_decode_auto`` (the one call a
user makes) with the per-step inputs copied from pinned host memory and the
output read back, inside the timed region.  ``cpu_baseline`` times the fp64
oracle on a bounded sample of the same workload on the host cores.

``--path prefill`` times the paged prefix-prefill kernel (TFLOP/s against
the bf16 tensor peak) and ``--path moe`` the MoE router + sort-by-expert
regroup + scatter-back (GB/s against the HBM peak; the step's six kernels
replay as one CUDA graph); both print a line of the same shape.  ``--impl reference`` times the oracle alone (the reference arm)
on the same workload, metric and unit.  Multi-GPU (torchrun): every rank runs its own
replica of the workload (no collective on the data path); time is the max
over ranks and the value is the total over ranks.
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention: KV-read GB/s and % of GB300 HBM peak; decode tokens/s"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
PREFILL_METRIC = "paged prefix-prefill attention: TFLOP/s on the bf16 tensor cores"
MOE_METRIC = ("MoE router + sort-by-expert regroup + scatter-back: GB/s of algorithmic HBM "
              "traffic; tokens/s")
# prefix-prefill workloads: (context tokens, chunk tokens, sequences, query heads,
# KV heads, head_dim); block 16, bf16.  The first three have the decode
# workloads' model shape (24 query / 4 KV heads, head_dim 128); the last the
# head_dim-256 attention of the pages' Qwen-family notes (16 query / 2 KV heads).
PREFILL_WORKLOADS = {
    "chunk2048_ctx16384_x16": (16384, 2048, 16, 24, 4, 128),
    "full100k_x1": (0, 100000, 1, 24, 4, 128),
    "chunk512_ctx4096_x64": (4096, 512, 64, 24, 4, 128),
    "d256_chunk2048_ctx16384_x8": (16384, 2048, 8, 16, 2, 256),
}


def prefill_workload_name(name):
    _, _, _, hq, hkv, d = PREFILL_WORKLOADS[name]
    return f"prefill_{name}_hq{hq}_hkv{hkv}_d{d}_bs16_bf16"


def prefill_kernel_name(name):
    # head_dim 256 runs on CTA pairs sharing 2-SM MMAs, the others on single CTAs
    return "pa_prefill_pair_kernel" if PREFILL_WORKLOADS[name][5] == 256 else "pa_prefill_tc_kernel"


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=4,
                    help="decode workload id: 1-5 (the five configurations), 6 (the mixed "
                         "batch with GQA 16), 7 (the mixed batch with block size 8)")
    ap.add_argument("--partition-size", type=int, default=None,
                    help="override the workload's (first) partition size (auto mode: 0 lets "
                         "the library's heuristic choose)")
    ap.add_argument("--mode", choices=["single", "partitioned", "auto"], default=None,
                    help="override the workload's decode mode")
    ap.add_argument("--single-pass-max-len", type=int, default=None,
                    help="override the workload's single-pass limit (auto mode; -1 lets the "
                         "library's heuristic choose)")
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="reduced batch of the same workload rule (for profiling captures)")
    ap.add_argument("--cpu-seconds", type=float, default=15.0,
                    help="target oracle CPU time of the cpu_baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--check", action="store_true",
                    help="also compare sampled sequences of the output with the oracle")
    ap.add_argument("--warmup-seconds", type=float, default=1.0,
                    help="minimum wall time of the warm-up (0 under a profiler, so the number "
                         "of launches before the timed steps is exactly known)")
    ap.add_argument("--path", choices=["decode", "prefill", "moe"], default="decode",
                    help="decode (default): the paged decode step; prefill: the paged "
                         "prefix-prefill kernel; moe: router + sort-by-expert regroup + "
                         "scatter-back")
    ap.add_argument("--prefill-workload", choices=sorted(PREFILL_WORKLOADS),
                    default="chunk2048_ctx16384_x16")
    return ap.parse_args()


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def kv_bytes(case) -> int:
    w = case.workload
    return case.total_tokens * 2 * w.num_kv_heads * w.head_dim * 2


def qo_bytes(case) -> int:
    w = case.workload
    return 2 * case.num_seqs * w.num_q_heads * w.head_dim * 2


# Sources each committed traffic figure depends on (a figure is dropped when
# any of them changes).
KERNEL_SOURCES = {
    "decode": ["pa_kernels.cuh", "pa_launch.cuh", "pa_launch.h", "pa_types.h", "pa_inst_bf16.cu",
               "pa_inst_f16.cu", "pa_aux.cu", "pa_api.cu", "../../include/pa_decode.h"],
    "prefill": ["pa_prefill_tc.cuh", "pa_prefill_pair.cuh", "pa_tc05.cuh", "pa_prefill.cu",
                "pa_kernels.cuh", "pa_launch.cuh", "pa_launch.h", "pa_types.h", "pa_api.cu",
                "../../include/pa_decode.h"],
    "moe": ["pa_moe.cu", "pa_types.h", "pa_api.cu", "../../include/pa_moe.h"],
}


def source_sha(path: str = "decode") -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_decode_partitioned_gb300", "csrc")
    for name in KERNEL_SOURCES[path]:
        with open(os.path.normpath(os.path.join(csrc, name)), "rb") as fh:
            h.update(os.path.basename(name).encode())
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_bf16_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured (MEASURED_PEAKS.json bf16_tflops, cuBLAS burst)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback (1.9 PFLOP/s, one earlier GB300 measurement)"


def measured_bf16_sustained():
    """The measured cuBLAS bf16 rate back to back for seconds (under the power cap), or None."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"])
    except (OSError, KeyError, ValueError):
        return None


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback (6.8 TB/s, one earlier GB300 measurement)"


def committed_traffic(wid, partition_size=None):
    """DRAM bytes per launch of a dominant kernel from the committed ncu summary
    (key ``workload{wid}_P{P}`` for decode, else the key itself), or None if the
    kernel sources changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    key = f"workload{wid}_P{partition_size}" if partition_size is not None else wid
    path = "decode" if partition_size is not None else str(wid).split("_")[0]
    e = d.get(key)
    if not e or e.get("source_sha") != source_sha(path if path in KERNEL_SOURCES else "decode"):
        return None
    return e.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms in the background."""

    FIELDS = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank: int):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES")
        self.gpu = vis.split(",")[local_rank] if vis else str(local_rank)
        self.proc = None
        self.file = None

    def start(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[1].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    frac = float("0." + parts[1].split(".")[1]) if "." in parts[1] else 0.0
                    rows.append({"t": ts + frac, "sm": float(parts[2]), "max": float(parts[3]),
                                 "reasons": {"hw_slowdown": parts[6], "hw_thermal_slowdown":
                                             parts[7], "sw_thermal_slowdown": parts[8],
                                             "sw_power_cap": parts[9]}})
                except (ValueError, IndexError):
                    continue
        os.unlink(self.file.name)
        return rows

    @staticmethod
    def summary(rows, t0, t1):
        inside = [r for r in rows if t0 <= r["t"] <= t1]
        window = "timed region"
        if len(inside) < 3:
            inside = [r for r in rows if r["t"] <= t1]
            window = "warm-up + timed region (timed region shorter than 3 samples)"
        if not inside:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": "no samples (nvidia-smi unavailable)"}
        reasons = sorted({k for r in inside for k, v in r["reasons"].items() if v == "Active"})
        return {"sm_mhz": statistics.median(r["sm"] for r in inside),
                "sm_max_mhz": max(r["max"] for r in inside), "reasons": reasons,
                "samples": len(inside), "window": window}


def host_subcase(case, seq_ids):
    """Host copies (query, caches, tables, lengths) of some sequences of a case.

    The blocks those sequences reference are copied into a compact host pool
    and their table rows relabelled to it; the result of the attention does
    not depend on which physical block holds a page."""
    import torch
    ids = torch.as_tensor(seq_ids, dtype=torch.long)
    bs = case.key_cache.shape[1]
    lens = [case.seq_lens_list[i] for i in seq_ids]
    bt = case.block_tables.cpu()[ids]
    need = [-(-L // bs) for L in lens]
    used = torch.cat([bt[j, :n] for j, n in enumerate(need)] + [torch.zeros(0, dtype=torch.int32)])
    uniq, inv = torch.unique(used.long(), return_inverse=True)
    idx = uniq.to(case.key_cache.device)
    kc = case.key_cache.index_select(0, idx).cpu()
    vc = case.value_cache.index_select(0, idx).cpu()
    nbt = torch.full((len(seq_ids), max(need + [1])), -1, dtype=torch.int32)
    off = 0
    for j, n in enumerate(need):
        nbt[j, :n] = inv[off:off + n].to(torch.int32)
        off += n
    q = case.query.index_select(0, ids.to(case.query.device)).cpu()
    return q, kc, vc, nbt, torch.tensor(lens, dtype=torch.int32)


def oracle_sample_plan(case, target_seconds: float, seed: int = 0):
    """Pick a sample of sequences whose oracle time is about target_seconds.

    A calibration run on a few short sequences gives the oracle's rate in
    (token x query head) per second on this host."""
    import numpy as np
    import oracle
    w = case.workload
    order = list(np.random.default_rng(seed).permutation(case.num_seqs))
    calib, tok = [], 0
    for i in sorted(order, key=lambda i: case.seq_lens_list[i]):
        calib.append(int(i))
        tok += case.seq_lens_list[i]
        if tok >= 4096:
            break
    q, kc, vc, bt, sl = host_subcase(case, calib)
    t = time.perf_counter()
    oracle.attention(q, kc, vc, bt, sl, w.scale)
    rate = max(1.0, tok * w.num_q_heads / max(time.perf_counter() - t, 1e-6))
    budget = target_seconds * rate / w.num_q_heads   # tokens
    sample, tok = [], 0
    for i in order:
        L = case.seq_lens_list[i]
        if sample and tok + L > budget:
            continue
        sample.append(int(i))
        tok += L
        if tok >= budget:
            break
    return sorted(sample), tok


def time_oracle(case, sample):
    import oracle
    w = case.workload
    q, kc, vc, bt, sl = host_subcase(case, sample)
    t = time.perf_counter()
    oracle.attention(q, kc, vc, bt, sl, w.scale)
    return time.perf_counter() - t


def one_core_oracle():
    """The oracle on one host core: workload 1 whole, and workload 3 cut to one
    of its 100,000-token sequences (GB/s of K+V and seconds of each)."""
    import torch
    import oracle
    from workloads import WORKLOADS, make_case
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    res = {}
    oracle.set_num_threads(1)
    try:
        for key, wid, kw in (("workload1", 1, {}), ("workload3_one_seq", 3,
                                                    {"lengths": [100000]})):
            case = make_case(WORKLOADS[wid], device=dev, seed=rank_seed(wid, 0), **kw)
            ids = list(range(case.num_seqs))
            secs = time_oracle(case, ids)
            res[key] = {"value": round(kv_bytes(case) / secs / 1e9, 4), "unit": "GB/s",
                        "seconds": round(secs, 4), "tokens": case.total_tokens}
            del case
    finally:
        oracle.set_num_threads(cpu_threads())
    return res


def cpu_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def rank_seed(wid: int, rank: int) -> int:
    """Seed of a rank's batch: rank 0 uses the workload's own seed and every
    other rank draws an independent batch of the same workload rule."""
    from workloads import SEED_BASE
    return SEED_BASE + wid + 1000 * rank


def make_inputs(wid, device, num_seqs=None, rank=0):
    from workloads import make_case, workload
    return make_case(workload(wid), device=device, num_seqs=num_seqs, seed=rank_seed(wid, rank))


def across_ranks(world: int, device, max_vals=(), sum_vals=()):
    """Max over ranks of each value of max_vals and sum over ranks of each of
    sum_vals (plain lists when world == 1).  Only timing and byte counts cross
    ranks; the decode itself has no collective."""
    max_vals, sum_vals = [float(v) for v in max_vals], [float(v) for v in sum_vals]
    if world == 1:
        return max_vals, sum_vals
    import torch
    import torch.distributed as dist
    out = []
    for vals, op in ((max_vals, dist.ReduceOp.MAX), (sum_vals, dist.ReduceOp.SUM)):
        t = torch.tensor(vals + [0.0], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=op)
        out.append(t.tolist()[:len(vals)])
    return out[0], out[1]


def whole_job(total_ms_max: float, steps: int, kv_bytes_sum: float, seqs_sum: float):
    """(ms per step, KV-read GB/s, decode tokens/s) of the whole job: every
    rank's bytes and sequences over the slowest rank's time (weak scaling)."""
    ms = total_ms_max / steps
    return ms, kv_bytes_sum / (ms * 1e-3) / 1e9, seqs_sum / (ms * 1e-3)


def run_reference(args, rank, world):
    """The oracle, as it stands, on the host cores (the reference arm)."""
    import torch
    if rank != 0:
        return
    import oracle
    oracle.build()
    # rank 0 alone runs the oracle, on every host core (torchrun sets
    # OMP_NUM_THREADS=1 for its ranks)
    oracle.set_num_threads(cpu_threads())
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    case = make_inputs(args.workload, dev, args.num_seqs)
    w = case.workload
    per_step = max(1.0, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
    sample, tok = oracle_sample_plan(case, per_step)
    kvb = tok * 2 * w.num_kv_heads * w.head_dim * 2
    for _ in range(args.warmup):
        time_oracle(case, sample)
    times = [time_oracle(case, sample) for _ in range(args.steps)]
    mean = sum(times) / len(times)
    value = kvb / mean / 1e9
    threads = cpu_threads()
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(mean * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "global_batch": case.num_seqs,
                   "seq_len": case.max_seq_len, "parallelism": "host threads (OpenMP)"},
        "decode_tokens_per_s": round(len(sample) / mean, 3),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{len(sample)} of {case.num_seqs} sequences, {tok} tokens "
                                   f"per step"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# The next rows of the path: prefix prefill and the MoE regrouping
# ---------------------------------------------------------------------------
def prefill_flops(ctx_lens, q_lens, num_q_heads, head_dim):
    """4 * d * Hq * (visible cache tokens summed over chunk rows): QK^T and PV."""
    vis = 0
    for c, n in zip(ctx_lens, q_lens):
        vis += n * c + n * (n + 1) // 2
    return 4.0 * head_dim * num_q_heads * vis


def graph_of(launches, stream):
    """The step's launches captured once into a CUDA graph (warmed up first on a
    side stream, as capture requires); returns its replay function."""
    import torch
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        for _, fn in launches:
            fn()
    stream.wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _, fn in launches:
            fn()
    torch.cuda.synchronize()
    return g.replay


def timed_steps(launches, K, warmup, flush_l2, stream, warmup_seconds=1.0, step_fn=None):
    """Run W (and at least 1 s of) warm-up steps, then K timed steps, each
    bracketed by its own two CUDA events; a spin kernel holds the stream while
    the host enqueues, so no host gap falls inside a step.  Per-launch times
    come from a second pass of K steps with an event after every launch (an
    event between two launches costs the step ~1 us, so the timed steps carry
    none).  ``step_fn`` (a CUDA-graph replay of the launches) runs the step in
    the warm-up and the timed steps when given.  Returns (per-step ms,
    per-launch mean ms, wall-clock start, end of the timed steps)."""
    import torch
    run_step = step_fn if step_fn is not None else (lambda: [fn() for _, fn in launches])
    t_soak, n = time.time(), 0
    while n < warmup or time.time() - t_soak < warmup_seconds:
        flush_l2()
        run_step()
        n += 1
        if n % 16 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(4):
        flush_l2()
        for _, fn in launches:
            fn()
    host_step = (time.perf_counter() - t0) / 4
    torch.cuda.synchronize()
    hold = int(min(2.0, 1.5 * K * host_step + 0.005) * 2.2e9)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    torch.cuda._sleep(hold)
    w0 = time.time()
    for k in range(K):
        flush_l2(k)
        ev[k][0].record(stream)
        run_step()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    w1 = time.time()
    step_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)]
    if len(launches) == 1:
        return step_ms, {launches[0][0]: sum(step_ms) / K}, w0, w1
    lev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(launches) + 1)]
           for _ in range(K)]
    torch.cuda._sleep(hold)
    for k in range(K):
        flush_l2(k)
        lev[k][0].record(stream)
        for j, (_, fn) in enumerate(launches):
            fn()
            lev[k][j + 1].record(stream)
    torch.cuda.synchronize()
    launch_ms = {name: sum(lev[k][j].elapsed_time(lev[k][j + 1]) for k in range(K)) / K
                 for j, (name, _) in enumerate(launches)}
    return step_ms, launch_ms, w0, w1


def timed_e2e(fn, K, flush_l2, stream):
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    e0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    e1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    for k in range(K):
        flush_l2(k)
        e0[k].record(stream)
        fn()
        e1[k].record(stream)
    torch.cuda.synchronize()
    return sum(e0[k].elapsed_time(e1[k]) for k in range(K))


def make_prefill_inputs(name, device, rank=0):
    import torch
    from workloads import custom_workload, make_prefill_case
    ctx, n, S, hq, hkv, d = PREFILL_WORKLOADS[name]
    w = custom_workload(num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=16,
                        dtype=torch.bfloat16, name=f"prefill_{name}")
    return make_prefill_case(w, ctx_lens=[ctx] * S, q_lens=[n] * S, device=device,
                             seed=20261400 + 1000 * rank), (ctx, n, S)


def oracle_prefill_sample(pc, rows: int):
    """The oracle's prefix prefill on the last ``rows`` chunk rows of sequence 0
    (they see the most context): host copies of that sequence's blocks."""
    import torch
    import oracle
    c = pc.case
    L = c.seq_lens_list[0]
    n = pc.q_lens[0]
    rows = max(1, min(rows, n))
    bs = c.key_cache.shape[1]
    nb = -(-L // bs)
    blocks = c.block_tables[0, :nb].long()
    kc = c.key_cache.index_select(0, blocks).cpu()
    vc = c.value_cache.index_select(0, blocks).cpu()
    bt = torch.arange(nb, dtype=torch.int32)[None, :]
    q = pc.query[n - rows:n].cpu()
    qs = torch.tensor([0, rows], dtype=torch.int32)
    sl = torch.tensor([L], dtype=torch.int32)
    t = time.perf_counter()
    oracle.prefill(q, kc, vc, bt, sl, qs, c.scale)
    secs = time.perf_counter() - t
    flops = 4.0 * c.workload.head_dim * c.workload.num_q_heads * sum(
        L - rows + i + 1 for i in range(rows))
    return secs, flops, rows


def run_next_path(args, rank, world, local_rank):
    """``--path prefill`` / ``--path moe``: one JSON line in the same contract."""
    import torch
    import torch.distributed as dist
    if args.impl == "reference":
        if rank != 0:
            return
        return run_next_reference(args, world)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the product path has no CPU fallback)")
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    from paged_kv_decode_partitioned_gb300 import build as pa_build
    if rank == 0:
        pa_build.build()
    if world > 1:
        dist.barrier()
    pa_build.build()
    import paged_kv_decode_partitioned_gb300 as pa
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(local_rank).L2_cache_size
    flush_w = torch.empty(max(2 * l2, 64 << 20), dtype=torch.uint8, device="cuda")
    flush_r = torch.ones(max(2 * l2, 64 << 20) // 4, dtype=torch.float32, device="cuda")
    flush_sink = torch.empty((), dtype=torch.float32, device="cuda")

    def flush_l2(k=1):
        flush_w.fill_(k & 0xFF)
        torch.sum(flush_r, dim=0, out=flush_sink)

    K = args.steps
    sampler = ClockSampler(local_rank)
    sampler.start()
    if args.path == "prefill":
        pc, (ctx, n, S) = make_prefill_inputs(args.prefill_workload, "cuda", rank)
        c = pc.case
        w = c.workload
        out = torch.empty_like(pc.query)

        def run():
            pa.prefill(pc.query, c.key_cache, c.value_cache, c.block_tables, c.seq_lens,
                       pc.q_start, c.scale, n, out=out)
        launches = [("prefill", run)]
        step_ms, launch_ms, w0, w1 = timed_steps(launches, K, args.warmup, flush_l2, stream,
                                                 args.warmup_seconds)
        if pa.device_status() != 0:
            raise SystemExit("device status flags raised")
        flops = prefill_flops([ctx] * S, [n] * S, w.num_q_heads, w.head_dim)
        (tot_ms,), (fl_all, tok_all) = across_ranks(world, "cuda", [sum(step_ms)],
                                                    [flops, n * S])
        ms = tot_ms / K
        value = fl_all / (ms * 1e-3) / 1e12
        peak, peak_src = measured_bf16_peak()
        sus = measured_bf16_sustained()
        achieved = flops / (launch_ms["prefill"] * 1e-3) / 1e12
        e2e = None
        if not args.no_e2e:
            hq = pc.query.cpu().pin_memory()
            hqs = pc.q_start.cpu().pin_memory()
            hsl = c.seq_lens.cpu().pin_memory()
            hbt = c.block_tables.cpu().pin_memory()
            hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
            h2d = (hq.numel() * 2 + hqs.numel() * 4 + hsl.numel() * 4 + hbt.numel() * 4)

            def e2e_step():
                pc.query.copy_(hq, non_blocking=True)
                pc.q_start.copy_(hqs, non_blocking=True)
                c.seq_lens.copy_(hsl, non_blocking=True)
                c.block_tables.copy_(hbt, non_blocking=True)
                run()
                hout.copy_(out, non_blocking=True)
            (e_ms,), _ = across_ranks(world, "cuda", [timed_e2e(e2e_step, K, flush_l2, stream)])
            e2e = {"value": round(fl_all / (e_ms / K * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                   "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(hout.numel() * 2),
                   "kv_cache": "resident in HBM; chunk query, tables and lengths copied in"}
        cpu = None
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            secs, fl, rows = oracle_prefill_sample(pc, 8)
            rows = max(1, min(n, int(rows * args.cpu_seconds / max(secs, 1e-3))))
            secs, fl, rows = oracle_prefill_sample(pc, rows)
            cpu = {"value": round(fl / secs / 1e12, 6), "unit": "TFLOP/s", "cores": cpu_threads(),
                   "kind": "oracle",
                   "sample": f"the last {rows} chunk rows of sequence 0 ({fl / 1e9:.1f} GFLOP), "
                             f"{secs:.1f} s"}
        name = prefill_workload_name(args.prefill_workload)
        line = {
            "metric": PREFILL_METRIC, "value": round(value, 2), "unit": "TFLOP/s",
            "n_gpus": world, "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": name, "global_batch": S * world, "context_tokens": ctx,
                       "chunk_tokens": n,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "flushed between steps (outside the events)"},
            "prefill_tokens_per_s": round(tok_all / (ms * 1e-3), 1),
            "roofline": {"bound": "tensor", "kernel": prefill_kernel_name(args.prefill_workload),
                         "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(achieved / peak, 4),
                         # the timed launches run back to back for seconds, under the
                         # power cap: the sustained cuBLAS rate is shown beside the burst
                         "sustained_peak": sus,
                         "frac_of_sustained": round(achieved / sus, 4) if sus else None,
                         "traffic": committed_traffic(f"prefill_{args.prefill_workload}"),
                         "algorithmic_flops_per_launch": flops,
                         "kernel_ms_per_launch": round(launch_ms["prefill"], 4),
                         "peak_source": peak_src},
            "cpu_baseline": cpu, "e2e": e2e,
            "launch_ms": {k: round(v, 4) for k, v in launch_ms.items()},
            "gpu_launches": K, "clocks": None,
        }
    else:
        from workloads import make_moe_case
        case = make_moe_case(device="cuda", seed=20261500 + 1000 * rank)
        T, E, K_, H = case.num_tokens, case.num_experts, case.topk, case.hidden.shape[1]
        P = T * K_
        w = torch.empty((T, K_), dtype=torch.float32, device="cuda")
        ids = torch.empty((T, K_), dtype=torch.int32, device="cuda")
        ws = torch.empty(pa.moe_sort_workspace_bytes(P, E), dtype=torch.uint8, device="cuda")
        sp = torch.empty(P, dtype=torch.int32, device="cuda")
        off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
        pos = torch.empty(P, dtype=torch.int32, device="cuda")
        y = torch.empty((P, H), dtype=case.hidden.dtype, device="cuda")
        out = torch.empty_like(case.hidden)
        launches = [
            ("topk_softmax", lambda: pa.topk_softmax(case.logits, K_, True, weights=w, ids=ids)),
            ("sort", lambda: pa.moe_sort(ids, E, workspace=ws, out=(sp, off, pos))),
            ("gather", lambda: pa.moe_gather(case.hidden, pos, K_, out=y)),
            ("scatter_back", lambda: pa.moe_scatter_back(y, pos, w, out=out)),
        ]
        # the step's six kernels replay as one CUDA graph (no launch gaps from the host)
        replay = graph_of(launches, stream)
        step_ms, launch_ms, w0, w1 = timed_steps(launches, K, args.warmup, flush_l2, stream,
                                                 args.warmup_seconds, step_fn=replay)
        if pa.device_status() != 0:
            raise SystemExit("device status flags raised")
        row = H * 2
        alg = {"topk_softmax": T * E * 2 + T * K_ * 8,
               "sort": 3 * P * 4 + 2 * P * 4,          # ids read by 3 launches; order + inverse
               "gather": P * row + T * row,
               "scatter_back": P * row + T * row + T * K_ * 8}
        step_bytes = sum(alg.values())
        (tot_ms,), (b_all, t_all) = across_ranks(world, "cuda", [sum(step_ms)], [step_bytes, T])
        ms = tot_ms / K
        value = b_all / (ms * 1e-3) / 1e9
        peak, peak_src = measured_peaks()
        dom = "gather"
        achieved = alg[dom] / (launch_ms[dom] * 1e-3) / 1e9
        e2e = None
        if not args.no_e2e:
            hl = case.logits.cpu().pin_memory()
            hh = case.hidden.cpu().pin_memory()
            hout = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)

            def e2e_step():
                case.logits.copy_(hl, non_blocking=True)
                case.hidden.copy_(hh, non_blocking=True)
                for _, fn in launches:
                    fn()
                hout.copy_(out, non_blocking=True)
            (e_ms,), _ = across_ranks(world, "cuda", [timed_e2e(e2e_step, K, flush_l2, stream)])
            e2e = {"value": round(b_all / (e_ms / K * 1e-3) / 1e9, 2), "unit": "GB/s",
                   "h2d_bytes_per_step": int(hl.numel() * 2 + hh.numel() * 2),
                   "d2h_bytes_per_step": int(hout.numel() * 2)}
        cpu = None
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            cpu = oracle_moe_sample(case, args.cpu_seconds)
        line = {
            "metric": MOE_METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": K, "warmup": args.warmup, "ms_per_step": round(ms, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": f"moe_T{T}_E{E}_top{K_}_H{H}_bf16_identity_expert",
                       "global_batch": T * world,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": "flushed between steps (outside the events)",
                       "launch": "the step's 6 kernels replayed as one CUDA graph",
                       "expert": "identity (the expert GEMMs need trained weights; not built)"},
            "tokens_per_s": round(t_all / (ms * 1e-3), 1),
            "roofline": {"bound": "hbm", "kernel": "pa_moe_gather_kernel",
                         "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4),
                         "traffic": committed_traffic("moe_gather"),
                         "algorithmic_bytes_per_launch": alg[dom],
                         "kernel_ms_per_launch": round(launch_ms[dom], 4),
                         "peak_source": peak_src,
                         "per_kernel_gbs": {k: round(alg[k] / (launch_ms[k] * 1e-3) / 1e9, 1)
                                            for k in alg}},
            "cpu_baseline": cpu, "e2e": e2e,
            "launch_ms": {k: round(v, 4) for k, v in launch_ms.items()},
            "gpu_launches": K * 6,   # router 1, sort 3, gather 1, scatter-back 1
            "clocks": None,
        }
    rows = sampler.stop()
    if rank != 0:
        return
    line["clocks"] = ClockSampler.summary(rows, w0, w1)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def oracle_moe_sample(case, target_seconds):
    """The oracle's router + sort + gather + scatter-back on the first tokens of
    the batch, sized to about target_seconds on the host cores."""
    import numpy as np
    import oracle
    oracle.build()

    def chain(t):
        logits = case.logits[:t].cpu()
        hidden = case.hidden[:t].cpu()
        s0 = time.perf_counter()
        w, ids = oracle.topk_softmax(logits, case.topk, True)
        sp, off, pos = oracle.moe_sort(ids, case.num_experts)
        y = oracle.moe_gather(hidden, sp, case.topk)
        import torch
        oracle.moe_scatter(torch.from_numpy(y.view(np.int16)).view(torch.bfloat16), pos, w,
                           case.topk)
        return time.perf_counter() - s0

    t = 256
    secs = chain(t)
    t = int(max(1, min(case.num_tokens, t * target_seconds / max(secs, 1e-3))))
    secs = chain(t)
    H = case.hidden.shape[1]
    P = t * case.topk
    byts = t * case.num_experts * 2 + 2 * (P * H * 2 + t * H * 2)
    return {"value": round(byts / secs / 1e9, 4), "unit": "GB/s", "cores": cpu_threads(),
            "kind": "oracle",
            "sample": f"the first {t} of {case.num_tokens} tokens, {secs:.1f} s"}


def run_next_reference(args, world):
    """``--impl reference`` for the prefill / MoE paths: the oracle on the host."""
    import torch
    import oracle
    oracle.set_num_threads(cpu_threads())   # every host core, whatever torchrun set
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    steps = []
    if args.path == "prefill":
        pc, (ctx, n, S) = make_prefill_inputs(args.prefill_workload, dev)
        per_step = max(1.0, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
        secs, fl, rows = oracle_prefill_sample(pc, 4)
        rows = max(1, min(n, int(rows * per_step / max(secs, 1e-3))))
        for _ in range(args.warmup + args.steps):
            secs, fl, rows = oracle_prefill_sample(pc, rows)
            steps.append(secs)
        steps = steps[args.warmup:]
        mean = sum(steps) / len(steps)
        value, unit = fl / mean / 1e12, "TFLOP/s"
        sample = f"the last {rows} chunk rows of sequence 0 per step"
        metric, wl = PREFILL_METRIC, prefill_workload_name(args.prefill_workload)
    else:
        from workloads import make_moe_case
        case = make_moe_case(device=dev, seed=20261500)
        per_step = max(1.0, min(10.0, 150.0 / max(1, args.steps + args.warmup)))
        vals = []
        for _ in range(args.warmup + args.steps):
            c = oracle_moe_sample(case, per_step)
            vals.append(c)
        vals = vals[args.warmup:]
        value = sum(v["value"] for v in vals) / len(vals)
        unit, sample = "GB/s", vals[-1]["sample"]
        mean = None
        metric = MOE_METRIC
        wl = f"moe_T{case.num_tokens}_E{case.num_experts}_top{case.topk}_H" \
             f"{case.hidden.shape[1]}_bf16_identity_expert"
    line = {
        "impl": "reference", "metric": metric, "value": round(value, 6), "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(mean * 1e3, 3) if mean else None, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl, "parallelism": "host threads (OpenMP)"},
        "cpu_baseline": {"value": round(value, 6), "unit": unit, "cores": cpu_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": unit, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    rank, world, local_rank = dist_env()
    if args.path != "decode":
        if args.impl == "ours" and (args.steps < 1 or args.warmup < 3):
            raise SystemExit("need --steps >= 1 and --warmup >= 3")
        run_next_path(args, rank, world, local_rank)
        return
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    if args.steps < 1 or args.warmup < 3:
        raise SystemExit("need --steps >= 1 and --warmup >= 3")

    import torch
    import torch.distributed as dist

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the product path has no CPU fallback)")
    torch.cuda.set_device(local_rank)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))

    def barrier():
        if world > 1:
            dist.barrier()

    from paged_kv_decode_partitioned_gb300 import build as pa_build
    if rank == 0:
        pa_build.build()
    barrier()
    pa_build.build()
    import paged_kv_decode_partitioned_gb300 as pa
    from paged_kv_decode_partitioned_gb300.step import DecodeStep

    case = make_inputs(args.workload, "cuda", args.num_seqs, rank)
    w = case.workload
    P = w.partition_sizes[0] if args.partition_size is None else args.partition_size
    mode = args.mode or w.mode
    thr = w.single_pass_max_len if args.single_pass_max_len is None else args.single_pass_max_len
    step = DecodeStep(mode, case.query, case.key_cache, case.value_cache, case.block_tables,
                      case.seq_lens, w.scale, max_seq_len=case.max_seq_len, partition_size=P,
                      single_pass_max_len=thr, max_total_tokens=case.total_tokens)
    launches = step.launches()
    stream = torch.cuda.current_stream()
    l2 = torch.cuda.get_device_properties(local_rank).L2_cache_size
    # L2 flush between steps: write one 2x-L2 buffer, then read another, so the
    # step starts with L2 full of clean lines (a write-only flush would leave
    # dirty lines whose write-back lands inside the next timed step).
    flush_w = torch.empty(max(2 * l2, 64 << 20), dtype=torch.uint8, device="cuda")
    flush_r = torch.ones(max(2 * l2, 64 << 20) // 4, dtype=torch.float32, device="cuda")
    flush_sink = torch.empty((), dtype=torch.float32, device="cuda")

    def flush_l2(k=1):
        flush_w.fill_(k & 0xFF)
        torch.sum(flush_r, dim=0, out=flush_sink)

    sampler = ClockSampler(local_rank)
    sampler.start()
    # W warm-up steps, continued for at least 1 s so the clock sampler sees
    # the same load before the timed region starts.
    t_soak, n = time.time(), 0
    while n < args.warmup or time.time() - t_soak < args.warmup_seconds:
        flush_l2()
        step()
        n += 1
        if n % 16 == 0:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    if pa.device_status() != 0:
        raise SystemExit("device status flags raised during warm-up")

    K = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    # Host cost of enqueuing one step (flush + launches + events), measured
    # while the GPU is busy, sizes the stream hold below.
    t0 = time.perf_counter()
    for _ in range(4):
        flush_l2()
        for _, fn in launches:
            fn()
    host_step = (time.perf_counter() - t0) / 4
    barrier()
    torch.cuda.synchronize()

    def hold_stream(steps):
        # A spin kernel holds the stream while the host enqueues the timed
        # steps, so no host-side launch gap can fall inside a step's events.
        secs = min(2.0, 1.5 * steps * host_step + 0.005)
        torch.cuda._sleep(int(secs * 2.2e9))

    hold_stream(K)
    t_wall0 = time.time()
    for k in range(K):   # the timed steps: each step's own two events only
        flush_l2(k)
        ev[k][0].record(stream)
        for _, fn in launches:
            fn()
        ev[k][1].record(stream)
    torch.cuda.synchronize()
    barrier()
    t_wall1 = time.time()
    rows = sampler.stop()
    step_ms = [ev[k][0].elapsed_time(ev[k][1]) for k in range(K)]

    # Per-launch times from a second pass with an event after every launch (an
    # event between two launches costs the step ~1 us, so the timed steps carry
    # none); with one launch per step the timed steps give it directly.
    names = [name for name, _ in launches]
    attn_idx = names.index("attention")
    if len(launches) == 1:
        attn_ms = step_ms
        launch_ms = {names[0]: round(sum(step_ms) / K, 4)}
    else:
        lev = [[torch.cuda.Event(enable_timing=True) for _ in range(len(launches) + 1)]
               for _ in range(K)]
        hold_stream(K)
        for k in range(K):
            flush_l2(k)
            lev[k][0].record(stream)
            for j, (_, fn) in enumerate(launches):
                fn()
                lev[k][j + 1].record(stream)
        torch.cuda.synchronize()
        attn_ms = [lev[k][attn_idx].elapsed_time(lev[k][attn_idx + 1]) for k in range(K)]
        # mean event time of each launch of the step (includes the gap before it)
        launch_ms = {n: round(sum(lev[k][j].elapsed_time(lev[k][j + 1]) for k in range(K)) / K, 4)
                     for j, n in enumerate(names)}
    kvb = kv_bytes(case)
    (total_ms,), (kvb_all, seqs_all) = across_ranks(world, "cuda", [sum(step_ms)],
                                                    [kvb, case.num_seqs])
    ms_per_step, value, tok_s = whole_job(total_ms, K, kvb_all, seqs_all)
    peak, peak_src = measured_peaks()
    alg = kvb + qo_bytes(case)
    attn_mean_ms = sum(attn_ms) / K
    achieved = alg / (attn_mean_ms * 1e-3) / 1e9

    # end to end through pa_decode_auto / the public calls with host buffers
    e2e = None
    if not args.no_e2e:
        hq = case.query.cpu().pin_memory()
        hbt = case.block_tables.cpu().pin_memory()
        hsl = case.seq_lens.cpu().pin_memory()
        hout = torch.empty(step.out.shape, dtype=step.out.dtype, pin_memory=True)
        h2d = hq.numel() * hq.element_size() + hbt.numel() * 4 + hsl.numel() * 4
        d2h = hout.numel() * hout.element_size()

        def e2e_step():
            case.query.copy_(hq, non_blocking=True)
            case.block_tables.copy_(hbt, non_blocking=True)
            case.seq_lens.copy_(hsl, non_blocking=True)
            step()
            hout.copy_(step.out, non_blocking=True)

        for _ in range(3):
            e2e_step()
        torch.cuda.synchronize()
        e0 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        e1 = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
        barrier()
        hold_stream(K)
        for k in range(K):
            flush_l2(k)
            e0[k].record(stream)
            e2e_step()
            e1[k].record(stream)
        torch.cuda.synchronize()
        (e2e_ms,), _ = across_ranks(world, "cuda", [sum(e0[k].elapsed_time(e1[k])
                                                      for k in range(K))])
        e2e = {"value": round(whole_job(e2e_ms, K, kvb_all, seqs_all)[1], 3), "unit": "GB/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "kv_cache": "resident in HBM (decode state); per-step inputs copied"}

    check = None
    if args.check and rank == 0:
        import numpy as np
        import oracle
        torch.cuda.synchronize()
        ids = sorted({int(np.argmax(case.seq_lens_list)), int(np.argmin(case.seq_lens_list)), 0})
        q, kc, vc, bt, sl = host_subcase(case, ids)
        ref = oracle.attention(q, kc, vc, bt, sl, w.scale)
        got = step.out.index_select(0, torch.as_tensor(ids, device="cuda")).float().cpu().double()
        err = (got.numpy() - ref)
        ok = bool((abs(err) <= 1e-2 + 1e-2 * abs(ref)).all())
        check = {"seqs": ids, "max_abs_err": float(abs(err).max()), "pass": ok}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        sample, tok = oracle_sample_plan(case, args.cpu_seconds)
        secs = time_oracle(case, sample)
        skv = tok * 2 * w.num_kv_heads * w.head_dim * 2
        cpu = {"value": round(skv / secs / 1e9, 4), "unit": "GB/s", "cores": cpu_threads(),
               "kind": "oracle",
               "sample": f"{len(sample)} of {case.num_seqs} sequences ({tok} tokens) of the "
                         f"same workload, {secs:.1f} s",
               "one_core": one_core_oracle()}

    if rank != 0:
        return
    clocks = ClockSampler.summary(rows, t_wall0, t_wall1)
    traffic = committed_traffic(args.workload, P)
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16"
        if w.dtype.__repr__().endswith("bfloat16") else "f16", "data": "synthetic",
        "config": {"workload": w.name if args.num_seqs is None else
                   f"{w.name} (reduced to {case.num_seqs} sequences)",
                   "global_batch": int(seqs_all),
                   "seq_len": case.max_seq_len, "total_tokens": case.total_tokens,
                   "mode": mode, "partition_size": step.resolved[1] if mode == "auto" else P,
                   "single_pass_max_len": step.resolved[0] if mode == "auto" else thr,
                   "launch_form": ("single", "dense", "worklist")[step.form]
                   if mode == "auto" else mode,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "l2": f"flushed between steps (outside the events): {flush_w.numel() >> 20} "
                         f"MiB written, then {flush_r.numel() * 4 >> 20} MiB read; "
                         f"K/V inputs {kvb / 2**30:.2f} GiB > L2"},
        "decode_tokens_per_s": round(tok_s, 1),
        "hbm_frac_kv": round(value / world / peak, 4),   # per GPU
        "hbm_frac_kvqo": round((alg / (ms_per_step * 1e-3) / 1e9) / peak, 4),
        "roofline": {"bound": "hbm", "kernel": step.attention_kernel,
                     "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "algorithmic_bytes_per_launch": alg,
                     "attention_ms_per_launch": round(attn_mean_ms, 4),
                     "peak_source": peak_src},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "launch_ms": launch_ms,
        "gpu_launches": K * len(launches),
        "clocks": clocks,
    }
    if check is not None:
        line["check"] = check
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
