"""Host-side logic of bench.py (no GPU): the roofline numerators, the clock
record that decides whether a run is kept, and the guard that drops a
committed traffic figure once the kernel sources change."""
import json
import random

import pytest
import torch

import bench
from workloads import WORKLOADS, custom_workload, make_case


def test_prefill_flops_counts_every_visible_pair():
    """4 * d * Hq per (chunk row, cache token it sees): row i of a chunk of n
    after ctx cached tokens sees ctx + i + 1 tokens (itself included)."""
    rng = random.Random(5)
    for _ in range(20):
        S = rng.randint(1, 5)
        ctx = [rng.randint(0, 300) for _ in range(S)]
        n = [rng.randint(0, 200) for _ in range(S)]
        hq, d = rng.choice([1, 6, 16]), rng.choice([64, 128, 256])
        brute = sum(c + i + 1 for c, m in zip(ctx, n) for i in range(m))
        assert bench.prefill_flops(ctx, n, hq, d) == 4.0 * d * hq * brute


def test_kv_bytes_is_one_key_and_one_value_row_per_token_and_kv_head():
    w = custom_workload(num_q_heads=24, num_kv_heads=4, head_dim=128, block_size=16,
                        dtype=torch.bfloat16)
    case = make_case(w, device="cpu", num_seqs=3, seed=1)
    lens = case.seq_lens.tolist()
    assert bench.kv_bytes(case) == sum(lens) * 2 * 4 * 128 * 2   # K and V, bf16
    assert bench.qo_bytes(case) == 2 * 3 * 24 * 128 * 2          # query in, output out


def test_workload_two_kv_bytes_match_its_lengths():
    case = make_case(WORKLOADS[2], device="cpu", num_seqs=4, seed=2)
    w = case.workload
    assert bench.kv_bytes(case) == int(case.seq_lens.sum()) * 2 * w.num_kv_heads * w.head_dim * 2


def _rows(ts, sm=2070.0, reasons=None):
    rows = []
    for k, t in enumerate(ts):
        r = {"hw_slowdown": "Not Active", "hw_thermal_slowdown": "Not Active",
             "sw_thermal_slowdown": "Not Active", "sw_power_cap": "Not Active"}
        if reasons and k in reasons:
            r[reasons[k]] = "Active"
        rows.append({"t": t, "sm": sm, "max": 2070.0, "reasons": r})
    return rows


def test_clock_summary_keeps_only_reasons_seen_in_the_timed_region():
    rows = _rows([0.0, 0.1, 1.0, 1.1, 1.2, 1.3, 5.0],
                 reasons={0: "hw_thermal_slowdown", 3: "sw_power_cap", 6: "hw_slowdown"})
    s = bench.ClockSampler.summary(rows, 1.0, 1.3)
    assert s["window"] == "timed region"
    assert s["samples"] == 4
    assert s["reasons"] == ["sw_power_cap"]   # the warm-up's and the tail's are outside
    assert s["sm_mhz"] == 2070.0 and s["sm_max_mhz"] == 2070.0


def test_clock_summary_falls_back_to_the_warm_up_for_a_short_timed_region():
    rows = _rows([0.0, 0.1, 0.2, 0.3, 1.05], reasons={1: "hw_slowdown"})
    s = bench.ClockSampler.summary(rows, 1.0, 1.1)
    assert s["window"].startswith("warm-up + timed region")
    assert s["samples"] == 5
    assert s["reasons"] == ["hw_slowdown"]


def test_clock_summary_without_samples():
    s = bench.ClockSampler.summary([], 0.0, 1.0)
    assert s["samples"] == 0 and s["sm_mhz"] is None and s["reasons"] == []


def test_clock_summary_median_of_the_samples():
    rows = _rows([1.0, 1.1, 1.2])
    for r, mhz in zip(rows, (1900.0, 2000.0, 2070.0)):
        r["sm"] = mhz
    assert bench.ClockSampler.summary(rows, 1.0, 1.2)["sm_mhz"] == 2000.0


def test_committed_traffic_is_dropped_when_the_sources_change(monkeypatch, tmp_path):
    """A committed ncu figure is reported only while the kernel sources it was
    taken on are unchanged (their hash is stored beside it)."""
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({
        "workload4_P512": {"dram_bytes_per_launch": 123, "source_sha": "a" * 16},
        "prefill_chunk": {"dram_bytes_per_launch": 456, "source_sha": "b" * 16}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    shas = {"decode": "a" * 16, "prefill": "b" * 16}
    monkeypatch.setattr(bench, "source_sha", lambda path="decode": shas.get(path, "c" * 16))
    assert bench.committed_traffic(4, partition_size=512) == 123
    assert bench.committed_traffic("prefill_chunk") == 456
    assert bench.committed_traffic(3, partition_size=512) is None   # no figure taken
    shas["decode"] = "d" * 16                                        # decode sources changed
    assert bench.committed_traffic(4, partition_size=512) is None
    assert bench.committed_traffic("prefill_chunk") == 456


def test_source_hash_covers_every_listed_source():
    for path, names in bench.KERNEL_SOURCES.items():
        assert len(bench.source_sha(path)) == 16
    # each path's hash changes with any one of its files (a byte appended here)
    import hashlib, os
    csrc = os.path.join(bench.ROOT, "paged_kv_decode_partitioned_gb300", "csrc")
    for path, names in bench.KERNEL_SOURCES.items():
        for drop in names:
            h = hashlib.sha256()
            for name in names:
                with open(os.path.normpath(os.path.join(csrc, name)), "rb") as fh:
                    data = fh.read()
                h.update(os.path.basename(name).encode())
                h.update(data + (b"x" if name == drop else b""))
            assert h.hexdigest()[:16] != bench.source_sha(path)


def test_whole_job_rates():
    ms, gbs, tok = bench.whole_job(100.0, 10, 5e9, 256)
    assert ms == 10.0
    assert gbs == pytest.approx(500.0)
    assert tok == pytest.approx(25600.0)


def test_prefill_sweep_flops_and_table():
    """The sweep tool's FLOP count agrees with the bench's brute-force-checked one,
    and its table has one row per shape and one column per batch."""
    from paged_kv_decode_partitioned_gb300 import prefill_sweep as ps
    for s, n, c in ps.BATCHES:
        assert ps.flops(s, n, c, 24, 128) == bench.prefill_flops([c] * s, [n] * s, 24, 128)
    rows = [{"head_dim": d, "num_q_heads": 8, "num_kv_heads": 2, "block_size": 16, "seqs": s,
             "chunk": n, "ctx": c, "ms": 1.0, "tflops": 1.0}
            for d in (64, 128) for s, n, c in ps.BATCHES[:2]]
    lines = ps.table(rows).splitlines()
    assert len(lines) == 2 + 2
    assert all(line.count("|") == 3 + 2 + 1 for line in lines)


def test_sustained_bf16_peak_is_read_when_present(monkeypatch, tmp_path):
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"bf16_tflops": 1900.0,
                                                             "bf16_tflops_sustained": 1700.0}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.measured_bf16_sustained() == 1700.0
    assert bench.measured_bf16_peak()[0] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"bf16_tflops": 1900.0}))
    assert bench.measured_bf16_sustained() is None
