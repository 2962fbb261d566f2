"""Seeded random shapes against the fp64 oracle: every decode entry point and the
prefill, element by element.

The hand-picked shapes of test_gpu_parity.py and test_gpu_prefill.py aim at known
edges; these draw (head_dim, KV heads, GQA group, block size, dtype, key scale,
lengths) from a fixed-seed generator, so combinations nobody picked get checked
too.  Lengths mix empty, one-token, short, tile-sized and long sequences; the
oracle's cost of each case is bounded, so the whole file runs in seconds.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_helpers import (assert_out_close, assert_partials_close, assert_stats_close)
from workloads import custom_workload, make_case, make_prefill_case

pytestmark = pytest.mark.gpu

N_DECODE = 48
N_PREFILL = 48
BLOCK_SIZES = [8, 16, 32, 48, 64, 128]
DTYPES = [torch.bfloat16, torch.float16]


@pytest.fixture(scope="module")
def pa():
    import paged_kv_decode_partitioned_gb300 as pa
    from paged_kv_decode_partitioned_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pa.load_library()
    return pa


def _length(rng, lo_cap=3000):
    kind = rng.integers(0, 6)
    if kind == 0:
        return 0
    if kind == 1:
        return 1
    if kind == 2:
        return int(rng.integers(2, 65))
    if kind == 3:   # around a 128-token tile edge
        return int(128 * rng.integers(1, 5) + rng.integers(-1, 2))
    if kind == 4:
        return int(rng.integers(65, 700))
    return int(rng.integers(700, lo_cap + 1))


def _decode_shape(i):
    rng = np.random.default_rng(7100 + i)
    while True:
        D = int(rng.choice([64, 128, 256]))
        Hkv = int(rng.choice([1, 2, 4, 8]))
        g = int(rng.choice([1, 2, 3, 5, 6, 8, 12, 16, 24, 32]))
        bs = int(rng.choice(BLOCK_SIZES))
        dt = DTYPES[int(rng.integers(0, 2))]
        ks = float(rng.choice([1.0, 2.0, 3.0]))
        S = int(rng.integers(1, 7))
        lengths = [_length(rng) for _ in range(S)]
        if max(lengths) == 0:
            lengths[0] = 1
        Hq = Hkv * g
        if Hq <= 64 and sum(lengths) * Hq * D <= 2e8:
            return lengths, Hq, Hkv, D, bs, dt, ks


def _prefill_shape(i):
    rng = np.random.default_rng(7300 + i)
    while True:
        D = int(rng.choice([64, 128, 256]))
        Hkv = int(rng.choice([1, 2, 4]))
        g = int(rng.choice([1, 2, 3, 4, 6, 8, 16, 32]))
        bs = int(rng.choice(BLOCK_SIZES))
        dt = DTYPES[int(rng.integers(0, 2))]
        S = int(rng.integers(1, 5))
        ctx = [int(rng.choice([0, rng.integers(1, 200), rng.integers(200, 1500)])) for _ in range(S)]
        ql = [int(rng.choice([0, 1, rng.integers(2, 64), rng.integers(64, 260)])) for _ in range(S)]
        if max(ql) == 0:
            ql[0] = int(rng.integers(1, 100))
        Hq = Hkv * g
        macs = sum(n * (c + (n + 1) / 2) for c, n in zip(ctx, ql)) * Hq * D
        if Hq <= 64 and macs <= 1.5e9:
            return ctx, ql, Hq, Hkv, D, bs, dt


def _id(shape, kind):
    if kind == "decode":
        lengths, Hq, Hkv, D, bs, dt, ks = shape
        return f"d{D}_hq{Hq}_hkv{Hkv}_bs{bs}_{str(dt)[6:]}_S{len(lengths)}"
    ctx, ql, Hq, Hkv, D, bs, dt = shape
    return f"d{D}_hq{Hq}_hkv{Hkv}_bs{bs}_{str(dt)[6:]}_S{len(ctx)}"


DECODE = [_decode_shape(i) for i in range(N_DECODE)]
PREFILL = [_prefill_shape(i) for i in range(N_PREFILL)]


@pytest.mark.parametrize("i", range(N_DECODE),
                         ids=[f"{k}_{_id(s, 'decode')}" for k, s in enumerate(DECODE)])
def test_decode_entry_points_on_random_shapes(pa, i):
    """pa_decode, pa_decode_partitioned + pa_partition_reduce (partials at 1e-4),
    and pa_decode_auto with the library's defaults, against the oracle."""
    lengths, Hq, Hkv, D, bs, dt, ks = DECODE[i]
    w = custom_workload(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=bs, dtype=dt,
                        k_scale=ks)
    host = make_case(w, lengths=lengths, seed=7200 + i)
    dev = host.to("cuda")
    ref = oracle.attention(host.query, host.key_cache, host.value_cache, host.block_tables,
                           host.seq_lens, host.scale)
    out = pa.decode(dev.query, dev.key_cache, dev.value_cache, dev.block_tables, dev.seq_lens,
                    host.scale)
    assert_out_close(out, ref, f"pa_decode, shape {i}")

    rng = np.random.default_rng(7400 + i)
    P = int(bs * rng.choice([1, 2, 4, 8, 16, 32]))
    NP = max(oracle.num_partitions(max(lengths), P), 1)
    tmp, es, ml = pa.decode_partitioned(dev.query, dev.key_cache, dev.value_cache,
                                        dev.block_tables, dev.seq_lens, host.scale, P, NP)
    red = pa.partition_reduce(tmp, es, ml, dev.seq_lens, P, dtype=dt)
    assert_out_close(red, ref, f"pa_decode_partitioned + reduce, P={P}, shape {i}")
    t_ref, e_ref, m_ref = oracle.partials(host.query, host.key_cache, host.value_cache,
                                          host.block_tables, host.seq_lens, host.scale, P, NP)
    if not np.isnan(e_ref).all():
        assert_stats_close(es, ml, e_ref, m_ref, f"partials, P={P}, shape {i}")
        assert_partials_close(tmp, t_ref, f"tmp_out, P={P}, shape {i}")

    auto = pa.decode_auto(dev.query, dev.key_cache, dev.value_cache, dev.block_tables,
                          dev.seq_lens, host.scale, max(lengths))
    assert_out_close(auto, ref, f"pa_decode_auto defaults, shape {i}")
    assert pa.device_status() == 0


@pytest.mark.parametrize("i", range(N_PREFILL),
                         ids=[f"{k}_{_id(s, 'prefill')}" for k, s in enumerate(PREFILL)])
def test_prefill_on_random_shapes(pa, i):
    ctx, ql, Hq, Hkv, D, bs, dt = PREFILL[i]
    w = custom_workload(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=bs, dtype=dt)
    host = make_prefill_case(w, ctx_lens=ctx, q_lens=ql, seed=7500 + i)
    dev = host.to("cuda")
    c = dev.case
    out = pa.prefill(dev.query, c.key_cache, c.value_cache, c.block_tables, c.seq_lens,
                     dev.q_start, c.scale, max(ql))
    hc = host.case
    ref = oracle.prefill(host.query, hc.key_cache, hc.value_cache, hc.block_tables, hc.seq_lens,
                         host.q_start, hc.scale)
    assert_out_close(out, ref, f"pa_prefill, shape {i}")
    assert pa.device_status() == 0
