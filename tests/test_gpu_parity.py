"""CUDA path against the fp64 oracle, element by element, on seeded inputs.

Every call goes through the C ABI (ctypes binding of libpadecode.so).  Small
shapes sweep head_dim, GQA group, block size, dtype and ragged lengths
(0, 1, one tile, one token past a tile, several partitions with a partial
last one); the five decode workloads run at reduced batch sizes here and at
full size (sampled) in test_gpu_workloads.py.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_helpers import (assert_out_close, assert_partials_close, assert_stats_close,
                               to_f64)
from workloads import custom_workload, make_case, make_dense_case

pytestmark = pytest.mark.gpu

# lengths, Hq, Hkv, D, bs, dtype, k_scale
SHAPES = [
    ([1, 15, 16, 17, 100, 0, 513], 8, 1, 128, 16, torch.bfloat16, 1.0),
    ([37, 1000, 250], 24, 4, 128, 16, torch.float16, 3.0),
    ([300, 64, 1, 545], 16, 2, 256, 32, torch.bfloat16, 1.0),
    ([77, 640, 31], 4, 4, 64, 16, torch.bfloat16, 2.0),
    ([33, 129, 2048], 12, 6, 64, 32, torch.float16, 1.0),
    ([5, 700], 6, 1, 256, 16, torch.float16, 1.0),
    # GQA groups above 8: 16 heads in one unit (head_dim 64 / 128), 12 (padded to
    # 16), and head groups (32 = 2 x 16; head_dim 256: 16 = 2 x 8)
    ([300, 1, 2000, 4097], 64, 4, 128, 16, torch.bfloat16, 1.0),
    ([1000, 17, 513], 48, 4, 128, 16, torch.float16, 2.0),
    ([700, 33], 16, 1, 64, 16, torch.bfloat16, 1.0),
    ([900, 5, 64], 32, 1, 128, 16, torch.bfloat16, 1.0),
    ([600, 40], 32, 2, 256, 32, torch.float16, 1.0),
    # block_size 8: a 16-token tile spans two blocks
    ([1, 7, 8, 9, 15, 16, 17, 1000], 24, 4, 128, 8, torch.bfloat16, 1.0),
    ([513, 31], 16, 2, 256, 8, torch.bfloat16, 1.0),
    ([129, 300], 32, 2, 64, 8, torch.float16, 2.0),
]
IDS = [f"d{s[3]}_hq{s[1]}_hkv{s[2]}_bs{s[4]}_{str(s[5])[6:]}" for s in SHAPES]
assert len(set(IDS)) == len(IDS)


@pytest.fixture(scope="module")
def pa():
    import paged_kv_decode_partitioned_gb300 as pa
    from paged_kv_decode_partitioned_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pa.load_library()
    return pa


def _case(i):
    lengths, Hq, Hkv, D, bs, dt, ks = SHAPES[i]
    w = custom_workload(num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=bs, dtype=dt,
                        k_scale=ks)
    return make_case(w, lengths=lengths, seed=1000 + i)


@pytest.fixture(scope="module", params=range(len(SHAPES)), ids=IDS)
def shaped(request):
    host = _case(request.param)
    return host, host.to("cuda"), oracle.attention(host.query, host.key_cache,
                                                   host.value_cache, host.block_tables,
                                                   host.seq_lens, host.scale)


def test_single_pass_matches_oracle(pa, shaped):
    host, dev, ref = shaped
    out = pa.decode(dev.query, dev.key_cache, dev.value_cache, dev.block_tables, dev.seq_lens,
                    host.scale)
    assert_out_close(out, ref, "pa_decode")
    assert pa.device_status() == 0


@pytest.mark.parametrize("pmul", [1, 4, 32])
def test_partitioned_partials_and_reduce_match_oracle(pa, shaped, pmul):
    host, dev, ref = shaped
    P = host.workload.block_size * pmul
    NP = max(1, oracle.num_partitions(host.max_seq_len, P))
    tmp, es, ml = pa.decode_partitioned(dev.query, dev.key_cache, dev.value_cache,
                                        dev.block_tables, dev.seq_lens, host.scale, P, NP)
    otmp, oes, oml = oracle.partials(host.query, host.key_cache, host.value_cache,
                                     host.block_tables, host.seq_lens, host.scale, P, NP)
    assert_stats_close(es, ml, oes, oml, f"partials P={P}")
    assert_partials_close(tmp, otmp, f"partials P={P}")
    out = pa.partition_reduce(tmp, es, ml, dev.seq_lens, P, dtype=host.query.dtype)
    assert_out_close(out, ref, f"reduce P={P}")
    # the merge of the oracle's own partials agrees with its single pass (pin)
    assert np.abs(oracle.lse_merge(otmp, oes, oml, host.seq_lens, P) - ref).max() < 1e-12
    assert pa.device_status() == 0


@pytest.mark.parametrize("thr_mul,pmul", [(0, 2), (2, 2), (3, 2), (1000, 2), (-1, 2), (-1, 0),
                                          (3, 0)])
def test_auto_matches_oracle(pa, shaped, thr_mul, pmul):
    """Every launch form of pa_decode_auto: thr 0 / 2bs (<= P: dense grid on these
    few-sequence batches), 3bs (> P: the work list with single-pass and partitioned
    sequences), huge (single pass), and the library's heuristic (thr = -1, P = 0)."""
    host, dev, ref = shaped
    bs = host.workload.block_size
    P = pmul * bs
    thr = -1 if thr_mul < 0 else thr_mul * bs
    out = pa.decode_auto(dev.query, dev.key_cache, dev.value_cache, dev.block_tables,
                         dev.seq_lens, host.scale, host.max_seq_len, thr, P)
    form = pa.auto_resolve(host.num_seqs, dev.key_cache.shape[2], dev.query.shape[2], bs,
                           host.max_seq_len, thr, P)[2]
    assert_out_close(out, ref, f"pa_decode_auto thr={thr} P={P} form={form}")
    assert pa.device_status() == 0


def test_auto_total_token_bound_and_its_overflow_flag(pa):
    """A correct total-token bound gives the same result from a smaller workspace; a
    bound below the batch's real total drops partitions and raises the flag (the
    planner caps the work list at the workspace's slots; no memory past it is used)."""
    lengths = [5000, 3000, 700, 12000, 9000, 100] * 6
    w = custom_workload(num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                        dtype=torch.bfloat16)
    host = make_case(w, lengths=lengths, seed=301)
    dev = host.to("cuda")
    ref = oracle.attention(host.query, host.key_cache, host.value_cache, host.block_tables,
                           host.seq_lens, host.scale)
    T = host.total_tokens
    thr, P = 1024, 512
    full = pa.auto_workspace_bytes(host.num_seqs, 8, 2, 128, 16, host.max_seq_len, 0, thr, P)
    tight = pa.auto_workspace_bytes(host.num_seqs, 8, 2, 128, 16, host.max_seq_len, T, thr, P)
    assert tight < full
    ws = torch.full((tight,), 0xAB, dtype=torch.uint8, device="cuda")
    out = pa.decode_auto(dev.query, dev.key_cache, dev.value_cache, dev.block_tables,
                         dev.seq_lens, host.scale, host.max_seq_len, thr, P, workspace=ws,
                         max_total_tokens=T)
    assert_out_close(out, ref, "auto with a total-token bound")
    assert pa.device_status() == 0
    # a bound far below the real total: the workspace is sized for too few slots
    small = T // 4
    need = pa.auto_workspace_bytes(host.num_seqs, 8, 2, 128, 16, host.max_seq_len, small, thr, P)
    guard = 1 << 20
    ws = torch.full((need + guard,), 0xCD, dtype=torch.uint8, device="cuda")
    out = pa.decode_auto(dev.query, dev.key_cache, dev.value_cache, dev.block_tables,
                         dev.seq_lens, host.scale, host.max_seq_len, thr, P,
                         workspace=ws[:need], max_total_tokens=small)
    torch.cuda.synchronize()
    assert pa.device_status() & pa.DEV_TOO_MANY_PARTITIONS
    assert bool((ws[need:] == 0xCD).all()), "the call wrote past its workspace"
    assert torch.isfinite(out.float()).all()
    # single-pass sequences are unaffected by the dropped partitions
    short = [i for i, L in enumerate(lengths) if L <= thr]
    assert_out_close(out[short], ref[short], "single-pass sequences under an overflow")
    assert pa.device_status() == 0


def test_gather_is_bit_exact(pa):
    for i, (D, bs, dt) in enumerate([(128, 16, torch.bfloat16), (256, 32, torch.float16),
                                      (64, 16, torch.float16), (128, 48, torch.bfloat16),
                                      (128, 8, torch.bfloat16), (256, 8, torch.float16)]):
        case, dk, dv = make_dense_case(lengths=[1, 16, 47, 130, 0], num_q_heads=4,
                                       num_kv_heads=2, head_dim=D, block_size=bs, dtype=dt,
                                       seed=50 + i)
        dev = case.to("cuda")
        max_len = max(case.seq_lens_list)
        kd, vd = pa.gather_kv(dev.key_cache, dev.value_cache, dev.block_tables, dev.seq_lens,
                              max_len)
        ok, ov = oracle.gather(case.key_cache, case.value_cache, case.block_tables,
                               case.seq_lens, max_len)
        kb = kd.cpu().view(torch.int16).numpy().view(np.uint16)
        vb = vd.cpu().view(torch.int16).numpy().view(np.uint16)
        assert np.array_equal(kb, ok) and np.array_equal(vb, ov), f"gather case {i}"
        for s, L in enumerate(case.seq_lens_list):
            assert torch.equal(kd[s, :L].cpu(), dk[s]) and torch.equal(vd[s, :L].cpu(), dv[s])


def test_block_permutation_gives_identical_bits(pa):
    host = _case(1)
    dev = host.to("cuda")
    a = pa.decode(dev.query, dev.key_cache, dev.value_cache, dev.block_tables, dev.seq_lens,
                  host.scale)
    nb = host.key_cache.shape[0]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(5))
    kc = torch.empty_like(host.key_cache)
    vc = torch.empty_like(host.value_cache)
    kc[perm] = host.key_cache
    vc[perm] = host.value_cache
    bt = host.block_tables.clone()
    m = bt >= 0
    bt[m] = perm[bt[m].long()].to(torch.int32)
    b = pa.decode(dev.query, kc.cuda(), vc.cuda(), bt.cuda(), dev.seq_lens, host.scale)
    assert torch.equal(a, b)


def test_seq_len_one_returns_v0_exactly(pa):
    for dt, D, bs in [(torch.bfloat16, 128, 16), (torch.float16, 256, 32)]:
        case, dk, dv = make_dense_case(lengths=[1, 1, 1], num_q_heads=8, num_kv_heads=1,
                                       head_dim=D, block_size=bs, dtype=dt, seed=7)
        dev = case.to("cuda")
        out = pa.decode(dev.query, dev.key_cache, dev.value_cache, dev.block_tables,
                        dev.seq_lens, 0.125).cpu()
        for s in range(3):
            assert torch.equal(out[s], dv[s][0, 0].expand(8, D))


def test_zero_query_gives_mean_of_v(pa):
    case, dk, dv = make_dense_case(lengths=[300, 17], num_q_heads=6, num_kv_heads=1,
                                   head_dim=128, block_size=16, dtype=torch.bfloat16, seed=8)
    case.query.zero_()
    dev = case.to("cuda")
    out = pa.decode(dev.query, dev.key_cache, dev.value_cache, dev.block_tables, dev.seq_lens,
                    0.1)
    for s in range(2):
        ref = dv[s].double().mean(dim=0).expand(6, 128).numpy()
        assert_out_close(out[s], ref, "zero query")


def test_partition_size_does_not_change_result(pa):
    host = _case(0)
    dev = host.to("cuda")
    outs = []
    for P in (16, 64, 512, 4096):
        NP = oracle.num_partitions(host.max_seq_len, P)
        tmp, es, ml = pa.decode_partitioned(dev.query, dev.key_cache, dev.value_cache,
                                            dev.block_tables, dev.seq_lens, host.scale, P, NP)
        outs.append(to_f64(pa.partition_reduce(tmp, es, ml, dev.seq_lens, P,
                                               dtype=host.query.dtype)))
    for o in outs[1:]:
        assert np.abs(o - outs[0]).max() <= 2e-2


def test_bad_table_entry_and_overlong_length_raise_flags(pa):
    host = _case(3)
    dev = host.to("cuda")
    bt = dev.block_tables.clone()
    bt[1, 2] = host.key_cache.shape[0] + 5       # outside the cache: read as zeros
    out = pa.decode(dev.query, dev.key_cache, dev.value_cache, bt, dev.seq_lens, host.scale)
    torch.cuda.synchronize()
    assert pa.device_status() & pa.DEV_BAD_BLOCK
    assert torch.isfinite(out.float()).all()
    sl = dev.seq_lens.clone()
    sl[0] = dev.block_tables.shape[1] * host.workload.block_size + 1   # longer than the table
    pa.decode(dev.query, dev.key_cache, dev.value_cache, dev.block_tables, sl, host.scale)
    assert pa.device_status() & pa.DEV_LEN_CLAMPED
    assert pa.device_status() == 0


def test_too_few_partition_slots_raise_flag(pa):
    host = _case(4)
    dev = host.to("cuda")
    P = 32
    NP = oracle.num_partitions(host.max_seq_len, P) - 1
    pa.decode_partitioned(dev.query, dev.key_cache, dev.value_cache, dev.block_tables,
                          dev.seq_lens, host.scale, P, NP)
    assert pa.device_status() & pa.DEV_TOO_MANY_PARTITIONS


def test_single_pass_with_many_equal_length_classes(pa):
    """Single-pass grid slots map to sequences longest first; ties (equal
    lengths or length classes) must still cover every sequence exactly once."""
    lengths = [100, 16, 100, 5000, 17, 100, 0, 5001, 16, 1, 4096, 4097, 100, 33, 5000, 2] * 3
    w = custom_workload(num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                        dtype=torch.bfloat16)
    host = make_case(w, lengths=lengths, seed=77)
    dev = host.to("cuda")
    ref = oracle.attention(host.query, host.key_cache, host.value_cache, host.block_tables,
                           host.seq_lens, host.scale)
    out = pa.decode(dev.query, dev.key_cache, dev.value_cache, dev.block_tables, dev.seq_lens,
                    host.scale)
    assert_out_close(out, ref, "pa_decode, tied lengths")
    assert pa.device_status() == 0


def test_wait_timeout_raises_flag_and_device_stays_usable(pa):
    """The bounded-wait failure path: a barrier nothing completes times out,
    raises PA_DEV_WAIT_TIMEOUT, and later launches still compute correctly."""
    assert pa.device_status() == 0
    pa.selftest_wait_timeout(20000)
    assert pa.device_status() & pa.DEV_WAIT_TIMEOUT
    assert pa.device_status() == 0
    host = _case(1)
    dev = host.to("cuda")
    ref = oracle.attention(host.query, host.key_cache, host.value_cache, host.block_tables,
                           host.seq_lens, host.scale)
    out = pa.decode(dev.query, dev.key_cache, dev.value_cache, dev.block_tables, dev.seq_lens,
                    host.scale)
    assert_out_close(out, ref, "decode after a time-out")


def test_long_sequence_single_pass_cluster_split(pa):
    """One 100K-token sequence in one pass: the cluster splits it 8 ways."""
    w = custom_workload(num_q_heads=24, num_kv_heads=4, head_dim=128, block_size=16,
                        dtype=torch.bfloat16, k_scale=3.0)
    host = make_case(w, lengths=[100000, 3], seed=91)
    dev = host.to("cuda")
    ref = oracle.attention(host.query, host.key_cache, host.value_cache, host.block_tables,
                           host.seq_lens, host.scale)
    out = pa.decode(dev.query, dev.key_cache, dev.value_cache, dev.block_tables, dev.seq_lens,
                    host.scale)
    assert_out_close(out, ref, "single pass, 100K tokens")
    assert pa.device_status() == 0


@pytest.mark.parametrize("bs", [48, 64, 80, 256])
def test_large_block_sizes(pa, bs):
    w = custom_workload(num_q_heads=16, num_kv_heads=2, head_dim=128, block_size=bs,
                        dtype=torch.float16)
    host = make_case(w, lengths=[1, bs - 1, bs, bs + 1, 3 * bs + 17], seed=92 + bs)
    dev = host.to("cuda")
    ref = oracle.attention(host.query, host.key_cache, host.value_cache, host.block_tables,
                           host.seq_lens, host.scale)
    out = pa.decode(dev.query, dev.key_cache, dev.value_cache, dev.block_tables, dev.seq_lens,
                    host.scale)
    assert_out_close(out, ref, f"single pass, bs={bs}")
    P = bs
    NP = oracle.num_partitions(host.max_seq_len, P)
    tmp, es, ml = pa.decode_partitioned(dev.query, dev.key_cache, dev.value_cache,
                                        dev.block_tables, dev.seq_lens, host.scale, P, NP)
    assert_out_close(pa.partition_reduce(tmp, es, ml, dev.seq_lens, P, dtype=torch.float16),
                     ref, f"partitioned, bs={bs}")
    out = pa.decode_auto(dev.query, dev.key_cache, dev.value_cache, dev.block_tables,
                         dev.seq_lens, host.scale, host.max_seq_len, bs, 2 * bs)
    assert_out_close(out, ref, f"auto, bs={bs}")
    assert pa.device_status() == 0


def test_many_short_sequences(pa):
    """1000 sequences: the planner's per-sequence loops and the compact list."""
    g = torch.Generator().manual_seed(93)
    lengths = [int(x) for x in torch.randint(0, 300, (1000,), generator=g)]
    w = custom_workload(num_q_heads=8, num_kv_heads=1, head_dim=64, block_size=16,
                        dtype=torch.bfloat16)
    host = make_case(w, lengths=lengths, seed=94)
    dev = host.to("cuda")
    ref = oracle.attention(host.query, host.key_cache, host.value_cache, host.block_tables,
                           host.seq_lens, host.scale)
    for thr in (0, 100, 10000):
        out = pa.decode_auto(dev.query, dev.key_cache, dev.value_cache, dev.block_tables,
                             dev.seq_lens, host.scale, host.max_seq_len, thr, 32)
        assert_out_close(out, ref, f"auto, 1000 sequences, thr={thr}")
    out = pa.decode(dev.query, dev.key_cache, dev.value_cache, dev.block_tables, dev.seq_lens,
                    host.scale)
    assert_out_close(out, ref, "single pass, 1000 sequences")
    assert pa.device_status() == 0


def test_planner_thousands_of_sequences(pa):
    """5000 sequences through the work list: the planner's chunked prefix sums (one CTA
    per 32 sequences) place single-pass and partition units of every sequence, including
    a chunk boundary falling inside runs of partitioned sequences."""
    g = torch.Generator().manual_seed(95)
    lengths = [int(x) for x in torch.randint(1, 400, (5000,), generator=g)]
    for i in range(0, 5000, 37):
        lengths[i] = 1500 + i % 700          # partitioned (> threshold 256)
    w = custom_workload(num_q_heads=8, num_kv_heads=2, head_dim=64, block_size=16,
                        dtype=torch.bfloat16)
    host = make_case(w, lengths=lengths, seed=96)
    dev = host.to("cuda")
    ref = oracle.attention(host.query, host.key_cache, host.value_cache, host.block_tables,
                           host.seq_lens, host.scale)
    out = pa.decode_auto(dev.query, dev.key_cache, dev.value_cache, dev.block_tables,
                         dev.seq_lens, host.scale, host.max_seq_len, 256, 128,
                         max_total_tokens=host.total_tokens)
    assert pa.auto_resolve(5000, 2, 64, 16, host.max_seq_len, 256, 128,
                           max_total_tokens=host.total_tokens)[2] == pa.AUTO_WORKLIST
    assert_out_close(out, ref, "auto, 5000 sequences")
    assert pa.device_status() == 0
