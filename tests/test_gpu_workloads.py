"""The five decode workloads on the GPU against the oracle.

Reduced batches are compared element by element; the full-size batches run
in exactly the launch configuration the benchmark times (``DecodeStep`` with
the workload's mode, partition size and single-pass limit) and a sample of
sequences -- the shortest, the longest, the ones nearest the single-pass
limit and two drawn at random -- is compared element by element.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_helpers import assert_out_close, host_subcase
from workloads import WORKLOADS, make_case

pytestmark = pytest.mark.gpu

REDUCED = {
    1: dict(),                                    # already small: full size
    2: dict(num_seqs=6),
    3: dict(lengths=[100000, 99991]),
    4: dict(num_seqs=16),
    5: dict(lengths=[32768, 32700, 5000]),
}


@pytest.fixture(scope="module")
def pa():
    import paged_kv_decode_partitioned_gb300 as pa
    from paged_kv_decode_partitioned_gb300 import build
    build.build()
    pa.load_library()
    return pa


def _steps(case_dev, w, max_seq_len):
    from paged_kv_decode_partitioned_gb300.step import DecodeStep
    for P in w.partition_sizes:
        yield P, DecodeStep(w.mode, case_dev.query, case_dev.key_cache, case_dev.value_cache,
                            case_dev.block_tables, case_dev.seq_lens, w.scale,
                            max_seq_len=max_seq_len, partition_size=P,
                            single_pass_max_len=w.single_pass_max_len)
        if w.mode == "single":
            break


@pytest.mark.parametrize("wid", sorted(WORKLOADS))
def test_workload_reduced_elementwise(pa, wid):
    w = WORKLOADS[wid]
    host = make_case(w, **REDUCED[wid])
    dev = host.to("cuda")
    ref = oracle.attention(host.query, host.key_cache, host.value_cache, host.block_tables,
                           host.seq_lens, w.scale)
    for P, step in _steps(dev, w, host.max_seq_len):
        out = step()
        assert_out_close(out, ref, f"workload {wid} reduced, P={P}")
    assert pa.device_status() == 0


def _sample(lengths, thr, k_random=2, seed=0):
    idx = {int(np.argmin(lengths)), int(np.argmax(lengths))}
    below = [i for i, L in enumerate(lengths) if L <= thr]
    above = [i for i, L in enumerate(lengths) if L > thr]
    if below:
        idx.add(max(below, key=lambda i: lengths[i]))
    if above:
        idx.add(min(above, key=lambda i: lengths[i]))
    rng = np.random.default_rng(seed)
    idx.update(int(i) for i in rng.choice(len(lengths), size=min(k_random, len(lengths)),
                                          replace=False))
    return sorted(idx)


@pytest.mark.parametrize("wid", sorted(WORKLOADS))
def test_workload_full_size_sampled(pa, wid):
    w = WORKLOADS[wid]
    dev = make_case(w, device="cuda")
    seq_ids = _sample(dev.seq_lens_list, w.single_pass_max_len, seed=wid)
    q, kc, vc, bt, sl = host_subcase(dev, seq_ids)
    ref = oracle.attention(q, kc, vc, bt, sl, w.scale)
    for P, step in _steps(dev, w, dev.max_seq_len):
        out = step()
        torch.cuda.synchronize()
        got = out.index_select(0, torch.as_tensor(seq_ids, device=out.device))
        assert_out_close(got, ref, f"workload {wid} full, P={P}, seqs {seq_ids}")
        assert torch.isfinite(out.float()).all()
    assert pa.device_status() == 0
    del dev
    torch.cuda.empty_cache()
