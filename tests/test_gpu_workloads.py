"""The five decode workloads on the GPU against the oracle, element by element.

Every workload runs at full size in exactly the launch configuration the
benchmark times (``DecodeStep`` with the workload's mode, partition sizes and
single-pass limit) and through ``pa_decode_auto`` with the library's default
heuristic; every output element of every sequence is compared with the
oracle.  The partitioned workloads also have their fp32 phase-1 partials
(max_logits, exp_sums: 1e-4 relative; tmp_out) compared slot by slot.
Reduced batches of the same rules run too (other launch shapes).
"""
import pytest
import torch

import oracle
from tests.gpu_helpers import (assert_out_close, assert_partials_close, assert_stats_close,
                               host_subcase)
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
                            single_pass_max_len=w.single_pass_max_len,
                            max_total_tokens=case_dev.total_tokens)
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


@pytest.fixture(scope="module", params=sorted(WORKLOADS))
def full(request):
    """A workload at full size on the device, the host copy of every sequence, and
    the oracle's output for all of them."""
    w = WORKLOADS[request.param]
    dev = make_case(w, device="cuda")
    ids = list(range(dev.num_seqs))
    host = host_subcase(dev, ids)
    ref = oracle.attention(*host, w.scale)
    yield w, dev, host, ref
    del dev
    torch.cuda.empty_cache()


def test_workload_full_size_every_element(pa, full):
    """The benchmark's launch configuration (DecodeStep with the workload's mode,
    partition sizes and single-pass limit) on the full batch, every output element
    against the oracle."""
    w, dev, host, ref = full
    for P, step in _steps(dev, w, dev.max_seq_len):
        out = step()
        assert_out_close(out, ref, f"workload {w.wid} full, P={P}, all {dev.num_seqs} seqs")
    assert pa.device_status() == 0


def test_workload_full_size_default_heuristic(pa, full):
    """pa_decode_auto with the library's defaults (threshold -1, partition size 0:
    the heuristic picks both and the launch form) on the full batch."""
    w, dev, host, ref = full
    thr, P, form = pa.auto_resolve(dev.num_seqs, w.num_kv_heads, w.head_dim, w.block_size,
                                   dev.max_seq_len, -1, 0, max_total_tokens=dev.total_tokens)
    out = pa.decode_auto(dev.query, dev.key_cache, dev.value_cache, dev.block_tables,
                         dev.seq_lens, w.scale, dev.max_seq_len, -1, 0,
                         max_total_tokens=dev.total_tokens)
    assert_out_close(out, ref, f"workload {w.wid} full, default heuristic (thr {thr}, P {P}, "
                               f"form {form})")
    assert pa.device_status() == 0


def test_workload_full_size_partials(pa, full):
    """Phase-1 partials of the partitioned workloads at full size: max_logits and
    exp_sums within 1e-4 relative of the oracle's (every written slot), tmp_out and
    the reduced output within the output tolerance."""
    w, dev, host, ref = full
    if w.mode != "partitioned":
        pytest.skip("the workload is not partitioned")
    for P in w.partition_sizes:
        NP = oracle.num_partitions(dev.max_seq_len, P)
        tmp, es, ml = pa.decode_partitioned(dev.query, dev.key_cache, dev.value_cache,
                                            dev.block_tables, dev.seq_lens, w.scale, P, NP)
        otmp, oes, oml = oracle.partials(*host, w.scale, P, NP)
        assert_stats_close(es, ml, oes, oml, f"workload {w.wid} partials P={P}")
        assert_partials_close(tmp, otmp, f"workload {w.wid} tmp_out P={P}")
        out = pa.partition_reduce(tmp, es, ml, dev.seq_lens, P, dtype=w.dtype)
        assert_out_close(out, ref, f"workload {w.wid} reduce of the partials, P={P}")
        del tmp, es, ml, otmp, oes, oml
    assert pa.device_status() == 0
