"""pa_decode_auto_static: the decode step for callers that cannot allocate.

Serving engines that reserve nearly all device memory for the KV cache, hot
loops that must avoid the synchronisation an allocation can cause, and plugin
hosts without an allocator cannot give the library a workspace; this entry
point keeps its scratch in a fixed device array inside the library instead.
These tests call it through the C ABI (ctypes) and compare it with the fp64
oracle and with pa_decode_auto, which uses a caller-provided workspace, on
different batches in a row (each call finds the previous call's leftovers in
the shared array), then once more on the first batch.  The file is named so
that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from tests.gpu_helpers import assert_out_close, host_subcase, to_f64
from workloads import WORKLOADS, make_case

pytestmark = pytest.mark.gpu

PA_ERR_WORKSPACE_TOO_SMALL = -4


@pytest.fixture(scope="module")
def pa():
    import paged_kv_decode_partitioned_gb300 as pa
    from paged_kv_decode_partitioned_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pa.load_library()
    return pa


def _static_call(lib, dev, out, thr, P, total=0):
    S, Hq, D = dev.query.shape
    nb, bs, Hkv, _ = dev.key_cache.shape
    dtype = 1 if dev.query.dtype == torch.bfloat16 else 0
    return lib.pa_decode_auto_static(
        out.data_ptr(), dev.query.data_ptr(), dev.key_cache.data_ptr(),
        dev.value_cache.data_ptr(), dev.block_tables.data_ptr(), dev.seq_lens.data_ptr(),
        S, Hq, Hkv, D, bs, nb, dev.block_tables.shape[1], ctypes.c_float(dev.scale),
        dev.max_seq_len, total, thr, P, dtype, torch.cuda.current_stream().cuda_stream)


def _oracle(dev):
    host = host_subcase(dev, list(range(dev.num_seqs)))
    return oracle.attention(*host, dev.scale)


def test_static_scratch_matches_workspace_entry_on_calls_in_a_row(pa):
    lib = pa.load_library()
    batches = [
        # partitioned long sequences (P=512, 196 partitions each)
        (make_case(WORKLOADS[3], lengths=[100000, 99991]).to("cuda"), 8192, 512),
        # mixed batch: single-pass and partitioned sequences in one work list
        (make_case(WORKLOADS[4], num_seqs=16).to("cuda"), 8192, 512),
        # a small head_dim-256 batch with a low threshold and P=256
        (make_case(WORKLOADS[5], lengths=[32768, 9000, 300]).to("cuda"), 4096, 256),
        # the library's heuristic (threshold, partition size and launch form)
        (make_case(WORKLOADS[4], num_seqs=5).to("cuda"), -1, 0),
    ]
    refs = [_oracle(dev) for dev, _, _ in batches]
    for (dev, thr, P), ref in list(zip(batches, refs)) + [(batches[0], refs[0])]:
        need = pa.auto_workspace_bytes(dev.num_seqs, dev.query.shape[1], dev.key_cache.shape[2],
                                       dev.query.shape[2], dev.key_cache.shape[1],
                                       dev.max_seq_len, 0, thr, P)
        assert need <= 96 << 20
        ws_out = pa.decode_auto(dev.query, dev.key_cache, dev.value_cache, dev.block_tables,
                                dev.seq_lens, dev.scale, dev.max_seq_len, thr, P)
        out = torch.full_like(dev.query, float("nan"))
        assert _static_call(lib, dev, out, thr, P) == 0
        torch.cuda.synchronize()
        assert_out_close(out, ref, f"static scratch vs oracle, thr={thr} P={P}")
        assert_out_close(out, to_f64(ws_out), f"static scratch vs workspace, thr={thr} P={P}")
        assert pa.device_status() == 0


def test_static_scratch_takes_the_mixed_256_batch_with_a_token_bound(pa):
    """The 256-sequence mixed batch (lengths 128..65536 log-uniform) fits the fixed
    scratch once the caller bounds its total tokens; every element against the oracle."""
    lib = pa.load_library()
    dev = make_case(WORKLOADS[4], device="cuda")
    need = pa.auto_workspace_bytes(256, 24, 4, 128, 16, dev.max_seq_len, dev.total_tokens,
                                   8192, 512)
    assert need <= 96 << 20
    out = torch.full_like(dev.query, float("nan"))
    assert _static_call(lib, dev, out, 8192, 512, dev.total_tokens) == 0
    torch.cuda.synchronize()
    assert_out_close(out, _oracle(dev), "static scratch, 256-sequence mixed batch")
    assert pa.device_status() == 0
    del dev
    torch.cuda.empty_cache()


def test_static_scratch_rejects_batches_beyond_its_size(pa):
    lib = pa.load_library()
    # 256 sequences of up to 65536 tokens at P=512 with no token bound need ~400 MB
    need = pa.auto_workspace_bytes(256, 24, 4, 128, 16, 65536, 0, 8192, 512)
    assert need > 96 << 20
    A = 1 << 20   # never dereferenced: the call must stop on the host
    st = lib.pa_decode_auto_static(A, A, A, A, A, A, 256, 24, 4, 128, 16, 100000, 4096,
                                   ctypes.c_float(0.088), 65536, 0, 8192, 512, 1, None)
    assert st == PA_ERR_WORKSPACE_TOO_SMALL
    assert lib.pa_status_string(st) == b"PA_ERR_WORKSPACE_TOO_SMALL"


def test_binding_wrapper_matches(pa):
    dev = make_case(WORKLOADS[4], num_seqs=8).to("cuda")
    a = pa.decode_auto_static(dev.query, dev.key_cache, dev.value_cache, dev.block_tables,
                              dev.seq_lens, dev.scale, dev.max_seq_len, 8192, 512)
    b = pa.decode_auto(dev.query, dev.key_cache, dev.value_cache, dev.block_tables,
                       dev.seq_lens, dev.scale, dev.max_seq_len, 8192, 512)
    assert np.abs(to_f64(a) - to_f64(b)).max() <= 1e-2
    assert_out_close(a, _oracle(dev), "binding wrapper vs oracle")
