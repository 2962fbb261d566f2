"""The C ABI without a GPU: the library loads, exports every declared entry
point, and rejects bad arguments on the host before touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in ("pa_decode.h", "pa_moe.h")]


@pytest.fixture(scope="module")
def lib():
    from paged_kv_decode_partitioned_gb300 import build
    build.build()
    import paged_kv_decode_partitioned_gb300 as pa
    return pa.load_library()


def declared_functions():
    text = "".join(open(h).read() for h in HEADERS)
    return sorted(set(re.findall(r"PA_API\s+[\w\s\*]*?\b(pa_\w+)\s*\(", text)))


def test_header_declares_the_three_operations():
    names = declared_functions()
    for n in ("pa_decode", "pa_decode_partitioned", "pa_partition_reduce"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} missing from libpadecode.so"


def test_binding_signatures_cover_header():
    import paged_kv_decode_partitioned_gb300 as pa
    assert sorted(n for n, _, _ in pa.SIGNATURES) == declared_functions()


def test_status_strings(lib):
    assert lib.pa_status_string(0) == b"PA_OK"
    assert lib.pa_status_string(-2) == b"PA_ERR_UNSUPPORTED"
    assert lib.pa_status_string(-99) == b"PA_ERR_UNKNOWN"
    assert lib.pa_version() >= 10000


# Fake, aligned, never-dereferenced device addresses: the library must reject
# the call on the host before it would use them.
A = 1 << 20


def _decode(lib, **kw):
    args = dict(out=A, q=A, k=A, v=A, bt=A, sl=A, S=2, Hq=24, Hkv=4, D=128, bs=16, nb=10,
                mb=4, scale=0.1, dtype=1)
    args.update(kw)
    return lib.pa_decode(args["out"], args["q"], args["k"], args["v"], args["bt"], args["sl"],
                         args["S"], args["Hq"], args["Hkv"], args["D"], args["bs"], args["nb"],
                         args["mb"], args["scale"], args["dtype"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(D=96), -2),                 # head_dim not supported
    (dict(bs=4), -2),                 # block_size neither 8 nor a multiple of 16
    (dict(bs=24), -2),
    (dict(Hq=256, Hkv=1), -2),        # GQA group 256 > 128
    (dict(Hq=10, Hkv=4), -1),         # Hq not a multiple of Hkv
    (dict(S=-1), -1),
    (dict(dtype=7), -1),
    (dict(q=0), -1),                  # null query
    (dict(out=0), -1),                # null out
    (dict(nb=0), -1),                 # empty cache
    (dict(k=A + 8), -3),              # misaligned cache
    (dict(out=A + 2), -3),            # misaligned out
    (dict(S=0), 0),                   # nothing to do
])
def test_decode_rejects_on_host(lib, kw, status):
    assert _decode(lib, **kw) == status


def test_partitioned_rejects_partition_not_multiple_of_block(lib):
    st = lib.pa_decode_partitioned(A, A, A, A, A, A, A, A, 2, 24, 4, 128, 16, 10, 4,
                                   ctypes.c_float(0.1), 40, 4, 1, None)
    assert st == -2
    st = lib.pa_decode_partitioned(A, A, A, A, A, A, A, A, 2, 24, 4, 128, 16, 10, 4,
                                   ctypes.c_float(0.1), 0, 4, 1, None)
    assert st == -1


def test_reduce_rejects_on_host(lib):
    assert lib.pa_partition_reduce(A, A, A, A, A, 2, 24, 100, 512, 4, 1, None) == -2
    assert lib.pa_partition_reduce(A, A, A, A, A, 2, 24, 128, 0, 4, 1, None) == -1
    assert lib.pa_partition_reduce(A, A + 4, A, A, A, 2, 24, 128, 512, 4, 1, None) == -3
    assert lib.pa_partition_reduce(A, A, A, A, A, 0, 24, 128, 512, 4, 1, None) == 0


def test_auto_rejects_small_workspace_before_launch(lib):
    need = lib.pa_auto_workspace_bytes(8, 24, 4, 128, 16, 100000, 0, 8192, 512)
    assert need > 0
    st = lib.pa_decode_auto(A, A, A, A, A, A, 8, 24, 4, 128, 16, 10, 6250, ctypes.c_float(0.1),
                            100000, 0, 8192, 512, A, need - 1, 1, None)
    assert st == -4
    st = lib.pa_decode_auto(A, A, A, A, A, A, 8, 24, 4, 128, 16, 10, 6250, ctypes.c_float(0.1),
                            100000, 0, 8192, 512, A + 16, need, 1, None)
    assert st == -3
    # a partition size that is not a multiple of the block size
    st = lib.pa_decode_auto(A, A, A, A, A, A, 8, 24, 4, 128, 16, 10, 6250, ctypes.c_float(0.1),
                            100000, 0, 8192, 520, A, need, 1, None)
    assert st == -2


def _payload(slots, S, Hq, Hkv, D):
    return slots * Hq * (D + 2) * 4 + (S + slots) * Hkv * 16 + S * 4 + S * 16


def test_auto_workspace_size_formula(lib):
    # 8 sequences of <=100000 tokens, P=512: 196 partition slots each.
    S, Hq, Hkv, D, P = 8, 24, 4, 128, 512
    need = lib.pa_auto_workspace_bytes(S, Hq, Hkv, D, 16, 100000, 0, 8192, P)
    payload = _payload(S * 196, S, Hq, Hkv, D)
    assert payload <= need <= payload + 7 * 256
    # nothing longer than the single-pass limit: no scratch at all
    assert lib.pa_auto_workspace_bytes(S, Hq, Hkv, D, 16, 8192, 0, 8192, P) == 256
    # a partition size that is not a multiple of the block size, a bad head split
    assert lib.pa_auto_workspace_bytes(S, Hq, Hkv, D, 16, 100000, 0, 8192, 520) == 0
    assert lib.pa_auto_workspace_bytes(S, 10, 4, D, 16, 100000, 0, 8192, P) == 0


def test_auto_workspace_shrinks_with_a_total_token_bound(lib):
    """The 256-sequence mixed batch: lengths up to 65536 but 2,854,935 tokens in all.
    With the bound, slots <= (T + S_p (P - 1)) / P, S_p = min(S, T / (thr + 1))."""
    S, Hq, Hkv, D, P, thr, T = 256, 24, 4, 128, 512, 8192, 2854935
    worst = lib.pa_auto_workspace_bytes(S, Hq, Hkv, D, 16, 65536, 0, thr, P)
    bound = lib.pa_auto_workspace_bytes(S, Hq, Hkv, D, 16, 65536, T, thr, P)
    assert worst >= _payload(S * 128, S, Hq, Hkv, D)
    sp = min(S, T // (thr + 1))
    slots = (T + sp * (P - 1)) // P
    assert slots == 5831
    assert _payload(slots, S, Hq, Hkv, D) <= bound <= _payload(slots, S, Hq, Hkv, D) + 7 * 256
    assert bound < 80e6 < 390e6 < worst
    # a bound above S * max_seq_len changes nothing
    assert lib.pa_auto_workspace_bytes(S, Hq, Hkv, D, 16, 65536, S * 65536 * 2, thr, P) == worst


def test_partition_workspace_bytes(lib):
    """The dense phase-1 partials: tmp_out, exp_sums, max_logits, 256-byte aligned."""
    up = lambda x: (x + 255) // 256 * 256
    for S, Hq, D, NP in [(8, 24, 128, 196), (32, 16, 256, 128), (1, 1, 64, 1), (3, 5, 64, 7)]:
        rows = S * Hq * NP
        want = up(up(up(rows * D * 4) + rows * 4) + rows * 4)
        assert lib.pa_partition_workspace_bytes(S, Hq, D, NP) == want
    assert lib.pa_partition_workspace_bytes(8, 24, 128, 0) == 0
    assert lib.pa_partition_workspace_bytes(-1, 24, 128, 4) == 0
    assert lib.pa_partition_workspace_bytes(8, 0, 128, 4) == 0


def test_binding_carves_partials_from_one_buffer():
    import paged_kv_decode_partitioned_gb300 as pa
    src = open(pa.__file__).read()
    assert "pa_partition_workspace_bytes" in src and "def partition_buffers" in src


def test_default_threshold_uses_sm_count(lib):
    # 64 seqs x 4 KV heads = 256 units: at least one per SM on 152 SMs, not on 300
    assert lib.pa_default_single_pass_max_len(64, 4, 512, 152) == 8192
    assert lib.pa_default_single_pass_max_len(64, 4, 512, 300) == 512
    assert lib.pa_default_single_pass_max_len(16, 4, 512, 152) == 512
    assert lib.pa_default_single_pass_max_len(256, 4, 256, 152) == 8192


@pytest.mark.parametrize("S,L,want", [
    # of 256 / 512 / 1024, the P minimising ceil(S * 4 * ceil(L / P) / 456) * (P + 256)
    # (152 SMs x 3 resident CTAs per wave), ties to the larger P
    (1, 1024, 256), (1, 16384, 256), (1, 32768, 512), (1, 65536, 1024),
    (4, 4096, 256), (4, 8192, 512), (4, 16384, 1024), (4, 65536, 1024),
    (16, 1024, 256), (16, 2048, 512), (16, 4096, 1024), (16, 65536, 1024),
    (256, 65536, 1024),
    # 512 units at P = 1024 are a wave and a bit: three waves of 512-token
    # partitions (2304) beat two of 1024 (2560)
    (4, 32768, 512), (16, 8192, 512),
])
def test_default_partition_size_from_units_and_sms(lib, S, L, want):
    assert lib.pa_default_partition_size(S, 4, 16, 128, L, 152) == want


def test_default_partition_size_is_a_multiple_of_the_block(lib):
    assert lib.pa_default_partition_size(1, 4, 48, 128, 1024, 152) == 288
    assert lib.pa_default_partition_size(1, 4, 2048, 128, 1024, 152) == 2048
    assert lib.pa_default_partition_size(1, 4, 16, 96, 1024, 152) == 0
    assert lib.pa_default_partition_size(1, 0, 16, 128, 1024, 152) == 0


def _resolve(lib, S, Hkv, L, thr, P, sms=152, bs=16, D=128, total=0):
    out = [ctypes.c_int(-9), ctypes.c_int(-9), ctypes.c_int(-9)]
    st = lib.pa_auto_resolve(S, Hkv, D, bs, L, total, thr, P, sms,
                             *[ctypes.byref(o) for o in out])
    return st, tuple(o.value for o in out)


def test_auto_resolve_launch_forms(lib):
    # few units: everything longer than one partition is split on the dense grid
    assert _resolve(lib, 1, 4, 65536, -1, 0) == (0, (1024, 1024, 1))
    assert _resolve(lib, 16, 4, 16384, -1, 0) == (0, (1024, 1024, 1))
    assert _resolve(lib, 1, 4, 200, -1, 0) == (0, (256, 256, 0))   # fits one partition
    # a batch whose single-pass grid (4 units x clusters of 8) fits a wave with at most a
    # partition per CTA: one launch, the threshold raised to max_seq_len
    assert _resolve(lib, 1, 4, 1000, -1, 0) == (0, (1000, 256, 0))
    assert _resolve(lib, 1, 4, 2048, -1, 0) == (0, (2048, 256, 0))
    assert _resolve(lib, 1, 4, 4096, -1, 0) == (0, (256, 256, 1))   # 512 tokens per CTA
    assert _resolve(lib, 16, 4, 1024, -1, 0) == (0, (256, 256, 1))  # 64 x 8 CTAs > a wave
    assert _resolve(lib, 1, 4, 1000, -1, 256) == (0, (1000, 256, 0))
    assert _resolve(lib, 1, 4, 1000, 256, 256) == (0, (256, 256, 1))  # explicit: kept
    # enough units: the pages' 8192 threshold, work list above it, single pass below
    assert _resolve(lib, 256, 4, 65536, -1, 512) == (0, (8192, 512, 2))
    assert _resolve(lib, 64, 4, 8192, -1, 512) == (0, (8192, 512, 0))
    assert _resolve(lib, 256, 4, 65536, -1, 0) == (0, (8192, 1024, 2))
    # explicit values are kept; a threshold above the partition size keeps the work list
    assert _resolve(lib, 2, 4, 5000, 100, 64) == (0, (100, 64, 2))
    assert _resolve(lib, 2, 4, 5000, 0, 64) == (0, (0, 64, 1))
    assert _resolve(lib, 64, 4, 5000, 0, 64) == (0, (0, 64, 2))   # 256 units >= 152 SMs
    # a token bound of nearly S * max_seq_len (equal lengths) and a unit per SM: one
    # pass; unequal lengths (the mixed batch's bound) keep the work list
    assert _resolve(lib, 64, 4, 16384, -1, 512, total=64 * 16384) == (0, (16384, 512, 0))
    assert _resolve(lib, 64, 4, 16384, -1, 512, total=-(-9 * 64 * 16384 // 10)) == \
        (0, (16384, 512, 0))
    assert _resolve(lib, 64, 4, 16384, -1, 512, total=int(0.8 * 64 * 16384)) == \
        (0, (8192, 512, 2))
    assert _resolve(lib, 256, 4, 65536, -1, 512, total=2854935) == (0, (8192, 512, 2))
    # too few units: still split, whatever the lengths
    assert _resolve(lib, 4, 4, 16384, -1, 0, total=4 * 16384) == (0, (1024, 1024, 1))
    # an explicit threshold is kept
    assert _resolve(lib, 64, 4, 16384, 8192, 512, total=64 * 16384) == (0, (8192, 512, 2))
    # bad values
    assert _resolve(lib, 2, 4, 5000, 0, 40)[0] == -2
    assert _resolve(lib, 2, 0, 5000, 0, 64)[0] == -1


def test_product_path_has_no_oracle_or_cpu_fallback():
    """The package never imports the oracle and has no non-CUDA compute path."""
    pkg = os.path.join(ROOT, "paged_kv_decode_partitioned_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f
                assert "pa_oracle" not in text, f


def _prefill(lib, **kw):
    args = dict(out=A, q=A, k=A, v=A, bt=A, sl=A, qs=A, S=2, R=40, mq=30, Hq=24, Hkv=4, D=128,
                bs=16, nb=10, mb=4, scale=0.1, dtype=1)
    args.update(kw)
    return lib.pa_prefill(args["out"], args["q"], args["k"], args["v"], args["bt"], args["sl"],
                          args["qs"], args["S"], args["R"], args["mq"], args["Hq"], args["Hkv"],
                          args["D"], args["bs"], args["nb"], args["mb"], args["scale"],
                          args["dtype"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(D=32), -2),                 # head_dim not supported by the prefill kernel
    (dict(D=96), -2),
    (dict(bs=24), -2),                # block_size neither 8 nor a multiple of 16
    (dict(bs=4), -2),
    (dict(Hq=256, Hkv=1), -2),        # more than 128 query heads per KV head
    (dict(Hq=10, Hkv=4), -1),         # Hq not a multiple of Hkv
    (dict(R=-1), -1),
    (dict(mq=-1), -1),
    (dict(dtype=7), -1),
    (dict(qs=0), -1),                 # null q_start
    (dict(out=0), -1),
    (dict(nb=0), -1),
    (dict(q=A + 8), -3),              # misaligned query
    (dict(qs=A + 2), -3),             # misaligned q_start
    (dict(S=0), 0),                   # nothing to do
    (dict(R=0), 0),
    (dict(mq=0), 0),
])
def test_prefill_rejects_on_host(lib, kw, status):
    assert _prefill(lib, **kw) == status


def test_moe_entry_points_reject_on_host(lib):
    # router: unsupported expert count, topk above 32 or E, bad dtype, misaligned logits
    assert lib.pa_topk_softmax(A, A, A, 16, 100, 8, 0, 1, None) == -2
    assert lib.pa_topk_softmax(A, A, A, 16, 256, 33, 0, 1, None) == -2
    assert lib.pa_topk_softmax(A, A, A, 16, 32, 33, 0, 1, None) == -2
    assert lib.pa_topk_softmax(A, A, A, 16, 256, 8, 0, 5, None) == -1
    assert lib.pa_topk_softmax(A, A, A + 4, 16, 256, 8, 0, 1, None) == -3
    assert lib.pa_topk_softmax(A, A, A, 0, 256, 8, 0, 1, None) == 0
    # sort: too many experts, missing workspace, workspace too small, misaligned
    need = lib.pa_moe_sort_workspace_bytes(131072, 256)
    assert need >= 64 * 256 * 4
    assert lib.pa_moe_sort_workspace_bytes(10, 2000) == 0
    assert lib.pa_moe_sort(A, A, A, A, 131072, 2000, A, need, None) == -2
    assert lib.pa_moe_sort(A, A, A, A, 131072, 256, 0, need, None) == -1
    assert lib.pa_moe_sort(A, A, A, A, 131072, 256, A, need - 1, None) == -4
    assert lib.pa_moe_sort(A, A, A, A, 131072, 256, A + 16, need, None) == -3
    # gather / scatter-back: row size, topk, alignment
    assert lib.pa_moe_gather(A, A, A, 100, 8, 800, 12, 1, None) == -2
    assert lib.pa_moe_gather(A, A, A, 100, 33, 3300, 2048, 1, None) == -2
    assert lib.pa_moe_gather(A + 8, A, A, 100, 8, 800, 2048, 1, None) == -3
    assert lib.pa_moe_gather(A, A, A + 2, 100, 8, 800, 2048, 1, None) == -3
    assert lib.pa_moe_gather(A, A, A, 0, 8, 0, 2048, 1, None) == 0
    assert lib.pa_moe_scatter_back(A, A, A, A, 16, 33, 2048, 1, None) == -2
    assert lib.pa_moe_scatter_back(A, A, A, A, 16, 8, 2044, 1, None) == -2
    assert lib.pa_moe_scatter_back(A, A, A, A, 16, 8, 2048, 3, None) == -1
    assert lib.pa_moe_scatter_back(A, A, A, A, 0, 8, 2048, 1, None) == 0
