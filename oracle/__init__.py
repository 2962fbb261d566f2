"""TEST INFRASTRUCTURE ONLY: the fp64 CPU oracle for paged-attention decode.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it and
shares no code with it; the C source ``pa_oracle.c`` is the whole computation,
this module only compiles it with the host C compiler and marshals arrays.

What each function computes, and the passage it follows, is stated in
``pa_oracle.c`` (page: project_6 commit cd0d9e1, "qwen3_6_scripts": the
forward_decode heuristic, phases 1 and 2 of the V2 description, the
pre-gather of context K/V through the block table, the prefix prefill, and
the MoE sort-by-expert regrouping; page: commit 490ff98, "Dockerfile": the
topk_softmax router).

Arrays are numpy arrays or CPU torch tensors.  16-bit floating-point inputs
(query, key/value caches) are passed as their bit patterns; the oracle widens
them to fp64 with its own decoder.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libpa_oracle.so")

F16 = 0
BF16 = 1

_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_i32p = ctypes.POINTER(ctypes.c_int32)
_int = ctypes.c_int


def build(force: bool = False) -> str:
    """Compile ``pa_oracle.c`` into ``_build/libpa_oracle.so`` (gcc, OpenMP)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_half_bits_to_f64.restype = ctypes.c_double
            lib.oracle_half_bits_to_f64.argtypes = [ctypes.c_uint16, _int]
            lib.oracle_bits_to_f64.restype = None
            lib.oracle_bits_to_f64.argtypes = [_u16p, _dp, ctypes.c_int64, _int]
            lib.oracle_attention.restype = _int
            lib.oracle_attention.argtypes = [_dp, _u16p, _u16p, _u16p, _i32p, _i32p] + \
                [_int] * 7 + [ctypes.c_float, _int]
            lib.oracle_partials.restype = _int
            lib.oracle_partials.argtypes = [_dp, _dp, _dp, _u16p, _u16p, _u16p, _i32p,
                                            _i32p] + [_int] * 7 + [ctypes.c_float] + \
                [_int] * 3
            lib.oracle_lse_merge.restype = _int
            lib.oracle_lse_merge.argtypes = [_dp, _dp, _dp, _dp, _i32p] + [_int] * 5
            lib.oracle_prefill.restype = _int
            lib.oracle_prefill.argtypes = [_dp, _u16p, _u16p, _u16p, _i32p, _i32p, _i32p] + \
                [_int] * 7 + [ctypes.c_float, _int]
            lib.oracle_topk_softmax.restype = _int
            lib.oracle_topk_softmax.argtypes = [_dp, _i32p, _dp] + [_int] * 4
            lib.oracle_moe_sort.restype = _int
            lib.oracle_moe_sort.argtypes = [_i32p, _i32p, _i32p, _i32p, _int, _int]
            lib.oracle_moe_gather.restype = _int
            lib.oracle_moe_gather.argtypes = [_u16p, _u16p, _i32p] + [_int] * 4
            lib.oracle_moe_scatter.restype = _int
            lib.oracle_moe_scatter.argtypes = [_dp, _u16p, _i32p, _dp] + [_int] * 5
            lib.oracle_gather.restype = _int
            lib.oracle_gather.argtypes = [_u16p, _u16p, _u16p, _u16p, _i32p, _i32p] + \
                [_int] * 7
            _lib = lib
    return _lib


def set_num_threads(n: int) -> None:
    """Set the OpenMP thread count the oracle uses (0 leaves the default)."""
    if n > 0:
        os.environ["OMP_NUM_THREADS"] = str(n)
        try:
            gomp = ctypes.CDLL("libgomp.so.1")
            gomp.omp_set_num_threads(ctypes.c_int(n))
        except OSError:
            pass


def _bits(x) -> np.ndarray:
    """16-bit float array (torch fp16/bf16 tensor or numpy uint16/float16) -> uint16 bits."""
    if hasattr(x, "detach"):  # torch tensor
        import torch
        x = x.detach()
        if x.device.type != "cpu":
            raise ValueError("the oracle reads host memory only")
        return np.ascontiguousarray(x.contiguous().view(torch.int16).numpy().view(np.uint16))
    x = np.asarray(x)
    if x.dtype == np.float16:
        x = x.view(np.uint16)
    if x.dtype != np.uint16:
        raise TypeError(f"expected 16-bit float bit patterns, got {x.dtype}")
    return np.ascontiguousarray(x)


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _dtype_code(x, dtype) -> int:
    if dtype is not None:
        return {"f16": F16, "fp16": F16, "float16": F16, "bf16": BF16,
                "bfloat16": BF16, F16: F16, BF16: BF16}[dtype]
    if hasattr(x, "dtype"):
        name = str(x.dtype)
        if "bfloat16" in name:
            return BF16
        if "float16" in name:
            return F16
    raise ValueError("cannot infer 16-bit float type; pass dtype='f16' or 'bf16'")


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its inputs (status {rc})")


def bits_to_f64(x, dtype=None) -> np.ndarray:
    """Widen 16-bit float bit patterns to fp64 with the oracle's own decoder."""
    code = _dtype_code(x, dtype)
    b = _bits(x)
    out = np.empty(b.shape, dtype=np.float64)
    _load().oracle_bits_to_f64(_ptr(b, ctypes.c_uint16), _ptr(out, ctypes.c_double),
                               b.size, code)
    return out


def _shapes(query, key_cache, block_tables):
    S, Hq, d = query.shape
    num_blocks, bs, Hkv, d2 = key_cache.shape
    if d2 != d:
        raise ValueError("head_dim mismatch between query and cache")
    if block_tables.ndim != 2 or block_tables.shape[0] != S:
        raise ValueError("block_tables must be [num_seqs, max_blocks_per_seq]")
    return S, Hq, Hkv, d, bs, num_blocks, block_tables.shape[1]


def attention(query, key_cache, value_cache, block_tables, seq_lens, scale,
              dtype=None) -> np.ndarray:
    """Single-pass decode output [S, Hq, d] in fp64 (see ``oracle_attention``)."""
    code = _dtype_code(query, dtype)
    q, k, v = _bits(query), _bits(key_cache), _bits(value_cache)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    S, Hq, Hkv, d, bs, nb, mb = _shapes(q, k, bt)
    out = np.empty((S, Hq, d), dtype=np.float64)
    rc = _load().oracle_attention(
        _ptr(out, ctypes.c_double), _ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
        _ptr(v, ctypes.c_uint16), _ptr(bt, ctypes.c_int32), _ptr(sl, ctypes.c_int32),
        S, Hq, Hkv, d, bs, nb, mb, ctypes.c_float(scale), code)
    _check(rc, "attention")
    return out


def num_partitions(seq_len: int, partition_size: int) -> int:
    """ceil(L / P): the partition count of one sequence."""
    return -(-int(seq_len) // int(partition_size))


def partials(query, key_cache, value_cache, block_tables, seq_lens, scale,
             partition_size, max_num_partitions=None, dtype=None):
    """Phase-1 partials (tmp_out [S,Hq,NP,d], exp_sums [S,Hq,NP], max_logits [S,Hq,NP]).

    Slots of partitions p >= ceil(L/P) are NaN.
    """
    code = _dtype_code(query, dtype)
    q, k, v = _bits(query), _bits(key_cache), _bits(value_cache)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    S, Hq, Hkv, d, bs, nb, mb = _shapes(q, k, bt)
    NP = max_num_partitions
    if NP is None:
        NP = max([num_partitions(x, partition_size) for x in sl] + [1])
    tmp = np.full((S, Hq, NP, d), np.nan)
    es = np.full((S, Hq, NP), np.nan)
    ml = np.full((S, Hq, NP), np.nan)
    rc = _load().oracle_partials(
        _ptr(tmp, ctypes.c_double), _ptr(es, ctypes.c_double), _ptr(ml, ctypes.c_double),
        _ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
        _ptr(bt, ctypes.c_int32), _ptr(sl, ctypes.c_int32), S, Hq, Hkv, d, bs, nb, mb,
        ctypes.c_float(scale), int(partition_size), int(NP), code)
    _check(rc, "partials")
    return tmp, es, ml


def lse_merge(tmp_out, exp_sums, max_logits, seq_lens, partition_size) -> np.ndarray:
    """Phase-2 log-sum-exp merge of fp64 partials -> [S, Hq, d]."""
    tmp = np.ascontiguousarray(tmp_out, dtype=np.float64)
    es = np.ascontiguousarray(exp_sums, dtype=np.float64)
    ml = np.ascontiguousarray(max_logits, dtype=np.float64)
    sl = _i32(seq_lens)
    S, Hq, NP, d = tmp.shape
    out = np.empty((S, Hq, d), dtype=np.float64)
    rc = _load().oracle_lse_merge(
        _ptr(out, ctypes.c_double), _ptr(tmp, ctypes.c_double), _ptr(es, ctypes.c_double),
        _ptr(ml, ctypes.c_double), _ptr(sl, ctypes.c_int32), S, Hq, d,
        int(partition_size), NP)
    _check(rc, "lse_merge")
    return out


def prefill(query, key_cache, value_cache, block_tables, seq_lens, q_start, scale,
            dtype=None) -> np.ndarray:
    """Prefix prefill output [q_start[-1], Hq, d] in fp64 (see ``oracle_prefill``)."""
    code = _dtype_code(query, dtype)
    q, k, v = _bits(query), _bits(key_cache), _bits(value_cache)
    bt, sl, qs = _i32(block_tables), _i32(seq_lens), _i32(q_start)
    R, Hq, d = q.shape
    num_blocks, bs, Hkv, d2 = k.shape
    S, mb = bt.shape
    if d2 != d or qs.shape != (S + 1,) or qs[-1] != R:
        raise ValueError("prefill shapes disagree")
    out = np.empty((R, Hq, d), dtype=np.float64)
    rc = _load().oracle_prefill(
        _ptr(out, ctypes.c_double), _ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
        _ptr(v, ctypes.c_uint16), _ptr(bt, ctypes.c_int32), _ptr(sl, ctypes.c_int32),
        _ptr(qs, ctypes.c_int32), S, Hq, Hkv, d, bs, num_blocks, mb, ctypes.c_float(scale), code)
    _check(rc, "prefill")
    return out


def gather(key_cache, value_cache, block_tables, seq_lens, max_len=None):
    """Dense per-sequence K/V bit patterns [S, max_len, Hkv, d] (uint16); rows t >= L are 0."""
    k, v = _bits(key_cache), _bits(value_cache)
    bt, sl = _i32(block_tables), _i32(seq_lens)
    nb, bs, Hkv, d = k.shape
    S, mb = bt.shape
    if max_len is None:
        max_len = int(sl.max()) if S else 0
    kd = np.zeros((S, max_len, Hkv, d), dtype=np.uint16)
    vd = np.zeros((S, max_len, Hkv, d), dtype=np.uint16)
    rc = _load().oracle_gather(
        _ptr(kd, ctypes.c_uint16), _ptr(vd, ctypes.c_uint16), _ptr(k, ctypes.c_uint16),
        _ptr(v, ctypes.c_uint16), _ptr(bt, ctypes.c_int32), _ptr(sl, ctypes.c_int32),
        S, Hkv, d, bs, nb, mb, int(max_len))
    _check(rc, "gather")
    return kd, vd


def _logits_f64(logits) -> np.ndarray:
    """Router logits (fp32, or 16-bit float bit patterns via their dtype) as exact fp64."""
    if isinstance(logits, np.ndarray) and logits.dtype in (np.float32, np.float64):
        return np.ascontiguousarray(logits, dtype=np.float64)
    import torch
    t = logits if isinstance(logits, torch.Tensor) else torch.as_tensor(logits)
    t = t.detach().cpu()
    if t.dtype in (torch.float16, torch.bfloat16):
        return bits_to_f64(t)
    return np.ascontiguousarray(t.to(torch.float64).numpy())


def topk_softmax(logits, k: int, renormalize: bool = False):
    """Router (see ``oracle_topk_softmax``): returns (weights fp64 [T,k], ids int32 [T,k])."""
    x = _logits_f64(logits)
    T, E = x.shape
    w = np.empty((T, k), dtype=np.float64)
    ids = np.empty((T, k), dtype=np.int32)
    rc = _load().oracle_topk_softmax(_ptr(w, ctypes.c_double), _ptr(ids, ctypes.c_int32),
                                     _ptr(x, ctypes.c_double), T, E, int(k), int(bool(renormalize)))
    _check(rc, "topk_softmax")
    return w, ids


def moe_sort(expert_ids, num_experts: int):
    """Stable sort of the flat pairs by expert (see ``oracle_moe_sort``):
    returns (sorted_pairs [P], offsets [E+1], pair_pos [P]), all int32."""
    ids = _i32(expert_ids).reshape(-1)
    P = ids.shape[0]
    sp = np.empty(P, dtype=np.int32)
    off = np.empty(num_experts + 1, dtype=np.int32)
    pos = np.empty(P, dtype=np.int32)
    rc = _load().oracle_moe_sort(_ptr(sp, ctypes.c_int32), _ptr(off, ctypes.c_int32),
                                 _ptr(pos, ctypes.c_int32), _ptr(ids, ctypes.c_int32), P,
                                 int(num_experts))
    _check(rc, "moe_sort")
    return sp, off, pos


def moe_gather(hidden, sorted_pairs, k: int) -> np.ndarray:
    """Rows of ``hidden`` [T,H] in sorted-pair order, as 16-bit bit patterns [P,H]."""
    h = _bits(hidden)
    T, H = h.shape
    sp = _i32(sorted_pairs).reshape(-1)
    out = np.empty((sp.shape[0], H), dtype=np.uint16)
    rc = _load().oracle_moe_gather(_ptr(out, ctypes.c_uint16), _ptr(h, ctypes.c_uint16),
                                   _ptr(sp, ctypes.c_int32), sp.shape[0], int(k), T, H)
    _check(rc, "moe_gather")
    return out


def moe_scatter(y, pair_pos, weights, k: int, dtype=None) -> np.ndarray:
    """Scatter-back (see ``oracle_moe_scatter``): fp64 [T,H] from per-pair rows ``y`` [P,H]."""
    code = _dtype_code(y, dtype)
    yb = _bits(y)
    P, H = yb.shape
    pos = _i32(pair_pos).reshape(-1)
    w = np.ascontiguousarray(np.asarray(weights, dtype=np.float64).reshape(-1))
    T = P // int(k)
    out = np.empty((T, H), dtype=np.float64)
    rc = _load().oracle_moe_scatter(_ptr(out, ctypes.c_double), _ptr(yb, ctypes.c_uint16),
                                    _ptr(pos, ctypes.c_int32), _ptr(w, ctypes.c_double), T,
                                    int(k), P, H, code)
    _check(rc, "moe_scatter")
    return out
