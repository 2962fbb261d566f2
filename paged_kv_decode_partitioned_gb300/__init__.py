"""Paged-attention decode for GB300 (sm_103a): the Python binding of libpadecode.so.

Every function here only marshals arguments (torch tensors -> device pointers,
the current CUDA stream) and calls the C ABI declared in ``include/pa_decode.h``;
all of the computation runs in the library's CUDA kernels.  There is no other
code path: if the compiled library is missing, importing a function raises.

The operation (page: project_6 commit cd0d9e1, "qwen3_6_scripts"): one decode
query per sequence attends over a block-paged KV cache through a
per-sequence block table; long sequences are split into partitions whose
partial results are merged with a log-sum-exp rescale (the V2 path of the
forward_decode heuristic, phases 1 and 2).
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Tuple

import torch

__all__ = [
    "PaError", "load_library", "library_path", "decode", "decode_partitioned",
    "partition_reduce", "decode_auto", "decode_auto_static", "auto_workspace_bytes",
    "default_single_pass_max_len", "default_partition_size", "auto_resolve",
    "partition_workspace_bytes", "AUTO_SINGLE_PASS", "AUTO_DENSE", "AUTO_WORKLIST",
    "prefill", "gather_kv", "device_status", "num_partitions", "version",
    "DEV_BAD_BLOCK", "DEV_LEN_CLAMPED", "DEV_WAIT_TIMEOUT", "DEV_TOO_MANY_PARTITIONS",
    "DEV_BAD_ROWS", "DEV_BAD_EXPERT", "topk_softmax", "moe_sort", "moe_gather",
    "moe_scatter_back", "moe_sort_workspace_bytes",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_lib", "libpadecode.so")

PA_F16, PA_BF16 = 0, 1
PHASE_PLAN, PHASE_ATTEND, PHASE_REDUCE = 1, 2, 4
AUTO_SINGLE_PASS, AUTO_DENSE, AUTO_WORKLIST = 0, 1, 2
DEV_BAD_BLOCK, DEV_LEN_CLAMPED, DEV_WAIT_TIMEOUT, DEV_TOO_MANY_PARTITIONS = 1, 2, 4, 8
DEV_BAD_ROWS = 16
DEV_BAD_EXPERT = 32
LOGITS_F16, LOGITS_BF16, LOGITS_F32 = 0, 1, 2

_lock = threading.Lock()
_lib = None

_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_ll = ctypes.c_longlong
_sz = ctypes.c_size_t
_ip = ctypes.POINTER(ctypes.c_int)

# (name, restype, argtypes) of every entry point in include/pa_decode.h and include/pa_moe.h
SIGNATURES = [
    ("pa_decode", _i, [_vp] * 6 + [_i] * 7 + [_f, _i, _vp]),
    ("pa_decode_partitioned", _i, [_vp] * 8 + [_i] * 7 + [_f, _i, _i, _i, _vp]),
    ("pa_partition_reduce", _i, [_vp] * 5 + [_i] * 6 + [_vp]),
    ("pa_partition_workspace_bytes", _sz, [_i] * 4),
    ("pa_default_single_pass_max_len", _i, [_i] * 4),
    ("pa_default_partition_size", _i, [_i] * 6),
    ("pa_auto_resolve", _i, [_i] * 5 + [_ll] + [_i] * 3 + [_ip] * 3),
    ("pa_auto_workspace_bytes", _sz, [_i] * 6 + [_ll, _i, _i]),
    ("pa_decode_auto", _i, [_vp] * 6 + [_i] * 7 + [_f, _i, _ll, _i, _i, _vp, _sz, _i, _vp]),
    ("pa_decode_auto_phases", _i, [_vp] * 6 + [_i] * 7 + [_f, _i, _ll, _i, _i, _vp, _sz, _i,
                                                           _vp, _i]),
    ("pa_decode_auto_static", _i, [_vp] * 6 + [_i] * 7 + [_f, _i, _ll, _i, _i, _i, _vp]),
    ("pa_prefill", _i, [_vp] * 7 + [_i] * 9 + [_f, _i, _vp]),
    ("pa_gather_kv", _i, [_vp] * 6 + [_i] * 7 + [_i, _vp]),
    ("pa_topk_softmax", _i, [_vp] * 3 + [_i] * 5 + [_vp]),
    ("pa_moe_sort_workspace_bytes", ctypes.c_size_t, [_i, _i]),
    ("pa_moe_sort", _i, [_vp] * 4 + [_i, _i, _vp, ctypes.c_size_t, _vp]),
    ("pa_moe_gather", _i, [_vp] * 3 + [_i] * 5 + [_vp]),
    ("pa_moe_scatter_back", _i, [_vp] * 4 + [_i] * 4 + [_vp]),
    ("pa_selftest_wait_timeout", _i, [_vp, _i]),
    ("pa_device_status", _i, [_vp, ctypes.POINTER(_i)]),
    ("pa_status_string", ctypes.c_char_p, [_i]),
    ("pa_version", _i, []),
]


class PaError(RuntimeError):
    """A non-zero status returned by the library."""

    def __init__(self, status: int, what: str):
        self.status = status
        name = _load().pa_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{what} failed: {name} ({status})")


def library_path() -> str:
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_LIB_PATH):
                raise ImportError(
                    f"libpadecode.so is not built ({_LIB_PATH}); run "
                    "`python -m paged_kv_decode_partitioned_gb300.build`")
            lib = ctypes.CDLL(_LIB_PATH)
            for name, res, args in SIGNATURES:
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def load_library():
    """Load (and return) the ctypes handle of libpadecode.so."""
    return _load()


def version() -> int:
    return _load().pa_version()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return PA_F16
    if t.dtype == torch.bfloat16:
        return PA_BF16
    raise TypeError(f"query/cache dtype must be float16 or bfloat16, got {t.dtype}")


def _dev(t: torch.Tensor, name: str) -> int:
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _i32(t: torch.Tensor, name: str) -> int:
    if t.dtype != torch.int32:
        raise TypeError(f"{name} must be int32")
    return _dev(t, name)


def _f32(t: torch.Tensor, name: str) -> int:
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32")
    return _dev(t, name)


def _stream(t: torch.Tensor) -> int:
    return torch.cuda.current_stream(t.device).cuda_stream


def _check(status: int, what: str) -> None:
    if status != 0:
        raise PaError(status, what)


def num_partitions(seq_len: int, partition_size: int) -> int:
    """ceil(seq_len / partition_size)."""
    return -(-int(seq_len) // int(partition_size))


def _shape(query, key_cache, block_tables):
    S, Hq, D = query.shape
    nb, bs, Hkv, D2 = key_cache.shape
    if D2 != D:
        raise ValueError("query and cache head_dim differ")
    return S, Hq, Hkv, D, bs, nb, block_tables.shape[1]


def decode(query, key_cache, value_cache, block_tables, seq_lens, scale: float,
           out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Single-pass decode (``pa_decode``); returns ``out`` [S, Hq, D]."""
    S, Hq, Hkv, D, bs, nb, mb = _shape(query, key_cache, block_tables)
    if out is None:
        out = torch.empty_like(query)
    with torch.cuda.device(query.device):
        st = _load().pa_decode(
            _dev(out, "out"), _dev(query, "query"), _dev(key_cache, "key_cache"),
            _dev(value_cache, "value_cache"), _i32(block_tables, "block_tables"),
            _i32(seq_lens, "seq_lens"), S, Hq, Hkv, D, bs, nb, mb, float(scale),
            _dtype_code(query), _stream(query))
    _check(st, "pa_decode")
    return out


def partition_workspace_bytes(num_seqs: int, num_q_heads: int, head_dim: int,
                              max_num_partitions: int) -> int:
    """Bytes of the dense phase-1 partials (``pa_partition_workspace_bytes``)."""
    return int(_load().pa_partition_workspace_bytes(int(num_seqs), int(num_q_heads),
                                                    int(head_dim), int(max_num_partitions)))


def partition_buffers(num_seqs: int, num_q_heads: int, head_dim: int, max_num_partitions: int,
                      device) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """(tmp_out, exp_sums, max_logits) as views of one buffer of
    ``partition_workspace_bytes`` bytes, in the layout the header states."""
    S, Hq, D, NP = int(num_seqs), int(num_q_heads), int(head_dim), int(max_num_partitions)
    total = partition_workspace_bytes(S, Hq, D, NP)
    if total == 0:
        raise ValueError("bad partition buffer shape")
    buf = torch.empty(total // 4, dtype=torch.float32, device=device)
    rows = S * Hq * NP

    def up(x):
        return (x + 255) // 256 * 256
    o_es = up(rows * D * 4)
    o_ml = up(o_es + rows * 4)
    tmp_out = buf[:rows * D].view(S, Hq, NP, D)
    exp_sums = buf[o_es // 4:o_es // 4 + rows].view(S, Hq, NP)
    max_logits = buf[o_ml // 4:o_ml // 4 + rows].view(S, Hq, NP)
    return tmp_out, exp_sums, max_logits


def decode_partitioned(query, key_cache, value_cache, block_tables, seq_lens, scale: float,
                       partition_size: int, max_num_partitions: int,
                       tmp_out=None, exp_sums=None, max_logits=None
                       ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Phase 1 (``pa_decode_partitioned``); returns (tmp_out, exp_sums, max_logits).

    Buffers not passed are carved from one allocation sized by
    ``pa_partition_workspace_bytes``."""
    S, Hq, Hkv, D, bs, nb, mb = _shape(query, key_cache, block_tables)
    NP = int(max_num_partitions)
    dev = query.device
    if tmp_out is None or exp_sums is None or max_logits is None:
        t, e, m = partition_buffers(S, Hq, D, NP, dev)
        tmp_out = t if tmp_out is None else tmp_out
        exp_sums = e if exp_sums is None else exp_sums
        max_logits = m if max_logits is None else max_logits
    with torch.cuda.device(dev):
        st = _load().pa_decode_partitioned(
            _f32(tmp_out, "tmp_out"), _f32(exp_sums, "exp_sums"), _f32(max_logits, "max_logits"),
            _dev(query, "query"), _dev(key_cache, "key_cache"), _dev(value_cache, "value_cache"),
            _i32(block_tables, "block_tables"), _i32(seq_lens, "seq_lens"),
            S, Hq, Hkv, D, bs, nb, mb, float(scale), int(partition_size), NP,
            _dtype_code(query), _stream(query))
    _check(st, "pa_decode_partitioned")
    return tmp_out, exp_sums, max_logits


def partition_reduce(tmp_out, exp_sums, max_logits, seq_lens, partition_size: int,
                     out: Optional[torch.Tensor] = None, dtype=torch.bfloat16) -> torch.Tensor:
    """Phase 2 (``pa_partition_reduce``); returns ``out`` [S, Hq, D] of ``dtype``."""
    S, Hq, NP, D = tmp_out.shape
    if out is None:
        out = torch.empty((S, Hq, D), dtype=dtype, device=tmp_out.device)
    with torch.cuda.device(tmp_out.device):
        st = _load().pa_partition_reduce(
            _dev(out, "out"), _f32(tmp_out, "tmp_out"), _f32(exp_sums, "exp_sums"),
            _f32(max_logits, "max_logits"), _i32(seq_lens, "seq_lens"), S, Hq, D,
            int(partition_size), NP, _dtype_code(out), _stream(tmp_out))
    _check(st, "pa_partition_reduce")
    return out


def default_single_pass_max_len(num_seqs: int, num_kv_heads: int, partition_size: int = 512,
                                num_sms: int = 0) -> int:
    return _load().pa_default_single_pass_max_len(num_seqs, num_kv_heads, partition_size,
                                                  num_sms)


def default_partition_size(num_seqs: int, num_kv_heads: int, block_size: int, head_dim: int,
                           max_seq_len: int, num_sms: int = 0) -> int:
    return _load().pa_default_partition_size(num_seqs, num_kv_heads, block_size, head_dim,
                                             max_seq_len, num_sms)


def auto_resolve(num_seqs: int, num_kv_heads: int, head_dim: int, block_size: int,
                 max_seq_len: int, single_pass_max_len: int = -1, partition_size: int = 0,
                 num_sms: int = 0, max_total_tokens: int = 0) -> Tuple[int, int, int]:
    """(single-pass threshold, partition size, launch form) that ``pa_decode_auto``
    takes for these host values (``pa_auto_resolve``)."""
    thr, P, form = ctypes.c_int(0), ctypes.c_int(0), ctypes.c_int(0)
    st = _load().pa_auto_resolve(int(num_seqs), int(num_kv_heads), int(head_dim),
                                 int(block_size), int(max_seq_len), int(max_total_tokens),
                                 int(single_pass_max_len), int(partition_size), int(num_sms),
                                 ctypes.byref(thr), ctypes.byref(P), ctypes.byref(form))
    _check(st, "pa_auto_resolve")
    return thr.value, P.value, form.value


def auto_workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                         block_size: int, max_seq_len: int, max_total_tokens: int = 0,
                         single_pass_max_len: int = -1, partition_size: int = 0) -> int:
    return int(_load().pa_auto_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                               block_size, max_seq_len, int(max_total_tokens),
                                               single_pass_max_len, partition_size))


def decode_auto(query, key_cache, value_cache, block_tables, seq_lens, scale: float,
                max_seq_len: int, single_pass_max_len: int = -1, partition_size: int = 0,
                workspace: Optional[torch.Tensor] = None,
                out: Optional[torch.Tensor] = None, phases: Optional[int] = None,
                max_total_tokens: int = 0) -> torch.Tensor:
    """Whole decode step with the per-sequence V1/V2 choice (``pa_decode_auto``).

    ``single_pass_max_len=-1`` and ``partition_size=0`` select the library's
    launch heuristic; ``max_total_tokens`` (> 0) bounds the batch's total
    tokens, which shrinks the workspace.  ``phases`` (a PHASE_* mask) calls
    ``pa_decode_auto_phases`` instead, to run only some of the step's launches;
    every phase needs the same arguments.
    """
    S, Hq, Hkv, D, bs, nb, mb = _shape(query, key_cache, block_tables)
    if workspace is None:
        need = auto_workspace_bytes(S, Hq, Hkv, D, bs, max_seq_len, max_total_tokens,
                                    single_pass_max_len, partition_size)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=query.device)
    if out is None:
        out = torch.empty_like(query)
    args = (_dev(out, "out"), _dev(query, "query"), _dev(key_cache, "key_cache"),
            _dev(value_cache, "value_cache"), _i32(block_tables, "block_tables"),
            _i32(seq_lens, "seq_lens"), S, Hq, Hkv, D, bs, nb, mb, float(scale),
            int(max_seq_len), int(max_total_tokens), int(single_pass_max_len),
            int(partition_size), _dev(workspace, "workspace"),
            workspace.numel() * workspace.element_size(), _dtype_code(query), _stream(query))
    with torch.cuda.device(query.device):
        if phases is None:
            st = _load().pa_decode_auto(*args)
        else:
            st = _load().pa_decode_auto_phases(*args, int(phases))
    _check(st, "pa_decode_auto")
    return out


def decode_auto_static(query, key_cache, value_cache, block_tables, seq_lens, scale: float,
                       max_seq_len: int, single_pass_max_len: int = -1,
                       partition_size: int = 0, out: Optional[torch.Tensor] = None,
                       max_total_tokens: int = 0) -> torch.Tensor:
    """``pa_decode_auto_static``: ``decode_auto`` with the library's fixed scratch.

    For callers that cannot allocate device memory: no workspace is passed and
    none is allocated.  Batches needing more than the library's fixed scratch
    are rejected (PaError with PA_ERR_WORKSPACE_TOO_SMALL).  Calls on one device
    share that scratch, so calls that overlap on the GPU must be serialised.
    """
    S, Hq, Hkv, D, bs, nb, mb = _shape(query, key_cache, block_tables)
    if out is None:
        out = torch.empty_like(query)
    with torch.cuda.device(query.device):
        st = _load().pa_decode_auto_static(
            _dev(out, "out"), _dev(query, "query"), _dev(key_cache, "key_cache"),
            _dev(value_cache, "value_cache"), _i32(block_tables, "block_tables"),
            _i32(seq_lens, "seq_lens"), S, Hq, Hkv, D, bs, nb, mb, float(scale),
            int(max_seq_len), int(max_total_tokens), int(single_pass_max_len),
            int(partition_size), _dtype_code(query), _stream(query))
    _check(st, "pa_decode_auto_static")
    return out


def prefill(query, key_cache, value_cache, block_tables, seq_lens, q_start, scale: float,
            max_q_len: int, out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Prefix prefill over the paged cache (``pa_prefill``); returns ``out`` [R, Hq, D].

    ``query`` holds the chunks of all sequences, R rows in all; ``q_start``
    (int32, S + 1) gives each sequence's first row, and ``max_q_len`` bounds
    every chunk's length.  The chunks' K/V must already be in the cache.
    """
    R, Hq, D = query.shape
    nb, bs, Hkv, D2 = key_cache.shape
    if D2 != D:
        raise ValueError("query and cache head_dim differ")
    S, mb = block_tables.shape
    if q_start.shape != (S + 1,):
        raise ValueError("q_start must have num_seqs + 1 entries")
    if out is None:
        out = torch.empty_like(query)
    with torch.cuda.device(query.device):
        st = _load().pa_prefill(
            _dev(out, "out"), _dev(query, "query"), _dev(key_cache, "key_cache"),
            _dev(value_cache, "value_cache"), _i32(block_tables, "block_tables"),
            _i32(seq_lens, "seq_lens"), _i32(q_start, "q_start"), S, R, int(max_q_len), Hq,
            Hkv, D, bs, nb, mb, float(scale), _dtype_code(query), _stream(query))
    _check(st, "pa_prefill")
    return out


def topk_softmax(gating_logits, topk: int, renormalize: bool = False,
                 weights: Optional[torch.Tensor] = None, ids: Optional[torch.Tensor] = None):
    """MoE router (``pa_topk_softmax``): returns (weights fp32 [T,k], ids int32 [T,k])."""
    T, E = gating_logits.shape
    code = {torch.float16: LOGITS_F16, torch.bfloat16: LOGITS_BF16,
            torch.float32: LOGITS_F32}.get(gating_logits.dtype)
    if code is None:
        raise TypeError("router logits must be float16, bfloat16 or float32")
    dev = gating_logits.device
    if weights is None:
        weights = torch.empty((T, topk), dtype=torch.float32, device=dev)
    if ids is None:
        ids = torch.empty((T, topk), dtype=torch.int32, device=dev)
    with torch.cuda.device(dev):
        st = _load().pa_topk_softmax(_f32(weights, "weights"), _i32(ids, "ids"),
                                     _dev(gating_logits, "gating_logits"), T, E, int(topk),
                                     int(bool(renormalize)), code, _stream(gating_logits))
    _check(st, "pa_topk_softmax")
    return weights, ids


def moe_sort_workspace_bytes(num_pairs: int, num_experts: int) -> int:
    return int(_load().pa_moe_sort_workspace_bytes(int(num_pairs), int(num_experts)))


def moe_sort(expert_ids, num_experts: int, workspace: Optional[torch.Tensor] = None, out=None):
    """Stable sort of the flat pairs by expert (``pa_moe_sort``): returns
    (sorted_pairs [P], expert_offsets [E+1], pair_pos [P]), int32."""
    flat = expert_ids.reshape(-1)
    P = flat.numel()
    dev = expert_ids.device
    if out is None:
        out = (torch.empty(P, dtype=torch.int32, device=dev),
               torch.empty(num_experts + 1, dtype=torch.int32, device=dev),
               torch.empty(P, dtype=torch.int32, device=dev))
    sp, off, pos = out
    need = moe_sort_workspace_bytes(P, num_experts)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    with torch.cuda.device(dev):
        st = _load().pa_moe_sort(_i32(sp, "sorted_pairs"), _i32(off, "expert_offsets"),
                                 _i32(pos, "pair_pos"), _i32(flat, "expert_ids"), P,
                                 int(num_experts), _dev(workspace, "workspace"),
                                 workspace.numel() * workspace.element_size(),
                                 _stream(expert_ids))
    _check(st, "pa_moe_sort")
    return sp, off, pos


def moe_gather(hidden, pair_pos, topk: int, out: Optional[torch.Tensor] = None):
    """Hidden rows in expert-sorted order (``pa_moe_gather``): row ``pair_pos[p]`` of
    the result is ``hidden[p // topk]``; returns [T * topk, H]."""
    T, H = hidden.shape
    if pair_pos.numel() != T * topk:
        raise ValueError("pair_pos must have num_tokens * topk entries")
    if out is None:
        out = torch.empty((T * topk, H), dtype=hidden.dtype, device=hidden.device)
    with torch.cuda.device(hidden.device):
        st = _load().pa_moe_gather(_dev(out, "sorted_hidden"), _dev(hidden, "hidden"),
                                   _i32(pair_pos, "pair_pos"), T, int(topk), out.shape[0], H,
                                   _dtype_code(hidden), _stream(hidden))
    _check(st, "pa_moe_gather")
    return out


def moe_scatter_back(expert_out, pair_pos, topk_weights, out: Optional[torch.Tensor] = None):
    """Weighted scatter-back of the per-pair rows (``pa_moe_scatter_back``): [T, H]."""
    P, H = expert_out.shape
    T, K = topk_weights.shape
    if P != T * K:
        raise ValueError("expert_out must have num_tokens * topk rows")
    if out is None:
        out = torch.empty((T, H), dtype=expert_out.dtype, device=expert_out.device)
    with torch.cuda.device(expert_out.device):
        st = _load().pa_moe_scatter_back(_dev(out, "out"), _dev(expert_out, "expert_out"),
                                         _i32(pair_pos, "pair_pos"),
                                         _f32(topk_weights, "topk_weights"), T, K, H,
                                         _dtype_code(expert_out), _stream(expert_out))
    _check(st, "pa_moe_scatter_back")
    return out


def gather_kv(key_cache, value_cache, block_tables, seq_lens, max_len: int):
    """Test entry ``pa_gather_kv``: dense K/V [S, max_len, Hkv, D] (rows >= L are 0)."""
    nb, bs, Hkv, D = key_cache.shape
    S, mb = block_tables.shape
    kd = torch.zeros((S, max_len, Hkv, D), dtype=key_cache.dtype, device=key_cache.device)
    vd = torch.zeros_like(kd)
    with torch.cuda.device(key_cache.device):
        st = _load().pa_gather_kv(
            _dev(kd, "k_dense"), _dev(vd, "v_dense"), _dev(key_cache, "key_cache"),
            _dev(value_cache, "value_cache"), _i32(block_tables, "block_tables"),
            _i32(seq_lens, "seq_lens"), S, Hkv, D, bs, nb, mb, int(max_len),
            _dtype_code(key_cache), _stream(key_cache))
    _check(st, "pa_gather_kv")
    return kd, vd


def selftest_wait_timeout(limit_us: int = 20000, device=None) -> None:
    """Launch the failure-path test kernel (``pa_selftest_wait_timeout``)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else \
        torch.device(device)
    with torch.cuda.device(dev):
        st = _load().pa_selftest_wait_timeout(torch.cuda.current_stream(dev).cuda_stream,
                                              int(limit_us))
    _check(st, "pa_selftest_wait_timeout")


def device_status(device=None) -> int:
    """Read and clear the PA_DEV_* flags raised on ``device`` (synchronises its stream)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else \
        torch.device(device)
    flags = ctypes.c_int(0)
    with torch.cuda.device(dev):
        st = _load().pa_device_status(torch.cuda.current_stream(dev).cuda_stream,
                                      ctypes.byref(flags))
    _check(st, "pa_device_status")
    return flags.value
