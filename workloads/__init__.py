"""Seeded synthetic inputs for paged-attention decode.

This module only draws random numbers and lays them out in the paged-cache
format; it holds none of the attention arithmetic.  It is the one module that
both the oracle-side tests and the CUDA-side tests and benchmark use, so that
both sides see identical input bits.

Shapes and value distributions follow the serving workload the pages
describe (page: project_6 commit 490ff98, "Dockerfile", the
computility-run.yaml notes: up to 256 concurrent sequences; page: blame of
optimizations/prefix_prefill_patch.py, the attention notes: head_dim 128
mostly and 256 rarely, GQA, fp16 or bf16, contexts up to 100K tokens) and
the five decode workloads below.  Recipe, for every workload:

* lengths are drawn on the host with ``torch.Generator`` seeded
  ``20261200 + workload id`` (uniform integers, log-uniform rounded, or fixed);
* the physical pool holds ``ceil(1.25 * sum ceil(L/bs))`` blocks unless the
  workload fixes it; a ``randperm`` of the pool is cut into consecutive runs,
  one run per sequence, which become its block-table row; unused table
  entries are -1;
* query, key and value values are fp32 ``randn`` (key multiplied by
  ``k_scale``) cast round-to-nearest-even to the workload's 16-bit type; every
  slot of the pool is filled, including unused blocks and the unused rows of
  each sequence's last block.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import Optional, Sequence

import torch

SEED_BASE = 20261200
_CHUNK = 1 << 26  # fp32 elements drawn per randn call (bounds temporary memory)


@dataclass(frozen=True)
class Workload:
    """One decode workload: shapes, length rule, dtype and the decode mode."""

    wid: int
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: torch.dtype
    lengths: tuple            # ("fixed", L) | ("uniform", lo, hi) | ("loguniform", lo, hi)
    mode: str                 # "single" | "partitioned" | "auto"
    partition_sizes: tuple = (512,)
    single_pass_max_len: int = 8192
    k_scale: float = 1.0
    pool_blocks: Optional[int] = None   # fixed pool size; else 1.25x the need
    pool_factor: float = 1.25

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def gqa(self) -> int:
        return self.num_q_heads // self.num_kv_heads


WORKLOADS = {
    1: Workload(1, "single_1x1000_hq24_hkv4_d128_bs16_fp16", 1, 24, 4, 128, 16,
                torch.float16, ("fixed", 1000), "single", pool_blocks=128),
    2: Workload(2, "batch64_L512-8192_hq24_hkv4_d128_bs16_bf16", 64, 24, 4, 128, 16,
                torch.bfloat16, ("uniform", 512, 8192), "single"),
    3: Workload(3, "long8x100000_hq24_hkv4_d128_bs16_bf16_P512", 8, 24, 4, 128, 16,
                torch.bfloat16, ("fixed", 100000), "partitioned", (512,), k_scale=3.0),
    4: Workload(4, "mixed256_L128-65536log_hq24_hkv4_d128_bs16_bf16_auto8192_P512", 256,
                24, 4, 128, 16, torch.bfloat16, ("loguniform", 128, 65536), "auto",
                (512,), single_pass_max_len=8192),
    5: Workload(5, "long32x32768_hq16_hkv2_d256_bs32_bf16_P256_P512", 32, 16, 2, 256, 32,
                torch.bfloat16, ("fixed", 32768), "partitioned", (256, 512)),
}


# More decode workloads of the same recipe, for the benchmark only (the parity
# tests sweep these shapes at reduced sizes): the mixed serving batch with a
# Qwen-style GQA group of 16 (64 query / 4 KV heads), and with block size 8.
EXTRA_WORKLOADS = {
    6: Workload(6, "mixed256_L128-65536log_hq64_hkv4_d128_bs16_bf16_auto8192_P512", 256,
                64, 4, 128, 16, torch.bfloat16, ("loguniform", 128, 65536), "auto",
                (512,), single_pass_max_len=8192),
    7: Workload(7, "mixed256_L128-65536log_hq24_hkv4_d128_bs8_bf16_auto8192_P512", 256,
                24, 4, 128, 8, torch.bfloat16, ("loguniform", 128, 65536), "auto",
                (512,), single_pass_max_len=8192),
}


def workload(wid: int) -> "Workload":
    """A decode workload by id: the five of WORKLOADS, or one of EXTRA_WORKLOADS."""
    return WORKLOADS[wid] if wid in WORKLOADS else EXTRA_WORKLOADS[wid]


@dataclass
class Case:
    """Materialised inputs of one workload (tensors on ``device``)."""

    workload: Workload
    query: torch.Tensor          # [S, Hq, d]
    key_cache: torch.Tensor      # [num_blocks, bs, Hkv, d]
    value_cache: torch.Tensor    # [num_blocks, bs, Hkv, d]
    block_tables: torch.Tensor   # [S, max_blocks_per_seq] int32
    seq_lens: torch.Tensor       # [S] int32
    seq_lens_list: list = field(default_factory=list)

    @property
    def num_seqs(self) -> int:
        return self.query.shape[0]

    @property
    def num_blocks(self) -> int:
        return self.key_cache.shape[0]

    @property
    def max_blocks_per_seq(self) -> int:
        return self.block_tables.shape[1]

    @property
    def max_seq_len(self) -> int:
        return max(self.seq_lens_list) if self.seq_lens_list else 0

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seq_lens_list))

    @property
    def scale(self) -> float:
        return self.workload.scale

    def to(self, device) -> "Case":
        return replace(self, query=self.query.to(device), key_cache=self.key_cache.to(device),
                       value_cache=self.value_cache.to(device),
                       block_tables=self.block_tables.to(device),
                       seq_lens=self.seq_lens.to(device))


def draw_lengths(w: Workload, gen: torch.Generator, num_seqs: Optional[int] = None) -> list:
    """Sequence lengths by the workload's rule (host generator)."""
    n = w.num_seqs if num_seqs is None else num_seqs
    kind = w.lengths[0]
    if kind == "fixed":
        return [int(w.lengths[1])] * n
    lo, hi = w.lengths[1], w.lengths[2]
    if kind == "uniform":   # integers, both ends inclusive
        return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen)]
    if kind == "loguniform":  # round(exp(U[ln lo, ln hi]))
        u = torch.rand(n, generator=gen, dtype=torch.float64)
        vals = torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))
        return [int(min(hi, max(lo, round(float(x))))) for x in vals]
    raise ValueError(f"unknown length rule {kind}")


def _fill_randn(t: torch.Tensor, gen: torch.Generator, mul: float = 1.0) -> None:
    """Fill a 16-bit tensor with fp32 randn * mul, cast round-to-nearest-even."""
    flat = t.view(-1)
    for i in range(0, flat.numel(), _CHUNK):
        n = min(_CHUNK, flat.numel() - i)
        x = torch.randn(n, generator=gen, device=t.device, dtype=torch.float32)
        if mul != 1.0:
            x.mul_(mul)
        flat[i:i + n].copy_(x)


def _tables(lengths: Sequence[int], bs: int, pool_blocks: Optional[int],
            pool_factor: float, gen: torch.Generator, max_blocks: Optional[int] = None):
    need = [-(-L // bs) for L in lengths]
    total = sum(need)
    nb = pool_blocks if pool_blocks is not None else max(1, math.ceil(pool_factor * total))
    if nb < total:
        raise ValueError("pool smaller than the blocks the sequences need")
    mb = max(need + [1]) if max_blocks is None else max_blocks
    perm = torch.randperm(nb, generator=gen)
    bt = torch.full((len(lengths), mb), -1, dtype=torch.int32)
    off = 0
    for s, n in enumerate(need):
        bt[s, :n] = perm[off:off + n].to(torch.int32)
        off += n
    return bt, nb


def make_case(w, *, device="cpu", seed: Optional[int] = None,
              num_seqs: Optional[int] = None, lengths: Optional[Sequence[int]] = None,
              max_blocks_per_seq: Optional[int] = None) -> Case:
    """Build the inputs of workload ``w`` (an id or a ``Workload``).

    ``num_seqs`` / ``lengths`` override the workload's batch (reduced-size
    variants for element-wise checks); everything else follows the recipe.
    Lengths and tables come from a host generator; values from a generator
    on ``device`` seeded the same way.
    """
    if isinstance(w, int):
        w = workload(w)
    seed = SEED_BASE + w.wid if seed is None else seed
    hgen = torch.Generator().manual_seed(seed)
    overridden = num_seqs is not None or lengths is not None
    if lengths is None:
        lengths = draw_lengths(w, hgen, num_seqs)
    lengths = [int(x) for x in lengths]
    pool_blocks = None if overridden else w.pool_blocks
    bt, nb = _tables(lengths, w.block_size, pool_blocks, w.pool_factor, hgen,
                     max_blocks_per_seq)
    dev = torch.device(device)
    vgen = torch.Generator(device=dev).manual_seed(seed)
    S = len(lengths)
    q = torch.empty((S, w.num_q_heads, w.head_dim), dtype=w.dtype, device=dev)
    kc = torch.empty((nb, w.block_size, w.num_kv_heads, w.head_dim), dtype=w.dtype,
                     device=dev)
    vc = torch.empty_like(kc)
    _fill_randn(q, vgen)
    _fill_randn(kc, vgen, w.k_scale)
    _fill_randn(vc, vgen)
    return Case(w, q, kc, vc, bt.to(dev), torch.tensor(lengths, dtype=torch.int32,
                                                       device=dev), list(lengths))


def custom_workload(*, num_q_heads: int, num_kv_heads: int, head_dim: int,
                    block_size: int, dtype=torch.bfloat16, k_scale: float = 1.0,
                    name: str = "custom", wid: int = 0) -> Workload:
    """A workload shell for hand-picked shapes (tests pass ``lengths=``)."""
    return Workload(wid, name, 0, num_q_heads, num_kv_heads, head_dim, block_size, dtype,
                    ("fixed", 0), "single", k_scale=k_scale)


def make_dense_case(*, lengths: Sequence[int], num_q_heads: int, num_kv_heads: int,
                    head_dim: int, block_size: int, dtype=torch.float16, seed: int = 0,
                    pool_factor: float = 1.5, k_scale: float = 1.0):
    """Draw dense per-sequence K/V first, then scatter them into a shuffled pool.

    Returns ``(case, dense_k, dense_v)`` with ``dense_k[s]`` of shape
    ``[L_s, Hkv, d]``: the arrays the paged cache was built from, so a dense
    attention over them is an independent statement of the same result.
    """
    gen = torch.Generator().manual_seed(seed)
    w = custom_workload(num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                        head_dim=head_dim, block_size=block_size, dtype=dtype,
                        k_scale=k_scale)
    lengths = [int(x) for x in lengths]
    bt, nb = _tables(lengths, block_size, None, pool_factor, gen)
    S = len(lengths)
    q = (torch.randn((S, num_q_heads, head_dim), generator=gen)).to(dtype)
    kc = (torch.randn((nb, block_size, num_kv_heads, head_dim), generator=gen)).to(dtype)
    vc = (torch.randn((nb, block_size, num_kv_heads, head_dim), generator=gen)).to(dtype)
    dense_k, dense_v = [], []
    for s, L in enumerate(lengths):
        dk = (torch.randn((L, num_kv_heads, head_dim), generator=gen) * k_scale).to(dtype)
        dv = torch.randn((L, num_kv_heads, head_dim), generator=gen).to(dtype)
        for t in range(L):
            b = int(bt[s, t // block_size])
            kc[b, t % block_size] = dk[t]
            vc[b, t % block_size] = dv[t]
        dense_k.append(dk)
        dense_v.append(dv)
    case = Case(w, q, kc, vc, bt, torch.tensor(lengths, dtype=torch.int32), lengths)
    return case, dense_k, dense_v


@dataclass
class PrefillCase:
    """Inputs of a prefix-prefill batch: the cache holds every sequence's
    context and its new chunk; ``query`` holds the chunk rows of all sequences
    (rows q_start[s] .. q_start[s+1]-1 belong to sequence s)."""

    case: Case                  # caches, tables, seq_lens (context + chunk lengths)
    query: torch.Tensor         # [q_start[-1], Hq, d]
    q_start: torch.Tensor       # [S + 1] int32
    q_lens: list = field(default_factory=list)

    def to(self, device) -> "PrefillCase":
        return PrefillCase(self.case.to(device), self.query.to(device),
                           self.q_start.to(device), list(self.q_lens))


def make_prefill_case(w, *, ctx_lens: Sequence[int], q_lens: Sequence[int], device="cpu",
                      seed: int = 0) -> PrefillCase:
    """Prefix-prefill inputs: sequence s has ctx_lens[s] cached tokens followed by
    q_lens[s] new ones (their K/V already in the cache); query rows are drawn
    for the new tokens.  Same recipe as ``make_case`` for the cache."""
    lengths = [int(c) + int(n) for c, n in zip(ctx_lens, q_lens)]
    case = make_case(w, lengths=lengths, device=device, seed=seed)
    gen = torch.Generator(device=torch.device(device)).manual_seed(seed + 1)
    rows = int(sum(q_lens))
    q = torch.empty((rows, w.num_q_heads, w.head_dim), dtype=w.dtype, device=device)
    _fill_randn(q, gen)
    qs = [0]
    for n in q_lens:
        qs.append(qs[-1] + int(n))
    return PrefillCase(case, q, torch.tensor(qs, dtype=torch.int32, device=device),
                       [int(n) for n in q_lens])


def make_dense_prefill_case(*, ctx_lens: Sequence[int], q_lens: Sequence[int],
                            num_q_heads: int, num_kv_heads: int, head_dim: int,
                            block_size: int, dtype=torch.float16, seed: int = 0):
    """Dense-first prefill inputs: returns ``(prefill_case, dense_k, dense_v)`` with
    the per-sequence dense K/V the paged cache was scattered from."""
    lengths = [int(c) + int(n) for c, n in zip(ctx_lens, q_lens)]
    case, dk, dv = make_dense_case(lengths=lengths, num_q_heads=num_q_heads,
                                   num_kv_heads=num_kv_heads, head_dim=head_dim,
                                   block_size=block_size, dtype=dtype, seed=seed)
    gen = torch.Generator().manual_seed(seed + 1)
    rows = int(sum(q_lens))
    q = torch.randn((rows, num_q_heads, head_dim), generator=gen).to(dtype)
    qs = [0]
    for n in q_lens:
        qs.append(qs[-1] + int(n))
    pc = PrefillCase(case, q, torch.tensor(qs, dtype=torch.int32), [int(n) for n in q_lens])
    return pc, dk, dv


# ---------------------------------------------------------------------------
# MoE routing workload (synthetic router logits and hidden states)
# ---------------------------------------------------------------------------
@dataclass
class MoeCase:
    """Router logits [T, E] and hidden states [T, H] of one MoE layer input."""

    logits: torch.Tensor
    hidden: torch.Tensor
    topk: int

    @property
    def num_tokens(self) -> int:
        return self.hidden.shape[0]

    @property
    def num_experts(self) -> int:
        return self.logits.shape[1]

    def to(self, device) -> "MoeCase":
        return MoeCase(self.logits.to(device), self.hidden.to(device), self.topk)


MOE_SEED = 20261300


def make_moe_case(*, num_tokens: int = 16384, num_experts: int = 256, topk: int = 8,
                  hidden_size: int = 2048, dtype=torch.bfloat16,
                  logits_dtype=torch.bfloat16, device="cpu", seed: int = MOE_SEED) -> MoeCase:
    """Seeded MoE inputs: router logits ~ N(0, 1) and hidden states ~ N(0, 1),
    both drawn in fp32 on ``device`` and rounded to their dtypes.  The default
    shape is the pages' MoE prefill batch: 16384 tokens, 256 experts, top-8;
    hidden size 2048 (the pages do not state it)."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev).manual_seed(seed)
    logits = torch.empty((num_tokens, num_experts), dtype=logits_dtype, device=dev)
    hidden = torch.empty((num_tokens, hidden_size), dtype=dtype, device=dev)
    _fill_randn(logits, gen)
    _fill_randn(hidden, gen)
    return MoeCase(logits, hidden, topk)
