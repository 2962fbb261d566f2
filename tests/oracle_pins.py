"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes an oracle module (the real one, or a copy built
from a source with a planted mistake) and raises ``AssertionError`` when the
oracle disagrees with what the mathematics or a library routine fixes:

* exhaustive 16-bit float decoding against numpy / torch conversions;
* brute-force dense attention through ``torch.nn.functional.scaled_dot_product_attention``
  (fp64) on the dense arrays the paged cache was scattered from;
* the bit-exact gather against those dense arrays;
* closed forms (seq_len = 1 returns v_0; a zero query or equal keys return
  the mean of V; a dominant logit returns its v);
* invariants (permuting physical blocks; partitioned + log-sum-exp merge equals
  single pass for any partition size; untouched unused partition slots);
* per-partition statistics against ``torch.max`` / ``torch.logsumexp`` of
  logits from a library matmul.
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F

from workloads import make_dense_case, make_dense_prefill_case

TOL = 1e-12

SHAPES = [
    # lengths, Hq, Hkv, d, bs, dtype
    ([1, 17, 40], 6, 1, 16, 4, torch.float16),
    ([33, 7], 4, 2, 8, 1, torch.bfloat16),
    ([40, 16, 3], 12, 2, 32, 16, torch.float16),
    ([25], 2, 2, 8, 4, torch.bfloat16),
]


def _f64(x: torch.Tensor) -> torch.Tensor:
    return x.to(torch.float64)


def _sdpa_dense(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, scale: float):
    """Library attention for one sequence: q [Hq,d], k/v [L,Hkv,d] -> [Hq,d] (fp64)."""
    Hq = q.shape[0]
    Hkv = k.shape[1]
    g = Hq // Hkv
    kk = _f64(k).permute(1, 0, 2).repeat_interleave(g, dim=0)   # [Hq, L, d]
    vv = _f64(v).permute(1, 0, 2).repeat_interleave(g, dim=0)
    qq = _f64(q)[:, None, :]                                       # [Hq, 1, d]
    o = F.scaled_dot_product_attention(qq[None], kk[None], vv[None], scale=scale)
    return o[0, :, 0, :]


def _logits_dense(q, k, scale):
    """Library matmul logits [Hq, L] for one sequence (fp64)."""
    Hq, Hkv = q.shape[0], k.shape[1]
    kk = _f64(k).permute(1, 0, 2).repeat_interleave(Hq // Hkv, dim=0)  # [Hq, L, d]
    return torch.einsum("hd,hld->hl", _f64(q), kk) * scale


def _scale_f32(d):
    return float(np.float32(1.0 / math.sqrt(d)))


def pin_decoder_exhaustive(orc):
    bits = np.arange(65536, dtype=np.uint16)
    got = orc.bits_to_f64(bits, "f16")
    ref = bits.view(np.float16).astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(got[m], ref[m]), "fp16 decoder differs from numpy"
    got = orc.bits_to_f64(bits, "bf16")
    ref = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    m = ~np.isnan(ref)
    assert np.array_equal(got[m], ref[m]), "bf16 decoder differs from torch"


def pin_dense_attention(orc):
    for i, (lengths, Hq, Hkv, d, bs, dt) in enumerate(SHAPES):
        case, dk, dv = make_dense_case(lengths=lengths, num_q_heads=Hq, num_kv_heads=Hkv,
                                       head_dim=d, block_size=bs, dtype=dt, seed=100 + i)
        scale = _scale_f32(d)
        out = orc.attention(case.query, case.key_cache, case.value_cache, case.block_tables,
                            case.seq_lens, scale)
        for s, L in enumerate(lengths):
            ref = _sdpa_dense(case.query[s], dk[s], dv[s], scale).numpy()
            err = np.abs(out[s] - ref).max()
            assert err <= TOL, f"shape {i} seq {s}: |oracle - sdpa| = {err}"


def pin_gather(orc):
    for i, (lengths, Hq, Hkv, d, bs, dt) in enumerate(SHAPES):
        case, dk, dv = make_dense_case(lengths=lengths, num_q_heads=Hq, num_kv_heads=Hkv,
                                       head_dim=d, block_size=bs, dtype=dt, seed=200 + i)
        kd, vd = orc.gather(case.key_cache, case.value_cache, case.block_tables,
                            case.seq_lens)
        for s, L in enumerate(lengths):
            ek = dk[s].view(torch.int16).numpy().view(np.uint16)
            ev = dv[s].view(torch.int16).numpy().view(np.uint16)
            assert np.array_equal(kd[s, :L], ek) and np.array_equal(vd[s, :L], ev)
            assert not kd[s, L:].any() and not vd[s, L:].any()


def pin_seq_len_one(orc):
    case, dk, dv = make_dense_case(lengths=[1, 1], num_q_heads=8, num_kv_heads=2,
                                   head_dim=16, block_size=4, dtype=torch.bfloat16, seed=3)
    out = orc.attention(case.query, case.key_cache, case.value_cache, case.block_tables,
                        case.seq_lens, _scale_f32(16))
    for s in range(2):
        for h in range(8):
            assert np.array_equal(out[s, h], _f64(dv[s][0, h // 4]).numpy())


def pin_zero_query_mean(orc):
    case, dk, dv = make_dense_case(lengths=[37, 5], num_q_heads=6, num_kv_heads=3,
                                   head_dim=8, block_size=4, dtype=torch.float16, seed=4)
    case.query.zero_()
    out = orc.attention(case.query, case.key_cache, case.value_cache, case.block_tables,
                        case.seq_lens, 0.3)
    for s in range(2):
        mean = _f64(dv[s]).mean(dim=0)           # [Hkv, d]
        ref = mean.repeat_interleave(2, dim=0).numpy()
        assert np.abs(out[s] - ref).max() <= TOL


def pin_equal_keys_mean(orc):
    case, dk, dv = make_dense_case(lengths=[29], num_q_heads=4, num_kv_heads=1,
                                   head_dim=16, block_size=4, dtype=torch.bfloat16, seed=5)
    row = case.key_cache[0, 0].clone()
    case.key_cache[:] = row
    out = orc.attention(case.query, case.key_cache, case.value_cache, case.block_tables,
                        case.seq_lens, _scale_f32(16))
    ref = _f64(dv[0]).mean(dim=0).repeat_interleave(4, dim=0).numpy()
    assert np.abs(out[0] - ref).max() <= TOL


def pin_dominant_logit(orc):
    # A scale this large makes the softmax one-hot at each head's largest
    # logit; without subtracting the maximum, exp overflows.
    case, dk, dv = make_dense_case(lengths=[23, 40], num_q_heads=4, num_kv_heads=2,
                                   head_dim=16, block_size=4, dtype=torch.float16, seed=6)
    scale = 3000.0
    out = orc.attention(case.query, case.key_cache, case.value_cache, case.block_tables,
                        case.seq_lens, scale)
    for s in range(2):
        lg = _logits_dense(case.query[s], dk[s], scale)           # [Hq, L]
        top2 = torch.topk(lg, 2, dim=1).values
        assert bool(((top2[:, 0] - top2[:, 1]) > 60).all()), "fixture lost its dominant logit"
        idx = lg.argmax(dim=1)
        for h in range(4):
            ref = _f64(dv[s][idx[h], h // 2]).numpy()
            assert np.abs(out[s, h] - ref).max() <= 1e-12


def pin_block_permutation(orc):
    case, dk, dv = make_dense_case(lengths=[50, 31, 9], num_q_heads=6, num_kv_heads=2,
                                   head_dim=16, block_size=4, dtype=torch.bfloat16, seed=7)
    scale = _scale_f32(16)
    a = orc.attention(case.query, case.key_cache, case.value_cache, case.block_tables,
                      case.seq_lens, scale)
    nb = case.key_cache.shape[0]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(8))
    kc2 = torch.empty_like(case.key_cache)
    vc2 = torch.empty_like(case.value_cache)
    kc2[perm] = case.key_cache
    vc2[perm] = case.value_cache
    bt = case.block_tables.clone()
    m = bt >= 0
    bt[m] = perm[bt[m].long()].to(torch.int32)
    b = orc.attention(case.query, kc2, vc2, bt, case.seq_lens, scale)
    assert np.array_equal(a, b)


def pin_partition_merge(orc):
    for i, (lengths, Hq, Hkv, d, bs, dt) in enumerate(SHAPES):
        case, dk, dv = make_dense_case(lengths=lengths, num_q_heads=Hq, num_kv_heads=Hkv,
                                       head_dim=d, block_size=bs, dtype=dt, seed=300 + i)
        scale = _scale_f32(d)
        single = orc.attention(case.query, case.key_cache, case.value_cache,
                               case.block_tables, case.seq_lens, scale)
        for P in sorted({bs, 2 * bs, 4 * bs, 8 * bs, 16 * bs, 64}):
            tmp, es, ml = orc.partials(case.query, case.key_cache, case.value_cache,
                                       case.block_tables, case.seq_lens, scale, P)
            merged = orc.lse_merge(tmp, es, ml, case.seq_lens, P)
            err = np.abs(merged - single).max()
            assert err <= TOL, f"shape {i} P={P}: |merge - single| = {err}"


def pin_partition_statistics(orc):
    for i, (lengths, Hq, Hkv, d, bs, dt) in enumerate(SHAPES):
        case, dk, dv = make_dense_case(lengths=lengths, num_q_heads=Hq, num_kv_heads=Hkv,
                                       head_dim=d, block_size=bs, dtype=dt, seed=400 + i,
                                       k_scale=3.0)
        scale = _scale_f32(d)
        P = 2 * bs if bs > 1 else 3
        tmp, es, ml = orc.partials(case.query, case.key_cache, case.value_cache,
                                   case.block_tables, case.seq_lens, scale, P)
        NP = tmp.shape[2]
        for s, L in enumerate(lengths):
            lg = _logits_dense(case.query[s], dk[s], scale)          # [Hq, L]
            n = -(-L // P)
            for p in range(n):
                t0, t1 = p * P, min(L, p * P + P)
                seg = lg[:, t0:t1]
                assert np.abs(ml[s, :, p] - seg.max(dim=1).values.numpy()).max() <= TOL
                lse = torch.logsumexp(seg, dim=1).numpy()
                assert np.abs(ml[s, :, p] + np.log(es[s, :, p]) - lse).max() <= TOL
                assert (es[s, :, p] >= 1.0).all()
                ref = _sdpa_dense(case.query[s], dk[s][t0:t1], dv[s][t0:t1], scale).numpy()
                assert np.abs(tmp[s, :, p] - ref).max() <= TOL
            assert np.isnan(tmp[s, :, n:]).all() and np.isnan(es[s, :, n:]).all()
            assert np.isnan(ml[s, :, n:]).all()
        assert NP == max(-(-L // P) for L in lengths)


def pin_zero_length(orc):
    case, dk, dv = make_dense_case(lengths=[0, 12], num_q_heads=2, num_kv_heads=1,
                                   head_dim=8, block_size=4, dtype=torch.float16, seed=9)
    out = orc.attention(case.query, case.key_cache, case.value_cache, case.block_tables,
                        case.seq_lens, 0.5)
    assert not out[0].any()
    ref = _sdpa_dense(case.query[1], dk[1], dv[1], 0.5).numpy()
    assert np.abs(out[1] - ref).max() <= TOL
    tmp, es, ml = orc.partials(case.query, case.key_cache, case.value_cache,
                               case.block_tables, case.seq_lens, 0.5, 4)
    merged = orc.lse_merge(tmp, es, ml, case.seq_lens, 4)
    assert not merged[0].any() and np.abs(merged[1] - ref).max() <= TOL


PREFILL_SHAPES = [
    # ctx_lens, q_lens, Hq, Hkv, d, bs, dtype
    ([0, 5, 17], [3, 9, 1], 6, 2, 16, 4, torch.float16),
    ([33, 0], [7, 12], 4, 1, 8, 16, torch.bfloat16),
    ([2, 40], [1, 4], 8, 4, 32, 1, torch.float16),
]


def _prefill_mask(ctx, n, L):
    """Visible cache tokens of each chunk row: t <= ctx + i (library-side mask)."""
    t = torch.arange(L)[None, :]
    i = torch.arange(n)[:, None]
    return t <= (L - n) + i


def pin_prefill_dense_sdpa(orc):
    for k, (ctx, ql, Hq, Hkv, d, bs, dt) in enumerate(PREFILL_SHAPES):
        pc, dk, dv = make_dense_prefill_case(ctx_lens=ctx, q_lens=ql, num_q_heads=Hq,
                                             num_kv_heads=Hkv, head_dim=d, block_size=bs,
                                             dtype=dt, seed=600 + k)
        c = pc.case
        scale = _scale_f32(d)
        out = orc.prefill(pc.query, c.key_cache, c.value_cache, c.block_tables, c.seq_lens,
                          pc.q_start, scale)
        g = Hq // Hkv
        for s, (cx, n) in enumerate(zip(ctx, ql)):
            L = cx + n
            r0 = int(pc.q_start[s])
            q = _f64(pc.query[r0:r0 + n]).permute(1, 0, 2)[None]           # [1, Hq, n, d]
            kk = _f64(dk[s]).permute(1, 0, 2).repeat_interleave(g, dim=0)[None]
            vv = _f64(dv[s]).permute(1, 0, 2).repeat_interleave(g, dim=0)[None]
            ref = F.scaled_dot_product_attention(q, kk, vv, attn_mask=_prefill_mask(cx, n, L),
                                                 scale=scale)[0].permute(1, 0, 2).numpy()
            err = np.abs(out[r0:r0 + n] - ref).max()
            assert err <= TOL, f"prefill shape {k} seq {s}: |oracle - sdpa| = {err}"


def pin_prefill_no_prefix_is_causal(orc):
    pc, dk, dv = make_dense_prefill_case(ctx_lens=[0, 0], q_lens=[13, 6], num_q_heads=4,
                                         num_kv_heads=2, head_dim=16, block_size=4,
                                         dtype=torch.bfloat16, seed=700)
    c = pc.case
    scale = _scale_f32(16)
    out = orc.prefill(pc.query, c.key_cache, c.value_cache, c.block_tables, c.seq_lens,
                      pc.q_start, scale)
    for s, n in enumerate([13, 6]):
        r0 = int(pc.q_start[s])
        q = _f64(pc.query[r0:r0 + n]).permute(1, 0, 2)[None]
        kk = _f64(dk[s]).permute(1, 0, 2).repeat_interleave(2, dim=0)[None]
        vv = _f64(dv[s]).permute(1, 0, 2).repeat_interleave(2, dim=0)[None]
        ref = F.scaled_dot_product_attention(q, kk, vv, is_causal=True,
                                             scale=scale)[0].permute(1, 0, 2).numpy()
        assert np.abs(out[r0:r0 + n] - ref).max() <= TOL


def pin_prefill_zero_query_prefix_means(orc):
    pc, dk, dv = make_dense_prefill_case(ctx_lens=[11], q_lens=[6], num_q_heads=2,
                                         num_kv_heads=1, head_dim=8, block_size=4,
                                         dtype=torch.float16, seed=701)
    pc.query.zero_()
    c = pc.case
    out = orc.prefill(pc.query, c.key_cache, c.value_cache, c.block_tables, c.seq_lens,
                      pc.q_start, 0.7)
    v = _f64(dv[0])[:, 0]                                     # [L, d]
    for i in range(6):
        ref = v[:11 + i + 1].mean(dim=0).numpy()
        assert np.abs(out[i, 0] - ref).max() <= TOL and np.abs(out[i, 1] - ref).max() <= TOL


def pin_prefill_single_row_is_decode(orc):
    """A chunk of one token per sequence is the decode of the pinned single pass."""
    pc, dk, dv = make_dense_prefill_case(ctx_lens=[0, 30, 7], q_lens=[1, 1, 1], num_q_heads=6,
                                         num_kv_heads=2, head_dim=16, block_size=4,
                                         dtype=torch.bfloat16, seed=702)
    c = pc.case
    scale = _scale_f32(16)
    a = orc.prefill(pc.query, c.key_cache, c.value_cache, c.block_tables, c.seq_lens,
                    pc.q_start, scale)
    b = orc.attention(pc.query, c.key_cache, c.value_cache, c.block_tables, c.seq_lens, scale)
    assert np.abs(a - b).max() <= TOL


ALL_PINS = [
    pin_prefill_dense_sdpa,
    pin_prefill_no_prefix_is_causal,
    pin_prefill_zero_query_prefix_means,
    pin_prefill_single_row_is_decode,
    pin_decoder_exhaustive,
    pin_dense_attention,
    pin_gather,
    pin_seq_len_one,
    pin_zero_query_mean,
    pin_equal_keys_mean,
    pin_dominant_logit,
    pin_block_permutation,
    pin_partition_merge,
    pin_partition_statistics,
    pin_zero_length,
]
