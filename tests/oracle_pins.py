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
  logits from a library matmul;
* the MoE router and regrouping: closed forms (equal logits, logits ln(e+1)),
  brute force over all k-subsets of a tiny router, torch.softmax / torch.topk,
  a hand-worked sort, numpy's stable argsort, and the identity expert (the
  scatter-back of the gathered rows with weights summing to one returns the
  hidden states).
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



# --------------------------------------------------------------------------
# MoE router (topk_softmax) and the sort-by-expert regrouping
# --------------------------------------------------------------------------

def pin_topk_equal_logits(o):
    """All logits equal: every p is 1/E, ties go to the lowest expert ids."""
    for E, k in [(256, 8), (7, 3)]:
        x = np.full((3, E), 0.25, dtype=np.float32)
        w, ids = o.topk_softmax(x, k)
        assert (ids == np.arange(k, dtype=np.int32)[None, :]).all(), ids
        assert np.abs(w - 1.0 / E).max() < TOL
        w2, _ = o.topk_softmax(x, k, renormalize=True)
        assert np.abs(w2 - 1.0 / k).max() < TOL


def pin_topk_log_integers(o):
    """logit_e = ln(e + 1): p_e = (e + 1) / (E (E + 1) / 2) in closed form, and the
    top-k are the last k experts in descending order."""
    E, k = 256, 8
    x = np.log(np.arange(1, E + 1, dtype=np.float64))[None, :].repeat(2, axis=0)
    w, ids = o.topk_softmax(x, k)
    want_ids = np.arange(E - 1, E - 1 - k, -1)
    assert (ids == want_ids[None, :]).all(), ids
    want_w = (want_ids + 1) / (E * (E + 1) / 2)
    assert np.abs(w - want_w[None, :]).max() < 1e-12
    w2, _ = o.topk_softmax(x, k, renormalize=True)
    assert np.abs(w2 - (want_ids + 1) / (want_ids + 1).sum()).max() < 1e-12


def pin_topk_brute_force(o):
    """Distinct random logits on a tiny router: the chosen set is the k-subset
    with the largest probability mass (itertools over all subsets), ordered by
    descending logit; weights from math.exp."""
    import itertools
    rng = np.random.default_rng(7)
    E, k = 7, 3
    x = rng.standard_normal((5, E)).astype(np.float32)
    w, ids = o.topk_softmax(x, k)
    for t in range(x.shape[0]):
        xs = [float(v) for v in x[t]]
        z = sum(math.exp(v) for v in xs)
        best = max(itertools.combinations(range(E), k), key=lambda c: sum(math.exp(xs[i]) for i in c))
        order = sorted(best, key=lambda i: -xs[i])
        assert list(ids[t]) == order, (ids[t], order)
        assert max(abs(w[t, j] - math.exp(xs[order[j]]) / z) for j in range(k)) < 1e-12


def pin_topk_large_logits_and_library(o):
    """Logits near 800 (exp overflows fp64 without the max shift) and a check
    against torch.softmax / torch.topk in fp64 on distinct bf16 logits."""
    x = np.array([[800.0, 799.0, 790.0, 0.0]], dtype=np.float32)
    w, ids = o.topk_softmax(x, 2)
    z = 1 + math.exp(-1) + math.exp(-10) + math.exp(-800)
    assert list(ids[0]) == [0, 1]
    assert abs(w[0, 0] - 1 / z) < 1e-12 and abs(w[0, 1] - math.exp(-1) / z) < 1e-12
    g = torch.Generator().manual_seed(11)
    xt = torch.randn((64, 256), generator=g).to(torch.bfloat16)
    xd = xt.to(torch.float64)
    distinct = torch.tensor([len(set(r.tolist())) == 256 for r in xd])
    w, ids = o.topk_softmax(xt, 8)
    p = torch.softmax(xd, dim=-1)
    tv, ti = torch.topk(p, 8, dim=-1)
    assert (torch.from_numpy(ids.astype(np.int64))[distinct] == ti[distinct]).all()
    assert np.abs(w - tv.numpy()).max() < 1e-12


def pin_moe_sort_worked_example(o):
    """ids [3, 1, 3, 0, 1] over 4 experts, worked by hand: expert 0 holds pair 3,
    expert 1 pairs 1 and 4, expert 2 none, expert 3 pairs 0 and 2."""
    sp, off, pos = o.moe_sort(np.array([3, 1, 3, 0, 1], dtype=np.int32), 4)
    assert list(sp) == [3, 1, 4, 0, 2]
    assert list(off) == [0, 1, 3, 3, 5]
    assert list(pos) == [3, 1, 4, 0, 2]


def pin_moe_sort_stable_library(o):
    """Random routing (16 tokens x 8 of 32 experts): numpy's stable argsort,
    bincount offsets, and the inverse permutation."""
    rng = np.random.default_rng(3)
    ids = np.stack([rng.choice(32, 8, replace=False) for _ in range(16)]).astype(np.int32)
    sp, off, pos = o.moe_sort(ids, 32)
    flat = ids.reshape(-1)
    assert (sp == np.argsort(flat, kind="stable")).all()
    assert (off == np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=32))])).all()
    assert (pos[sp] == np.arange(flat.size)).all()


def pin_moe_gather_and_identity_scatter(o):
    """Gather puts hidden row p // K at sorted position pos[p]; scattering the
    gathered rows back with weights that sum to one per token returns the
    hidden states (an identity expert); a hand-worked K = 2 case checks the
    weighting."""
    rng = np.random.default_rng(5)
    T, K, E, H = 6, 3, 8, 16
    ids = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    hidden = torch.randn((T, H), generator=torch.Generator().manual_seed(2)).to(torch.bfloat16)
    sp, off, pos = o.moe_sort(ids, E)
    y = o.moe_gather(hidden, sp, K)
    hb = hidden.view(torch.int16).numpy().view(np.uint16)
    for p in range(T * K):
        assert (y[pos[p]] == hb[p // K]).all()
    w = rng.random((T, K))
    w /= w.sum(axis=1, keepdims=True)
    out = o.moe_scatter(torch.from_numpy(y.view(np.int16)).view(torch.bfloat16), pos, w, K)
    assert np.abs(out - hidden.to(torch.float64).numpy()).max() < 1e-12
    # K = 2, two tokens, rows [1, 2] and [3, 4] per pair: out = w0 y0 + w1 y1
    y2 = torch.tensor([[1.0, 2.0], [3.0, 4.0], [5.0, 6.0], [7.0, 8.0]], dtype=torch.float16)
    pos2 = np.array([2, 0, 3, 1], dtype=np.int32)   # token 0 -> rows 2, 0; token 1 -> rows 3, 1
    w2 = np.array([[0.5, 0.25], [1.0, -1.0]])
    out2 = o.moe_scatter(y2, pos2, w2, 2)
    assert np.abs(out2 - np.array([[2.75, 3.5], [4.0, 4.0]])).max() < TOL


ALL_PINS = [
    pin_topk_equal_logits,
    pin_topk_log_integers,
    pin_topk_brute_force,
    pin_topk_large_logits_and_library,
    pin_moe_sort_worked_example,
    pin_moe_sort_stable_library,
    pin_moe_gather_and_identity_scatter,
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
