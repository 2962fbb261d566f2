"""Shared helpers of the GPU parity tests (comparison bounds, host sub-cases)."""
from __future__ import annotations

import numpy as np
import torch

# Output tolerance for bf16/fp16 results: |gpu - ref| <= ATOL + RTOL * |ref|.
ATOL = 1e-2
RTOL = 1e-2
# fp32 partial statistics: relative 1e-4 (max_logits against max(|ref|, 1)).
STAT_RTOL = 1e-4


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().double().numpy()


def assert_out_close(gpu: torch.Tensor, ref: np.ndarray, what: str) -> dict:
    g = to_f64(gpu)
    assert g.shape == ref.shape, f"{what}: shape {g.shape} vs {ref.shape}"
    err = np.abs(g - ref)
    bad = err > ATOL + RTOL * np.abs(ref)
    info = {"max_abs": float(err.max()) if err.size else 0.0,
            "max_rel_norm": float(err.max() / max(np.abs(ref).max(), 1e-30)) if err.size else 0.0}
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {bad.size} elements outside "
                           f"{ATOL}+{RTOL}|ref|; max abs err {info['max_abs']:.3e}")
    assert np.isfinite(g).all(), f"{what}: non-finite output"
    return info


def assert_stats_close(es_gpu, ml_gpu, es_ref, ml_ref, what: str) -> None:
    """Compare exp_sums / max_logits on the slots the oracle wrote (non-NaN)."""
    es_g, ml_g = to_f64(es_gpu), to_f64(ml_gpu)
    m = ~np.isnan(es_ref)
    assert m.any()
    e_err = np.abs(es_g[m] - es_ref[m]) / es_ref[m]
    assert e_err.max() <= STAT_RTOL, f"{what}: exp_sums rel err {e_err.max():.3e}"
    l_err = np.abs(ml_g[m] - ml_ref[m]) / np.maximum(np.abs(ml_ref[m]), 1.0)
    assert l_err.max() <= STAT_RTOL, f"{what}: max_logits rel err {l_err.max():.3e}"


def assert_partials_close(tmp_gpu, tmp_ref, what: str) -> None:
    g = to_f64(tmp_gpu)
    m = ~np.isnan(tmp_ref)
    err = np.abs(g[m] - tmp_ref[m])
    bad = err > ATOL + RTOL * np.abs(tmp_ref[m])
    assert not bad.any(), f"{what}: tmp_out max abs err {err.max():.3e}"


def host_subcase(case, seq_ids):
    """Host copies of a few sequences of a device-resident case.

    The referenced physical blocks are copied into a compact host pool and
    the block-table rows are relabelled to it (the attention result does not
    depend on which physical block holds a page: the oracle's
    block-permutation pin).  Returns (query, key_cache, value_cache,
    block_tables, seq_lens) on the host.
    """
    ids = torch.as_tensor(seq_ids, dtype=torch.long)
    bs = case.key_cache.shape[1]
    lens = [case.seq_lens_list[i] for i in seq_ids]
    bt = case.block_tables.cpu()[ids]
    need = [-(-L // bs) for L in lens]
    used = torch.cat([bt[j, :n] for j, n in enumerate(need)] + [torch.zeros(0, dtype=torch.int32)])
    uniq, inv = torch.unique(used.long(), return_inverse=True)
    dev_idx = uniq.to(case.key_cache.device)
    kc = case.key_cache.index_select(0, dev_idx).cpu()
    vc = case.value_cache.index_select(0, dev_idx).cpu()
    nbt = torch.full((len(seq_ids), max(need + [1])), -1, dtype=torch.int32)
    off = 0
    for j, n in enumerate(need):
        nbt[j, :n] = inv[off:off + n].to(torch.int32)
        off += n
    q = case.query.index_select(0, ids.to(case.query.device)).cpu()
    return q, kc, vc, nbt, torch.tensor(lens, dtype=torch.int32)
