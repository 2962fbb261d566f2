"""MoE router and regrouping kernels against the fp64 oracle.

Integer results (router ids, sorted pair order, expert offsets, the inverse
permutation) and the gather are compared bit for bit; router weights within
1e-6 + 1e-5 |ref| (fp32 softmax); the scatter-back within the 16-bit output
tolerance.  Cases sweep the expert count (32 .. 512, 1024 for the sort), top-k
(1 .. 32), logits dtype, renormalisation, ragged token counts, tied logits,
skewed routing, out-of-range ids, and the pages' full MoE batch (16384 tokens,
256 experts, top-8, hidden 2048).
"""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_helpers import assert_out_close, to_f64
from workloads import make_moe_case

pytestmark = pytest.mark.gpu

W_ATOL, W_RTOL = 1e-6, 1e-5


@pytest.fixture(scope="module")
def pa():
    import paged_kv_decode_partitioned_gb300 as pa
    from paged_kv_decode_partitioned_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    pa.load_library()
    return pa


def _check_router(w_gpu, ids_gpu, w_ref, ids_ref, what):
    ids = ids_gpu.cpu().numpy()
    assert (ids == ids_ref).all(), f"{what}: {int((ids != ids_ref).sum())} ids differ"
    w = w_gpu.cpu().double().numpy()
    err = np.abs(w - w_ref)
    assert (err <= W_ATOL + W_RTOL * np.abs(w_ref)).all(), f"{what}: weight err {err.max():.3e}"


@pytest.mark.parametrize("E,k,ldt,renorm,T", [
    (256, 8, torch.bfloat16, False, 1000),
    (256, 8, torch.float32, True, 77),
    (128, 4, torch.float16, True, 33),
    (512, 32, torch.float32, False, 9),
    (64, 1, torch.bfloat16, False, 300),
    (32, 32, torch.float16, True, 5),
    (256, 2, torch.float32, True, 1),
])
def test_topk_softmax_matches_oracle(pa, E, k, ldt, renorm, T):
    case = make_moe_case(num_tokens=T, num_experts=E, topk=k, hidden_size=8,
                         logits_dtype=ldt, seed=4000 + E + k)
    w, ids = pa.topk_softmax(case.logits.cuda(), k, renorm)
    w_ref, ids_ref = oracle.topk_softmax(case.logits, k, renorm)
    _check_router(w, ids, w_ref, ids_ref, f"E={E} k={k}")
    assert pa.device_status() == 0


def test_topk_ties_and_extremes(pa):
    """Tied logits (all equal, pairs equal), a very large and a very negative
    logit: ids follow the lower-index rule exactly."""
    x = torch.zeros((4, 256), dtype=torch.float32)
    x[1, :] = torch.arange(256) // 2          # pairs of equal logits
    x[2, 100] = 3e4
    x[2, 7] = 3e4                              # tie at the top
    x[3, :] = -1e30
    x[3, 200] = 0.0
    x[3, 100] = -0.0                           # equal to +0: the lower id comes first
    for renorm in (False, True):
        w, ids = pa.topk_softmax(x.cuda(), 8, renorm)
        w_ref, ids_ref = oracle.topk_softmax(x.numpy(), 8, renorm)
        _check_router(w, ids, w_ref, ids_ref, f"ties renorm={renorm}")
    assert list(ids[0].cpu()) == list(range(8))
    assert list(ids[2].cpu()[:2]) == [7, 100]
    assert list(ids[3].cpu()[:2]) == [100, 200]


@pytest.mark.parametrize("ldt", [torch.bfloat16, torch.float16])
def test_topk_ties_and_extremes_16bit(pa, ldt):
    """The 16-bit router: all-equal rows, pairs of equal logits, a tie at the
    top, -0 against +0, the largest finite and most negative values, and a row
    whose top-k spans all 32 lanes' first choices."""
    big = 3.0e38 if ldt == torch.bfloat16 else 65504.0
    x = torch.zeros((6, 256), dtype=torch.float32)
    x[1, :] = torch.arange(256) // 2
    x[2, 100] = 30.0
    x[2, 7] = 30.0
    x[3, :] = -big
    x[3, 200] = 0.0
    x[3, 100] = -0.0
    x[4, :] = -5.0
    x[4, 255] = big
    x[5, :] = -(torch.arange(256) % 8).float()   # every lane's first logit is 0
    xl = x.to(ldt)
    for renorm in (False, True):
        w, ids = pa.topk_softmax(xl.cuda(), 8, renorm)
        w_ref, ids_ref = oracle.topk_softmax(xl, 8, renorm)
        _check_router(w, ids, w_ref, ids_ref, f"16-bit ties renorm={renorm}")
    assert list(ids[0].cpu()) == list(range(8))
    assert list(ids[2].cpu()[:2]) == [7, 100]
    assert list(ids[3].cpu()[:2]) == [100, 200]
    assert list(ids[5].cpu()) == [8 * i for i in range(8)]
    assert pa.device_status() == 0


def _routing(T, E, K, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.stack([torch.randperm(E, generator=g)[:K] for _ in range(T)]).to(torch.int32)


@pytest.mark.parametrize("T,E,K", [(1, 256, 8), (300, 256, 8), (5000, 32, 4), (100, 1024, 16),
                                   (2049, 2, 1), (0, 16, 2)])
def test_moe_sort_is_bit_exact(pa, T, E, K):
    ids = _routing(T, E, K, 4100 + T) if T else torch.zeros((0, K), dtype=torch.int32)
    sp, off, pos = pa.moe_sort(ids.cuda(), E)
    rsp, roff, rpos = oracle.moe_sort(ids, E)
    assert (sp.cpu().numpy() == rsp).all()
    assert (off.cpu().numpy() == roff).all()
    assert (pos.cpu().numpy() == rpos).all()
    assert pa.device_status() == 0


def test_moe_sort_large(pa):
    """3.2 M pairs (1563 chunks of 2048, more than the GPU holds at once): the
    sort stays bit-exact against the oracle."""
    g = torch.Generator().manual_seed(4150)
    ids = torch.randint(0, 64, (400000 * 8,), generator=g, dtype=torch.int32)
    sp, off, pos = pa.moe_sort(ids.cuda(), 64)
    rsp, roff, rpos = oracle.moe_sort(ids, 64)
    assert (sp.cpu().numpy() == rsp).all() and (off.cpu().numpy() == roff).all()
    assert (pos.cpu().numpy() == rpos).all()
    assert pa.device_status() == 0


def test_moe_sort_skewed_routing(pa):
    """Every pair on one expert, then on two alternating experts: the sort keeps
    the flat order (stability) across chunks of the kernel."""
    for ids in (torch.full((10000,), 5, dtype=torch.int32),
                (torch.arange(9000, dtype=torch.int32) % 2) * 255):
        sp, off, pos = pa.moe_sort(ids.cuda(), 256)
        rsp, roff, rpos = oracle.moe_sort(ids, 256)
        assert (sp.cpu().numpy() == rsp).all() and (off.cpu().numpy() == roff).all()
        assert (pos.cpu().numpy() == rpos).all()


def test_moe_sort_out_of_range_ids_flagged_and_skipped(pa):
    ids = _routing(500, 64, 4, 4200).reshape(-1)
    bad = torch.tensor([3, 999, 1500], dtype=torch.long)
    ids[bad[0]] = -1
    ids[bad[1]] = 64
    ids[bad[2]] = 1 << 30
    sp, off, pos = pa.moe_sort(ids.cuda(), 64)
    assert pa.device_status() & pa.DEV_BAD_EXPERT
    pos = pos.cpu().numpy()
    assert (pos[bad.numpy()] == -1).all()
    keep = np.ones(ids.numel(), dtype=bool)
    keep[bad.numpy()] = False
    valid = np.nonzero(keep)[0]
    rsp, roff, _ = oracle.moe_sort(ids[keep], 64)      # the valid pairs, renumbered
    assert (sp.cpu().numpy()[:valid.size] == valid[rsp]).all()
    assert (off.cpu().numpy() == roff).all()


@pytest.mark.parametrize("H,dt", [(2048, torch.bfloat16), (136, torch.float16), (8, torch.bfloat16)])
def test_moe_gather_bit_exact_and_scatter_matches_oracle(pa, H, dt):
    T, E, K = 333, 64, 6
    case = make_moe_case(num_tokens=T, num_experts=E, topk=K, hidden_size=H, dtype=dt,
                         seed=4300 + H)
    dev = case.to("cuda")
    w, ids = pa.topk_softmax(dev.logits, K, True)
    sp, off, pos = pa.moe_sort(ids, E)
    y = pa.moe_gather(dev.hidden, pos, K)
    # the reference chain runs on the oracle alone
    w_ref, ids_ref = oracle.topk_softmax(case.logits, K, True)
    rsp, roff, rpos = oracle.moe_sort(ids_ref, E)
    y_ref = oracle.moe_gather(case.hidden, rsp, K)
    assert (y.cpu().view(torch.int16).numpy().view(np.uint16) == y_ref).all()
    # scatter-back of independent per-pair rows with the router's weights
    yy = torch.randn((T * K, H), generator=torch.Generator().manual_seed(9)).to(dt)
    out = pa.moe_scatter_back(yy.cuda(), pos, w)
    ref = oracle.moe_scatter(yy, rpos, w_ref, K)
    assert_out_close(out, ref, f"scatter-back H={H}")
    assert pa.device_status() == 0


def test_identity_expert_round_trip(pa):
    """router (renormalised) -> sort -> gather -> scatter-back of the gathered rows
    returns the hidden states (the weights of a token sum to one)."""
    case = make_moe_case(num_tokens=4096, num_experts=256, topk=8, hidden_size=512, seed=4400)
    dev = case.to("cuda")
    w, ids = pa.topk_softmax(dev.logits, 8, True)
    sp, off, pos = pa.moe_sort(ids, 256)
    out = pa.moe_scatter_back(pa.moe_gather(dev.hidden, pos, 8), pos, w)
    h = to_f64(case.hidden)
    err = np.abs(to_f64(out) - h)
    assert (err <= 2 ** -7 * np.abs(h) + 1e-30).all(), err.max()   # at most 1 bf16 ulp


def test_full_moe_batch(pa):
    """The pages' batch: 16384 tokens x top-8 of 256 experts, hidden 2048 (bf16)."""
    case = make_moe_case(seed=4500)
    dev = case.to("cuda")
    w, ids = pa.topk_softmax(dev.logits, 8, True)
    w_ref, ids_ref = oracle.topk_softmax(case.logits, 8, True)
    _check_router(w, ids, w_ref, ids_ref, "full batch router")
    sp, off, pos = pa.moe_sort(ids, 256)
    rsp, roff, rpos = oracle.moe_sort(ids_ref, 256)
    assert (sp.cpu().numpy() == rsp).all() and (off.cpu().numpy() == roff).all()
    assert (pos.cpu().numpy() == rpos).all()
    y = pa.moe_gather(dev.hidden, pos, 8)
    rows = torch.randint(0, y.shape[0], (512,), generator=torch.Generator().manual_seed(1))
    y_ref = oracle.moe_gather(case.hidden, rsp[rows.numpy()], 8)
    assert (y[rows.cuda()].cpu().view(torch.int16).numpy().view(np.uint16) == y_ref).all()
    out = pa.moe_scatter_back(y, pos, w)
    # oracle chain for sampled tokens: their pairs' rows of the oracle's gather,
    # scattered with the oracle's weights
    toks = torch.randint(0, 16384, (256,), generator=torch.Generator().manual_seed(2)).numpy()
    pairs = (toks[:, None] * 8 + np.arange(8)[None, :]).reshape(-1)
    yr = oracle.moe_gather(case.hidden, pairs.astype(np.int32), 8)   # row of pair p = hidden[p // 8]
    ref = oracle.moe_scatter(torch.from_numpy(yr.view(np.int16)).view(torch.bfloat16),
                             np.arange(pairs.size, dtype=np.int32), w_ref[toks], 8)
    assert_out_close(out[torch.from_numpy(toks).cuda()], ref, "full batch scatter-back")
    assert pa.device_status() == 0


def test_moe_gather_skips_pairs_that_were_not_placed(pa):
    """Pairs at -1 (an out-of-range expert id in the sort) write nothing; the
    other rows are still the oracle's."""
    T, E, K, H = 64, 16, 4, 64
    ids = _routing(T, E, K, 4600).reshape(-1)
    ids[5] = E            # out of range: not placed
    hidden = torch.randn((T, H), generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    sp, off, pos = pa.moe_sort(ids.cuda(), E)
    assert pa.device_status() & pa.DEV_BAD_EXPERT
    y = torch.full((T * K, H), 7.0, dtype=torch.bfloat16, device="cuda")
    pa.moe_gather(hidden.cuda(), pos, K, out=y)
    placed = int(off[-1])
    keep = np.ones(T * K, dtype=bool)
    keep[5] = False
    valid = np.nonzero(keep)[0]
    rsp, _, _ = oracle.moe_sort(ids[keep], E)
    y_ref = oracle.moe_gather(hidden, valid[rsp].astype(np.int32), K)
    assert (y[:placed].cpu().view(torch.int16).numpy().view(np.uint16) == y_ref).all()
    assert bool((y[placed:] == 7.0).all())


def test_moe_chain_replays_in_a_cuda_graph(pa):
    """The whole chain (router, sort, gather, scatter-back) captured once into a
    CUDA graph and replayed on new inputs gives bit for bit what direct calls give
    (the bench times the step this way)."""
    T, E, K, H = 2048, 256, 8, 512
    a = make_moe_case(num_tokens=T, num_experts=E, topk=K, hidden_size=H, seed=4700).to("cuda")
    b = make_moe_case(num_tokens=T, num_experts=E, topk=K, hidden_size=H, seed=4701).to("cuda")
    logits, hidden = a.logits.clone(), a.hidden.clone()
    w = torch.empty((T, K), dtype=torch.float32, device="cuda")
    ids = torch.empty((T, K), dtype=torch.int32, device="cuda")
    ws = torch.empty(pa.moe_sort_workspace_bytes(T * K, E), dtype=torch.uint8, device="cuda")
    sp = torch.empty(T * K, dtype=torch.int32, device="cuda")
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    pos = torch.empty(T * K, dtype=torch.int32, device="cuda")
    y = torch.empty((T * K, H), dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(hidden)

    def chain():
        pa.topk_softmax(logits, K, True, weights=w, ids=ids)
        pa.moe_sort(ids, E, workspace=ws, out=(sp, off, pos))
        pa.moe_gather(hidden, pos, K, out=y)
        pa.moe_scatter_back(y, pos, w, out=out)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        chain()
    torch.cuda.current_stream().wait_stream(side)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chain()
    for case in (b, a):   # replay on new inputs, then on the first ones again
        logits.copy_(case.logits)
        hidden.copy_(case.hidden)
        g.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (w, ids, sp, off, pos, out)]
        chain()
        torch.cuda.synchronize()
        for x, r in zip(got, (w, ids, sp, off, pos, out)):
            assert torch.equal(x, r)
    assert pa.device_status() == 0
