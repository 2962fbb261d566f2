"""The benchmark's multi-rank path on CPU: two gloo ranks.

With N GPUs every rank decodes its own batch (replicas; the decode has no
collective). Only the slowest rank's time and the byte / sequence totals
cross ranks; these tests run that host logic with world_size 2 on gloo.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # rank r took (10 + 5r) ms for its K steps over (100 + r) MB and (3 + r) sequences
        (t,), (b, n) = bench.across_ranks(world, "cpu", [10.0 + 5 * rank],
                                          [100e6 + 1e6 * rank, 3 + rank])
        assert t == 15.0, t                                  # the slowest rank's time
        assert b == 201e6 and n == 7, (b, n)                 # totals over both ranks
        ms, gbs, tok = bench.whole_job(t, 5, b, n)
        assert abs(ms - 3.0) < 1e-12
        assert abs(gbs - 201e6 / 3e-3 / 1e9) < 1e-9
        assert abs(tok - 7 / 3e-3) < 1e-9
        # every rank draws its own batch; rank 0 keeps the workload's seed
        from workloads import SEED_BASE
        assert bench.rank_seed(4, 0) == SEED_BASE + 4
        seeds = [None, None]
        dist.all_gather_object(seeds, bench.rank_seed(4, rank))
        assert seeds[0] != seeds[1]
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_time_and_bytes():
    mp.spawn(_rank_main, args=(2, _free_port()), nprocs=2, join=True)


def test_single_rank_needs_no_process_group():
    import bench
    assert not dist.is_initialized()
    (t,), (b,) = bench.across_ranks(1, "cpu", [4.0], [8.0])
    assert (t, b) == (4.0, 8.0)


def test_replica_batches_are_independent_draws():
    import bench
    from workloads import WORKLOADS, make_case
    a = make_case(WORKLOADS[2], seed=bench.rank_seed(2, 0), num_seqs=4)
    b = make_case(WORKLOADS[2], seed=bench.rank_seed(2, 1), num_seqs=4)
    assert a.seq_lens_list != b.seq_lens_list or not torch.equal(a.query, b.query)
