"""The benchmark's multi-rank path on CPU: two gloo ranks.

Each rank processes its own shard of requests (its own seed; weak scaling,
no data-path collective).  The job's time is the slowest rank's (a MAX
all-reduce), and the job-wide rate counts every rank's steps.  The shards'
plans are computed by the oracle here, so the test needs no GPU.
"""

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from conftest import ROOT


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    from confidence_scheduled_speculative_gb300 import workloads as wl
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank plans its own shard
        step = wl.make_step(wl.QWEN, seed=bench.rank_seed(7, rank))
        r = oracle.plan_step(step)
        lens = torch.from_numpy(np.asarray(r.verify_lens, np.int64))
        gathered = [torch.zeros_like(lens) for _ in range(world)]
        dist.all_gather(gathered, lens)
        # a rank-dependent "elapsed time": the job takes the largest
        elapsed = 0.5 + rank
        t_job = bench.max_over_ranks(elapsed, torch.device("cpu"), world)
        rate = bench.job_rate(100, world, t_job)
        np.save(os.path.join(out_dir, f"rank{rank}.npy"),
                np.array([t_job, rate] + [x for g in gathered for x in g.tolist()], np.float64))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path, orc):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    res = [np.load(tmp_path / f"rank{r}.npy") for r in range(world)]
    from confidence_scheduled_speculative_gb300 import workloads as wl
    import bench
    for r in range(world):
        assert res[r][0] == 1.5                   # the slowest rank's time, on every rank
        assert res[r][1] == world * 100 / 1.5      # every rank's steps in that time
    # the shards are independent plans: each equals the oracle on its own seed
    B = wl.QWEN.B
    for q in range(world):
        ref = orc.plan_step(wl.make_step(wl.QWEN, seed=bench.rank_seed(7, q)))
        for r in range(world):
            np.testing.assert_array_equal(res[r][2 + q * B: 2 + (q + 1) * B], ref.verify_lens)
    # different seeds: the ranks hold different requests
    a, b = (wl.make_step(wl.QWEN, seed=bench.rank_seed(7, q)) for q in range(world))
    assert not np.array_equal(a.conf_logits, b.conf_logits)


def test_single_rank_helpers():
    import bench
    assert bench.max_over_ranks(3.25, None, 1) == 3.25
    assert bench.job_rate(300, 1, 0.5) == 600.0
    assert bench.rank_seed(5, 0) == 5 and bench.rank_seed(5, 3) == 8


def _tier_rank_main(rank, world, port, out_dir):
    """One data-parallel rank of the shared-tier exchange: plan and pack its
    own shard (the oracle stands in for the kernels), then the exchange of
    engine.share_tier (a gloo MAX all-reduce of totals[1]) and the pad to the
    shared tier."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    from confidence_scheduled_speculative_gb300 import workloads as wl
    from confidence_scheduled_speculative_gb300.engine import share_tier
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank 0 runs a small forced budget: its local tier is below rank 1's
        step = wl.make_step(wl.QWEN, seed=bench.rank_seed(7, rank),
                            forced_budget=40 if rank == 0 else None)
        r = oracle.plan_step(step)
        p = oracle.pack(step.anchor, step.draft, step.prefix_lens, r.verify_lens, step.tiers,
                        step.capacity)
        totals = torch.tensor([p.total, p.padded], dtype=torch.int32)
        tier = int(share_tier(totals)[0])
        q = oracle.pad_to_tier(p, tier, step.capacity)
        np.savez(os.path.join(out_dir, f"tier{rank}.npz"), local=[p.total, p.padded],
                 shared=[q.total, q.padded, q.status], ids=q.ids, pos=q.pos, req=q.req,
                 src=q.src, ids0=p.ids, req0=p.req)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_the_largest_verify_tier(tmp_path, orc):
    """[AVS] §六 / [SGL] "Ragged verify": two ranks with different packed
    totals both replay the largest local tier; the smaller rank's extra rows
    are pad rows (id 0, position 0, request -1, source -1), its real rows
    and everything past the shared tier are as its own pack left them."""
    world = 2
    mp.start_processes(_tier_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    res = [np.load(tmp_path / f"tier{r}.npz") for r in range(world)]
    import bench
    from confidence_scheduled_speculative_gb300 import workloads as wl
    # the local tiers, recomputed here from the oracle's plans
    local = []
    for q in range(world):
        step = wl.make_step(wl.QWEN, seed=bench.rank_seed(7, q),
                            forced_budget=40 if q == 0 else None)
        r = orc.plan_step(step)
        p = orc.pack(step.anchor, step.draft, step.prefix_lens, r.verify_lens, step.tiers,
                     step.capacity)
        local.append((p.total, p.padded))
    assert local[0][1] < local[1][1]  # the ranks need different tiers
    shared = max(t for _, t in local)
    for q in range(world):
        total, padded = local[q]
        assert list(res[q]["local"]) == [total, padded]
        assert list(res[q]["shared"]) == [total, shared, 0]
        for k in ("ids", "pos"):
            assert np.all(res[q][k][total:shared] == 0), (q, k)
        for k in ("req", "src"):
            assert np.all(res[q][k][total:shared] == -1), (q, k)
        np.testing.assert_array_equal(res[q]["ids"][:total], res[q]["ids0"][:total])
        np.testing.assert_array_equal(res[q]["req"][:total], res[q]["req0"][:total])
        np.testing.assert_array_equal(res[q]["req"][shared:], res[q]["req0"][shared:])


def test_share_tier_without_a_process_group_is_a_no_op():
    from confidence_scheduled_speculative_gb300.engine import share_tier
    totals = torch.tensor([37, 40], dtype=torch.int32)
    assert int(share_tier(totals)[0]) == 40 and totals.tolist() == [37, 40]
