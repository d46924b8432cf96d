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
