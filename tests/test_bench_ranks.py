"""bench.py's multi-rank bookkeeping on CPU: two gloo ranks with different
step times agree on the slowest rank's time, and the whole-job value counts
every rank's steps over that time (replicas, weak scaling)."""
import os
import tempfile

import numpy as np
import torch.multiprocessing as mp


def _rank(rank, world, port, outdir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 100.0 + 50.0 * rank                # rank 1 is slower
        slowest = bench.max_over_ranks(ms, world)
        value = bench.whole_job_gbs(47_579_136, 1000, world, slowest)
        np.save(os.path.join(outdir, f"r{rank}.npy"), np.array([slowest, value]))
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time():
    world = 2
    with tempfile.TemporaryDirectory() as d:
        port = 31000 + (os.getpid() % 2000)
        mp.start_processes(_rank, args=(world, port, d), nprocs=world, start_method="spawn")
        got = [np.load(os.path.join(d, f"r{r}.npy")) for r in range(world)]
    for slowest, value in got:
        assert slowest == 150.0
        assert abs(value - 47_579_136 * 1000 * 2 / 0.150 / 1e9) < 1e-6


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(12.5, 1) == 12.5
    assert abs(bench.whole_job_gbs(1e9, 10, 1, 1000.0) - 10.0) < 1e-12
