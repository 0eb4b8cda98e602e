"""The bench's multi-rank host logic on CPU: two gloo ranks reduce their step times to the
slowest rank's, and the job's throughput counts every rank's work (weak scaling).  One GPU
per rank runs an independent replica of the whole path; these ranks exchange only the
timings."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port),
                       "RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r: kernel leg 10 + r ms, end-to-end leg 20 - r ms
        ms, e2e = bench.job_times([10.0 + rank, 20.0 - rank], dist)
        dist.barrier()
    finally:
        dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{ms} {e2e}")


def test_two_gloo_ranks_take_the_slowest(tmp_path):
    port = _free_port()
    mp.start_processes(_rank, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for rank in (0, 1):
        ms, e2e = (float(v) for v in (tmp_path / f"rank{rank}.txt").read_text().split())
        assert (ms, e2e) == (11.0, 20.0)


def test_single_rank_and_job_value():
    assert bench.job_times([3.5, 7.0]) == [3.5, 7.0]
    # two ranks of 1 TFLOP each per step in 2 ms: 1 PFLOP/s for the job
    assert bench.job_value(2, 1e12, 2.0) == pytest.approx(1000.0)
    assert bench.job_value(1, 1e12, 2.0) == pytest.approx(500.0)
