"""The benchmark's multi-process logic on CPU (gloo, two ranks): each rank times its own
replica, the job takes the slowest rank's time, and the whole-job throughput counts every
rank's bytes. No GPU: the replicas' kernels are not involved."""
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r measured (1 + r) ms per step and 10 - r ms end to end
        ms, ms_e2e = bench.max_over_ranks([1.0 + rank, 10.0 - rank], dist, "cpu")
        out[rank] = (ms, ms_e2e)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    # every rank sees the slowest rank's times
    assert res[0] == res[1] == (2.0, 10.0)
    # 7.29 GB per replica in the slowest rank's 2 ms, two replicas
    assert bench.job_throughput(7.29e9, 2.0, world) == pytest.approx(2 * 7.29e9 / 2e-3 / 1e9)
    assert bench.job_throughput(7.29e9, 2.0, 1) == pytest.approx(3645.0)


def test_oracle_sample_runs_one_child_per_core():
    # two single-threaded children, one pass each, started together: the job's bytes are
    # both children's, over the slower child's time
    r = bench.run_oracle_sample(passes=1, cores=2)
    assert r["cores"] == 2 and r["kind"] == "oracle" and r["unit"] == bench.UNIT
    assert "2 single-threaded processes" in r["sample"] and "2 passes" in r["sample"]
    assert r["value"] == pytest.approx(2 * 2.80e6 / r["seconds_per_pass"] / 1e9, rel=0.01)
