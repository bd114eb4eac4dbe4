"""The bench's multi-rank host logic on CPU (gloo, world size 2): replicas only,
so the only exchange is the max over ranks of the step time; the whole-job
throughput counts every rank's bytes over that time; each rank draws its own
synthetic batch."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from compressed_cache_decode_gb300 import inputs
        local_ms = [3.0, 7.5][rank]
        t = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
        w = inputs.WORKLOADS[next(iter(inputs.WORKLOADS))]
        case = inputs.make_decode_inputs(w, seed=rank)
        out[rank] = (t, float(case["q"].double().sum()))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_per_rank_inputs_gloo():
    world = 2
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    assert out[0][0] == 7.5 and out[1][0] == 7.5      # the job takes as long as its slowest rank
    assert out[0][1] != out[1][1]                     # rank-seeded inputs: each rank its own batch


def test_job_throughput_counts_all_ranks():
    import bench
    assert bench.job_gbs(1e9, 1, 1000.0) == pytest.approx(1.0)
    assert bench.job_gbs(1e9, 4, 1000.0) == pytest.approx(4.0)   # weak scaling: 4 replicas
    assert bench.max_over_ranks(2.5, 1, None) == 2.5
