"""The bench's multi-rank host logic on CPU: two gloo ranks stand in for two GPUs. Each rank
is an independent replica (weak scaling): the step time is the slowest rank's, throughput is
the sum over ranks, and the reference arm runs on rank 0 alone."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took (r + 1) ms per step; every rank must see the slowest
        out[rank] = bench.max_over_ranks(float(rank + 1), dist, "cpu")
        dist.barrier()
        # the reference arm: rank 0 runs the oracle sample, the others return without work
        args = type("A", (), {"steps": 1, "warmup": 1})()
        from synthetic import gen
        res = bench.run_reference(args, gen.TINY_FP32, "tiny-fp32-b1-t512")
        out[world + rank] = None if res is None else res["impl"]
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step_and_only_rank0_reports():
    import torch.multiprocessing as mp
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        assert out[0] == out[1] == 2.0
        assert out[world + 0] == "reference" and out[world + 1] is None


def test_job_throughput_is_weak_scaling_sum():
    import bench
    one = bench.job_throughput_gbs(1, 35_651_584, 0.040)
    assert one == pytest.approx(35_651_584 / 1e9 / 40e-6)
    assert bench.job_throughput_gbs(4, 35_651_584, 0.040) == pytest.approx(4 * one)
    assert bench.max_over_ranks(3.5) == 3.5
