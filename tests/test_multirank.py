"""The bench's multi-rank host logic on two gloo ranks (CPU, no GPU).

Under torchrun every rank runs an independent replica of the workload; the
ranks share only a barrier and the max of their elapsed times, and the line
reports all ranks' work over the slowest rank's time.
"""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    assert bench.dist_setup() == (world, rank, rank)
    ms = bench.barrier_max(10.0 + 5.0 * rank, world)          # rank 1 is the slower one
    dist.barrier()
    value = bench.aggregate_tflops(2.0e12, 4, world, ms)
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{ms} {value}\n")
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    got = [open(tmp_path / f"rank{r}.txt").read().split() for r in range(world)]
    for ms, value in got:
        assert float(ms) == 15.0                     # max over ranks
        # 2 TFLOP per step x 4 steps x 2 ranks / 15 ms
        assert float(value) == pytest.approx(2.0e12 * 4 * 2 / 15e-3 / 1e12)


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        workload, steps, warmup, ref_budget = "sgemm_128", 3, 3, 1.0
    assert bench.run_reference(Args(), world=2, rank=1) == 0


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.barrier_max(3.25, 1) == 3.25
    assert bench.aggregate_tflops(1e12, 10, 1, 1000.0) == pytest.approx(10.0)
