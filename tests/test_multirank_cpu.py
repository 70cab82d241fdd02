"""The benchmark's multi-rank path on CPU: two processes in a gloo group, as
`bench.py --gpus 2` runs two replicas (one per GPU, weak scaling, no collective
on the data path).  The step time every rank reports is the slowest rank's,
and the job's throughput counts the tokens of every replica."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    from selective_state_space_ssd_gb300.configs import CONFIGS

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        own_ms = 100.0 + 7.0 * rank  # this replica's time for its steps
        slowest = bench.max_over_ranks(own_ms, world, "cpu")
        value = bench.job_tokens_per_s(CONFIGS["mamba2_2p7b_bf16"], world, 20, slowest)
        dist.barrier()
    finally:
        dist.destroy_process_group()
    with open(os.path.join(out_dir, f"rank{rank}.txt"), "w") as f:
        f.write(f"{slowest} {value}\n")


def test_two_ranks_report_the_slowest_replica(tmp_path):
    world = 2
    mp.start_processes(_rank, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True,
                       start_method="spawn")
    got = [tuple(map(float, open(tmp_path / f"rank{r}.txt").read().split())) for r in range(world)]
    tokens = 4 * 4096
    for slowest, value in got:
        assert slowest == 107.0
        assert value == pytest.approx(world * tokens * 20 / 0.107)


def test_one_rank_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5
