"""Multi-rank logic of bench.py on the CPU: two gloo ranks (world size 2).

Every rank times its own batch (weak scaling, no collective on the data path); the job's
step time is the maximum over the ranks, the throughput counts the units of all ranks,
the batches of the ranks differ only in their seeds, and the reference arm runs on
rank 0 alone.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        import bench
        assert bench.dist_env() == (rank, world, rank)
        # the slowest rank sets the job's time
        ms = bench.max_over_ranks(10.0 + 3.0 * rank, world, "cpu")
        assert ms == 10.0 + 3.0 * (world - 1)
        # weak scaling: all ranks' queries over that time
        assert bench.weak_value(64, world, 10, ms) == pytest.approx(64 * world * 10 / (ms / 1e3))
        # each rank gets a batch of the same shape under its own seed
        wl = bench.make_workload("tiny", rank)
        shapes = [None] * world
        dist.all_gather_object(shapes, (wl.seed, wl.B, wl.Q, list(map(int, wl.q_pos))))
        seeds = {s[0] for s in shapes}
        assert len(seeds) == world
        assert all(s[1:] == shapes[0][1:] for s in shapes)
        # the reference arm: rank 0 only; the other ranks return without work
        if rank != 0:
            class Args:
                config, steps, warmup = "tiny", 1, 0
            assert bench.run_reference(Args()) is None
        with open(os.path.join(out_dir, f"rank{rank}.ok"), "w") as f:
            f.write("ok")
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    assert sorted(os.listdir(tmp_path)) == ["rank0.ok", "rank1.ok"]
