"""The bench's multi-GPU mode runs independent replicas; its only cross-rank step is the
max-over-ranks timing reduction.  Checked here with world size 2 on the gloo backend (CPU)."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.replica_max(10.0 + rank, world, "cpu")  # rank 1 is slower
        dist.barrier()
        results[rank] = (t, bench.aggregate_gbs(1_000_000_000, world, t))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_aggregate():
    world = 2
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    results = mgr.dict()
    mp.spawn(_rank_main, args=(world, port, results), nprocs=world, join=True)
    assert results[0][0] == results[1][0] == 11.0
    # 2 replicas x 1 GB each in 11 ms
    assert results[0][1] == pytest.approx(2e9 / 11e-3 / 1e9)


def test_single_rank_passthrough():
    import bench
    assert bench.replica_max(3.5, 1, "cpu") == 3.5
    assert bench.aggregate_gbs(10**9, 1, 1.0) == pytest.approx(1000.0)


def test_reference_arm_nonzero_rank_does_nothing(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr("sys.argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    bench.main()
    assert capsys.readouterr().out == ""
