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


def test_reference_step_samples_stay_within_small_budgets():
    """The reference arm sizes each step's oracle sample to its share of a fixed total: with a
    budget no request fits, a step takes the shortest request alone; a larger budget takes
    more requests, never one whose estimated time would overrun it."""
    import bench
    import workloads
    inp = workloads.make_workload("tiny", device="cpu")
    per_token = bench.oracle_seconds_per_token(inp, 2)
    v, cores, desc = bench.cpu_oracle_rate(inp, 1e-9, rng_seed=0, threads=2, per_token=per_token, fit=True)
    assert v > 0 and cores == 2
    assert desc.startswith("1 of 4 requests (17 of ")  # the shortest length is 17
    lens = inp["seq_lens"].numpy()
    eff = min(2, inp["num_kv_heads"] * len(lens))
    budget = per_token * (17 + 200) * inp["num_kv_heads"] / eff  # room for the two shortest
    _, _, desc = bench.cpu_oracle_rate(inp, budget * 1.0001, rng_seed=3, threads=2, per_token=per_token, fit=True)
    n = int(desc.split(" ")[0])
    tokens = int(desc.split("(")[1].split(" ")[0])
    assert 1 <= n <= 2 and tokens <= 17 + 200
