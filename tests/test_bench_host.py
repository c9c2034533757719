"""The benchmark's byte counts, on which every GB/s and roofline fraction rests, checked
against counts made by hand for small configurations; and the host-CPU record."""
import os

import bench
import workloads


def test_kv_bytes_by_hand():
    # bf16: K and V rows of 128 two-byte values per (token, KV head)
    assert workloads.kv_bytes([17, 64, 200], 2, "bf16") == (17 + 64 + 200) * 2 * (2 * 128 * 2)
    # E4M3: K and V rows of 128 bytes plus one fp32 scale each
    assert workloads.kv_bytes([17, 64, 200], 2, "fp8") == (17 + 64 + 200) * 2 * (128 + 128 + 4 + 4)
    # a negative length counts as no tokens (the kernels skip it and set a status bit)
    assert workloads.kv_bytes([5, -3], 1, "bf16") == 5 * 512
    # the bench reads the lengths of a workload dict
    inp = workloads.make_workload("tiny", device="cpu")
    assert bench.kv_bytes(inp) == (17 + 64 + 200 + 1500) * 1 * 512


def test_prologue_bytes_by_hand():
    # one token, 2 Q heads and 1 KV head (4 rows), rotary_dim 128
    rows = 2 + 2 * 1
    read = rows * 128 * 2 + 4 + 4 + 128 * 4  # qkv rows, position, slot, the cos/sin row
    assert bench.prologue_bytes(1, 2, 1, False) == read + rows * 128 * 2
    # E4M3: one-byte codes and one fp32 scale per row written
    assert bench.prologue_bytes(1, 2, 1, True) == read + rows * 128 + rows * 4
    # linear in the token count; the rotary dim only changes the table row read
    assert bench.prologue_bytes(7, 64, 8, True) == 7 * bench.prologue_bytes(1, 64, 8, True)
    assert bench.prologue_bytes(1, 2, 1, False, rot=64) == bench.prologue_bytes(1, 2, 1, False) - 64 * 4


def test_host_cpu_record():
    rec = bench.host_cpu()
    assert rec["hardware_concurrency"] == os.cpu_count()
    assert isinstance(rec["cpu_arch"], str) and rec["cpu_arch"]
    assert "cpu_model" in rec
