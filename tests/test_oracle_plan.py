"""Pins for the oracle's task map (the assign step) and the static split rule.

The task map is a scheduling heuristic: the oracle walks it tile by tile as the
HPC-Ops × SGLang blog states it (section "围绕活跃 KV 工作进行调度").  These tests
pin that walk to things other than itself: hand-worked examples, invariants the
rule implies (every tile covered once, bins within one tile of the real-valued
budget, the minimum-work floor), closed forms for special cases, and brute force
over all tiny inputs.
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "plan_worked_examples.json")
TILE = 64


def check_invariants(lens, hkv, C, m, tm):
    lens = np.asarray(lens, np.int64)
    n = np.repeat((np.maximum(lens, 0) + TILE - 1) // TILE, hkv)  # tiles per unit, u = b*hkv + h
    U = n.shape[0]
    T = int(n.sum())
    T_, C_eff, nd, status = (int(x) for x in tm["meta"])
    assert T_ == T
    assert status == (1 if (lens < 0).any() else 0)
    if T == 0:
        assert C_eff == 0 and nd == 0
        assert (tm["cta_desc_begin"] == 0).all()
        return
    assert C_eff == min(C, max(1, T // m))
    descs = tm["descs"]
    assert descs.shape == (nd, 4)
    assert nd <= U + C - 1
    begin = tm["cta_desc_begin"]
    assert begin[0] == 0 and begin[C] == nd
    assert (np.diff(begin) >= 0).all()
    # global tile positions of each descriptor
    P = np.concatenate([[0], np.cumsum(n)])
    g0 = P[descs[:, 0]] + descs[:, 1]
    g1 = P[descs[:, 0]] + descs[:, 2]
    assert (descs[:, 1] < descs[:, 2]).all()
    assert (descs[:, 2] <= n[descs[:, 0]]).all()
    # exact cover, in global tile order
    assert g0[0] == 0 and g1[-1] == T
    assert (g0[1:] == g1[:-1]).all()
    # bins: sizes within one tile of the budget T/C_eff; only the first C_eff are used
    sizes = []
    for i in range(C):
        a, b = begin[i], begin[i + 1]
        if i >= C_eff:
            assert a == b
            continue
        assert b > a
        lo, hi = g0[a], g1[b - 1]
        sizes.append(hi - lo)
        # bin boundaries are the cumulative floors of the budget
        assert lo == (i * T) // C_eff and hi == ((i + 1) * T) // C_eff
        # each descriptor of the bin belongs to a different unit, in order
        assert (np.diff(descs[a:b, 0]) > 0).all()
    sizes = np.array(sizes)
    assert sizes.sum() == T
    assert sizes.min() >= T // C_eff and sizes.max() <= -(-T // C_eff)
    if T >= m:
        assert sizes.min() >= m
    # per-unit partial bookkeeping
    upb, unp = tm["unit_partial_begin"], tm["unit_num_partials"]
    seen = 0
    for u in range(U):
        assert upb[u] == seen
        assert unp[u] == (0 if n[u] == 0 else int((descs[:, 0] == u).sum()))
        for k in range(unp[u]):
            assert descs[seen + k, 0] == u and descs[seen + k, 3] == k
        seen += unp[u]
    assert seen == nd


def golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


@pytest.mark.parametrize("case", golden_cases(), ids=lambda c: c["name"])
def test_hand_worked_examples(case):
    tm = oracle.plan(case["seq_lens"], case["num_kv_heads"], case["num_ctas"], TILE,
                     case["min_tiles_per_split"])
    assert tm["meta"].tolist() == case["meta"]
    assert tm["cta_desc_begin"].tolist() == case["cta_desc_begin"]
    assert tm["descs"].tolist() == case["descs"]
    assert tm["unit_partial_begin"].tolist() == case["unit_partial_begin"]
    assert tm["unit_num_partials"].tolist() == case["unit_num_partials"]
    check_invariants(case["seq_lens"], case["num_kv_heads"], case["num_ctas"],
                     case["min_tiles_per_split"], tm)


def test_16k_request_carries_16x_the_tiles_of_1k():
    # "Attention：变长 decode 的负载均衡": a 16K-token request has about 16x the KV work of a 1K one
    tm = oracle.plan([16384], 1, 1, TILE, 1)
    tm1 = oracle.plan([1024], 1, 1, TILE, 1)
    assert tm["meta"][0] == 16 * tm1["meta"][0]


def test_exhaustive_tiny():
    # every length vector over a small alphabet, several CTA counts and floors
    alphabet = [0, 1, 63, 64, 65, 200]
    for B in (1, 2, 3):
        for lens in itertools.product(alphabet, repeat=B):
            for hkv in (1, 2):
                for C in (1, 2, 3, 5, 8):
                    for m in (1, 2, 4):
                        check_invariants(lens, hkv, C, m, oracle.plan(list(lens), hkv, C, TILE, m))


def test_random_invariants():
    rng = np.random.default_rng(1234)
    for _ in range(300):
        B = int(rng.integers(1, 40))
        lens = np.exp(rng.uniform(0, np.log(40000), B)).astype(np.int64)
        lens[rng.random(B) < 0.1] = 0
        hkv = int(rng.choice([1, 2, 4, 8]))
        C = int(rng.integers(1, 200))
        m = int(rng.integers(1, 17))
        check_invariants(lens, hkv, C, m, oracle.plan(lens, hkv, C, TILE, m))


def test_small_total_uses_floor():
    # T <= C*m gives C_eff = floor(T/m) bins, each of at least m tiles
    tm = oracle.plan([64 * 10], 1, 16, TILE, 4)
    assert tm["meta"][1] == 2
    assert tm["descs"].tolist() == [[0, 0, 5, 0], [0, 5, 10, 1]]


def test_single_request_equal_slices():
    # one request, T divisible by C: equal slices, one descriptor per bin
    tm = oracle.plan([131072], 1, 16, TILE, 4)
    assert tm["meta"].tolist() == [2048, 16, 16, 0]
    assert tm["descs"][:, 2].tolist() == [128 * (i + 1) for i in range(16)]
    assert (tm["descs"][:, 2] - tm["descs"][:, 1] == 128).all()


def test_uniform_lengths_no_fragments():
    # uniform lengths where every bin holds whole units: no unit is split
    tm = oracle.plan([512] * 64, 1, 16, TILE, 4)  # 64 units x 8 tiles, 4 units per bin
    assert tm["meta"].tolist() == [512, 16, 64, 0]
    assert (tm["unit_num_partials"] == 1).all()
    assert tm["cta_desc_begin"].tolist() == list(range(0, 65, 4))


def test_long_request_spans_bins_in_proportion():
    # a long sequence spans CTAs in proportion to its length
    lens = [65536] + [1024] * 127
    tm = oracle.plan(lens, 8, 152, TILE, 4)
    T, C_eff = tm["meta"][0], tm["meta"][1]
    share = 8 * 1024 / T  # tiles of the long request (8 units) over all tiles
    nbins = len(set(np.searchsorted(tm["cta_desc_begin"], np.flatnonzero(tm["descs"][:, 0] < 8), "right") - 1))
    assert abs(nbins - share * C_eff) <= 8 + 1


@pytest.mark.parametrize("mode,param", [(0, 16), (0, 3), (1, 4096), (1, 128)])
def test_static_split_cover(mode, param):
    for max_len in (1, 64, 100, 4096, 5000, 131072):
        S = oracle.static_num_splits(mode, param, max_len)
        if mode == 0:
            assert S == param
        else:
            assert S == max(1, -(-max_len // param))
        for length in sorted({0, 1, 63, max_len // 2, max_len}):
            n = -(-length // TILE)
            ranges = [oracle.static_split(mode, param, TILE, S, n, s) for s in range(S)]
            # contiguous exact cover of [0, n)
            covered = [t for a, b in ranges for t in range(a, b)]
            assert covered == list(range(n))
            sizes = [b - a for a, b in ranges]
            if mode == 0:
                assert max(sizes) <= -(-n // S)  # a fixed count: heavy chunks for long requests
            else:
                assert all(sz <= param // TILE for sz in sizes)  # fixed chunk size
                nonempty = [sz for sz in sizes if sz]
                assert all(sz == param // TILE for sz in nonempty[:-1])
