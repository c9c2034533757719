"""Pins for the oracle's attention and merge.

Attention is computed exactly by definition; the pins are a dense brute force
with scipy's softmax/logsumexp over a densely gathered K/V (tests/brute.py),
closed forms, page-pool permutation invariance and the split/merge invariant
(merged log-sum-exp partials of any split equal unsplit attention).
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import brute

HQ, HKV = 8, 2


def tiny(lens, kv="bf16", seed=0, hq=HQ, hkv=HKV, q_len=1, page=64, layout="HND"):
    inp = workloads.make_inputs(np.array(lens), hq, hkv, kv, seed=seed, device="cpu", q_len=q_len,
                                page_size=page, kv_layout=layout)
    h = workloads.host_view(inp)
    return inp, h


def problem(h, inp):
    return oracle.Problem(h["q"], h["k_pages"], h["v_pages"], h["block_table"], h["seq_lens"],
                          inp["num_q_heads"], inp["num_kv_heads"], inp["sm_scale"],
                          q_scale=h["q_scale"], k_scale=h["k_scale"], v_scale=h["v_scale"],
                          q_len=inp.get("q_len", 1), page_size=inp["page_size"], kv_layout=inp["kv_layout"])


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_matches_dense_brute_force(kv):
    lens = [0, 1, 63, 64, 65, 130, 200, 333]
    inp, h = tiny(lens, kv, seed=3)
    out, lse = problem(h, inp).attention()
    ref, ref_lse = brute.dense_attention(h, HQ, HKV, inp["sm_scale"])
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)
    assert (out[0] == 0).all() and np.isneginf(lse[0]).all()  # empty request


def test_q_zero_gives_mean_of_v():
    lens = [5, 77, 130]
    inp, h = tiny(lens)
    h["q"] = np.zeros_like(h["q"])
    out, lse = problem(h, inp).attention()
    v = brute.decode_bf16(h["v_pages"])
    for b, n in enumerate(lens):
        rows = [v[h["block_table"][b, t // 64], :, t % 64] for t in range(n)]  # [n][Hkv][d]
        mean = np.mean(rows, axis=0)
        for j in range(HQ):
            np.testing.assert_allclose(out[b, j], mean[j // (HQ // HKV)], rtol=0, atol=1e-13)
            assert abs(lse[b, j] - math.log(n)) < 1e-13


def test_constant_v_rows():
    lens = [9, 150]
    inp, h = tiny(lens)
    c = np.float32(0.375)  # exact in bf16
    h["v_pages"] = np.full_like(h["v_pages"], torch.tensor([c]).to(torch.bfloat16).view(torch.int16).item())
    out, _ = problem(h, inp).attention()
    np.testing.assert_allclose(out, 0.375, rtol=0, atol=1e-14)


def test_single_token():
    inp, h = tiny([1, 1])
    out, lse = problem(h, inp).attention()
    q = brute.decode_bf16(h["q"])
    k = brute.decode_bf16(h["k_pages"])
    v = brute.decode_bf16(h["v_pages"])
    for b in range(2):
        p = h["block_table"][b, 0]
        for j in range(HQ):
            hk = j // (HQ // HKV)
            np.testing.assert_array_equal(out[b, j], v[p, hk, 0])
            assert abs(lse[b, j] - inp["sm_scale"] * float(q[b, j] @ k[p, hk, 0])) < 1e-12


def test_gqa_head_mapping_probe():
    # V of KV head h is the constant h: query head j must read floor(j / G)
    hq, hkv = 16, 4
    inp, h = tiny([40, 100], hq=hq, hkv=hkv)
    vv = np.zeros(h["v_pages"].shape, np.float32)
    for hh in range(hkv):
        vv[:, hh] = hh
    h["v_pages"] = torch.from_numpy(vv).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    out, _ = oracle.Problem(h["q"], h["k_pages"], h["v_pages"], h["block_table"], h["seq_lens"],
                            hq, hkv, inp["sm_scale"]).attention()
    for j in range(hq):
        np.testing.assert_allclose(out[:, j], j // (hq // hkv), rtol=0, atol=1e-13)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_page_pool_permutation_invariance(kv):
    inp, h = tiny([70, 129, 300], kv, seed=5)
    out, lse = problem(h, inp).attention()
    rng = np.random.default_rng(9)
    n = h["k_pages"].shape[0]
    perm = rng.permutation(n)  # new page p holds old page perm[p]
    inv = np.argsort(perm)
    h2 = dict(h)
    for key in ("k_pages", "v_pages", "k_scale", "v_scale"):
        if h[key] is not None:
            h2[key] = np.ascontiguousarray(h[key][perm])
    bt = h["block_table"].copy()
    bt[bt >= 0] = inv[bt[bt >= 0]]
    h2["block_table"] = bt
    out2, lse2 = problem(h2, inp).attention()
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(lse, lse2)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_split_merge_equals_unsplit(kv):
    lens = [1, 64, 257, 1000]
    inp, h = tiny(lens, kv, seed=7)
    prob = problem(h, inp)
    out, lse = prob.attention()
    rng = np.random.default_rng(11)
    G = HQ // HKV
    for b, n in enumerate(lens):
        for hk in range(HKV):
            for _ in range(4):
                cuts = sorted(set(rng.integers(0, n + 1, rng.integers(0, 6)).tolist()) | {0, n})
                parts = [prob.span(b, hk, a, c) for a, c in zip(cuts, cuts[1:])]
                # add an empty partial: it must not change the result
                parts.append(prob.span(b, hk, n, n))
                mo, ml = oracle.merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
                np.testing.assert_allclose(mo, out[b, hk * G:(hk + 1) * G], rtol=0, atol=1e-12)
                np.testing.assert_allclose(ml, lse[b, hk * G:(hk + 1) * G], rtol=0, atol=1e-12)


def test_merge_of_nothing():
    mo, ml = oracle.merge(np.zeros((2, 3, 4)), np.full((2, 3), -np.inf))
    assert (mo == 0).all() and np.isneginf(ml).all()


def test_units_subset_and_threads():
    lens = [100, 200, 300]
    inp, h = tiny(lens)
    prob = problem(h, inp)
    full, full_lse = prob.attention(n_threads=1)
    sub, sub_lse = prob.attention(units=[5, 0], n_threads=3)
    G = HQ // HKV
    for u in (5, 0):
        b, hk = divmod(u, HKV)
        rows = slice(hk * G, (hk + 1) * G)
        np.testing.assert_array_equal(sub[b, rows], full[b, rows])
    assert np.isnan(sub[0, G:]).all()


# ---------------------------------------------------------------- multi-token queries
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("q_len", [2, 3, 6])
def test_multi_token_matches_causal_brute_force(kv, q_len):
    lens = [0, 1, 4, 6, 63, 64, 65, 130, 200]
    inp, h = tiny(lens, kv, seed=5, q_len=q_len)
    out, lse = problem(h, inp).attention()
    ref, ref_lse = brute.dense_attention_multi(h, HQ, HKV, inp["sm_scale"], q_len)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)
    # query tokens before the request's first token see nothing
    for b, n in enumerate(lens):
        for i in range(q_len):
            if n - q_len + i < 0:
                assert (out[b, i] == 0).all() and np.isneginf(lse[b, i]).all()


@pytest.mark.parametrize("q_len", [2, 5])
def test_multi_token_row_is_single_token_on_truncated_request(q_len):
    """Query token i of a request of length n is a one-token decode over the first
    n - q_len + i + 1 tokens: the same bytes through the q_len = 1 oracle."""
    lens = [7, 64, 99, 140]
    inp, h = tiny(lens, "fp8", seed=8, q_len=q_len)
    out, lse = problem(h, inp).attention()
    for i in range(q_len):
        trunc = np.maximum(np.array(lens) - q_len + i + 1, 0).astype(np.int32)
        one = oracle.Problem(np.ascontiguousarray(h["q"][:, i]), h["k_pages"], h["v_pages"], h["block_table"],
                             trunc, HQ, HKV, inp["sm_scale"], q_scale=np.ascontiguousarray(h["q_scale"][:, i]),
                             k_scale=h["k_scale"], v_scale=h["v_scale"])
        o1, l1 = one.attention()
        np.testing.assert_allclose(out[:, i], o1, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse[:, i], l1, rtol=0, atol=1e-13)


def test_multi_token_split_merge():
    q_len = 4
    lens = [3, 70, 257]
    inp, h = tiny(lens, "bf16", seed=9, q_len=q_len)
    prob = problem(h, inp)
    out, lse = prob.attention()
    rng = np.random.default_rng(0)
    G = HQ // HKV
    for b, n in enumerate(lens):
        for hk in range(HKV):
            cuts = np.unique(np.concatenate([[0, n], rng.integers(0, n + 1, 3)]))
            parts = [prob.span(b, hk, a, c) for a, c in zip(cuts[:-1], cuts[1:])]
            o = np.stack([p[0] for p in parts])
            ls = np.stack([p[1] for p in parts])
            mo, ml = oracle.merge(o, ls)
            ref = out[b][:, hk * G:(hk + 1) * G].reshape(q_len * G, -1)
            np.testing.assert_allclose(mo, ref, rtol=0, atol=1e-12)
            np.testing.assert_allclose(ml, lse[b][:, hk * G:(hk + 1) * G].reshape(-1), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- page layouts and sizes
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("page,layout", [(16, "HND"), (32, "NHD"), (64, "NHD"), (16, "NHD")])
def test_layouts_match_dense_brute_force(kv, page, layout):
    lens = [0, 1, 15, 16, 17, 63, 64, 65, 130, 333]
    inp, h = tiny(lens, kv, seed=11, page=page, layout=layout)
    out, lse = problem(h, inp).attention()
    ref, ref_lse = brute.dense_attention(h, HQ, HKV, inp["sm_scale"], page=page, layout=layout)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def repage(h, lens, page, new_page, layout, rng):
    """The same tokens moved into pages of new_page tokens (randomly placed) and the
    given layout: [num_pages, Hkv, P, d] (HND) or [num_pages, P, Hkv, d] (NHD)."""
    hkv, d = h["k_pages"].shape[1], h["k_pages"].shape[-1]
    pieces_k, pieces_v, pieces_ks, pieces_vs, rows = [], [], [], [], []
    for b, n in enumerate(lens):
        for t0 in range(0, n, new_page):
            pieces = []
            for t in range(t0, t0 + new_page):
                src_page = h["block_table"][b, min(t, max(n - 1, 0)) // page]
                slot = min(t, max(n - 1, 0)) % page
                pieces.append((src_page, slot))
            rows.append((b, t0 // new_page, pieces))
    order = rng.permutation(len(rows))
    npages = len(rows)
    k = np.zeros((npages, hkv, new_page, d), h["k_pages"].dtype)
    v = np.zeros_like(k)
    fp8 = h.get("k_scale") is not None
    ks = np.zeros((npages, hkv, new_page), np.float32) if fp8 else None
    vs = np.zeros_like(ks) if fp8 else None
    bt = np.full((len(lens), max(1, max(-(-n // new_page) for n in lens))), -1, np.int32)
    for dst, i in enumerate(order):
        b, j, pieces = rows[i]
        bt[b, j] = dst
        for s_, (sp, sl) in enumerate(pieces):
            k[dst, :, s_] = h["k_pages"][sp, :, sl]
            v[dst, :, s_] = h["v_pages"][sp, :, sl]
            if fp8:
                ks[dst, :, s_] = h["k_scale"][sp, :, sl]
                vs[dst, :, s_] = h["v_scale"][sp, :, sl]
    if layout == "NHD":
        k, v = np.ascontiguousarray(k.transpose(0, 2, 1, 3)), np.ascontiguousarray(v.transpose(0, 2, 1, 3))
    return dict(h, k_pages=k, v_pages=v, k_scale=ks, v_scale=vs, block_table=bt)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_page_size_and_layout_do_not_change_the_result(kv):
    """The same tokens in 16- or 32-token pages, HND or NHD, give exactly the 64-token HND result."""
    lens = [1, 40, 64, 100, 257]
    inp, h = tiny(lens, kv, seed=12)
    out, lse = problem(h, inp).attention()
    rng = np.random.default_rng(3)
    for new_page in (16, 32):
        for layout in ("HND", "NHD"):
            h2 = repage(h, lens, 64, new_page, layout, rng)
            p2 = oracle.Problem(h2["q"], h2["k_pages"], h2["v_pages"], h2["block_table"], h2["seq_lens"], HQ, HKV,
                                inp["sm_scale"], q_scale=h2["q_scale"], k_scale=h2["k_scale"], v_scale=h2["v_scale"],
                                page_size=new_page, kv_layout=layout)
            o2, l2 = p2.attention()
            assert np.array_equal(o2, out) and np.array_equal(l2, lse), (new_page, layout)
