"""Persistent decode + combine, and the static split-KV path, on the GPU vs the fp64 oracle.

Small cases are checked element by element (several tiles per request, ragged last
tiles, many and few CTAs, GQA groups 1-8, bf16 and E4M3); the five full-size
workloads are checked on sampled requests in the bench's launch configuration.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import load_balanced_paged_gb300 as m
    return m


def sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


def make(lens, hq=64, hkv=8, kv="bf16", seed=0):
    return workloads.make_inputs(np.asarray(lens), hq, hkv, kv, seed=seed, device="cuda")


def run_dynamic(dsa, inp, C, m=4, out_dtype=torch.bfloat16):
    out, lse, tm, po, pl = dsa.attention(inp, C, min_tiles_per_split=m, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out, lse, tm, po, pl


SMALL = [
    ([17, 64, 200, 1500], 8, 1, "bf16"),
    ([1, 63, 64, 65, 127, 500, 1000, 3000], 64, 8, "bf16"),
    ([1, 63, 64, 65, 127, 500, 1000, 3000], 64, 8, "fp8"),
    ([0, 5, 0, 700, 129], 16, 4, "bf16"),
    ([0, 5, 0, 700, 129], 16, 4, "fp8"),
    ([33, 4000], 8, 8, "bf16"),      # G = 1
    ([300, 2222, 77], 12, 4, "bf16"),  # G = 3
    ([300, 2222, 77], 12, 4, "fp8"),
]


def resolve_ctas(C):
    """None: one bin per SM; "2x": two bins per SM (the two-CTAs-per-SM kernel shape)."""
    if C is None:
        return sm_count()
    if C == "2x":
        return 2 * sm_count()
    return C


@pytest.mark.parametrize("lens,hq,hkv,kv", SMALL)
@pytest.mark.parametrize("C,m", [(3, 1), (None, 4), (300, 1), ("2x", 4)])
def test_small_vs_oracle(dsa, lens, hq, hkv, kv, C, m):
    inp = make(lens, hq, hkv, kv, seed=len(lens))
    C = resolve_ctas(C)
    out, lse, tm, po, pl = run_dynamic(dsa, inp, C, m)
    assert dsa.get_status(tm) == 0
    h = workloads.host_view(inp)
    ref_map = oracle.plan(h["seq_lens"], hkv, C, 64, m)
    got_map = tm.host()
    for k in ref_map:
        assert np.array_equal(got_map[k], ref_map[k]), k
    prob = parity.problem_from_host(h, inp)
    ref, ref_lse = prob.attention()
    out32 = dsa.combine(tm, po, pl, hq, out_dtype=torch.float32)
    parity.check_outputs(out.float().cpu().numpy(), out32.cpu().numpy(), ref, kv, "dynamic")
    parity.assert_lse_close(lse.cpu().numpy(), ref_lse, "out lse")


@pytest.mark.parametrize("scale", [-0.3, 0.0])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_any_finite_scale(dsa, scale, kv):
    """The softmax scale may be any finite number (the header asks only that): with a
    negative scale the smallest raw score weighs most, with a zero scale every visible
    token weighs the same.  The persistent decode (one and two CTAs per SM), the fused
    decode + combine and the static split-KV path must all match the oracle."""
    lens = [17, 300, 1500, 64, 1]
    inp = make(lens, 16, 2, kv, seed=31)
    inp["sm_scale"] = scale
    h = workloads.host_view(inp)
    ref, ref_lse = parity.problem_from_host(h, inp).attention()
    for C in (7, "2x"):
        out, lse, tm, po, pl = run_dynamic(dsa, inp, resolve_ctas(C), 1)
        assert dsa.get_status(tm) == 0
        out32 = dsa.combine(tm, po, pl, 16, out_dtype=torch.float32)
        parity.check_outputs(out.float().cpu().numpy(), out32.cpu().numpy(), ref, kv, f"scale {scale}, C {C}")
        parity.assert_lse_close(lse.cpu().numpy(), ref_lse, f"scale {scale}, C {C}")
    kw = dict(q_scale=inp["q_scale"], k_scale=inp["k_scale"], v_scale=inp["v_scale"])
    tm = dsa.plan(inp["seq_lens"], 2, 7, 1)
    outf = dsa.decode_fused(inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"], inp["seq_lens"], tm,
                            scale, out_dtype=torch.float32, **kw)
    torch.cuda.synchronize()
    assert dsa.get_status(tm) == 0
    parity.assert_close(outf.cpu().numpy(), ref, kv, f"fused, scale {scale}", round_ref=False)
    po, pl, S, status = dsa.static_splitkv(0, 16, max(lens), inp["q"], inp["k_pages"], inp["v_pages"],
                                           inp["block_table"], inp["seq_lens"], 2, scale, **kw)
    out32 = dsa.static_combine(S, po, pl, len(lens), 16, 2, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert dsa.read_status(status) == 0
    parity.assert_close(out32.cpu().numpy(), ref, kv, f"static, scale {scale}", round_ref=False)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_partials_each_descriptor(dsa, kv):
    """Each GPU partial equals attention over its descriptor's tokens, and the oracle's
    merge of the GPU partials equals unsplit attention (checks decode without combine)."""
    lens = [70, 1000, 2500, 64]
    inp = make(lens, 32, 4, kv, seed=11)
    _, _, tm, po, pl = run_dynamic(dsa, inp, 7, 1)
    h = workloads.host_view(inp)
    prob = parity.problem_from_host(h, inp)
    ref, ref_lse = prob.attention()
    m = tm.host()
    po, pl = po.cpu().numpy(), pl.cpu().numpy()
    G = 8
    for x, (u, t0, t1, k) in enumerate(m["descs"]):
        b, hk = divmod(int(u), 4)
        o, l = prob.span(b, hk, 64 * t0, min(64 * t1, lens[b]))
        parity.assert_close(po[x], o, kv, f"partial {x}", round_ref=False)
        parity.assert_lse_close(pl[x], l, f"partial lse {x}")
    for u in range(len(lens) * 4):
        b, hk = divmod(u, 4)
        beg, n = m["unit_partial_begin"][u], m["unit_num_partials"][u]
        mo, ml = oracle.merge(po[beg:beg + n].astype(np.float64), pl[beg:beg + n].astype(np.float64))
        parity.assert_close(mo, ref[b, hk * G:(hk + 1) * G], kv, f"merged unit {u}", round_ref=False)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("mode,param", [(0, 16), (0, 3), (1, 4096), (1, 128)])
def test_static_vs_oracle(dsa, kv, mode, param):
    lens = [1, 63, 64, 65, 127, 500, 1000, 5000]
    inp = make(lens, 64, 8, kv, seed=5)
    max_len = max(lens)
    po, pl, S, status = dsa.static_splitkv(mode, param, max_len, inp["q"], inp["k_pages"], inp["v_pages"],
                                           inp["block_table"], inp["seq_lens"], 8, inp["sm_scale"],
                                           q_scale=inp["q_scale"], k_scale=inp["k_scale"], v_scale=inp["v_scale"])
    lse = torch.empty(len(lens), 64, dtype=torch.float32, device="cuda")
    out = dsa.static_combine(S, po, pl, len(lens), 64, 8, out_lse=lse)
    out32 = dsa.static_combine(S, po, pl, len(lens), 64, 8, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert dsa.read_status(status) == 0
    assert S == oracle.static_num_splits(mode, param, max_len)
    h = workloads.host_view(inp)
    prob = parity.problem_from_host(h, inp)
    ref, ref_lse = prob.attention()
    parity.check_outputs(out.float().cpu().numpy(), out32.cpu().numpy(), ref, kv, "static")
    parity.assert_lse_close(lse.cpu().numpy(), ref_lse, "static lse")
    # every split's partial against the oracle over that split's tokens
    po, pl = po.cpu().numpy(), pl.cpu().numpy()
    for b, n in enumerate(lens):
        nt = -(-n // 64)
        for hk in (0, 7):
            for s in range(S):
                t0, t1 = oracle.static_split(mode, param, 64, S, nt, s)
                o, l = prob.span(b, hk, 64 * t0, min(64 * t1, n))
                slot = (b * 8 + hk) * S + s
                parity.assert_close(po[slot], o, kv, f"static partial {slot}", round_ref=False)
                parity.assert_lse_close(pl[slot], l, f"static partial lse {slot}")


@pytest.mark.parametrize("name", ["tiny", "mixed", "long", "tail", "fp8"])
def test_full_size_workloads_sampled(dsa, name):
    """Full-size workloads in the bench's launch configuration, checked on sampled requests;
    the task map is checked whole."""
    w = workloads.WORKLOADS[name]
    inp = workloads.make_workload(name, device="cuda")
    C = w.num_ctas(sm_count())
    out, lse, tm, po, pl = run_dynamic(dsa, inp, C, 4)
    out32 = dsa.combine(tm, po, pl, w.num_q_heads, out_dtype=torch.float32)
    assert dsa.get_status(tm) == 0
    lens = inp["seq_lens"].cpu().numpy()
    ref_map = oracle.plan(lens, w.num_kv_heads, C, 64, 4)
    got_map = tm.host()
    for k in ref_map:
        assert np.array_equal(got_map[k], ref_map[k]), k
    order = np.argsort(lens, kind="stable")
    picks = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])})
    prob = parity.sub_problem(inp, picks)
    ref, ref_lse = prob.attention()
    parity.check_outputs(out[picks].float().cpu().numpy(), out32[picks].cpu().numpy(), ref, w.kv_dtype,
                         f"{name} sampled")
    parity.assert_lse_close(lse[picks].cpu().numpy(), ref_lse, f"{name} sampled lse")


def test_static_full_size_long(dsa):
    """Single 131072-token request: both static forms vs the oracle on the full output."""
    inp = workloads.make_workload("long", device="cuda")
    prob = parity.sub_problem(inp, [0])
    ref, _ = prob.attention()
    for mode, param in ((0, 16), (1, 4096)):
        po, pl, S, status = dsa.static_splitkv(mode, param, 131072, inp["q"], inp["k_pages"], inp["v_pages"],
                                               inp["block_table"], inp["seq_lens"], 8, inp["sm_scale"])
        out = dsa.static_combine(S, po, pl, 1, 64, 8)
        out32 = dsa.static_combine(S, po, pl, 1, 64, 8, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert dsa.read_status(status) == 0
        parity.check_outputs(out.float().cpu().numpy(), out32.cpu().numpy(), ref, "bf16", f"static mode {mode}")


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_masked_tail_garbage_is_ignored(dsa, kv):
    """Slots past a request's length in its last page hold NaN: the output must not change."""
    lens = [70, 129, 1]
    inp = make(lens, 16, 2, kv, seed=3)
    ref_out, _, _, _, _ = run_dynamic(dsa, inp, 5, 1)
    bt = inp["block_table"].cpu().numpy()
    for b, n in enumerate(lens):
        last = bt[b, (n - 1) // 64]
        for key in ("k_pages", "v_pages"):
            t = inp[key]
            if kv == "bf16":
                t[last, :, n % 64 or 64:] = float("nan")
            else:
                t[last, :, n % 64 or 64:] = 0x7F  # E4M3 NaN
    out, _, tm, _, _ = run_dynamic(dsa, inp, 5, 1)
    assert dsa.get_status(tm) == 0
    assert torch.equal(out, ref_out)


def test_empty_requests(dsa):
    inp = make([0, 0, 100, 0], 16, 2, "bf16")
    out, lse, tm, _, _ = run_dynamic(dsa, inp, 4, 1)
    o = out.float().cpu()
    assert (o[[0, 1, 3]] == 0).all()
    assert torch.isneginf(lse[[0, 1, 3]].cpu()).all()
    assert torch.isfinite(o[2]).all()
    inp = make([0, 0], 16, 2, "bf16")
    out, lse, tm, _, _ = run_dynamic(dsa, inp, 4, 1)
    assert (out.float() == 0).all() and torch.isneginf(lse).all()
    assert tm.host()["meta"].tolist() == [0, 0, 0, 0]


def test_bad_page_id_sets_status(dsa):
    """A block-table entry outside the pool is reported in the status word; nothing faults
    (the kernel skips the tile instead of loading it)."""
    inp = make([300, 200], 16, 2, "bf16")
    inp["block_table"][0, 2] = inp["num_pages"] + 5
    _, _, tm, _, _ = run_dynamic(dsa, inp, 4, 1)
    assert dsa.get_status(tm) & dsa.DEV_BAD_PAGE
    # the context is still usable
    inp2 = make([300, 200], 16, 2, "bf16")
    _, _, tm2, _, _ = run_dynamic(dsa, inp2, 4, 1)
    assert dsa.get_status(tm2) == 0


def test_length_beyond_block_table_sets_status(dsa):
    inp = make([100, 200], 16, 2, "bf16")
    inp["seq_lens"][1] = 64 * inp["max_pages"] + 10  # more tokens than the block table can hold
    _, _, tm, _, _ = run_dynamic(dsa, inp, 4, 1)
    assert dsa.get_status(tm) & dsa.DEV_BAD_SEQLEN


def test_host_validation(dsa):
    inp = make([100], 16, 2, "bf16")
    tm = dsa.plan(inp["seq_lens"], 2, 4)
    with pytest.raises(dsa.DSAError) as e:  # head_dim 64 is not built
        dsa.decode(inp["q"][..., :64].contiguous(), inp["k_pages"][..., :64].contiguous(),
                   inp["v_pages"][..., :64].contiguous(), inp["block_table"], inp["seq_lens"], tm, 0.1)
    assert e.value.code == dsa.ERR_UNSUPPORTED
    with pytest.raises(dsa.DSAError) as e:  # E4M3 K/V without scales
        dsa.decode(inp["q"].view(torch.uint8)[..., :128].contiguous(), inp["k_pages"].view(torch.uint8)[..., :128].contiguous(),
                   inp["v_pages"].view(torch.uint8)[..., :128].contiguous(), inp["block_table"], inp["seq_lens"], tm, 0.1)
    assert e.value.code == dsa.ERR_INVALID_ARG


# ---------------------------------------------------------------- fused decode + combine

@pytest.mark.parametrize("lens,hq,hkv,kv", SMALL[:6])
@pytest.mark.parametrize("C,m", [(3, 1), (None, 4), (300, 1), ("2x", 4)])
def test_fused_vs_oracle(dsa, lens, hq, hkv, kv, C, m):
    inp = make(lens, hq, hkv, kv, seed=len(lens) + 100)
    C = resolve_ctas(C)
    out, lse, tm = dsa.attention_fused(inp, C, m)
    out32, _, _ = dsa.attention_fused(inp, C, m, out_dtype=torch.float32, task_map=tm)
    torch.cuda.synchronize()
    assert dsa.get_status(tm) == 0
    assert (tm.unit_counters() == 0).all()  # every unit's counter returned to zero
    prob = parity.problem_from_host(workloads.host_view(inp), inp)
    ref, ref_lse = prob.attention()
    parity.check_outputs(out.float().cpu().numpy(), out32.cpu().numpy(), ref, kv, "fused")
    parity.assert_lse_close(lse.cpu().numpy(), ref_lse, "fused lse")


def test_fused_matches_separate_combine(dsa):
    """The fused epilogue and the separate combine kernel merge the same partials."""
    inp = make([100, 5000, 64, 2000, 129], 64, 8, "bf16", seed=21)
    sep, sep_lse, _, _, _ = run_dynamic(dsa, inp, 40, 1, out_dtype=torch.float32)
    fused, fused_lse, _ = dsa.attention_fused(inp, 40, 1, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert (fused - sep).abs().max().item() <= 1e-5
    fin = torch.isfinite(sep_lse)
    assert torch.equal(fin, torch.isfinite(fused_lse))
    assert (fused_lse[fin] - sep_lse[fin]).abs().max().item() <= 1e-5


@pytest.mark.parametrize("name", ["mixed", "tail", "fp8"])
def test_fused_full_size_sampled(dsa, name):
    w = workloads.WORKLOADS[name]
    inp = workloads.make_workload(name, device="cuda")
    C = w.num_ctas(sm_count())
    tm = dsa.plan(inp["seq_lens"], w.num_kv_heads, C, 4)
    kw = dict(q_scale=inp["q_scale"], k_scale=inp["k_scale"], v_scale=inp["v_scale"])
    outs = []
    for dt in (torch.bfloat16, torch.float32, torch.float32):  # the last two: a repeated step
        outs.append(dsa.decode_fused(inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"],
                                     inp["seq_lens"], tm, inp["sm_scale"], out_dtype=dt, **kw))
    torch.cuda.synchronize()
    assert dsa.get_status(tm) == 0
    assert torch.equal(outs[1], outs[2])
    lens = inp["seq_lens"].cpu().numpy()
    order = np.argsort(lens, kind="stable")
    picks = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])})
    ref, _ = parity.sub_problem(inp, picks).attention()
    parity.check_outputs(outs[0][picks].float().cpu().numpy(), outs[1][picks].cpu().numpy(), ref, w.kv_dtype,
                         f"{name} fused sampled")


def test_bounded_wait_times_out_and_context_survives(dsa):
    """A wait on a barrier nothing arrives at ends after its limit with DSA_DEV_TIMEOUT; the
    other waiting warp leaves on the abort flag; the device keeps working afterwards."""
    import time
    t0 = time.time()
    status = dsa.selftest_wait_timeout(limit_ns=20_000_000)  # 20 ms
    assert time.time() - t0 < 10
    assert status & dsa.DEV_TIMEOUT
    assert status & (1 << 16)
    inp = make([300, 200], 16, 2, "bf16")
    _, _, tm, _, _ = run_dynamic(dsa, inp, 4, 1)
    assert dsa.get_status(tm) == 0


def test_batch_zero_is_a_no_op(dsa):
    inp = make([], 16, 2, "bf16")
    tm = dsa.plan(inp["seq_lens"], 2, 8)
    po, pl = dsa.decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"], inp["seq_lens"], tm,
                        inp["sm_scale"])
    out = dsa.combine(tm, po, pl, 16)
    torch.cuda.synchronize()
    assert out.shape == (0, 16, 128)
    assert tm.host()["meta"].tolist() == [0, 0, 0, 0]


# ---------------------------------------------------------------- per-CTA timestamps

@pytest.mark.parametrize("C", [None, "2x", 7])
def test_cta_times_leave_results_unchanged(dsa, C):
    """dsa_decode_ex with a timestamp buffer: every CTA reports start <= end, and the
    partials are bit-identical to a launch without timestamps."""
    inp = make([1, 63, 700, 3000, 129], 64, 8, "bf16", seed=9)
    C = resolve_ctas(C)
    tm = dsa.plan(inp["seq_lens"], 8, C, 1)
    po0, pl0 = dsa.decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"], inp["seq_lens"], tm,
                          inp["sm_scale"])
    times = torch.zeros(C, 2, dtype=torch.int64, device="cuda")
    po1, pl1 = dsa.decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"], inp["seq_lens"], tm,
                          inp["sm_scale"], cta_times=times)
    torch.cuda.synchronize()
    assert dsa.get_status(tm) == 0
    nd = len(tm.host()["descs"])
    assert torch.equal(po0[:nd], po1[:nd]) and torch.equal(pl0[:nd], pl1[:nd])
    t = times.cpu().numpy()
    assert (t[:, 0] > 0).all() and (t[:, 1] >= t[:, 0]).all()
    assert (t[:, 1] - t[:, 0]).max() < 10 ** 9  # under a second


def test_static_cta_times(dsa):
    lens = [1, 63, 700, 3000]
    inp = make(lens, 16, 2, "fp8", seed=10)
    S = dsa.static_num_splits(0, 4, max(lens))
    times = torch.zeros(len(lens) * 2 * S, 2, dtype=torch.int64, device="cuda")
    po, pl, S, status = dsa.static_splitkv(0, 4, max(lens), inp["q"], inp["k_pages"], inp["v_pages"],
                                           inp["block_table"], inp["seq_lens"], 2, inp["sm_scale"],
                                           q_scale=inp["q_scale"], k_scale=inp["k_scale"], v_scale=inp["v_scale"],
                                           cta_times=times)
    torch.cuda.synchronize()
    assert dsa.read_status(status) == 0
    t = times.cpu().numpy()
    assert (t[:, 0] > 0).all() and (t[:, 1] >= t[:, 0]).all()
