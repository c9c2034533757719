"""Multi-token queries (dsa_decode_multi + dsa_combine_multi) on the GPU vs the fp64 oracle.

q_len query tokens per request, each seeing the KV tokens up to its own position (the
last q_len positions of the request).  Outputs, LSEs and every descriptor's partial
rows are compared with the oracle (parity.check_outputs: the stated tolerance of the KV
dtype on the fp32 output, and the bf16 output equal to its round-to-nearest-even).  bf16
K/V runs on the tensor-memory kernel, E4M3 K/V on the mma.sync kernel.
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


def make(lens, q_len, hq=64, hkv=8, seed=0, kv="bf16"):
    return workloads.make_inputs(np.asarray(lens), hq, hkv, kv, seed=seed, device="cuda", q_len=q_len)


def problem(inp):
    return parity.problem_from_host(workloads.host_view(inp), inp)


def run(dsa, inp, C, m=4):
    q_len = inp["q_len"]
    out32, lse, tm, po, pl = dsa.attention_multi(inp, C, min_tiles_per_split=m, out_dtype=torch.float32)
    out16 = dsa.combine_multi(q_len, tm, po, pl, inp["num_q_heads"], out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert dsa.get_status(tm) == 0
    return out16, out32, lse, tm, po, pl


CASES = [
    # lengths, q_len, Hq, Hkv   (rows per unit q_len * Hq/Hkv: 16, 32, 48, 64, 24, 6)
    ([17, 64, 200, 1500, 6, 1], 2, 64, 8),
    ([17, 64, 200, 1500, 6, 1], 4, 64, 8),
    ([1, 63, 64, 65, 127, 500, 3000], 6, 64, 8),
    ([5, 70, 130, 2048], 8, 64, 8),
    ([300, 2222, 77, 3], 6, 16, 4),
    ([33, 4000, 64], 6, 8, 8),
]


@pytest.mark.parametrize("lens,q_len,hq,hkv", CASES)
@pytest.mark.parametrize("C,m", [(3, 1), (None, 4), (300, 1)])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_multi_vs_oracle(dsa, lens, q_len, hq, hkv, C, m, kv):
    inp = make(lens, q_len, hq, hkv, seed=q_len + len(lens), kv=kv)
    C = sm_count() if C is None else C
    out16, out32, lse, tm, po, pl = run(dsa, inp, C, m)
    ref, ref_lse = problem(inp).attention()
    what = f"{kv} q_len {q_len} lens {lens} C {C}"
    parity.check_outputs(out16.float().cpu().numpy(), out32.cpu().numpy(), ref, kv, what)
    parity.assert_lse_close(lse.cpu().numpy(), ref_lse, what)
    # query tokens before the request's first token see nothing: exactly zero, lse -inf
    for b, n in enumerate(lens):
        for i in range(q_len):
            if n - q_len + i < 0:
                assert (out32[b, i] == 0).all() and torch.isneginf(lse[b, i]).all()


@pytest.mark.parametrize("scale", [-0.3, 0.0])
@pytest.mark.parametrize("q_len", [2, 6])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_multi_any_finite_scale(dsa, scale, q_len, kv):
    """The softmax scale may be any finite number (the header asks only that): a negative
    scale turns the largest raw score into the smallest scaled one, and a zero scale gives
    every visible token the same weight.  Both kernels must take the maximum over the
    scaled scores and mask after scaling."""
    inp = make([17, 300, 1500, 64], q_len, 64, 8, seed=21, kv=kv)
    inp["sm_scale"] = scale
    out16, out32, lse, tm, po, pl = run(dsa, inp, 40, 1)
    ref, ref_lse = problem(inp).attention()
    what = f"{kv} q_len {q_len} scale {scale}"
    parity.check_outputs(out16.float().cpu().numpy(), out32.cpu().numpy(), ref, kv, what)
    parity.assert_lse_close(lse.cpu().numpy(), ref_lse, what)


@pytest.mark.parametrize("q_len", [2, 3, 6])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_multi_partials_each_descriptor(dsa, q_len, kv):
    inp = make([40, 129, 1000, 2500], q_len, 64, 8, seed=7, kv=kv)
    _, _, _, tm, po, pl = run(dsa, inp, 37, 1)
    prob = problem(inp)
    h = tm.host()
    R = q_len * 8
    spd = int(dsa.lib().dsa_multi_slots_per_desc(q_len, 8))
    po, pl = po.cpu().numpy(), pl.cpu().numpy()
    for x, (u, t0, t1, k) in enumerate(h["descs"]):
        b, hk = divmod(int(u), 8)
        o, lse = prob.span(b, hk, 64 * int(t0), min(64 * int(t1), int(inp["seq_lens"][b])))
        # slots of the descriptor (two: softmax teams, or token halves for E4M3), merged by the oracle
        got_o, got_l = oracle.merge(po[spd * x:spd * x + spd, :R], pl[spd * x:spd * x + spd, :R])
        parity.assert_close(got_o, o, kv, f"descriptor {x}", round_ref=False)
        parity.assert_lse_close(got_l, lse, f"descriptor {x}")


def test_multi_full_size_sampled(dsa):
    """The mixed-length workload's lengths with 6 query tokens per request (1 + 5 draft
    tokens), in the one-CTA-per-SM configuration; 6 requests checked."""
    w = workloads.WORKLOADS["mixed"]
    rng = np.random.default_rng(w.seed)
    lens = workloads.draw_lengths(w.name, w.batch, rng)
    inp = workloads.make_inputs(lens, w.num_q_heads, w.num_kv_heads, "bf16", w.seed, "cuda", rng=rng, q_len=6)
    out16, out32, lse, tm, po, pl = run(dsa, inp, w.num_ctas(sm_count()), 4)
    prob = problem(inp)
    pick = np.argsort(lens)[[0, 1, len(lens) // 2, -2, -1]].tolist() + [3]
    units = [b * w.num_kv_heads + h for b in pick for h in range(w.num_kv_heads)]
    ref, ref_lse = prob.attention(units=units)
    parity.check_outputs(out16[pick].float().cpu().numpy(), out32[pick].cpu().numpy(), ref[pick], "bf16",
                         "mixed, q_len 6")
    parity.assert_lse_close(lse[pick].cpu().numpy(), ref_lse[pick], "mixed, q_len 6")


@pytest.mark.parametrize("q_len", [2, 6])
def test_multi_full_size_fp8_sampled(dsa, q_len):
    """The FP8 workload's lengths (64 requests, mean 68k tokens) with 2 query tokens per
    request (16 rows: mma.sync kernel) or 6 (48 rows: tensor-memory kernel), one bin per
    SM; the shortest, median and longest requests checked."""
    w = workloads.WORKLOADS["fp8"]
    rng = np.random.default_rng(w.seed)
    lens = workloads.draw_lengths(w.name, w.batch, rng)
    inp = workloads.make_inputs(lens, w.num_q_heads, w.num_kv_heads, "fp8", w.seed, "cuda", rng=rng, q_len=q_len)
    out16, out32, lse, tm, po, pl = run(dsa, inp, sm_count(), 4)
    order = np.argsort(lens, kind="stable")
    picks = sorted({int(order[0]), int(order[len(order) // 2]), int(order[-1])})
    ref, ref_lse = parity.sub_problem(inp, picks).attention()
    parity.check_outputs(out16[picks].float().cpu().numpy(), out32[picks].cpu().numpy(), ref, "fp8",
                         f"fp8, q_len {q_len}")
    parity.assert_lse_close(lse[picks].cpu().numpy(), ref_lse, f"fp8, q_len {q_len}")


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_multi_masked_tail_garbage_is_ignored(dsa, kv):
    """Rows of the last page past the request's length hold NaN (bf16 NaN; E4M3 code 0x7F
    and NaN scales): no output may see them."""
    inp = make([70, 200], 4, 16, 2, seed=3, kv=kv)
    bt = inp["block_table"].cpu().numpy()
    for b, n in enumerate([70, 200]):
        last = bt[b, (n - 1) // 64]
        if kv == "bf16":
            inp["v_pages"][last, :, n % 64:] = float("nan")
            inp["k_pages"][last, :, n % 64:] = float("nan")
        else:
            inp["v_pages"][last, :, n % 64:] = 0x7F
            inp["k_pages"][last, :, n % 64:] = 0x7F
            inp["k_scale"][last, :, n % 64:] = float("nan")
            inp["v_scale"][last, :, n % 64:] = float("nan")
    out16, out32, lse, *_ = run(dsa, inp, 5, 1)
    assert torch.isfinite(out32).all()
    ref, _ = problem(inp).attention()
    parity.check_outputs(out16.float().cpu().numpy(), out32.cpu().numpy(), ref, kv, "NaN tail")


def test_multi_one_token_is_decode(dsa):
    inp = make([17, 64, 200, 1500], 1, 64, 8, seed=2)
    C = sm_count()
    a16, a32, alse, *_ = run(dsa, inp, C, 4)
    out, lse, *_ = dsa.attention(inp, C, min_tiles_per_split=4, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert torch.equal(a32.reshape(out.shape), out) and torch.equal(alse.reshape(lse.shape), lse)


@pytest.mark.parametrize("q_len,kv", [(2, "bf16"), (6, "bf16"), (6, "fp8")])
def test_multi_cta_times_leave_results_unchanged(dsa, q_len, kv):
    """dsa_decode_ex for q_len > 1 with a timestamp buffer: every CTA reports start <= end,
    and the partials are bit-identical to a launch without timestamps."""
    inp = make([1, 63, 700, 3000, 129], q_len, 64, 8, seed=11, kv=kv)
    C = 7
    tm = dsa.plan(inp["seq_lens"], 8, C, 1)
    kw = dict(q_scale=inp.get("q_scale"), k_scale=inp.get("k_scale"), v_scale=inp.get("v_scale"))
    po0, pl0 = dsa.decode_multi(q_len, inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"],
                                inp["seq_lens"], tm, inp["sm_scale"], **kw)
    times = torch.zeros(C, 2, dtype=torch.int64, device="cuda")
    po1, pl1 = dsa.decode_multi(q_len, inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"],
                                inp["seq_lens"], tm, inp["sm_scale"], cta_times=times, **kw)
    torch.cuda.synchronize()
    assert dsa.get_status(tm) == 0
    assert torch.equal(po0, po1) and torch.equal(pl0, pl1)
    t = times.cpu().numpy()
    assert (t[:, 0] > 0).all() and (t[:, 1] >= t[:, 0]).all()
    assert (t[:, 1] - t[:, 0]).max() < 10 ** 9  # under a second


def test_multi_rejects_unsupported(dsa):
    inp = make([100, 200], 9, 64, 8)                   # 72 rows per unit
    tm = dsa.plan(inp["seq_lens"], 8, 4)
    with pytest.raises(dsa.DSAError) as e:
        dsa.decode_multi(9, inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"], inp["seq_lens"], tm,
                         inp["sm_scale"])
    assert e.value.code == dsa.ERR_UNSUPPORTED
    f8 = workloads.make_inputs(np.array([100, 200]), 64, 8, "fp8", device="cuda", q_len=9)
    tm = dsa.plan(f8["seq_lens"], 8, 4)
    with pytest.raises(dsa.DSAError) as e:
        dsa.decode_multi(9, f8["q"], f8["k_pages"], f8["v_pages"], f8["block_table"], f8["seq_lens"], tm,
                         f8["sm_scale"], q_scale=f8["q_scale"], k_scale=f8["k_scale"], v_scale=f8["v_scale"])
    assert e.value.code == dsa.ERR_UNSUPPORTED
