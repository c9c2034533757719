"""dsa_decode_step_noalloc: the allocation-free whole step, for callers that cannot call
cudaMalloc (e.g. code running under another framework's memory pool or allocator hooks).

It keeps its task map and partial outputs in a fixed device array inside the library and
runs the same plan, decode and combine kernels as the ordinary path (whose buffers the
caller allocates).  So on the same inputs, CTA count and floor its outputs must equal that
path's bit for bit, on every call of a sequence (each call reuses what the previous one
left in the array), and lie within the stated tolerance of the fp64 oracle.  Device input
errors reach the caller's status word; a step the fixed array cannot hold, or one with an
argument the kernels would refuse, is refused before anything is launched.
This file is collected last so that a failure here leaves every other test already run.
"""
import numpy as np
import pytest
import torch

import workloads
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import load_balanced_paged_gb300 as m
    return m


def allocating_step(dsa, inp, ctas, out_dtype):
    tm = dsa.plan(inp["seq_lens"], inp["num_kv_heads"], ctas, 4)
    po, pl = dsa.decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"], inp["seq_lens"], tm,
                        inp["sm_scale"], q_scale=inp["q_scale"], k_scale=inp["k_scale"], v_scale=inp["v_scale"])
    lse = torch.empty(inp["seq_lens"].shape[0], inp["num_q_heads"], dtype=torch.float32, device="cuda")
    out = dsa.combine(tm, po, pl, inp["num_q_heads"], out_lse=lse, out_dtype=out_dtype)
    torch.cuda.synchronize()
    return out, lse, dsa.get_status(tm)


def noalloc_step(dsa, inp, ctas, out_dtype, with_lse=True):
    B, hq = inp["seq_lens"].shape[0], inp["num_q_heads"]
    fill = float("nan") if out_dtype == torch.float32 else 7.0
    out = torch.full((B, hq, 128), fill, dtype=out_dtype, device="cuda")
    lse = torch.full((B, hq), float("nan"), dtype=torch.float32, device="cuda") if with_lse else None
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    dsa.decode_step_noalloc(inp, ctas, out, out_lse=lse, status=status)
    torch.cuda.synchronize()
    return out, lse, int(status.item())


CASES = [((17, 64, 200, 1500, 0, 3000), 64, 8, "bf16", 1), ((5000, 1, 640, 129), 32, 4, "fp8", 2)]


def test_calls_in_a_row_equal_the_allocating_path_and_the_oracle(dsa):
    ctas = torch.cuda.get_device_properties(0).multi_processor_count
    for lens, hq, hkv, kv, seed in CASES:  # each call over what the previous one left behind
        inp = workloads.make_inputs(np.array(lens), hq, hkv, kv, seed=seed, device="cuda")
        for out_dtype in (torch.float32, torch.bfloat16):
            out, lse, st = noalloc_step(dsa, inp, ctas, out_dtype)
            assert st == 0
            ref, ref_lse, ref_st = allocating_step(dsa, inp, ctas, out_dtype)
            assert ref_st == 0
            assert torch.equal(out, ref), f"{kv} {out_dtype}: outputs differ from the allocating path"
            assert torch.equal(lse, ref_lse), f"{kv} {out_dtype}: LSEs differ from the allocating path"
        # the fp64 oracle on the same bytes (fp32 output: the stated tolerance, unrounded)
        out32, lse32, _ = noalloc_step(dsa, inp, ctas, torch.float32)
        prob = parity.problem_from_host(workloads.host_view(inp), inp)
        oref, olse = prob.attention()
        parity.assert_close(out32.cpu().numpy(), oref, kv, f"no-alloc {kv} vs oracle", round_ref=False)
        parity.assert_lse_close(lse32.cpu().numpy(), olse, f"no-alloc {kv} lse vs oracle")


def test_device_status_reaches_the_caller(dsa):
    """A negative length is device-resident bad input: the plan skips that request and sets
    DSA_DEV_BAD_SEQLEN, which the step copies into the caller's status word; the other
    requests still equal the allocating path's."""
    inp = workloads.make_inputs(np.array([300, 900, 64]), 16, 2, "bf16", seed=4, device="cuda")
    inp["seq_lens"][1] = -5
    out, lse, st = noalloc_step(dsa, inp, 20, torch.float32)
    assert st & dsa.DEV_BAD_SEQLEN
    ref, ref_lse, ref_st = allocating_step(dsa, inp, 20, torch.float32)
    assert ref_st & dsa.DEV_BAD_SEQLEN
    keep = torch.tensor([0, 2], device="cuda")
    assert torch.equal(out[keep], ref[keep]) and torch.equal(lse[keep], ref_lse[keep])
    # the next good step clears it again
    inp["seq_lens"][1] = 900
    _, _, st = noalloc_step(dsa, inp, 20, torch.float32)
    assert st == 0


def test_without_out_lse_and_with_an_empty_batch(dsa):
    inp = workloads.make_inputs(np.array([77, 4096, 1]), 24, 3, "bf16", seed=6, device="cuda")
    out_a, _, st = noalloc_step(dsa, inp, 9, torch.float32, with_lse=False)
    assert st == 0
    out_b, _, _ = noalloc_step(dsa, inp, 9, torch.float32)
    assert torch.equal(out_a, out_b)
    empty = workloads.make_inputs(np.zeros(0, np.int64), 24, 3, "bf16", seed=6, device="cuda")
    out, lse, st = noalloc_step(dsa, empty, 9, torch.bfloat16)
    assert st == 0 and out.numel() == 0


def test_refuses_before_any_launch(dsa):
    # 2048 requests x 8 KV heads x 8 query heads per KV head need far more than the fixed array
    inp = workloads.make_inputs(np.full(2048, 1, np.int64), 64, 8, "bf16", seed=3, device="cuda")
    out = torch.zeros(2048, 64, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dsa.DSAError) as e:
        dsa.decode_step_noalloc(inp, 152, out)
    assert e.value.code == dsa.ERR_BUFFER_TOO_SMALL
    assert (out == 0).all()
    # an output the combine kernel would refuse (not 16-byte aligned): nothing runs, the
    # status word is not written
    small = workloads.make_inputs(np.array([100, 200]), 8, 1, "bf16", seed=5, device="cuda")
    base = torch.zeros(2 * 8 * 128 + 4, dtype=torch.float32, device="cuda")
    misaligned = base[1:1 + 2 * 8 * 128].view(2, 8, 128)
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    with pytest.raises(dsa.DSAError) as e:
        dsa.decode_step_noalloc(small, 4, misaligned, status=status)
    assert e.value.code == dsa.ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert status.item() == -1 and (base == 0).all()
