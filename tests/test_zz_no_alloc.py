"""dsa_decode_step_noalloc: the allocation-free whole step, for callers that cannot call
cudaMalloc (e.g. code running under another framework's memory pool or allocator hooks).

It keeps its task map and partial outputs in a fixed device array inside the library.
Two calls in a row, on different inputs, must each give the same output as the
ordinary plan / decode / combine path (whose buffers the caller allocates), within the
parity tolerance; a step too large for the fixed array is refused before any launch.
This file is collected last so that a failure here leaves every other test already run.
"""
import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu

TOL = {"bf16": (2e-3, 1e-3), "fp8": (2e-2, 1e-2)}  # max-abs, per-row rel-L2 (fp32 outputs)


@pytest.fixture(scope="module")
def dsa():
    import load_balanced_paged_gb300 as m
    return m


def close(a: torch.Tensor, b: torch.Tensor, kv: str):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    atol, rtol = TOL[kv]
    err = np.abs(a - b).max()
    den = np.linalg.norm(b, axis=-1)
    rel = np.where(den > 0, np.linalg.norm(a - b, axis=-1) / np.where(den > 0, den, 1), 0).max()
    assert err <= atol and rel <= rtol, (err, rel)


def test_two_calls_match_the_allocating_path(dsa):
    ctas = torch.cuda.get_device_properties(0).multi_processor_count
    cases = [
        (workloads.make_inputs(np.array([17, 64, 200, 1500, 0, 3000]), 64, 8, "bf16", seed=1, device="cuda"), "bf16"),
        (workloads.make_inputs(np.array([5000, 1, 640, 129]), 32, 4, "fp8", seed=2, device="cuda"), "fp8"),
    ]
    for inp, kv in cases:  # two calls in a row, the second over what the first left behind
        B, hq = inp["seq_lens"].shape[0], inp["num_q_heads"]
        out = torch.full((B, hq, 128), float("nan"), dtype=torch.float32, device="cuda")
        lse = torch.full((B, hq), float("nan"), dtype=torch.float32, device="cuda")
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        dsa.decode_step_noalloc(inp, ctas, out, out_lse=lse, status=status)
        torch.cuda.synchronize()
        assert status.item() == 0

        ref_tm = dsa.plan(inp["seq_lens"], inp["num_kv_heads"], ctas, 4)
        po, pl = dsa.decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"], inp["seq_lens"], ref_tm,
                            inp["sm_scale"], q_scale=inp["q_scale"], k_scale=inp["k_scale"], v_scale=inp["v_scale"])
        ref_lse = torch.empty_like(lse)
        ref = dsa.combine(ref_tm, po, pl, hq, out_lse=ref_lse, out_dtype=torch.float32)
        torch.cuda.synchronize()
        close(out, ref, kv)
        fin = torch.isfinite(ref_lse)
        assert torch.equal(fin, torch.isfinite(lse))
        assert (lse[fin] - ref_lse[fin]).abs().max().item() <= 1e-3


def test_refuses_steps_beyond_the_fixed_scratch(dsa):
    # 2048 requests x 8 KV heads x 8 query heads per KV head need far more than the fixed array
    inp = workloads.make_inputs(np.full(2048, 1, np.int64), 64, 8, "bf16", seed=3, device="cuda")
    out = torch.zeros(2048, 64, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(dsa.DSAError) as e:
        dsa.decode_step_noalloc(inp, 152, out)
    assert e.value.code == dsa.ERR_BUFFER_TOO_SMALL
    assert (out == 0).all()
