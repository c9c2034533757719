"""Randomised decode steps on the GPU against the fp64 oracle.

Each case draws, from its own seed: batch size, lengths (zeros, single tokens, tile
boundaries, ragged tails, a few long requests), heads per KV head, page size and layout,
KV dtype, query tokens per request, bins and the minimum-work floor; the step runs through
plan -> decode -> combine (or the multi-token calls) and must meet the stated tolerances,
with a clean device status word.
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


def draw_case(seed):
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 9))
    kinds = rng.integers(0, 5, B)
    lens = []
    for k in kinds:
        if k == 0:
            lens.append(int(rng.choice([0, 1, 63, 64, 65, 128])))
        elif k == 1:
            lens.append(int(rng.integers(1, 200)))
        elif k == 2:
            lens.append(int(rng.integers(200, 1200)))
        elif k == 3:
            lens.append(int(rng.integers(1200, 4000)))
        else:
            lens.append(64 * int(rng.integers(1, 40)))
    hkv = int(rng.choice([1, 2, 4, 8]))
    G = int(rng.choice([g for g in (1, 2, 3, 4, 6, 8) if g * hkv <= 64]))
    page = int(rng.choice([16, 32, 64]))
    layout = str(rng.choice(["HND", "NHD"]))
    q_len = int(rng.choice([1, 1, 2, 3, 6])) if G * 6 <= 64 else 1
    kv = str(rng.choice(["bf16", "fp8"]))
    C = int(rng.choice([1, 3, 17, 148, 300]))
    m = int(rng.choice([1, 2, 4, 16]))
    return dict(lens=lens, hkv=hkv, hq=G * hkv, page=page, layout=layout, q_len=q_len, kv=kv, C=C, m=m)


@pytest.mark.parametrize("seed", range(80))
def test_random_step_vs_oracle(dsa, seed):
    c = draw_case(seed)
    inp = workloads.make_inputs(np.asarray(c["lens"]), c["hq"], c["hkv"], c["kv"], seed=seed, device="cuda",
                                page_size=c["page"], kv_layout=c["layout"], q_len=c["q_len"])
    if c["q_len"] == 1:
        out32, lse, tm, po, pl = dsa.attention(inp, c["C"], min_tiles_per_split=c["m"], out_dtype=torch.float32)
        out16 = dsa.combine(tm, po, pl, c["hq"], out_dtype=torch.bfloat16)
    else:
        out32, lse, tm, po, pl = dsa.attention_multi(inp, c["C"], min_tiles_per_split=c["m"],
                                                     out_dtype=torch.float32)
        out16 = dsa.combine_multi(c["q_len"], tm, po, pl, c["hq"], out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert dsa.get_status(tm) == 0, c
    ref, ref_lse = parity.problem_from_host(workloads.host_view(inp), inp).attention()
    what = f"case {seed}: {c}"
    parity.check_outputs(out16.float().cpu().numpy(), out32.cpu().numpy(), ref, c["kv"], what)
    parity.assert_lse_close(lse.cpu().numpy(), ref_lse, what)
