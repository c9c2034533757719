"""The prologue parity rule (parity.assert_encoded) on the CPU: an fp32 emulation of the
chain in plain PyTorch passes it, and planted mistakes (a wrong code, a wrong scale) fail."""
import numpy as np
import pytest
import scipy.linalg
import torch

import workloads
from oracle import prologue as P
from tests.parity import PROLOGUE_ERR, assert_encoded


def fp32_chain(inp, hq, hkv):
    n = inp["qkv"].shape[0]
    x = inp["qkv"].float().reshape(n, hq + 2 * hkv, 128)
    cs = inp["cos_sin"][inp["positions"].long()][:, None]
    H = torch.tensor(scipy.linalg.hadamard(128), dtype=torch.float32) * np.float32(128 ** -0.5)

    def chain(t, w):
        t = t / torch.sqrt((t * t).mean(-1, keepdim=True) + 1e-6) * w
        a, b = t[..., :64], t[..., 64:]
        t = torch.cat([a * cs[..., :64] - b * cs[..., 64:], b * cs[..., :64] + a * cs[..., 64:]], -1)
        return t @ H.T
    return chain(x[:, :hq], inp["q_norm_weight"])


@pytest.fixture(scope="module")
def case():
    hq, hkv = 16, 2
    inp = workloads.make_prologue_inputs(200, hq, hkv, 8, seed=3)
    q32 = fp32_chain(inp, hq, hkv)
    q64, _, _ = P.prologue(inp["qkv"].view(torch.int16).numpy().view(np.uint16), hq, hkv,
                           inp["positions"].numpy(), inp["cos_sin"].numpy(), 128, "neox",
                           inp["q_norm_weight"].double().numpy(), None, 1e-6, True)
    amax = q32.abs().amax(-1)
    codes = (q32 * (448.0 / amax)[..., None]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    scale = (amax / 448.0).numpy()
    err = PROLOGUE_ERR * np.abs(q64.reshape(-1, 128)).max(1)
    return q32, q64, codes, scale, err


def test_fp32_chain_passes(case):
    q32, q64, codes, scale, err = case
    assert_encoded(codes, scale, q64, "e4m3", err, "fp32 chain e4m3")
    assert_encoded(q32.to(torch.bfloat16).view(torch.int16).numpy(), None, q64, "bf16", err, "fp32 chain bf16")


def test_planted_mistakes_fail(case):
    q32, q64, codes, scale, err = case
    bad = codes.copy().reshape(-1, 128)
    bad[5, 7] = (int(bad[5, 7]) & 0x80) | min((int(bad[5, 7]) & 0x7F) + 2, 0x7E) if (bad[5, 7] & 0x7F) < 0x7C else bad[5, 7] - 2
    with pytest.raises(AssertionError):
        assert_encoded(bad, scale, q64, "e4m3", err, "code two steps off")
    with pytest.raises(AssertionError):
        assert_encoded(codes, scale * 1.001, q64, "e4m3", err, "scale off")
    with pytest.raises(AssertionError):   # the chain without the Hadamard rotation
        q64_nohad = P.hadamard(q64)
        assert_encoded(codes, scale, q64_nohad, "e4m3", err, "wrong chain")
