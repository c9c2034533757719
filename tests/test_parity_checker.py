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


# ---------------------------------------------------------------------------------------
# Every branch of the oracle's chain, pinned against a second statement of the chain in
# fp32 PyTorch that shares no code with oracle/prologue.py: RoPE as multiplication of
# complex pairs by e^(i*angle) (the pairs (i, i + rot/2) for neox, (2i, 2i + 1) for
# interleaved), RMSNorm per head with the weight of its head kind (Q: q_norm_weight,
# K: k_norm_weight), V passed through (HPC-Ops × SGLang blog, "融合式 attention 前导":
# QK-Norm on Q and K before RoPE; Hy3 preview write-up 2.2.1).

def complex_rope(t, cs, rot, style):
    """Rotate the first `rot` dims of t [n, heads, 128] by the angles of cs [n, 1, rot]."""
    h = rot // 2
    rotor = torch.complex(cs[..., :h], cs[..., h:rot])
    if style == "interleaved":
        z = torch.view_as_complex(t[..., :rot].reshape(*t.shape[:-1], h, 2).contiguous())
        r = torch.view_as_real(z * rotor).reshape(*t.shape[:-1], rot)
    else:
        z = torch.complex(t[..., :h], t[..., h:rot])
        w = z * rotor
        r = torch.cat([w.real, w.imag], -1)
    return torch.cat([r, t[..., rot:]], -1)


def fp32_heads(inp, hq, hkv, rot, style, had):
    """(q, k, v) of the chain in fp32: Q and K heads normalised with their own weights."""
    n = inp["qkv"].shape[0]
    x = inp["qkv"].float().reshape(n, hq + 2 * hkv, 128)
    cs = inp["cos_sin"][inp["positions"].long()][:, None]
    H = torch.tensor(scipy.linalg.hadamard(128), dtype=torch.float32) * np.float32(128 ** -0.5)

    def branch(t, w):
        t = t * torch.rsqrt((t * t).mean(-1, keepdim=True) + 1e-6) * w
        if rot:
            t = complex_rope(t, cs, rot, style)
        return t @ H.T if had else t
    return (branch(x[:, :hq], inp["q_norm_weight"]), branch(x[:, hq:hq + hkv], inp["k_norm_weight"]),
            x[:, hq + hkv:])


def oracle_heads(inp, hq, hkv, rot, style, had, q_w="q", k_w="k"):
    """The oracle's chain; q_w / k_w name the weight each head kind is given (a planted
    mistake passes the other kind's weight, or None for no normalisation)."""
    wt = {"q": inp["q_norm_weight"].double().numpy(), "k": inp["k_norm_weight"].double().numpy(), None: None}
    return P.prologue(inp["qkv"].view(torch.int16).numpy().view(np.uint16), hq, hkv, inp["positions"].numpy(),
                      inp["cos_sin"].numpy(), rot, style, wt[q_w], wt[k_w], 1e-6, had)


def assert_rows_close(got64, ref32, what):
    """Per row of 128: |oracle - fp32 restatement| <= 2e-5 x the row's amax (the fp32
    chain's own error is below 1e-6 of amax)."""
    g = np.asarray(got64).reshape(-1, 128)
    r = ref32.double().numpy().reshape(-1, 128)
    tol = 2e-5 * np.abs(r).max(1, keepdims=True)
    bad = np.abs(g - r) > tol
    assert not bad.any(), f"{what}: {int(bad.sum())} values off, worst {np.abs(g - r).max():.3e}"


BRANCH_CASES = [(128, "neox", True), (64, "interleaved", True), (64, "neox", False), (128, "interleaved", False)]


@pytest.fixture(scope="module", params=BRANCH_CASES, ids=lambda c: f"rot{c[0]}-{c[1]}-had{int(c[2])}")
def branches(request):
    rot, style, had = request.param
    hq, hkv = 8, 2
    inp = workloads.make_prologue_inputs(96, hq, hkv, 4, seed=11, rotary_dim=rot)
    return inp, hq, hkv, rot, style, had, fp32_heads(inp, hq, hkv, rot, style, had)


def test_every_head_kind_matches_the_fp32_restatement(branches):
    inp, hq, hkv, rot, style, had, (q32, k32, v32) = branches
    q, k, v = oracle_heads(inp, hq, hkv, rot, style, had)
    assert_rows_close(q, q32, "Q")
    assert_rows_close(k, k32, "K")
    assert np.array_equal(v, v32.double().numpy()), "V must pass through unchanged"


def test_planted_k_branch_mistakes_fail(branches):
    inp, hq, hkv, rot, style, had, (q32, k32, v32) = branches
    # K normalised with the Q weight, K not normalised, Q normalised with the K weight
    for q_w, k_w, which in (("q", "q", "K"), ("q", None, "K"), ("k", "k", "Q")):
        q, k, _ = oracle_heads(inp, hq, hkv, rot, style, had, q_w=q_w, k_w=k_w)
        with pytest.raises(AssertionError):
            if which == "K":
                assert_rows_close(k, k32, f"K with weight {k_w}")
            else:
                assert_rows_close(q, q32, f"Q with weight {q_w}")
    # the other RoPE pairing
    other = "neox" if style == "interleaved" else "interleaved"
    _, k, _ = oracle_heads(inp, hq, hkv, rot, other, had)
    with pytest.raises(AssertionError):
        assert_rows_close(k, k32, f"K with {other} pairs")
