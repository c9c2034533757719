"""Pins for the prologue oracle (QK-Norm -> RoPE -> Hadamard -> quantise -> cache slot).

Each step is pinned to something other than itself: library routines (torch's RNE
casts to float8_e4m3fn and bf16, scipy's Hadamard matrix), closed forms (a rotation of
(1, 0) by θ, RMS = 1 after RMSNorm, H·H = I) and invariants the pages' chain implies
(RoPE scores depend only on the position difference; an orthogonal rotation of Q and K
keeps every q·k).
"""
import numpy as np
import pytest
import scipy.linalg
import torch

import oracle
from oracle import prologue as P

D = 128


def rotary_table(max_pos, rot, theta=10000.0):
    inv = theta ** (-np.arange(0, rot, 2, dtype=np.float64) / rot)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1)


# ---------------------------------------------------------------- encoders
def test_e4m3_rounding_matches_torch_cast():
    vals, codes = P._e4m3_table()
    mids = (vals[:-1] + vals[1:]) / 2                     # exact in fp32: ties to even
    rng = np.random.default_rng(0)
    rand = rng.uniform(-448, 448, 20000)
    small = rng.uniform(-2 ** -5, 2 ** -5, 5000)          # subnormal range
    x = np.concatenate([vals, -vals, mids, -mids, rand, small]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn)
    got_val, got_code = P.round_e4m3(x.astype(np.float64))
    assert np.array_equal(got_val, ref.to(torch.float64).numpy())
    ref_code = ref.view(torch.uint8).numpy().astype(np.int64)
    nz = x != 0                                            # torch keeps the sign of zero the same way
    assert np.array_equal(got_code[nz], ref_code[nz])


def test_e4m3_saturates_and_ties_to_even():
    assert P.round_e4m3(np.array([460.0]))[0][0] == 448.0
    assert P.round_e4m3(np.array([-1e6]))[0][0] == -448.0
    # 1.0625 is the midpoint of 1.0 (mantissa 000) and 1.125 (mantissa 001): goes to 1.0
    assert P.round_e4m3(np.array([1.0625]))[0][0] == 1.0
    # 1.1875 is the midpoint of 1.125 (001) and 1.25 (010): goes to 1.25
    assert P.round_e4m3(np.array([1.1875]))[0][0] == 1.25
    assert P.round_e4m3(np.array([2 ** -10]))[0][0] == 0.0   # half the smallest subnormal: to even 0


def test_bf16_rounding_matches_torch_cast():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal(50000) * np.exp2(rng.integers(-60, 60, 50000))).astype(np.float32)
    vals, _ = P._bf16_table()
    mids = ((vals[1000:1400] + vals[1001:1401]) / 2).astype(np.float32)
    x = np.concatenate([x, mids, -mids])
    ref = torch.from_numpy(x).to(torch.bfloat16)
    got_val, got_code = P.round_bf16(x.astype(np.float64))
    assert np.array_equal(got_val, ref.to(torch.float64).numpy())
    assert np.array_equal(got_code.astype(np.uint16), ref.view(torch.int16).numpy().view(np.uint16))


def test_bf16_decoder_matches_c_oracle():
    codes = np.arange(0, 1 << 16, 97, dtype=np.uint16)
    got = P.bf16_to_double(codes)
    ref = np.array([oracle.bf16_to_double(int(c)) for c in codes])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()


# ---------------------------------------------------------------- RMSNorm
def test_rms_norm_unit_rms_scale_invariance_and_weight():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((7, 3, D))
    y = P.rms_norm(x, np.ones(D), 0.0)
    assert np.allclose(np.mean(y * y, axis=-1), 1.0, rtol=0, atol=1e-12)
    assert np.allclose(P.rms_norm(5.5 * x, np.ones(D), 0.0), y, rtol=0, atol=1e-12)
    w = rng.standard_normal(D)
    assert np.allclose(P.rms_norm(x, w, 0.0), y * w, rtol=0, atol=1e-12)
    # eps enters under the root: a constant row c gives c / sqrt(c² + eps)
    c = np.full((1, 1, D), 0.5)
    assert np.allclose(P.rms_norm(c, np.ones(D), 0.75), 0.5 / np.sqrt(0.25 + 0.75), atol=1e-15)


# ---------------------------------------------------------------- RoPE
@pytest.mark.parametrize("style", ["neox", "interleaved"])
def test_rope_rotates_unit_vector_by_the_table_angle(style):
    rot = 32
    cs = rotary_table(50, rot)
    for i in (0, 5, rot // 2 - 1):
        x = np.zeros((1, 1, D))
        a, b = (i, i + rot // 2) if style == "neox" else (2 * i, 2 * i + 1)
        x[0, 0, a] = 1.0
        y = P.rope(x, np.array([37]), cs, rot, style)
        expect = np.zeros(D)
        expect[a], expect[b] = cs[37, i], cs[37, rot // 2 + i]   # (cos θ, sin θ)
        assert np.allclose(y[0, 0], expect, atol=1e-15)


@pytest.mark.parametrize("style", ["neox", "interleaved"])
@pytest.mark.parametrize("rot", [32, 64, 128])
def test_rope_scores_depend_on_position_difference_only(style, rot):
    rng = np.random.default_rng(3)
    cs = rotary_table(4096, rot)
    q, k = rng.standard_normal((2, 1, 1, D))
    def score(pq, pk):
        return float(np.sum(P.rope(q, np.array([pq]), cs, rot, style) * P.rope(k, np.array([pk]), cs, rot, style)))
    s0 = score(100, 37)
    for shift in (1, 250, 3000):
        assert abs(score(100 + shift, 37 + shift) - s0) < 1e-9
    assert abs(score(100, 38) - s0) > 1e-6                    # and it does depend on the difference


def test_rope_identity_at_position_zero_and_tail_untouched():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((3, 2, D))
    cs = rotary_table(8, 64)
    assert np.array_equal(P.rope(x, np.zeros(3, np.int64), cs, 64, "neox"), x)
    y = P.rope(x, np.array([1, 2, 3]), cs, 64, "neox")
    assert np.array_equal(y[..., 64:], x[..., 64:])
    # rotation keeps the norm of each rotated pair
    assert np.allclose(y[..., :32] ** 2 + y[..., 32:64] ** 2, x[..., :32] ** 2 + x[..., 32:64] ** 2, atol=1e-12)


def test_rope_interleaved_is_neox_on_deinterleaved_dims():
    rng = np.random.default_rng(5)
    rot = 64
    x = rng.standard_normal((4, 3, D))
    cs = rotary_table(100, rot)
    pos = np.array([0, 9, 55, 99])
    perm = np.concatenate([np.arange(0, rot, 2), np.arange(1, rot, 2), np.arange(rot, D)])
    a = P.rope(x, pos, cs, rot, "interleaved")[..., perm]
    b = P.rope(x[..., perm], pos, cs, rot, "neox")
    assert np.allclose(a, b, atol=1e-15)


# ---------------------------------------------------------------- Hadamard
@pytest.mark.parametrize("d", [2, 8, 128])
def test_hadamard_matches_scipy_and_is_an_involution(d):
    rng = np.random.default_rng(6)
    x = rng.standard_normal((5, d))
    H = scipy.linalg.hadamard(d).astype(np.float64) / np.sqrt(d)
    assert np.allclose(P.hadamard(x), x @ H.T, atol=1e-13)
    assert np.allclose(P.hadamard(P.hadamard(x)), x, atol=1e-13)


# ---------------------------------------------------------------- the chain
def make_qkv(n, hq, hkv, seed=7):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, (hq + 2 * hkv) * D)).astype(np.float32)
    return torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_chain_splits_heads_and_hadamard_keeps_scores():
    n, hq, hkv = 5, 8, 2
    qkv = make_qkv(n, hq, hkv)
    cs = rotary_table(64, 128)
    pos = np.array([3, 0, 63, 17, 8])
    rng = np.random.default_rng(8)
    wq, wk = rng.uniform(0.5, 1.5, D), rng.uniform(0.5, 1.5, D)
    q0, k0, v0 = P.prologue(qkv, hq, hkv, pos, cs, 128, "neox", wq, wk, 1e-6, False)
    q1, k1, v1 = P.prologue(qkv, hq, hkv, pos, cs, 128, "neox", wq, wk, 1e-6, True)
    x = P.bf16_to_double(qkv).reshape(n, hq + 2 * hkv, D)
    assert np.array_equal(v0, x[:, hq + hkv:]) and np.array_equal(v1, v0)   # V only passes through
    # without norm and rope, Q and K are the input heads
    q2, k2, _ = P.prologue(qkv, hq, hkv, pos, cs, 0, "neox", None, None, 0.0, False)
    assert np.array_equal(q2, x[:, :hq]) and np.array_equal(k2, x[:, hq:hq + hkv])
    s0 = np.einsum("nhd,ngd->nhg", q0, k0)
    s1 = np.einsum("nhd,ngd->nhg", q1, k1)
    assert np.allclose(s0, s1, atol=1e-10)
    assert not np.allclose(q0, q1)


def test_quantize_rows_scale_amax_and_zero_row():
    rng = np.random.default_rng(9)
    y = rng.standard_normal((6, D)) * rng.uniform(0.01, 30, (6, 1))
    y[2] = 0.0
    val, code, scale = P.quantize_rows(y, "e4m3")
    assert scale[2] == 1.0 and (code[2] == 0).all()
    for r in (0, 1, 3, 4, 5):
        assert np.max(np.abs(val[r])) == 448.0
        assert scale[r] == np.max(np.abs(y[r])) / 448.0
    # every stored value is within half an E4M3 step of y/scale (relative 2^-4 for normals)
    v = y / scale[:, None]
    err = np.abs(val - v)
    assert (err <= np.maximum(np.abs(v) * 2 ** -4, 2 ** -10) + 1e-12).all()
    bval, bcode, bscale = P.quantize_rows(y, "bf16")
    assert bscale is None and np.array_equal(bval, P.bf16_to_double(bcode))
    assert (np.abs(bval - y) <= np.abs(y) * 2 ** -8 + 1e-300).all()


def test_cache_writes():
    assert P.cache_writes(np.array([130, -1, 0, 63]), 64) == {0: (2, 2), 2: (0, 0), 3: (0, 63)}
