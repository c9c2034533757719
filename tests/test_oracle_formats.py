"""Pins for the oracle's own bf16 and FP8-E4M3 decoders.

Checked code by code against torch's conversions (a library routine) and against
values fixed by the formats' definitions (OCP 8-bit floating point, E4M3 "fn":
bias 7, largest finite 448, no infinities, S.1111.111 = NaN).
"""
import math

import numpy as np
import torch

import oracle


def test_bf16_all_codes_match_torch():
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_double(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()


def test_bf16_spec_values():
    assert oracle.bf16_to_double(0x3F80) == 1.0
    assert oracle.bf16_to_double(0xC000) == -2.0
    assert oracle.bf16_to_double(0x0001) == 2.0 ** -133
    assert oracle.bf16_to_double(0x7F7F) == (2 - 2 ** -7) * 2.0 ** 127
    assert math.isinf(oracle.bf16_to_double(0x7F80))


def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert nan.sum() == 2  # 0x7F and 0xFF only
    assert (np.isnan(got) == nan).all()
    assert (got[~nan] == ref[~nan]).all()


def test_e4m3_spec_values():
    assert oracle.e4m3_to_double(0x7E) == 448.0
    assert oracle.e4m3_to_double(0x08) == 2.0 ** -6  # smallest normal
    assert oracle.e4m3_to_double(0x01) == 2.0 ** -9  # smallest subnormal
    assert oracle.e4m3_to_double(0x38) == 1.0
    assert oracle.e4m3_to_double(0xB8) == -1.0
    assert math.isnan(oracle.e4m3_to_double(0x7F))
    assert math.isnan(oracle.e4m3_to_double(0xFF))
    pos = [oracle.e4m3_to_double(c) for c in range(0x7F)]
    assert all(a < b for a, b in zip(pos, pos[1:]))  # strictly increasing over finite codes
