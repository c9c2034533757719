"""fp64 oracle of the fused attention prologue (test infrastructure only).

Only the test suite and ``__graft_entry__.smoke()`` may use this module; nothing on
the product path imports it, and it shares no code with the CUDA library.

What it computes, per token n and head j of the QKV projection output:

- HPC-Ops × SGLang blog, section "融合式 attention 前导": QK-Norm is applied before
  RoPE; Q leaves in FP8 with one scale per (token, head); K and V are written straight
  into the paged FP8 cache, and the quantised Q with its scales goes to the attention
  kernel as is.
- Hy3 preview write-up, §2.2.1 "Fused Rope+Norm+[Hadamard]+Quant+Store KV": the same
  element-wise chain with an optional Hadamard product, quantised online before the
  cache write; §2.6.1 "Hadamard在线旋转变换": an orthogonal rotation applied to Q and K
  before they are quantised, to spread outlier channels.

Readings where the pages are silent (each one is the plainest form of the step):

1. Input: the bf16 projection output ``qkv`` [n_tokens, (Hq + 2·Hkv)·d], heads in the
   order Q heads, K heads, V heads.
2. QK-Norm is RMSNorm over the d values of one head, y = x / sqrt(mean(x²) + eps) · w,
   with one weight vector for Q and one for K, shared by all heads.  V is not normalised.
3. RoPE takes a table ``cos_sin`` [max_position, rot]: cos in columns [0, rot/2), sin in
   [rot/2, rot).  "neox" rotates the pairs (i, i + rot/2), "interleaved" the pairs
   (2i, 2i + 1), each by the angle of row ``positions[n]``, column i; dims ≥ rot pass.
4. The Hadamard product is x ↦ H_d·x/√d with H_d the Sylvester Hadamard matrix, applied
   to the whole head vector of Q and of K after RoPE.  It is orthogonal, so it leaves
   every q·k unchanged.
5. Quantisation is per (token, head): scale = amax/448 (1 when amax = 0), stored value =
   E4M3 round-to-nearest-even of y/scale, evaluated as (y·448)/amax so that the only
   rounding before the decision is that of the quotient.  A bf16 output is the bf16
   round-to-nearest-even of y.
6. The cache slot of token n is ``slot_mapping[n]`` = page·page_size + offset; −1 means
   the token writes no K/V.  K/V scales live at [page, kv_head, offset].
"""
from __future__ import annotations

import numpy as np

import oracle

E4M3_MAX = 448.0

_E4M3_POS = None   # (values, codes) of the non-negative finite E4M3 codes, ascending
_BF16_POS = None


def _e4m3_table():
    global _E4M3_POS
    if _E4M3_POS is None:
        codes = np.arange(0, 0x7F, dtype=np.int64)          # 0x00 .. 0x7E: +0 .. 448
        vals = np.array([oracle.e4m3_to_double(int(c)) for c in codes])
        assert np.all(np.diff(vals) > 0)
        _E4M3_POS = (vals, codes)
    return _E4M3_POS


def _bf16_table():
    global _BF16_POS
    if _BF16_POS is None:
        codes = np.arange(0, 0x7F80, dtype=np.int64)        # +0 .. largest finite
        vals = bf16_to_double(codes.astype(np.uint16))
        assert np.all(np.diff(vals) > 0)
        _BF16_POS = (vals, codes)
    return _BF16_POS


def bf16_to_double(u16) -> np.ndarray:
    """bf16 bit patterns -> values: a bf16 is the high half of an IEEE binary32."""
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):                       # NaN codes stay NaN
        return u.view(np.float32).astype(np.float64)


def _round_to_table(v, table, sign_bit: int, saturate: bool):
    """Nearest representable value, ties to the even code (the code whose last mantissa
    bit is 0), looked up in the ascending table of non-negative finite values."""
    vals, codes = table
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    hi = np.clip(np.searchsorted(vals, a, side="left"), 0, len(vals) - 1)
    lo = np.clip(hi - 1, 0, None)
    d_lo = np.abs(a - vals[lo])
    d_hi = np.abs(vals[hi] - a)
    take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (codes[hi] % 2 == 0))
    idx = np.where(take_hi, hi, lo)
    over = a > vals[-1]
    if not saturate and over.any():
        raise ValueError("value beyond the format's largest finite")
    idx = np.where(over, len(vals) - 1, idx)                   # saturate at the largest
    code = codes[idx] | np.where(np.signbit(v), sign_bit, 0)
    val = np.copysign(vals[idx], v)
    return val, code


def round_e4m3(v):
    """(value, code) of E4M3 round-to-nearest-even, saturating at ±448."""
    return _round_to_table(v, _e4m3_table(), 0x80, saturate=True)


def round_bf16(v):
    """(value, code) of bf16 round-to-nearest-even (finite range only)."""
    return _round_to_table(v, _bf16_table(), 0x8000, saturate=False)


def rms_norm(x, w, eps: float):
    """RMSNorm over the last axis: x / sqrt(mean(x²) + eps) · w."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(w, dtype=np.float64)


def rope(x, positions, cos_sin, rotary_dim: int, style: str):
    """Rotary embedding over the first ``rotary_dim`` dims of the last axis.

    x: [n, heads, d]; positions: [n]; cos_sin: [max_position, rotary_dim]."""
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    if rotary_dim == 0:
        return out
    half = rotary_dim // 2
    cs = np.asarray(cos_sin, dtype=np.float64)[np.asarray(positions)]   # [n, rot]
    cos = cs[:, None, :half]
    sin = cs[:, None, half:rotary_dim]
    if style == "neox":
        a, b = x[..., :half], x[..., half:rotary_dim]
        out[..., :half] = a * cos - b * sin
        out[..., half:rotary_dim] = b * cos + a * sin
    elif style == "interleaved":
        a, b = x[..., 0:rotary_dim:2], x[..., 1:rotary_dim:2]
        out[..., 0:rotary_dim:2] = a * cos - b * sin
        out[..., 1:rotary_dim:2] = b * cos + a * sin
    else:
        raise ValueError(style)
    return out


def hadamard(x):
    """H_d·x/√d over the last axis, by the Walsh–Hadamard butterfly (Sylvester order):
    at each stride h the pair (x[i], x[i+h]) becomes (x[i] + x[i+h], x[i] − x[i+h])."""
    x = np.array(x, dtype=np.float64)
    d = x.shape[-1]
    assert d & (d - 1) == 0
    h = 1
    while h < d:
        y = x.reshape(x.shape[:-1] + (d // (2 * h), 2, h))
        a, b = y[..., 0, :].copy(), y[..., 1, :].copy()
        y[..., 0, :] = a + b
        y[..., 1, :] = a - b
        x = y.reshape(x.shape)
        h *= 2
    return x / np.sqrt(d)


def quantize_rows(y, dtype: str):
    """Per-row (last axis) output encoding.  Returns (stored values, codes, scales);
    scales are None for bf16."""
    if dtype == "bf16":
        val, code = round_bf16(y)
        return val, code.astype(np.uint16), None
    amax = np.max(np.abs(y), axis=-1, keepdims=True)
    pos = amax > 0
    scale = np.where(pos, amax / E4M3_MAX, 1.0)
    # y / scale written as (y * 448) / amax: one rounding of the exact quotient, so a value
    # exactly on a rounding midpoint (common for bf16 inputs) is decided to even
    v = np.where(pos, y * E4M3_MAX / np.where(pos, amax, 1.0), y)
    val, code = round_e4m3(v)
    return val, code.astype(np.uint8), scale[..., 0]


def prologue(qkv_u16, num_q_heads: int, num_kv_heads: int, positions, cos_sin, rotary_dim: int,
             rope_style: str, q_norm_weight, k_norm_weight, eps: float, use_hadamard: bool):
    """The chain up to (not including) the encoding: returns fp64 (q, k, v) of shapes
    [n, Hq, d], [n, Hkv, d], [n, Hkv, d]."""
    n = qkv_u16.shape[0]
    x = bf16_to_double(qkv_u16).reshape(n, num_q_heads + 2 * num_kv_heads, -1)
    q = x[:, :num_q_heads]
    k = x[:, num_q_heads:num_q_heads + num_kv_heads]
    v = x[:, num_q_heads + num_kv_heads:]
    if q_norm_weight is not None:
        q = rms_norm(q, q_norm_weight, eps)
    if k_norm_weight is not None:
        k = rms_norm(k, k_norm_weight, eps)
    q = rope(q, positions, cos_sin, rotary_dim, rope_style)
    k = rope(k, positions, cos_sin, rotary_dim, rope_style)
    if use_hadamard:
        q, k = hadamard(q), hadamard(k)
    return q, k, v.copy()


def cache_writes(slot_mapping, page_size: int):
    """{token n: (page, offset)} for every token that writes the cache."""
    out = {}
    for n, s in enumerate(np.asarray(slot_mapping).tolist()):
        if s >= 0:
            out[n] = (s // page_size, s % page_size)
    return out
