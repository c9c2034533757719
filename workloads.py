"""Seeded synthetic decode-step inputs shared by the tests, the smoke check and the bench.

This module draws random inputs and lays them out; it holds none of the method's
arithmetic (no tiling, scheduling, softmax or merging).  Both the CUDA path and
the CPU oracle consume the exact bytes it produces.

Draw order for a workload with seed s:
  1. lengths        numpy Generator(PCG64(s))
  2. page permutation  same numpy Generator, continued
  3. Q, then K, then V   torch.Generator(device).manual_seed(s), fp32 ~ N(0, 1),
                         cast to bf16, or quantised to FP8-E4M3 with one fp32
                         scale per (token, head) = amax / 448.

Paged layout: K/V pools are [num_pages, Hkv, page, d] (one contiguous
page x head block per (page, KV head)), scales [num_pages, Hkv, page],
Q [B, Hq, d], Q scale [B, Hq], block_table [B, max_pages] int32 with the pages of
request b in its first ceil(len_b / page) entries and -1 after them.  The pool
has exactly sum_b ceil(len_b / page) pages, randomly permuted over requests.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

HEAD_DIM = 128
PAGE = 64
E4M3_MAX = 448.0


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    description: str
    batch: int
    num_q_heads: int
    num_kv_heads: int
    kv_dtype: str  # "bf16" or "fp8"
    ctas: int | None  # persistent CTAs (bins); None = ctas_per_sm x the device's SM count
    seed: int = 0
    ctas_per_sm: int = 1

    def num_ctas(self, sm_count: int) -> int:
        return self.ctas or self.ctas_per_sm * sm_count

    def lengths(self) -> np.ndarray:
        return draw_lengths(self.name, self.batch, np.random.default_rng(self.seed))


# The five decode workloads.
WORKLOADS = {
    "tiny": Workload("tiny", "batch 4, KV lengths {17,64,200,1500}, 8 q / 1 KV head, bf16",
                     4, 8, 1, "bf16", None),
    "mixed": Workload("mixed", "batch 32, KV lengths log-uniform 128-32768, 64 q / 8 KV heads, bf16, 148 CTAs",
                      32, 64, 8, "bf16", 148),
    "long": Workload("long", "batch 1, KV length 131072, 64 q / 8 KV heads, bf16",
                     1, 64, 8, "bf16", None),
    "tail": Workload("tail", "batch 128: 127 KV lengths uniform 512-2048 plus one 65536, 64 q / 8 KV heads, bf16",
                     128, 64, 8, "bf16", None, ctas_per_sm=2),
    "fp8": Workload("fp8", "batch 64, KV lengths lognormal (mean 68k, cap 192k, min 1k), 64 q / 8 KV heads, FP8-E4M3 Q/K/V",
                    64, 64, 8, "fp8", None, ctas_per_sm=2),
}

# lognormal location chosen so that the mean after clipping to [1024, 196608] is 69632 (68k)
FP8_LOGNORMAL_MU = 10.814848
FP8_LOGNORMAL_SIGMA = 1.0


def draw_lengths(name: str, batch: int, rng: np.random.Generator) -> np.ndarray:
    if name == "tiny":
        lens = np.array([17, 64, 200, 1500], np.int64)
    elif name == "mixed":
        lens = np.floor(np.exp(rng.uniform(math.log(128), math.log(32769), batch)))
        lens = np.clip(lens, 128, 32768)
    elif name == "long":
        lens = np.array([131072], np.int64)
    elif name == "tail":
        lens = rng.integers(512, 2049, batch - 1)
        pos = int(rng.integers(0, batch))
        lens = np.insert(lens, pos, 65536)
    elif name == "fp8":
        lens = np.rint(rng.lognormal(FP8_LOGNORMAL_MU, FP8_LOGNORMAL_SIGMA, batch))
        lens = np.clip(lens, 1024, 196608)
    else:
        raise KeyError(name)
    return lens.astype(np.int32)


def _fill_normal(shape, gen, device, chunk_rows, out_fn):
    """Draw N(0,1) fp32 in row chunks along dim 0 and hand each chunk to out_fn."""
    rows = shape[0]
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=gen, device=device, dtype=torch.float32)
        out_fn(r0, r1, x)


def _quantize_e4m3(x: torch.Tensor):
    """Per-row (last dim) symmetric E4M3 quantisation: scale = amax / 448."""
    amax = x.abs().amax(dim=-1)
    scale = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    q = (x / scale.unsqueeze(-1)).clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return q.view(torch.uint8), scale


def make_inputs(lengths, num_q_heads: int, num_kv_heads: int, kv_dtype: str = "bf16",
                seed: int = 0, device="cpu", head_dim: int = HEAD_DIM, page_size: int = PAGE,
                rng: np.random.Generator | None = None, chunk_pages: int = 2048, q_len: int = 1,
                kv_layout: str = "HND") -> dict:
    """Build one decode step's inputs on `device`.

    `rng` continues the numpy stream used for the lengths (draw order above); if
    None a fresh Generator(seed) is used for the page permutation.  q_len > 1 gives
    each request q_len query tokens (a multi-token verify step): Q [B, q_len, Hq, d]
    (Q scale [B, q_len, Hq]), drawn in that order from the same stream.  kv_layout "NHD"
    stores each page token-major, [num_pages, page, Hkv, d] (the values drawn as for "HND",
    then transposed); the FP8 scales stay [num_pages, Hkv, page].
    """
    lens = np.asarray(lengths, np.int64)
    B = int(lens.shape[0])
    if rng is None:
        rng = np.random.default_rng(seed)
    pages_per_req = (np.maximum(lens, 0) + page_size - 1) // page_size
    num_pages = int(pages_per_req.sum())
    max_pages = max(int(pages_per_req.max()) if B else 0, 1)
    perm = rng.permutation(num_pages).astype(np.int32)
    bt = np.full((max(B, 1), max_pages), -1, np.int32)[:B]
    off = 0
    for b in range(B):
        n = int(pages_per_req[b])
        bt[b, :n] = perm[off:off + n]
        off += n

    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    fp8 = kv_dtype == "fp8"
    pool_pages = max(num_pages, 1)
    out = {
        "seq_lens": torch.from_numpy(lens.astype(np.int32)).to(device),
        "block_table": torch.from_numpy(np.ascontiguousarray(bt)).to(device),
        "num_pages": num_pages,
        "max_pages": max_pages,
        "num_q_heads": num_q_heads,
        "num_kv_heads": num_kv_heads,
        "head_dim": head_dim,
        "page_size": page_size,
        "kv_dtype": kv_dtype,
        "kv_layout": kv_layout,
        "sm_scale": 1.0 / math.sqrt(head_dim),
        "q_len": q_len,
    }
    # Q
    qshape = (B, num_q_heads, head_dim) if q_len == 1 else (B, q_len, num_q_heads, head_dim)
    qf = torch.randn(qshape, generator=gen, device=device, dtype=torch.float32)
    if fp8:
        out["q"], out["q_scale"] = _quantize_e4m3(qf)
    else:
        out["q"], out["q_scale"] = qf.to(torch.bfloat16), None
    # K then V, drawn in page chunks to bound the fp32 intermediate
    shape = (pool_pages, num_kv_heads, page_size, head_dim)
    for name in ("k", "v"):
        if fp8:
            pool = torch.empty(shape, dtype=torch.uint8, device=device)
            scale = torch.empty(shape[:3], dtype=torch.float32, device=device)

            def put(r0, r1, x, pool=pool, scale=scale):
                qq, ss = _quantize_e4m3(x)
                pool[r0:r1] = qq
                scale[r0:r1] = ss
            _fill_normal(shape, gen, device, chunk_pages, put)
            out[name + "_pages"], out[name + "_scale"] = pool, scale
        else:
            pool = torch.empty(shape, dtype=torch.bfloat16, device=device)

            def put(r0, r1, x, pool=pool):
                pool[r0:r1] = x.to(torch.bfloat16)
            _fill_normal(shape, gen, device, chunk_pages, put)
            out[name + "_pages"], out[name + "_scale"] = pool, None
    if kv_layout == "NHD":
        for name in ("k_pages", "v_pages"):
            out[name] = out[name].permute(0, 2, 1, 3).contiguous()
    return out


def make_workload(name: str, device="cpu", seed: int | None = None, max_requests: int | None = None) -> dict:
    """The named workload; max_requests keeps only its first requests (small profiling cases)."""
    w = WORKLOADS[name]
    s = w.seed if seed is None else seed
    rng = np.random.default_rng(s)
    lens = draw_lengths(w.name, w.batch, rng)
    if max_requests is not None:
        lens = lens[:max_requests]
    inp = make_inputs(lens, w.num_q_heads, w.num_kv_heads, w.kv_dtype, s, device, rng=rng)
    inp["workload"] = w
    return inp


def kv_bytes(lengths, num_kv_heads: int, kv_dtype: str, head_dim: int = HEAD_DIM) -> int:
    """Algorithmic KV bytes of one decode step: every valid token's K and V row
    of every KV head read once (plus its two fp32 scales for FP8)."""
    per = 2 * head_dim * 2 if kv_dtype == "bf16" else 2 * head_dim + 2 * 4
    return int(np.maximum(np.asarray(lengths, np.int64), 0).sum()) * num_kv_heads * per


def host_view(inp: dict) -> dict:
    """Numpy copies of the exact bytes (bf16 as uint16, E4M3 as uint8)."""
    def np_bytes(t):
        if t is None:
            return None
        t = t.detach().cpu().contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.numpy()
    keys = ("q", "q_scale", "k_pages", "v_pages", "k_scale", "v_scale", "block_table", "seq_lens")
    return {k: np_bytes(inp[k]) for k in keys}


def rotary_table(max_position: int, rotary_dim: int, theta: float = 10000.0) -> np.ndarray:
    """The usual RoPE cos/sin table [max_position, rotary_dim] as fp32: column i <
    rotary_dim/2 holds cos(p * theta^(-2i/rotary_dim)), column rotary_dim/2 + i its sin.
    An input of the prologue (a model constant), computed once here in fp64."""
    inv = theta ** (-np.arange(0, rotary_dim, 2, dtype=np.float64) / rotary_dim)
    ang = np.arange(max_position, dtype=np.float64)[:, None] * inv[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def make_prologue_inputs(n_tokens: int, num_q_heads: int, num_kv_heads: int, num_pages: int, seed: int = 0,
                         device="cpu", rotary_dim: int = 128, max_position: int = 8192,
                         skip_fraction: float = 0.1, outlier_channels: int = 4) -> dict:
    """Inputs of the fused prologue for n_tokens tokens.

    Draw order: numpy Generator(PCG64(seed)) gives the positions (uniform in
    [0, max_position)), distinct cache slots in [0, num_pages * 64) with a fraction
    set to -1 (tokens that write no K/V), and the outlier channels; then
    torch.Generator(device).manual_seed(seed) gives qkv ~ N(0, 1) with the outlier
    channels of every Q/K head scaled by 20 (the outliers a Hadamard rotation spreads),
    cast to bf16, and the Q/K norm weights ~ U(0.5, 1.5) in fp32."""
    rng = np.random.default_rng(seed)
    positions = rng.integers(0, max_position, n_tokens).astype(np.int32)
    slots = rng.choice(num_pages * PAGE, n_tokens, replace=False).astype(np.int32)
    slots[rng.random(n_tokens) < skip_fraction] = -1
    chans = rng.choice(HEAD_DIM, outlier_channels, replace=False)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    H = num_q_heads + 2 * num_kv_heads
    x = torch.randn((n_tokens, H, HEAD_DIM), generator=gen, device=device, dtype=torch.float32)
    x[:, :num_q_heads + num_kv_heads, torch.as_tensor(chans, device=device)] *= 20.0
    qw = torch.rand(HEAD_DIM, generator=gen, device=device, dtype=torch.float32) + 0.5
    kw = torch.rand(HEAD_DIM, generator=gen, device=device, dtype=torch.float32) + 0.5
    return {
        "qkv": x.reshape(n_tokens, H * HEAD_DIM).to(torch.bfloat16).contiguous(),
        "positions": torch.from_numpy(positions).to(device),
        "slot_mapping": torch.from_numpy(slots).to(device),
        "cos_sin": torch.from_numpy(rotary_table(max_position, rotary_dim)).to(device),
        "q_norm_weight": qw,
        "k_norm_weight": kw,
        "num_q_heads": num_q_heads,
        "num_kv_heads": num_kv_heads,
        "num_pages": num_pages,
        "rotary_dim": rotary_dim,
    }

