"""Dense brute-force attention for pinning the oracle (tests only).

Decodes bytes with torch's own bf16 / float8_e4m3fn conversions (not the
oracle's decoders), gathers each request's K/V rows densely through the block
table, and applies scipy's softmax / logsumexp to the full score matrix.
"""
import numpy as np
import torch
from scipy.special import logsumexp, softmax


def decode_bf16(u16: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(u16).view(np.int16)).view(torch.bfloat16)
    return t.to(torch.float64).numpy()


def decode_e4m3(u8: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.ascontiguousarray(u8)).view(torch.float8_e4m3fn)
    return t.to(torch.float64).numpy()


def values(h: dict, key: str) -> np.ndarray:
    a = h[key]
    return decode_e4m3(a) if a.dtype == np.uint8 else decode_bf16(a)


def hnd_pools(h: dict, layout: str = "HND"):
    """Decoded K and V pools as [num_pages, Hkv, page, d] (scales applied); an NHD pool
    [num_pages, page, Hkv, d] is transposed first.  Scales are [num_pages, Hkv, page]."""
    k = values(h, "k_pages")
    v = values(h, "v_pages")
    if layout == "NHD":
        k, v = k.transpose(0, 2, 1, 3), v.transpose(0, 2, 1, 3)
    if h.get("k_scale") is not None:
        k = k * h["k_scale"].astype(np.float64)[..., None]
        v = v * h["v_scale"].astype(np.float64)[..., None]
    return k, v


def dense_attention(h: dict, num_q_heads: int, num_kv_heads: int, sm_scale: float, page: int = 64,
                    layout: str = "HND"):
    q = values(h, "q")
    if h.get("q_scale") is not None:
        q = q * h["q_scale"].astype(np.float64)[..., None]
    k, v = hnd_pools(h, layout)
    B = h["seq_lens"].shape[0]
    G = num_q_heads // num_kv_heads
    d = q.shape[-1]
    out = np.zeros((B, num_q_heads, d))
    lse = np.full((B, num_q_heads), -np.inf)
    for b in range(B):
        n = int(h["seq_lens"][b])
        if n <= 0:
            continue
        pages = h["block_table"][b, : (n + page - 1) // page]
        kb = k[pages].transpose(1, 0, 2, 3).reshape(num_kv_heads, -1, d)[:, :n]  # [Hkv, n, d]
        vb = v[pages].transpose(1, 0, 2, 3).reshape(num_kv_heads, -1, d)[:, :n]
        for j in range(num_q_heads):
            s = sm_scale * (kb[j // G] @ q[b, j])
            out[b, j] = softmax(s) @ vb[j // G]
            lse[b, j] = logsumexp(s)
    return out, lse


def dense_attention_multi(h: dict, num_q_heads: int, num_kv_heads: int, sm_scale: float, q_len: int,
                          page: int = 64, layout: str = "HND"):
    """q [B, q_len, Hq, d]: query token i of request b (length n) stands at position
    n - q_len + i and sees the tokens t <= that position; the score matrix of each
    (request, query head) is masked to that causal pattern before scipy's softmax and
    logsumexp."""
    q = values(h, "q").reshape(-1, q_len, num_q_heads, h["q"].shape[-1])
    if h.get("q_scale") is not None:
        q = q * h["q_scale"].astype(np.float64).reshape(q.shape[:3])[..., None]
    k, v = hnd_pools(h, layout)
    B = h["seq_lens"].shape[0]
    G = num_q_heads // num_kv_heads
    d = q.shape[-1]
    out = np.zeros((B, q_len, num_q_heads, d))
    lse = np.full((B, q_len, num_q_heads), -np.inf)
    for b in range(B):
        n = int(h["seq_lens"][b])
        if n <= 0:
            continue
        pages = h["block_table"][b, : (n + page - 1) // page]
        kb = k[pages].transpose(1, 0, 2, 3).reshape(num_kv_heads, -1, d)[:, :n]
        vb = v[pages].transpose(1, 0, 2, 3).reshape(num_kv_heads, -1, d)[:, :n]
        t = np.arange(n)
        for i in range(q_len):
            visible = t <= n - q_len + i
            if not visible.any():
                continue
            for j in range(num_q_heads):
                s = sm_scale * (kb[j // G] @ q[b, i, j])
                s = np.where(visible, s, -np.inf)
                out[b, i, j] = softmax(s) @ vb[j // G]
                lse[b, i, j] = logsumexp(s)
    return out, lse
