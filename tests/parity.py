"""Helpers for GPU-vs-oracle parity tests (error metrics, sampled full-size checks)."""
import numpy as np
import torch

import oracle
import workloads

# Tolerances for decode outputs against the fp64 oracle.
TOL = {"bf16": (2e-3, 1e-3), "fp8": (2e-2, 1e-2)}  # (max-abs, max per-row rel-L2)
LSE_ATOL = 1e-3


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round fp64 values once to bf16 (round to nearest even), back to fp64."""
    return torch.from_numpy(np.ascontiguousarray(x)).to(torch.bfloat16).to(torch.float64).numpy()


def errors(got: np.ndarray, ref: np.ndarray):
    """(max-abs, max over rows of ||got-ref|| / ||ref||) over the last axis; rows whose
    reference is exactly zero must match exactly (their rel error is counted as inf otherwise)."""
    got = got.astype(np.float64)
    diff = got - ref
    max_abs = float(np.abs(diff).max()) if diff.size else 0.0
    num = np.linalg.norm(diff, axis=-1)
    den = np.linalg.norm(ref, axis=-1)
    rel = np.where(den > 0, num / np.where(den > 0, den, 1), np.where(num > 0, np.inf, 0.0))
    return max_abs, float(rel.max()) if rel.size else 0.0


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |x| (8 significant bits): 2^(floor(log2|x|) - 7)."""
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.exp2(e - 7), 0.0)


def assert_close(got: np.ndarray, ref: np.ndarray, kv: str, what: str = "", round_ref: bool = True):
    """The stated tolerance: max-abs and max per-row rel-L2 against the oracle (rounded to
    bf16 first when `round_ref`, for bf16-stored outputs)."""
    atol, rtol = TOL[kv]
    r = round_bf16(ref) if round_ref else ref
    ma, rel = errors(got, r)
    assert ma <= atol and rel <= rtol, f"{what}: max-abs {ma:.3e} (<= {atol}), rel-L2 {rel:.3e} (<= {rtol})"
    return ma, rel


def assert_bf16_is_rounded(got_bf16: np.ndarray, got_fp32: np.ndarray, what: str = ""):
    """The bf16 output is the fp32 output of the same merge rounded to nearest even, bit for bit."""
    r = round_bf16(got_fp32.astype(np.float64))
    g = got_bf16.astype(np.float64)
    bad = ~((g == r) | (np.isnan(g) & np.isnan(r)))
    assert not bad.any(), f"{what}: {int(bad.sum())} bf16 outputs are not the rounded fp32 outputs"


def check_outputs(got_bf16, got_fp32, ref, kv: str, what: str = ""):
    """Gate for one decode output.  The stated tolerance (max-abs, max per-row rel-L2) applies
    to the kernels' fp32 output against the exact oracle.  A bf16-stored output cannot meet it
    against the exact value (one bf16 rounding of an O(1) output is up to 7.8e-3; a single
    rounding flip on a row's largest element is ~1.2e-3 rel-L2), so the bf16 output is checked
    to be exactly the round-to-nearest-even of that fp32 output."""
    assert_close(got_fp32, ref, kv, what + " fp32 out", round_ref=False)
    if got_bf16 is not None:
        assert_bf16_is_rounded(got_bf16, got_fp32, what + " bf16 out")


def assert_lse_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    got = got.astype(np.float64)
    inf = np.isneginf(ref)
    assert (np.isneginf(got) == inf).all(), f"{what}: -inf lse pattern differs"
    if (~inf).any():
        err = float(np.abs(got[~inf] - ref[~inf]).max())
        assert err <= LSE_ATOL, f"{what}: lse error {err:.3e}"


def problem_from_host(h: dict, inp: dict) -> oracle.Problem:
    return oracle.Problem(h["q"], h["k_pages"], h["v_pages"], h["block_table"], h["seq_lens"],
                          inp["num_q_heads"], inp["num_kv_heads"], inp["sm_scale"],
                          q_scale=h["q_scale"], k_scale=h["k_scale"], v_scale=h["v_scale"],
                          page_size=inp.get("page_size", 64), q_len=inp.get("q_len", 1),
                          kv_layout=inp.get("kv_layout", "HND"))


def np_bytes(t):
    """Host numpy copy of a tensor's exact bytes (bf16 as uint16)."""
    if t is None:
        return None
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def sub_problem(inp: dict, requests) -> oracle.Problem:
    """Oracle problem over a few requests of a (large, device-resident) workload: only their
    pages are copied to the host and renumbered (the oracle is pinned to be invariant under
    a permutation of the page pool).  Request i of the result is requests[i]."""
    requests = [int(b) for b in requests]
    lens = inp["seq_lens"][requests].cpu().numpy()
    P = inp["page_size"]
    npages = [(int(n) + P - 1) // P for n in lens]
    idx = torch.cat([inp["block_table"][b, :n] for b, n in zip(requests, npages)]).long()
    pools = {k: (None if inp[k] is None else np_bytes(inp[k].index_select(0, idx)))
             for k in ("k_pages", "v_pages", "k_scale", "v_scale")}
    new_bt = np.full((len(requests), max(max(npages), 1)), -1, np.int32)
    off = 0
    for i, n in enumerate(npages):
        new_bt[i, :n] = np.arange(off, off + n)
        off += n
    qs = None if inp["q_scale"] is None else np_bytes(inp["q_scale"][requests])
    return oracle.Problem(np_bytes(inp["q"][requests]), pools["k_pages"], pools["v_pages"], new_bt, lens,
                          inp["num_q_heads"], inp["num_kv_heads"], inp["sm_scale"], q_scale=qs,
                          k_scale=pools["k_scale"], v_scale=pools["v_scale"], page_size=P,
                          q_len=inp.get("q_len", 1), kv_layout=inp.get("kv_layout", "HND"))


# ---------------------------------------------------------------- prologue encodings
# Bound on the fp32 prologue chain's absolute error, as a fraction of the row's largest
# |value|: the sum of 128 squares, one reciprocal square root, two products (RMSNorm), two
# products and a sum (RoPE) and seven butterfly stages (Hadamard) leave a few fp32 ulps of
# the row's scale; 5e-5 leaves a wide margin and is still far below an E4M3 step (2^-4
# relative) or a bf16 step (2^-8 relative) for all but the row's tiniest values.
PROLOGUE_ERR = 5e-5


def _e4m3_lut():
    return np.array([oracle.e4m3_to_double(c) for c in range(256)])


def assert_encoded(got_codes, got_scale, y, kind: str, err_abs, what: str = ""):
    """GPU encodings of the oracle rows y [rows, 128] (fp64, before encoding).

    err_abs [rows] bounds the kernel's fp32 error in y.  A code is accepted when its value
    lies between the round-to-nearest-even of the two ends of the interval y can have
    moved in, so a rounding decision is only allowed to differ from the exact one where y
    sits within that error of a rounding midpoint; the fraction of such differences must
    stay below 1e-3.  E4M3: the scale must be amax/448 within the same error."""
    from oracle import prologue as P
    y = np.asarray(y, np.float64).reshape(-1, 128)
    E = np.asarray(err_abs, np.float64).reshape(-1, 1)
    if kind == "bf16":
        got = P.bf16_to_double(np.asarray(got_codes).view(np.uint16).reshape(-1, 128))
        lo, hi, exact = P.round_bf16(y - E)[0], P.round_bf16(y + E)[0], P.round_bf16(y)[0]
    else:
        got = _e4m3_lut()[np.asarray(got_codes).view(np.uint8).reshape(-1, 128)]
        amax = np.abs(y).max(axis=1, keepdims=True)
        s = np.where(amax > 0, amax / 448.0, 1.0)
        gs = np.asarray(got_scale, np.float64).reshape(-1, 1)
        s_tol = (E + amax * 2.0 ** -22) / 448.0
        bad_s = np.abs(gs - s) > s_tol
        assert not bad_s.any(), f"{what}: {int(bad_s.sum())} scales off (first row {int(np.argmax(bad_s))})"
        v = np.where(amax > 0, y * 448.0 / np.where(amax > 0, amax, 1.0), y)
        rel = np.where(amax > 0, E / np.where(amax > 0, amax, 1.0), 0.0) + 2.0 ** -21
        d = E / s + np.abs(v) * rel
        lo, hi, exact = P.round_e4m3(v - d)[0], P.round_e4m3(v + d)[0], P.round_e4m3(v)[0]
    ties = np.zeros(y.shape, bool)
    if kind != "bf16":
        # values exactly on an E4M3 rounding midpoint (frequent when y has few significant
        # bits, e.g. bf16 V rows): the kernel evaluates y / scale as y * (448 / amax), whose
        # last-bit rounding decides these either way, so both neighbours count as exact
        tv, _ = P._e4m3_table()
        mids = (tv[:-1] + tv[1:]) / 2
        ties = np.isin(np.abs(v), mids)
    bad = ~((got >= lo) & (got <= hi))
    if bad.any():
        r, c = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} codes outside the rounding interval; row {r} dim {c}: "
                             f"got {got[r, c]!r}, allowed [{lo[r, c]!r}, {hi[r, c]!r}]")
    flips = float(np.mean((got != exact) & ~ties))
    assert flips < 1e-3, f"{what}: {flips:.2e} of the codes differ from the exact rounding"
    return flips
