"""dsa_prologue on the GPU vs the fp64 prologue oracle: Q rows, cache rows and scales.

The encodings are compared with the rounding-interval rule of ``parity.assert_encoded``;
V rows, which go through no arithmetic, must be the exact rounding of the input.  Slots
that no token maps to must keep their old contents.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import prologue as P
from tests.parity import PROLOGUE_ERR, assert_encoded, check_outputs, problem_from_host

pytestmark = pytest.mark.gpu

D = 128
EPS = 1e-6
SENTINEL_BF16 = 3.0
SENTINEL_U8 = 0x5A
SENTINEL_SCALE = -7.0


@pytest.fixture(scope="module")
def dsa():
    import load_balanced_paged_gb300 as m
    return m


def host_u16(t):
    return t.cpu().view(torch.int16).numpy().view(np.uint16)


def empty_cache(num_pages, hkv, kind, page=64, layout="HND"):
    """num_pages pages of 64 tokens' worth of slots, held in pages of `page` tokens."""
    num_pages = num_pages * 64 // page
    shape = (num_pages, page, hkv, D) if layout == "NHD" else (num_pages, hkv, page, D)
    if kind == "bf16":
        kp = torch.full(shape, SENTINEL_BF16, dtype=torch.bfloat16, device="cuda")
        vp = torch.full(shape, SENTINEL_BF16, dtype=torch.bfloat16, device="cuda")
        return kp, vp, None, None
    kp = torch.full(shape, SENTINEL_U8, dtype=torch.uint8, device="cuda")
    vp = torch.full(shape, SENTINEL_U8, dtype=torch.uint8, device="cuda")
    ks = torch.full((num_pages, hkv, page), SENTINEL_SCALE, dtype=torch.float32, device="cuda")
    vs = torch.full((num_pages, hkv, page), SENTINEL_SCALE, dtype=torch.float32, device="cuda")
    return kp, vp, ks, vs


def run(dsa, n, hq, hkv, q_kind, kv_kind, rot, style, norm, had, seed=0, max_position=4096, page=64,
        layout="HND"):
    num_pages = math.ceil(n / 64) + 3
    inp = workloads.make_prologue_inputs(n, hq, hkv, num_pages, seed=seed, device="cuda",
                                         rotary_dim=rot or 128, max_position=max_position)
    inp["page_size"], inp["kv_layout"] = page, layout
    kp, vp, ks, vs = empty_cache(num_pages, hkv, kv_kind, page, layout)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, qs = dsa.prologue(inp["qkv"], hq, hkv, inp["slot_mapping"], kp, vp, ks, vs,
                         positions=inp["positions"] if rot else None,
                         cos_sin=inp["cos_sin"] if rot else None, rotary_dim=rot, rope_style=style,
                         q_norm_weight=inp["q_norm_weight"] if norm else None,
                         k_norm_weight=inp["k_norm_weight"] if norm else None, eps=EPS, hadamard=had,
                         q_dtype=torch.uint8 if q_kind == "e4m3" else torch.bfloat16, status=status,
                         kv_layout=layout)
    torch.cuda.synchronize()
    assert dsa.read_status(status) == 0
    return inp, (q, qs, kp, vp, ks, vs)


def check(inp, got, q_kind, kv_kind, rot, style, norm, had, what):
    q, qs, kp, vp, ks, vs = got
    hq, hkv = inp["num_q_heads"], inp["num_kv_heads"]
    qw = inp["q_norm_weight"].cpu().numpy().astype(np.float64) if norm else None
    kw = inp["k_norm_weight"].cpu().numpy().astype(np.float64) if norm else None
    q64, k64, v64 = P.prologue(host_u16(inp["qkv"]), hq, hkv, inp["positions"].cpu().numpy(),
                               inp["cos_sin"].cpu().numpy(), rot, style, qw, kw, EPS, had)
    n = q64.shape[0]

    def err(y):
        return PROLOGUE_ERR * np.abs(y.reshape(-1, D)).max(axis=1)

    def codes(t):
        return host_u16(t) if t.dtype == torch.bfloat16 else t.cpu().numpy()

    assert_encoded(codes(q), None if qs is None else qs.cpu().numpy(), q64, q_kind, err(q64), what + " Q")
    slots = inp["slot_mapping"].cpu().numpy()
    page, nhd = inp.get("page_size", 64), inp.get("kv_layout", "HND") == "NHD"
    writes = P.cache_writes(slots, page)
    toks = np.array(sorted(writes), dtype=np.int64)
    pages = np.array([writes[t][0] for t in toks], dtype=np.int64)
    offs = np.array([writes[t][1] for t in toks], dtype=np.int64)
    kc, vc = codes(kp), codes(vp)                         # [pages, hkv, P, D] or [pages, P, hkv, D]
    if nhd:
        gk, gv = kc[pages, offs], vc[pages, offs]         # [tokens, hkv, D]
    else:
        gk, gv = kc[pages, :, offs], vc[pages, :, offs]
    gks = None if ks is None else ks.cpu().numpy()[pages, :, offs]
    gvs = None if vs is None else vs.cpu().numpy()[pages, :, offs]
    assert_encoded(gk, gks, k64[toks], kv_kind, err(k64[toks]), what + " K")
    assert_encoded(gv, gvs, v64[toks], kv_kind, np.zeros(len(toks) * hkv), what + " V")
    if kv_kind == "bf16":   # no arithmetic on V: the bf16 input bits come back unchanged
        x = host_u16(inp["qkv"]).reshape(n, hq + 2 * hkv, D)[toks, hq + hkv:]
        assert np.array_equal(gv, x)
    # slots no token maps to keep their old contents
    untouched = np.ones(kc.shape[0] * page, bool)
    untouched[pages * page + offs] = False
    sent = np.uint16(0x4040) if kv_kind == "bf16" else np.uint8(SENTINEL_U8)
    for c in (kc, vc):
        rest = (c if nhd else c.transpose(0, 2, 1, 3)).reshape(-1, hkv, D)[untouched]
        assert (rest == sent).all()
    for s_ in (ks, vs):
        if s_ is not None:
            rest = s_.cpu().numpy().transpose(0, 2, 1).reshape(-1, hkv)[untouched]
            assert (rest == SENTINEL_SCALE).all()
    return len(toks)


CASES = [
    # n, Hq, Hkv, Q, KV, rotary_dim, style, QK-Norm, Hadamard
    (37, 8, 1, "bf16", "bf16", 128, "neox", True, False),
    (37, 64, 8, "e4m3", "e4m3", 128, "neox", True, True),
    (50, 16, 2, "e4m3", "bf16", 64, "interleaved", True, False),
    (20, 8, 2, "bf16", "e4m3", 32, "neox", False, True),
    (9, 4, 4, "e4m3", "e4m3", 0, "neox", True, False),
    (64, 32, 4, "bf16", "bf16", 16, "interleaved", False, True),
    (129, 8, 8, "e4m3", "e4m3", 128, "interleaved", True, True),
    (40, 8, 1, "e4m3", "bf16", 64, "neox", True, True),
    (12, 8, 2, "bf16", "bf16", 16, "neox", True, False),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_prologue_vs_oracle(dsa, case):
    n, hq, hkv, qk, kvk, rot, style, norm, had = case
    inp, got = run(dsa, n, hq, hkv, qk, kvk, rot, style, norm, had, seed=n)
    written = check(inp, got, qk, kvk, rot, style, norm, had, str(case))
    assert written > 0


@pytest.mark.parametrize("page,layout", [(16, "HND"), (16, "NHD"), (32, "NHD"), (64, "NHD")])
@pytest.mark.parametrize("kinds", [("e4m3", "e4m3"), ("bf16", "bf16")])
def test_prologue_page_layouts(dsa, page, layout, kinds):
    """Cache writes into pages of 16 / 32 / 64 tokens in either layout."""
    inp, got = run(dsa, 300, 16, 4, kinds[0], kinds[1], 128, "neox", True, True, seed=page, page=page,
                   layout=layout)
    check(inp, got, kinds[0], kinds[1], 128, "neox", True, True, f"P {page} {layout}")


@pytest.mark.parametrize("n", [2048, 4097])
@pytest.mark.parametrize("kinds", [("e4m3", "e4m3"), ("bf16", "bf16")])
def test_prologue_prefill_size(dsa, kinds, n):
    # 2048 tokens x 80 heads: enough work items for blocks of 8 heads per warp and several
    # grid-stride passes; 4097 tokens: the CTA shape of large batches (above 4096 tokens)
    inp, got = run(dsa, n, 64, 8, kinds[0], kinds[1], 128, "neox", True, True, seed=11)
    check(inp, got, kinds[0], kinds[1], 128, "neox", True, True, f"prefill {n}")


def test_bad_position_and_slot_set_status(dsa):
    n, hq, hkv = 8, 8, 1
    inp = workloads.make_prologue_inputs(n, hq, hkv, 2, seed=5, device="cuda", max_position=100,
                                         skip_fraction=0.0)
    inp["positions"][3] = 100                  # past the table
    inp["slot_mapping"][5] = 2 * 64            # past the pool
    kp, vp, ks, vs = empty_cache(2, hkv, "e4m3")
    q = torch.full((n, hq, D), SENTINEL_U8, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    dsa.prologue(inp["qkv"], hq, hkv, inp["slot_mapping"], kp, vp, ks, vs, positions=inp["positions"],
                 cos_sin=inp["cos_sin"], q_norm_weight=inp["q_norm_weight"], k_norm_weight=inp["k_norm_weight"],
                 q_dtype=torch.uint8, q_out=q, status=status)
    st = dsa.read_status(status)
    assert st == dsa.DEV_BAD_POSITION | dsa.DEV_BAD_PAGE
    qh = q.cpu().numpy()
    assert (qh[3] == SENTINEL_U8).all()                       # token 3: no Q
    assert not (qh[np.arange(n) != 3] == SENTINEL_U8).all(axis=(1, 2)).any()
    s3 = int(inp["slot_mapping"][3])
    kh, vh = kp.cpu().numpy(), vp.cpu().numpy()
    assert (kh[s3 // 64, :, s3 % 64] == SENTINEL_U8).all()    # token 3: no K ...
    assert not (vh[s3 // 64, :, s3 % 64] == SENTINEL_U8).all()  # ... but its V is written
    writes = int((kh != SENTINEL_U8).any(axis=(1, 3)).sum())
    assert writes == n - 2                                    # tokens 3 and 5 wrote no K


def test_host_validation(dsa):
    inp = workloads.make_prologue_inputs(4, 8, 1, 1, device="cuda")
    kp, vp, ks, vs = empty_cache(1, 1, "bf16")
    args = dict(positions=inp["positions"], cos_sin=inp["cos_sin"])
    with pytest.raises(dsa.DSAError) as e:
        dsa.prologue(inp["qkv"], 8, 1, inp["slot_mapping"], kp, vp, rotary_dim=48, **args)
    assert e.value.code == dsa.ERR_UNSUPPORTED
    with pytest.raises(dsa.DSAError) as e:
        dsa.prologue(inp["qkv"], 8, 1, inp["slot_mapping"], kp, vp, eps=-1.0, **args)
    assert e.value.code == dsa.ERR_INVALID_ARG
    with pytest.raises(dsa.DSAError) as e:     # FP8 cache without scales
        k8, v8, _, _ = empty_cache(1, 1, "e4m3")
        dsa.prologue(inp["qkv"], 8, 1, inp["slot_mapping"], k8, v8, **args)
    assert e.value.code == dsa.ERR_INVALID_ARG
    with pytest.raises(dsa.DSAError) as e:     # pages of 8 tokens
        k8, v8, _, _ = empty_cache(1, 1, "bf16", page=8)
        dsa.prologue(inp["qkv"], 8, 1, inp["slot_mapping"], k8, v8, **args)
    assert e.value.code == dsa.ERR_UNSUPPORTED
    q, _ = dsa.prologue(inp["qkv"][:0], 8, 1, inp["slot_mapping"][:0], kp, vp, **args)   # no tokens
    assert q.shape[0] == 0


@pytest.mark.parametrize("page,layout", [(64, "HND"), (16, "NHD"), (32, "HND")])
def test_prologue_feeds_decode(dsa, page, layout):
    """The prologue writes each request's newest token (Q, and K/V at its cache slot) into
    an FP8 decode step; the step's output matches the oracle on the bytes it read."""
    lens = [17, 64, 200, 1500, 1]
    hq, hkv = 16, 2
    inp = workloads.make_inputs(lens, hq, hkv, "fp8", seed=21, device="cuda", page_size=page, kv_layout=layout)
    B = len(lens)
    bt = inp["block_table"].cpu().numpy()
    pos = np.array([L - 1 for L in lens], np.int32)
    slots = np.array([bt[b, p // page] * page + p % page for b, p in enumerate(pos)], np.int32)
    pro = workloads.make_prologue_inputs(B, hq, hkv, 1, seed=22, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, qs = dsa.prologue(pro["qkv"], hq, hkv, torch.from_numpy(slots).cuda(), inp["k_pages"], inp["v_pages"],
                         inp["k_scale"], inp["v_scale"], positions=torch.from_numpy(pos).cuda(),
                         cos_sin=pro["cos_sin"], q_norm_weight=pro["q_norm_weight"],
                         k_norm_weight=pro["k_norm_weight"], hadamard=True, q_dtype=torch.uint8, status=status,
                         kv_layout=layout)
    assert dsa.read_status(status) == 0
    inp["q"], inp["q_scale"] = q, qs
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    out, lse, tm, po, pl = dsa.attention(inp, sms, out_dtype=torch.float32)
    out_b = dsa.combine(tm, po, pl, hq, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    ref_o, ref_lse = problem_from_host(workloads.host_view(inp), inp).attention()
    check_outputs(out_b.float().cpu().numpy(), out.cpu().numpy(), ref_o, "fp8", "prologue -> decode")
