"""Page sizes 16 / 32 / 64 and the HND / NHD page layouts on the GPU vs the fp64 oracle.

A serving runtime's paged KV store comes in its own page size and dimension order (HPC-Ops ×
SGLang blog, "从 HPC-Ops kernel 到 SGLang": the attention kernel reads that store as it is).
The kernels keep the 64-token tile; a tile spans 64 / P pages, each loaded by its own
tensor-map box.  Checked here: outputs and LSEs against the oracle for every (P, layout,
KV dtype); bit-identical partials when the same tokens are re-paged into another page size
and layout; page-id checks per sub-page; the multi-token, split-KV and fused paths.
"""
import numpy as np
import pytest
import torch

import workloads
from tests import parity

pytestmark = pytest.mark.gpu

LAYOUTS = [(16, "HND"), (16, "NHD"), (32, "HND"), (32, "NHD"), (64, "NHD")]
LENS = [1, 15, 16, 17, 33, 64, 65, 100, 700, 2049, 0, 4000]


@pytest.fixture(scope="module")
def dsa():
    import load_balanced_paged_gb300 as m
    return m


def sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


def make(lens, hq, hkv, kv, page, layout, seed=0, q_len=1):
    return workloads.make_inputs(np.asarray(lens), hq, hkv, kv, seed=seed, device="cuda", page_size=page,
                                 kv_layout=layout, q_len=q_len)


def oracle_of(inp):
    return parity.problem_from_host(workloads.host_view(inp), inp)


def repage(inp, page, layout, seed):
    """The same tokens (and FP8 scales) moved into randomly placed pages of `page` tokens in
    `layout`; inp holds 64-token HND pages."""
    lens = inp["seq_lens"].cpu().numpy()
    bt = inp["block_table"].cpu().numpy()
    src_pg, src_sl, owner = [], [], []
    for b, n in enumerate(lens):
        for j in range(-(-int(n) // page)):
            t = np.minimum(np.arange(j * page, (j + 1) * page), n - 1)
            src_pg.append(bt[b, t // 64])
            src_sl.append(t % 64)
            owner.append((b, j))
    npages = len(owner)
    perm = np.random.default_rng(seed).permutation(npages)
    new_bt = np.full((len(lens), max(1, max(-(-int(n) // page) for n in lens))), -1, np.int32)
    for i, (b, j) in enumerate(owner):
        new_bt[b, j] = perm[i]
    dev = inp["k_pages"].device
    where = torch.from_numpy(np.argsort(perm)).to(dev)  # new page id -> row of the gathered pool
    pg = torch.from_numpy(np.stack(src_pg).astype(np.int64)).to(dev)[where]
    sl = torch.from_numpy(np.stack(src_sl).astype(np.int64)).to(dev)[where]
    out = dict(inp)
    for name in ("k_pages", "v_pages"):
        x = inp[name][pg, :, sl, :]  # [pages, P, Hkv, d]
        out[name] = (x if layout == "NHD" else x.permute(0, 2, 1, 3)).contiguous()
    for name in ("k_scale", "v_scale"):
        if inp[name] is not None:
            out[name] = inp[name][pg, :, sl].permute(0, 2, 1).contiguous()  # [pages, Hkv, P]
    out["block_table"] = torch.from_numpy(new_bt).to(dev)
    out.update(num_pages=npages, max_pages=new_bt.shape[1], page_size=page, kv_layout=layout)
    return out


@pytest.mark.parametrize("page,layout", LAYOUTS)
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("hq,hkv,C,m", [(32, 4, 5, 1), (64, 8, None, 4), (8, 8, 300, 1)])
def test_layout_vs_oracle(dsa, page, layout, kv, hq, hkv, C, m):
    inp = make(LENS, hq, hkv, kv, page, layout, seed=page + hq)
    C = sm_count() if C is None else C
    out32, lse, tm, po, pl = dsa.attention(inp, C, min_tiles_per_split=m, out_dtype=torch.float32)
    out16 = dsa.combine(tm, po, pl, hq, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert dsa.get_status(tm) == 0  # block-table entries past a request's pages are never read
    ref, ref_lse = oracle_of(inp).attention()
    what = f"P {page} {layout} {kv} C {C}"
    parity.check_outputs(out16.float().cpu().numpy(), out32.cpu().numpy(), ref, kv, what)
    parity.assert_lse_close(lse.cpu().numpy(), ref_lse, what)


@pytest.mark.parametrize("page,layout", LAYOUTS)
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_repaged_tokens_give_the_same_bits(dsa, page, layout, kv):
    """Only the token order within a request matters: partials are bit-identical."""
    base = make(LENS, 64, 8, kv, 64, "HND", seed=11)
    other = repage(base, page, layout, seed=page)
    C = sm_count()
    a = dsa.attention(base, C, min_tiles_per_split=2, out_dtype=torch.float32)
    b = dsa.attention(other, C, min_tiles_per_split=2, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert dsa.get_status(a[2]) == 0 and dsa.get_status(b[2]) == 0
    nd = len(a[2].host()["descs"])  # slots past the descriptors are never written
    assert nd == len(b[2].host()["descs"])
    for x, y in ((a[0], b[0]), (a[1], b[1]), (a[3][:nd], b[3][:nd]), (a[4][:nd], b[4][:nd])):
        assert torch.equal(x, y)


@pytest.mark.parametrize("page,layout", [(16, "NHD"), (32, "HND")])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("q_len", [2, 6])
def test_multi_token_repaged_tokens_give_the_same_bits(dsa, page, layout, kv, q_len):
    """Multi-token steps too: the same tokens in other pages give bit-identical partials."""
    base = make(LENS, 64, 8, kv, 64, "HND", seed=12, q_len=q_len)
    other = repage(base, page, layout, seed=page + q_len)
    a = dsa.attention_multi(base, 37, min_tiles_per_split=1, out_dtype=torch.float32)
    b = dsa.attention_multi(other, 37, min_tiles_per_split=1, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert dsa.get_status(a[2]) == 0 and dsa.get_status(b[2]) == 0
    nd = 2 * len(a[2].host()["descs"])  # two slots per descriptor
    for x, y in ((a[0], b[0]), (a[1], b[1]), (a[3][:nd], b[3][:nd]), (a[4][:nd], b[4][:nd])):
        assert torch.equal(x, y)


@pytest.mark.parametrize("layout", ["HND", "NHD"])
def test_bad_sub_page_is_flagged(dsa, layout):
    lens = [100, 200, 40]
    inp = make(lens, 16, 2, "bf16", 16, layout, seed=4)
    # entries past a request's last page, inside its last tile: never read, never checked
    bt = inp["block_table"]
    assert int(bt[0, 7]) == -1 and int(bt[2, 3]) == -1
    bt[0, 7] = 10 ** 6
    bt[2, 3] = -7
    out32, lse, tm, *_ = dsa.attention(inp, 7, min_tiles_per_split=1, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert dsa.get_status(tm) == 0
    inp2 = dict(inp)
    bt2 = bt.clone()
    bt2[0, 7] = -1
    bt2[2, 3] = -1
    inp2["block_table"] = bt2
    ref, _ = oracle_of(inp2).attention()
    parity.check_outputs(out32.to(torch.bfloat16).float().cpu().numpy(), out32.cpu().numpy(), ref, "bf16",
                         "garbage past the last page")
    # a page id outside the pool for the second 16-token page of request 1's second tile
    bt2[1, 5] = inp["num_pages"] + 3
    inp2["block_table"] = bt2
    _, _, tm2, *_ = dsa.attention(inp2, 7, min_tiles_per_split=1, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert dsa.get_status(tm2) & dsa.DEV_BAD_PAGE


@pytest.mark.parametrize("page,layout", [(16, "NHD"), (32, "HND"), (64, "NHD")])
@pytest.mark.parametrize("q_len,hq,hkv", [(2, 64, 8), (6, 64, 8), (3, 16, 4)])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_multi_token_layouts(dsa, page, layout, q_len, hq, hkv, kv):
    lens = [1, 40, 64, 129, 1000, 3000]
    inp = make(lens, hq, hkv, kv, page, layout, seed=q_len, q_len=q_len)
    out32, lse, tm, po, pl = dsa.attention_multi(inp, 37, min_tiles_per_split=1, out_dtype=torch.float32)
    out16 = dsa.combine_multi(q_len, tm, po, pl, hq, out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert dsa.get_status(tm) == 0
    ref, ref_lse = oracle_of(inp).attention()
    what = f"{kv} q_len {q_len} P {page} {layout}"
    parity.check_outputs(out16.float().cpu().numpy(), out32.cpu().numpy(), ref, kv, what)
    parity.assert_lse_close(lse.cpu().numpy(), ref_lse, what)


@pytest.mark.parametrize("page", [16, 32])
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_static_and_fused_small_pages(dsa, page, kv):
    lens = [1, 63, 64, 65, 127, 500, 1000, 5000]
    inp = make(lens, 64, 8, kv, page, "HND", seed=page + 1)
    ref, ref_lse = oracle_of(inp).attention()
    po, pl, S, status = dsa.static_splitkv(1, 1024, max(lens), inp["q"], inp["k_pages"], inp["v_pages"],
                                           inp["block_table"], inp["seq_lens"], 8, inp["sm_scale"],
                                           q_scale=inp["q_scale"], k_scale=inp["k_scale"], v_scale=inp["v_scale"])
    out32 = dsa.static_combine(S, po, pl, len(lens), 64, 8, out_dtype=torch.float32)
    out16 = dsa.static_combine(S, po, pl, len(lens), 64, 8)
    torch.cuda.synchronize()
    assert dsa.read_status(status) == 0
    parity.check_outputs(out16.float().cpu().numpy(), out32.cpu().numpy(), ref, kv, f"static P {page}")
    f16, flse, tm = dsa.attention_fused(inp, 40, 1)
    f32, _, _ = dsa.attention_fused(inp, 40, 1, out_dtype=torch.float32, task_map=tm)
    torch.cuda.synchronize()
    assert dsa.get_status(tm) == 0
    parity.check_outputs(f16.float().cpu().numpy(), f32.cpu().numpy(), ref, kv, f"fused P {page}")
    parity.assert_lse_close(flse.cpu().numpy(), ref_lse, f"fused P {page}")
