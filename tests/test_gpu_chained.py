"""dsa_decode_chained: the KV gather started before the layer's Q is ready (SGLang Low-Latency
Mode: Kernels and Runtime, section 2, item 1), in a chain of layers that share one task map.

Each layer has its own paged cache; per layer the fused prologue writes Q and the newest token
of every request (position len - 1) into the cache, then the decode and the combine run, all
in one stream with no synchronisation between layers.  The chained decode loads the tiles that
hold none of those newest tokens while the prologue still runs, so a tile read too early would
see the cache slot's previous contents.  Its outputs must equal the same chain run with the
plain dsa_decode bit for bit, and the fp64 oracle on the cache the prologue left.
"""
import numpy as np
import pytest
import torch

import workloads
from tests import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import load_balanced_paged_gb300 as m
    return m


def make_layers(lens, hq, hkv, kv, n_layers, seed):
    """Per layer: the cache (older tokens drawn at random) and the prologue inputs of the step's
    new token of each request, at position len - 1, whose slot is in the request's last page."""
    layers = []
    lens = np.asarray(lens)
    for layer in range(n_layers):
        inp = workloads.make_inputs(lens, hq, hkv, kv, seed=seed + layer, device="cuda")
        B = len(lens)
        pin = workloads.make_prologue_inputs(B, hq, hkv, inp["num_pages"], seed=seed + 100 + layer, device="cuda",
                                             skip_fraction=0.0, max_position=int(lens.max()) + 1)
        bt = inp["block_table"].cpu().numpy()
        pos = lens - 1
        slots = np.array([bt[b, p // 64] * 64 + p % 64 for b, p in enumerate(pos)], np.int32)
        pin["positions"] = torch.from_numpy(pos.astype(np.int32)).cuda()
        pin["slot_mapping"] = torch.from_numpy(slots).cuda()
        layers.append((inp, pin))
    return layers


def run_chain(dsa, layers, tm, chained, new_tokens=1, with_prologue=True):
    """prologue -> decode -> combine per layer, one stream; returns the fp32 outputs and LSEs."""
    outs = []
    for layer, (inp, pin) in enumerate(layers):
        hq, hkv = inp["num_q_heads"], inp["num_kv_heads"]
        fp8 = inp["kv_dtype"] == "fp8"
        B = inp["seq_lens"].shape[0]
        if with_prologue:
            qdt = torch.uint8 if fp8 else torch.bfloat16
            q = torch.empty(B, hq, 128, dtype=qdt, device="cuda")
            qs = torch.empty(B, hq, dtype=torch.float32, device="cuda") if fp8 else None
            dsa.prologue(pin["qkv"], hq, hkv, pin["slot_mapping"], inp["k_pages"], inp["v_pages"], inp["k_scale"],
                         inp["v_scale"], positions=pin["positions"], cos_sin=pin["cos_sin"],
                         q_norm_weight=pin["q_norm_weight"], k_norm_weight=pin["k_norm_weight"], hadamard=True,
                         q_dtype=qdt, q_out=q, q_scale=qs)
            inp["q"], inp["q_scale"] = q, qs
        kw = dict(q_scale=inp["q_scale"], k_scale=inp["k_scale"], v_scale=inp["v_scale"])
        args = (inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"], inp["seq_lens"], tm, inp["sm_scale"])
        if chained and layer > 0:  # the first layer's map comes from the plan just before it
            po, pl = dsa.decode_chained(new_tokens, *args, **kw)
        else:
            po, pl = dsa.decode(*args, **kw)
        lse = torch.empty(B, hq, dtype=torch.float32, device="cuda")
        out = dsa.combine(tm, po, pl, hq, out_lse=lse, out_dtype=torch.float32)
        outs.append((out, lse))
    torch.cuda.synchronize()
    assert dsa.get_status(tm) == 0
    return outs


CASES = [((1500, 64, 17, 3000, 700, 129), 64, 8, "bf16"), ((5000, 65, 640, 2), 32, 4, "fp8"),
         ((9000,) * 3 + (63,) * 5, 16, 2, "bf16")]


@pytest.mark.parametrize("lens,hq,hkv,kv", CASES)
def test_chained_layers_equal_plain_and_oracle(dsa, lens, hq, hkv, kv):
    ctas = torch.cuda.get_device_properties(0).multi_processor_count
    layers = make_layers(lens, hq, hkv, kv, n_layers=4, seed=len(lens))
    seq = layers[0][0]["seq_lens"]
    tm = dsa.plan(seq, hkv, ctas, 4)
    # the chained chain first, on caches whose newest slots still hold other values (a tile read
    # before the prologue's write would see them); then the plain chain on the same caches again
    keys = ("k_pages", "v_pages", "k_scale", "v_scale")
    snap = [{k: inp[k].clone() for k in keys if inp[k] is not None} for inp, _ in layers]
    chained = run_chain(dsa, layers, tm, chained=True)
    for (inp, _), sv in zip(layers, snap):
        for k, t in sv.items():
            inp[k].copy_(t)
    plain = run_chain(dsa, layers, tm, chained=False)
    for layer, ((o1, l1), (o2, l2)) in enumerate(zip(plain, chained)):
        assert torch.equal(o1, o2), f"layer {layer}: outputs differ from the plain decode"
        assert torch.equal(l1, l2), f"layer {layer}: LSEs differ from the plain decode"
    # the oracle on the cache and Q the prologue left for layer 2
    inp = layers[2][0]
    prob = parity.problem_from_host(workloads.host_view(inp), inp)
    ref, ref_lse = prob.attention()
    parity.assert_close(chained[2][0].cpu().numpy(), ref, kv, "chained layer 2", round_ref=False)
    parity.assert_lse_close(chained[2][1].cpu().numpy(), ref_lse, "chained layer 2 lse")


def test_chained_with_every_tile_early(dsa):
    """new_tokens = 0: nothing before the decode writes the cache, every tile may be loaded
    early; the results are still the plain decode's."""
    ctas = 40
    layers = make_layers((2000, 64, 777, 1), 32, 4, "bf16", n_layers=2, seed=9)  # Q as drawn, no prologue
    tm = dsa.plan(layers[0][0]["seq_lens"], 4, ctas, 2)
    plain = run_chain(dsa, layers, tm, chained=False, with_prologue=False)
    chained = run_chain(dsa, layers, tm, chained=True, new_tokens=0, with_prologue=False)
    for (o1, l1), (o2, l2) in zip(plain, chained):
        assert torch.equal(o1, o2) and torch.equal(l1, l2)
