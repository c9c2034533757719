"""dsa_plan on the GPU vs the oracle's greedy tile walk: bit-exact task maps."""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dsa():
    import load_balanced_paged_gb300 as m
    return m


def sm_count():
    return torch.cuda.get_device_properties(0).multi_processor_count


def check_plan(dsa, lens, hkv, C, m):
    lens = np.asarray(lens, np.int32)
    seq = torch.from_numpy(lens).cuda()
    tm = dsa.plan(seq, hkv, C, min_tiles_per_split=m)
    got = tm.host()
    ref = oracle.plan(lens, hkv, C, 64, m)
    for k in ref:
        assert np.array_equal(got[k], ref[k]), (k, lens.tolist()[:8], hkv, C, m)
    return got


@pytest.mark.parametrize("name", list(workloads.WORKLOADS))
@pytest.mark.parametrize("m", [1, 4, 16])
def test_workload_maps_bit_exact(dsa, name, m):
    w = workloads.WORKLOADS[name]
    C = w.num_ctas(sm_count())
    got = check_plan(dsa, w.lengths(), w.num_kv_heads, C, m)
    assert got["meta"][3] == 0


def test_fuzz_bit_exact(dsa):
    rng = np.random.default_rng(2024)
    for _ in range(150):
        B = int(rng.integers(1, 257))
        hkv = int(rng.choice([1, 2, 4, 8]))
        lens = np.exp(rng.uniform(0, np.log(200_000), B)).astype(np.int64)
        lens[rng.random(B) < 0.1] = 0
        C = int(rng.integers(1, 321))
        m = int(rng.integers(1, 17))
        check_plan(dsa, lens, hkv, C, m)


@pytest.mark.parametrize("units,ctas", [(256, 1), (257, 600), (1024, 4000), (1025, 152), (2048, 8191),
                                         (2048, 8192), (2049, 304), (3000, 12288)])
def test_kernel_shapes_bit_exact(dsa, units, ctas):
    """Maps at the edges of each plan kernel: one warp (up to 256 units), 4 and 8 warps (1024,
    2048), the bin table at its shared-memory limit (12287 CTAs), and the block kernel beyond
    (more units, or more CTAs); lengths with empty requests and negative ones."""
    rng = np.random.default_rng(units + ctas)
    for hkv in (1, 8):
        if units % hkv:
            continue
        B = units // hkv
        lens = np.exp(rng.uniform(0, np.log(300_000), B)).astype(np.int64)
        lens[rng.random(B) < 0.15] = 0
        for m in (1, 4):
            check_plan(dsa, lens, hkv, ctas, m)
    lens = np.full(units, 100, np.int64)
    lens[units // 2] = -7
    got = check_plan(dsa, lens, 1, ctas, 2)
    assert got["meta"][3] == dsa.DEV_BAD_SEQLEN


def test_edge_cases(dsa):
    check_plan(dsa, [0, 0, 0], 2, 5, 4)            # no work
    check_plan(dsa, [1], 1, 1, 1)                  # one tile, one CTA
    check_plan(dsa, [64 * 7], 1, 300, 1)           # more CTAs than tiles
    check_plan(dsa, [5000] * 2048, 8, 152, 4)      # 16384 units, the largest map
    got = check_plan(dsa, [100, -3, 70], 2, 4, 1)  # negative length: zero tiles, status bit
    assert got["meta"][3] == dsa.DEV_BAD_SEQLEN


def test_rejects_bad_arguments(dsa):
    seq = torch.tensor([10, 20], dtype=torch.int32, device="cuda")
    with pytest.raises(dsa.DSAError) as e:
        dsa.plan(seq, 1, 4, tile=32)
    assert e.value.code == dsa.ERR_UNSUPPORTED
    with pytest.raises(dsa.DSAError) as e:
        dsa.plan(seq, 1, 4, min_tiles_per_split=0)
    assert e.value.code == dsa.ERR_INVALID_ARG
    small = dsa.TaskMap(2, 1, 4)
    small.struct.max_descs = 2
    with pytest.raises(dsa.DSAError) as e:
        dsa.plan(seq, 1, 4, task_map=small)
    assert e.value.code == dsa.ERR_BUFFER_TOO_SMALL
    with pytest.raises(dsa.DSAError) as e:
        dsa.plan(seq, 1, 5, task_map=dsa.TaskMap(2, 1, 4))  # map sized for another CTA count
    assert e.value.code == dsa.ERR_INVALID_ARG
