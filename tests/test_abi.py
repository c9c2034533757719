"""The C ABI without a GPU: the library loads, exports every entry point the header
declares, and rejects bad host arguments before launching anything."""
import ctypes
import os
import re
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__._builder().build()
    return ctypes.CDLL(os.path.join(ROOT, "load_balanced_paged_gb300", "libdsa.so"))


def declared_functions():
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(dsa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("dsa_plan", "dsa_decode", "dsa_combine", "dsa_static_splitkv", "dsa_static_combine",
              "dsa_max_descs", "dsa_static_num_splits", "dsa_get_status", "dsa_read_status",
              "dsa_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_sizing_helpers(lib):
    lib.dsa_max_descs.restype = ctypes.c_int32
    assert lib.dsa_max_descs(32, 8, 148) == 32 * 8 + 147
    assert lib.dsa_max_descs(0, 8, 1) == 0
    assert lib.dsa_max_descs(1, 0, 1) == -1
    assert lib.dsa_max_descs(1 << 30, 8, 1) == -1
    lib.dsa_static_num_splits.restype = ctypes.c_int32
    assert lib.dsa_static_num_splits(0, 16, 131072) == 16
    assert lib.dsa_static_num_splits(1, 4096, 131072) == 32
    assert lib.dsa_static_num_splits(1, 4096, 4097) == 2
    assert lib.dsa_static_num_splits(1, 4096, 0) == 1
    assert lib.dsa_static_num_splits(1, 100, 1000) == -1  # chunk must be whole tiles
    assert lib.dsa_static_num_splits(2, 16, 100) == -1


class TaskMap(ctypes.Structure):
    _fields_ = [("cta_desc_begin", ctypes.c_void_p), ("descs", ctypes.c_void_p),
                ("unit_partial_begin", ctypes.c_void_p), ("unit_num_partials", ctypes.c_void_p),
                ("meta", ctypes.c_void_p), ("max_descs", ctypes.c_int32), ("num_ctas", ctypes.c_int32),
                ("num_units", ctypes.c_int32)]


def test_plan_host_checks(lib):
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: every call below fails its host checks
    tm = TaskMap(fake, fake, fake, fake, fake, 10, 4, 2)
    V = ctypes.c_void_p
    lib.dsa_plan.argtypes = [V, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                             ctypes.c_int32, ctypes.POINTER(TaskMap), V]
    assert lib.dsa_plan(fake, 2, 1, 4, 64, 4, None, None) == 1             # no map
    assert lib.dsa_plan(fake, 2, 1, 4, 32, 4, ctypes.byref(tm), None) == 2  # tile != 64
    assert lib.dsa_plan(fake, 2, 1, 4, 64, 0, ctypes.byref(tm), None) == 1  # floor < 1
    assert lib.dsa_plan(None, 2, 1, 4, 64, 4, ctypes.byref(tm), None) == 1  # no lengths
    assert lib.dsa_plan(fake, 2, 1, 5, 64, 4, ctypes.byref(tm), None) == 1  # CTA count mismatch
    tm.max_descs = 4
    assert lib.dsa_plan(fake, 2, 1, 4, 64, 4, ctypes.byref(tm), None) == 3  # too small
    assert lib.dsa_plan(fake, 20000, 1, 4, 64, 4, ctypes.byref(tm), None) == 2  # too many units


def test_decode_host_checks(lib):
    fake = ctypes.c_void_p(0x10000)
    tm = TaskMap(fake, fake, fake, fake, fake, 10, 4, 16)
    i, f, V = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p
    lib.dsa_decode.argtypes = [V, i, V, V, V, i, V, V, V, i, i, V, i, i, i, i, i, f,
                               ctypes.POINTER(TaskMap), V, V, V]

    def call(q_dt=0, kv_dt=0, hq=64, hkv=8, d=128, page=64, scales=None, batch=2, sm=0.1):
        return lib.dsa_decode(fake, q_dt, scales, fake, fake, kv_dt, scales, scales, fake, 4, 8, fake,
                              batch, hq, hkv, d, page, sm, ctypes.byref(tm), fake, fake, None)
    assert call(d=64) == 2
    assert call(page=8) == 2               # page sizes 16, 32 and 64 only
    assert call(page=48) == 2
    assert call(page=128) == 2
    assert call(hq=63) == 1
    assert call(hq=128, hkv=8) == 2        # G = 16 not built
    assert call(q_dt=0, kv_dt=1) == 2      # mixed dtypes not built
    assert call(q_dt=1, kv_dt=1) == 1      # E4M3 without scales
    assert call(sm=float("nan")) == 1
    assert call(batch=3) == 1              # map sized for another batch


def test_decode_ex_host_checks(lib):
    fake = ctypes.c_void_p(0x10000)
    tm = TaskMap(fake, fake, fake, fake, fake, 10, 4, 16)
    i, f, V = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p
    lib.dsa_decode_ex.argtypes = [i, i, V, i, V, V, V, i, V, V, V, i, i, V, i, i, i, i, i, f,
                                  ctypes.POINTER(TaskMap), V, V, V, V]

    def call(q_len=1, layout=1, kv_dt=0, hq=64, hkv=8, page=16, q_dt=0, scales=None):
        return lib.dsa_decode_ex(q_len, layout, fake, q_dt, scales, fake, fake, kv_dt, scales, scales, fake, 4, 8,
                                 fake, 2, hq, hkv, 128, page, 0.1, ctypes.byref(tm), fake, fake, None, None)
    assert call(layout=2) == 1              # not a dsa_kv_layout
    assert call(layout=-1) == 1
    assert call(page=8) == 2
    assert call(q_len=0) == 1
    assert call(q_len=9) == 2               # 9 x 8 = 72 query rows per unit
    assert call(q_len=2, kv_dt=1) == 2      # bf16 Q over E4M3 K/V not built
    assert call(q_len=2, q_dt=1, kv_dt=1) == 1  # E4M3 multi-token without scales
    misaligned = ctypes.c_void_p(0x10004)
    assert call(q_len=6, q_dt=1, kv_dt=1, scales=misaligned) == 1  # scale pools must be 16-byte aligned
    assert call(q_len=9, q_dt=1, kv_dt=1, scales=fake) == 2  # 72 query rows per unit


def test_chained_decode_host_checks(lib):
    fake = ctypes.c_void_p(0x10000)
    tm = TaskMap(fake, fake, fake, fake, fake, 10, 4, 16)
    i, f, V = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p
    lib.dsa_decode_chained.argtypes = [i, V, i, V, V, V, i, V, V, V, i, i, V, i, i, i, i, i, f,
                                       ctypes.POINTER(TaskMap), V, V, V]

    def call(new_tokens=1, d=128, page=64, hq=64, batch=2):
        return lib.dsa_decode_chained(new_tokens, fake, 0, None, fake, fake, 0, None, None, fake, 4, 8, fake, batch,
                                      hq, 8, d, page, 0.1, ctypes.byref(tm), fake, fake, None)
    assert call(new_tokens=-1) == 1
    assert call(d=64) == 2
    assert call(page=8) == 2
    assert call(hq=63) == 1
    assert call(batch=3) == 1              # map sized for another batch


def test_noalloc_host_checks(lib):
    """dsa_decode_step_noalloc refuses, before it touches the device, every argument that one
    of its three kernels' entry points would refuse, so a step is never half enqueued."""
    fake = ctypes.c_void_p(0x10000)
    i, f, V = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p
    lib.dsa_decode_step_noalloc.argtypes = [V, i, V, V, V, i, V, V, V, i, i, V, i, i, i, i, i, f,
                                            i, i, V, i, V, V, V]

    def call(out=fake, batch=2, ctas=4, floor=4, out_dt=0, hq=64, hkv=8):
        return lib.dsa_decode_step_noalloc(fake, 0, None, fake, fake, 0, None, None, fake, 4, 8, fake, batch,
                                           hq, hkv, 128, 64, 0.1, ctas, floor, out, out_dt, None, None, None)
    assert call(out=ctypes.c_void_p(0x10004)) == 1   # out not 16-byte aligned (dsa_combine's rule)
    assert call(out=None) == 1
    assert call(out_dt=1) == 2                         # E4M3 output not built
    assert call(floor=0) == 1
    assert call(ctas=0) == 1
    assert call(batch=0, ctas=2 ** 31 - 1) == 2        # above the plan's CTA limit, no overflow
    assert call(batch=4096, hkv=8, hq=64) == 2         # 32768 units: above the plan's unit limit
    assert call(batch=2048, hkv=8, hq=64) == 3         # fits the plan, not the fixed scratch


def test_status_strings(lib):
    lib.dsa_status_string.restype = ctypes.c_char_p
    assert lib.dsa_status_string(0) == b"DSA_OK"
    for code in range(1, 6):
        assert lib.dsa_status_string(code).startswith(b"DSA_ERR_")
    assert lib.dsa_status_string(99) == b"unknown dsa_status"
    lib.dsa_read_status.argtypes = [ctypes.c_void_p, ctypes.c_void_p]
    assert lib.dsa_read_status(None, None) == 1


def test_package_fails_loudly_without_library(tmp_path, lib):
    pkg = tmp_path / "load_balanced_paged_gb300"
    pkg.mkdir()
    shutil.copy(os.path.join(ROOT, "load_balanced_paged_gb300", "__init__.py"), pkg / "__init__.py")
    r = subprocess.run([sys.executable, "-c", "import load_balanced_paged_gb300"], cwd=tmp_path,
                       capture_output=True, text=True)
    assert r.returncode != 0 and "libdsa.so is missing" in r.stderr
