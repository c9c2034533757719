"""fp64 CPU oracle for load-balanced paged-KV decode attention (test infrastructure).

Only the test suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  It is independent of the CUDA library: the C source
``oracle.c`` decodes bf16/E4M3 by itself and restates the method from the pages
(HPC-Ops × SGLang blog, sections "Attention：变长 decode 的负载均衡" and
"围绕活跃 KV 工作进行调度"; Hy3 preview write-up, section 2.1.1).

Every function takes host numpy arrays holding the exact bytes the GPU reads
(bf16 as uint16, E4M3 as uint8) and returns fp64 results.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

BF16 = 0
E4M3 = 1

_i32p = ctypes.POINTER(ctypes.c_int32)
_f64p = ctypes.POINTER(ctypes.c_double)
_f32p = ctypes.POINTER(ctypes.c_float)
_vp = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (plain gcc, fp64, no fast-math)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-Wall", "-shared", "-fPIC", "-pthread",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB_PATH)
            L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_double.restype = ctypes.c_double
            L.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
            L.oracle_e4m3_to_double.restype = ctypes.c_double
            L.oracle_plan.argtypes = [_i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                      _i32p, _i32p, _i32p, _i32p, _i32p]
            L.oracle_plan.restype = ctypes.c_int
            L.oracle_static_num_splits.argtypes = [ctypes.c_int32] * 3
            L.oracle_static_num_splits.restype = ctypes.c_int32
            L.oracle_static_split.argtypes = [ctypes.c_int32] * 6 + [_i32p, _i32p]
            L.oracle_static_split.restype = None
            common = [_vp, ctypes.c_int32, _f32p, _vp, _vp, ctypes.c_int32, _f32p, _f32p,
                      _i32p, ctypes.c_int32, ctypes.c_int32, _i32p, ctypes.c_int32,
                      ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                      ctypes.c_double, ctypes.c_int32, ctypes.c_int32]
            L.oracle_attention_span.argtypes = common + [ctypes.c_int32, ctypes.c_int32,
                                                         ctypes.c_int64, ctypes.c_int64, _f64p, _f64p]
            L.oracle_attention_span.restype = ctypes.c_int
            L.oracle_attention.argtypes = common + [_i32p, ctypes.c_int64, ctypes.c_int32, _f64p, _f64p]
            L.oracle_attention.restype = ctypes.c_int
            L.oracle_default_threads.argtypes = []
            L.oracle_default_threads.restype = ctypes.c_int32
            L.oracle_merge.argtypes = [_f64p, _f64p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                       _f64p, _f64p]
            L.oracle_merge.restype = None
            _lib = L
    return _lib


def _p(a, ptype):
    return None if a is None else a.ctypes.data_as(ptype)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def bf16_to_double(bits: int) -> float:
    return lib().oracle_bf16_to_double(int(bits))


def e4m3_to_double(bits: int) -> float:
    return lib().oracle_e4m3_to_double(int(bits))


def max_descs(batch: int, num_kv_heads: int, num_ctas: int) -> int:
    """Upper bound on descriptors: each bin boundary splits at most one unit."""
    return batch * num_kv_heads + num_ctas - 1


def plan(seq_lens, num_kv_heads: int, num_ctas: int, tile: int = 64, min_tiles_per_split: int = 4):
    """Task map by the greedy tile walk.  Returns a dict of numpy int32 arrays:
    cta_desc_begin [C+1], descs [num_descs, 4] = (u, t0, t1, k),
    unit_partial_begin [U], unit_num_partials [U], meta [4] = (T, C_eff, num_descs, status)."""
    sl = _c(seq_lens, np.int32)
    B = int(sl.shape[0])
    U = B * num_kv_heads
    md = max(max_descs(B, num_kv_heads, num_ctas), 1)
    begin = np.zeros(num_ctas + 1, np.int32)
    descs = np.zeros((md, 4), np.int32)
    upb = np.zeros(max(U, 1), np.int32)
    unp = np.zeros(max(U, 1), np.int32)
    meta = np.zeros(4, np.int32)
    rc = lib().oracle_plan(_p(sl, _i32p), B, num_kv_heads, num_ctas, tile, min_tiles_per_split, md,
                           _p(begin, _i32p), _p(descs, _i32p), _p(upb, _i32p), _p(unp, _i32p),
                           _p(meta, _i32p))
    if rc != 0:
        raise ValueError(f"oracle_plan failed with {rc}")
    return {"cta_desc_begin": begin, "descs": descs[: meta[2]].copy(),
            "unit_partial_begin": upb[:U].copy(), "unit_num_partials": unp[:U].copy(), "meta": meta}


def static_num_splits(mode: int, param: int, max_seq_len: int) -> int:
    return int(lib().oracle_static_num_splits(mode, param, max_seq_len))


def static_split(mode: int, param: int, tile: int, num_splits: int, n_tiles: int, s: int):
    a = ctypes.c_int32()
    b = ctypes.c_int32()
    lib().oracle_static_split(mode, param, tile, num_splits, n_tiles, s, ctypes.byref(a), ctypes.byref(b))
    return a.value, b.value


class Problem:
    """Host copies of one decode step's inputs (exact bytes).  q_len > 1: each request
    has q_len query tokens, q [B, q_len, Hq, d] (q_scale [B, q_len, Hq]), the last q_len
    positions of the request, each seeing the tokens up to its own position."""

    def __init__(self, q, k_pages, v_pages, block_table, seq_lens, num_q_heads, num_kv_heads,
                 sm_scale, q_scale=None, k_scale=None, v_scale=None, head_dim=128, page_size=64, q_len=1,
                 kv_layout=0):
        self.q_dtype = E4M3 if q.dtype == np.uint8 else BF16
        self.kv_dtype = E4M3 if k_pages.dtype == np.uint8 else BF16
        self.q = np.ascontiguousarray(q)
        self.k_pages = np.ascontiguousarray(k_pages)
        self.v_pages = np.ascontiguousarray(v_pages)
        self.q_scale = _c(q_scale, np.float32)
        self.k_scale = _c(k_scale, np.float32)
        self.v_scale = _c(v_scale, np.float32)
        self.block_table = _c(block_table, np.int32)
        self.seq_lens = _c(seq_lens, np.int32)
        self.batch = int(self.seq_lens.shape[0])
        self.max_pages = int(self.block_table.shape[1]) if self.block_table.ndim == 2 else 0
        self.num_pages = int(self.k_pages.shape[0])
        self.num_q_heads = int(num_q_heads)
        self.num_kv_heads = int(num_kv_heads)
        self.head_dim = int(head_dim)
        self.page_size = int(page_size)
        self.sm_scale = float(sm_scale)
        self.q_len = int(q_len)
        self.kv_layout = 1 if kv_layout in (1, "NHD") else 0
        if self.q.size != self.batch * self.q_len * self.num_q_heads * self.head_dim:
            raise ValueError("q does not hold B x q_len x Hq x d values")
        if self.q_dtype == E4M3 and self.q_scale is None:
            raise ValueError("FP8 Q needs q_scale")
        if self.kv_dtype == E4M3 and (self.k_scale is None or self.v_scale is None):
            raise ValueError("FP8 K/V need k_scale and v_scale")

    def _common(self):
        return [self.q.ctypes.data, self.q_dtype, _p(self.q_scale, _f32p),
                self.k_pages.ctypes.data, self.v_pages.ctypes.data, self.kv_dtype,
                _p(self.k_scale, _f32p), _p(self.v_scale, _f32p),
                _p(self.block_table, _i32p), self.max_pages, self.num_pages,
                _p(self.seq_lens, _i32p), self.batch, self.num_q_heads, self.num_kv_heads,
                self.head_dim, self.page_size, self.sm_scale, self.q_len, self.kv_layout]

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def attention(self, units=None, n_threads: int = 0):
        """Unsplit attention.  Returns (out [B, Hq, d], lse [B, Hq]) in fp64, or [B, q_len,
        Hq, d] / [B, q_len, Hq] for q_len > 1; rows of units not listed are left NaN."""
        lead = (self.batch,) if self.q_len == 1 else (self.batch, self.q_len)
        out = np.full(lead + (self.num_q_heads, self.head_dim), np.nan, np.float64)
        lse = np.full(lead + (self.num_q_heads,), np.nan, np.float64)
        u = _c(units, np.int32)
        n = 0 if u is None else int(u.shape[0])
        rc = lib().oracle_attention(*self._common(), _p(u, _i32p), n, int(n_threads),
                                    _p(out, _f64p), _p(lse, _f64p))
        if rc != 0:
            raise ValueError(f"oracle_attention failed with {rc}")
        return out, lse

    def span(self, b: int, h: int, tok0: int, tok1: int):
        """Attention of the G query heads on KV head h of request b over tokens
        [tok0, tok1) (each query token further limited to its own position).  Returns
        (o [q_len*G, d], lse [q_len*G]), row i*G + g."""
        R = self.q_len * self.group
        o = np.zeros((R, self.head_dim), np.float64)
        lse = np.zeros(R, np.float64)
        rc = lib().oracle_attention_span(*self._common(), int(b), int(h), int(tok0), int(tok1),
                                         _p(o, _f64p), _p(lse, _f64p))
        if rc != 0:
            raise ValueError(f"oracle_attention_span failed with {rc}")
        return o, lse


def default_threads() -> int:
    return int(lib().oracle_default_threads())


def merge(o, lse):
    """LSE merge of partials o [n, rows, d], lse [n, rows] -> (o [rows, d], lse [rows])."""
    o = np.ascontiguousarray(o, np.float64)
    lse = np.ascontiguousarray(lse, np.float64)
    n, rows, d = o.shape
    out = np.zeros((rows, d), np.float64)
    out_lse = np.zeros(rows, np.float64)
    lib().oracle_merge(_p(o, _f64p), _p(lse, _f64p), n, rows, d, _p(out, _f64p), _p(out_lse, _f64p))
    return out, out_lse
