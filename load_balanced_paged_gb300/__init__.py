"""Python binding of libdsa: load-balanced paged-KV GQA decode attention on GB300.

Argument marshalling only: every step runs in the CUDA kernels of libdsa.so
(include/dsa.h).  PyTorch supplies device memory and streams.  There is no CPU
fallback: importing this package fails if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it first (python load_balanced_paged_gb300/build.py, or __graft_entry__.build())")

_lib = ctypes.CDLL(LIB_PATH)

# dsa_status
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_BUFFER_TOO_SMALL, ERR_CUDA, ERR_DEVICE_INPUT = range(6)
# device status bits
DEV_BAD_SEQLEN, DEV_BAD_PAGE, DEV_TIMEOUT, DEV_BAD_MAP, DEV_BAD_POSITION = 1, 2, 4, 8, 32
# dsa_rope_style
ROPE_NEOX, ROPE_INTERLEAVED = 0, 1
# dsa_dtype
BF16, FP8_E4M3, FP32 = 0, 1, 2

TILE = 64
HEAD_DIM = 128


class DSAError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {_lib.dsa_status_string(code).decode()}")


class TaskMapStruct(ctypes.Structure):
    _fields_ = [("cta_desc_begin", ctypes.c_void_p), ("descs", ctypes.c_void_p),
                ("unit_partial_begin", ctypes.c_void_p), ("unit_num_partials", ctypes.c_void_p),
                ("meta", ctypes.c_void_p), ("max_descs", ctypes.c_int32), ("num_ctas", ctypes.c_int32),
                ("num_units", ctypes.c_int32)]


_i32, _f32, _vp = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p
_TMP = ctypes.POINTER(TaskMapStruct)
_attn_args = [_vp, _i32, _vp, _vp, _vp, _i32, _vp, _vp, _vp, _i32, _i32, _vp, _i32, _i32, _i32, _i32, _i32, _f32]

_lib.dsa_max_descs.argtypes = [_i32, _i32, _i32]
_lib.dsa_max_descs.restype = _i32
_lib.dsa_plan.argtypes = [_vp, _i32, _i32, _i32, _i32, _i32, _TMP, _vp]
_lib.dsa_plan.restype = ctypes.c_int
_lib.dsa_decode.argtypes = _attn_args + [_TMP, _vp, _vp, _vp]
_lib.dsa_decode.restype = ctypes.c_int
_lib.dsa_decode_fused.argtypes = _attn_args + [_TMP, _vp, _vp, _vp, _vp, _i32, _vp, _vp]
_lib.dsa_decode_fused.restype = ctypes.c_int
_lib.dsa_combine.argtypes = [_TMP, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _i32, _vp, _vp]
_lib.dsa_combine.restype = ctypes.c_int
_lib.dsa_multi_slots_per_desc.argtypes = [_i32, _i32]
_lib.dsa_multi_slots_per_desc.restype = _i32
_lib.dsa_decode_multi.argtypes = [_i32] + _attn_args + [_TMP, _vp, _vp, _vp]
_lib.dsa_decode_multi.restype = ctypes.c_int
_lib.dsa_decode_ex.argtypes = [_i32, _i32] + _attn_args + [_TMP, _vp, _vp, _vp, _vp]
_lib.dsa_decode_ex.restype = ctypes.c_int
_lib.dsa_decode_chained.argtypes = [_i32] + _attn_args + [_TMP, _vp, _vp, _vp]
_lib.dsa_decode_chained.restype = ctypes.c_int
_lib.dsa_combine_multi.argtypes = [_i32, _TMP, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _i32, _vp, _vp]
_lib.dsa_combine_multi.restype = ctypes.c_int
_lib.dsa_static_num_splits.argtypes = [_i32, _i32, _i32]
_lib.dsa_static_num_splits.restype = _i32
_lib.dsa_static_splitkv.argtypes = [_i32, _i32, _i32] + _attn_args + [_vp, _vp, _vp, _vp, _vp]
_lib.dsa_static_splitkv.restype = ctypes.c_int
_lib.dsa_static_combine.argtypes = [_i32, _vp, _vp, _i32, _i32, _i32, _i32, _vp, _i32, _vp, _vp]
_lib.dsa_static_combine.restype = ctypes.c_int
_lib.dsa_read_status.argtypes = [_vp, ctypes.POINTER(_i32)]
_lib.dsa_read_status.restype = ctypes.c_int
_lib.dsa_get_status.argtypes = [_TMP, ctypes.POINTER(_i32)]
_lib.dsa_get_status.restype = ctypes.c_int
_lib.dsa_decode_step_noalloc.argtypes = _attn_args + [_i32, _i32, _vp, _i32, _vp, _vp, _vp]
_lib.dsa_decode_step_noalloc.restype = ctypes.c_int
_lib.dsa_selftest_wait_timeout.argtypes = [_vp, ctypes.c_int64, _vp]
_lib.dsa_selftest_wait_timeout.restype = ctypes.c_int
_lib.dsa_prologue.argtypes = [_vp, _i32, _i32, _i32, _i32, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _f32, _i32, _vp,
                              _vp, _i32, _vp, _vp, _vp, _i32, _vp, _vp, _i32, _i32, _i32, _vp, _vp]
_lib.dsa_prologue.restype = ctypes.c_int
_lib.dsa_status_string.argtypes = [ctypes.c_int]
_lib.dsa_status_string.restype = ctypes.c_char_p


def lib():
    return _lib


def _check(rc: int, what: str):
    if rc != OK:
        raise DSAError(rc, what)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dtype_code(t) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype in (torch.uint8, torch.float8_e4m3fn):
        return FP8_E4M3
    if t.dtype == torch.float32:
        return FP32
    raise TypeError(f"unsupported dtype {t.dtype}")


def max_descs(batch: int, num_kv_heads: int, num_ctas: int) -> int:
    return int(_lib.dsa_max_descs(batch, num_kv_heads, num_ctas))


class TaskMap:
    """Device buffers of one task map plus the C struct that points at them."""

    def __init__(self, batch: int, num_kv_heads: int, num_ctas: int, device="cuda"):
        md = max_descs(batch, num_kv_heads, num_ctas)
        if md < 0:
            raise DSAError(ERR_INVALID_ARG, "dsa_max_descs")
        units = batch * num_kv_heads
        i32 = dict(dtype=torch.int32, device=device)
        self.cta_desc_begin = torch.zeros(num_ctas + 1, **i32)
        self.descs = torch.zeros(max(md, 1), 4, **i32)
        self.unit_partial_begin = torch.zeros(max(units, 1), **i32)
        self.unit_num_partials = torch.zeros(max(units, 1), **i32)
        self.meta = torch.zeros(4, **i32)
        self.max_descs, self.num_ctas, self.num_units = md, num_ctas, units
        self.batch, self.num_kv_heads = batch, num_kv_heads
        self.struct = TaskMapStruct(self.cta_desc_begin.data_ptr(), self.descs.data_ptr(),
                                    self.unit_partial_begin.data_ptr(), self.unit_num_partials.data_ptr(),
                                    self.meta.data_ptr(), md, num_ctas, units)

    def unit_counters(self) -> torch.Tensor:
        """Zeroed [B*Hkv] int32 counters for dsa_decode_fused, kept with the map."""
        c = getattr(self, "_unit_counters", None)
        if c is None:
            c = torch.zeros(max(self.num_units, 1), dtype=torch.int32, device=self.meta.device)
            self._unit_counters = c
        return c

    def host(self) -> dict:
        """Copies of the map (synchronises): the same keys as the oracle's plan."""
        meta = self.meta.cpu().numpy()
        nd = int(meta[2])
        return {"cta_desc_begin": self.cta_desc_begin.cpu().numpy(),
                "descs": self.descs[:nd].cpu().numpy(),
                "unit_partial_begin": self.unit_partial_begin[:self.num_units].cpu().numpy(),
                "unit_num_partials": self.unit_num_partials[:self.num_units].cpu().numpy(),
                "meta": meta}


def plan(seq_lens: torch.Tensor, num_kv_heads: int, num_persistent_ctas: int, min_tiles_per_split: int = 4,
         tile: int = TILE, task_map: TaskMap | None = None, stream=None) -> TaskMap:
    """dsa_plan: build the step's task map on the device."""
    batch = int(seq_lens.shape[0])
    tm = task_map or TaskMap(batch, num_kv_heads, num_persistent_ctas, seq_lens.device)
    rc = _lib.dsa_plan(_ptr(seq_lens), batch, num_kv_heads, num_persistent_ctas, tile, min_tiles_per_split,
                       ctypes.byref(tm.struct), _stream(stream))
    _check(rc, "dsa_plan")
    return tm


KV_LAYOUTS = {"HND": 0, "NHD": 1}  # dsa_kv_layout


def _attn_args(q, k_pages, v_pages, block_table, seq_lens, num_kv_heads, sm_scale, q_scale, k_scale, v_scale,
               kv_layout="HND"):
    batch, hq, d = q.shape[0], q.shape[-2], q.shape[-1]
    if kv_layout == "NHD":  # [num_pages, P, Hkv, d]
        num_pages, page, hkv, d2 = k_pages.shape
    else:                   # [num_pages, Hkv, P, d]
        num_pages, hkv, page, d2 = k_pages.shape
    if hkv != num_kv_heads:
        raise ValueError("k_pages head count differs from num_kv_heads")
    return [_ptr(q), _dtype_code(q), _ptr(q_scale), _ptr(k_pages), _ptr(v_pages), _dtype_code(k_pages),
            _ptr(k_scale), _ptr(v_scale), _ptr(block_table), int(block_table.shape[1]), num_pages,
            _ptr(seq_lens), batch, hq, num_kv_heads, d, page, float(sm_scale)]


def partial_buffers(max_slots: int, group: int, device="cuda"):
    o = torch.empty(max(max_slots, 1), group, HEAD_DIM, dtype=torch.float32, device=device)
    lse = torch.empty(max(max_slots, 1), group, dtype=torch.float32, device=device)
    return o, lse


def decode(q, k_pages, v_pages, block_table, seq_lens, task_map: TaskMap, sm_scale: float,
           partial_o=None, partial_lse=None, q_scale=None, k_scale=None, v_scale=None, stream=None,
           kv_layout="HND", cta_times=None):
    """dsa_decode (dsa_decode_ex for NHD pages or per-CTA timestamps, cta_times uint64-sized
    [num_ctas, 2]): persistent kernel writing one partial (o, lse) per descriptor."""
    G = q.shape[1] // task_map.num_kv_heads
    if partial_o is None:
        partial_o, partial_lse = partial_buffers(task_map.max_descs, G, q.device)
    args = _attn_args(q, k_pages, v_pages, block_table, seq_lens, task_map.num_kv_heads, sm_scale,
                      q_scale, k_scale, v_scale, kv_layout)
    if kv_layout == "HND" and cta_times is None:
        rc = _lib.dsa_decode(*args, ctypes.byref(task_map.struct), _ptr(partial_o), _ptr(partial_lse),
                             _stream(stream))
    else:
        rc = _lib.dsa_decode_ex(1, KV_LAYOUTS[kv_layout], *args, ctypes.byref(task_map.struct), _ptr(partial_o),
                                _ptr(partial_lse), _ptr(cta_times), _stream(stream))
    _check(rc, "dsa_decode")
    return partial_o, partial_lse


def decode_chained(new_tokens: int, q, k_pages, v_pages, block_table, seq_lens, task_map: TaskMap, sm_scale: float,
                   partial_o=None, partial_lse=None, q_scale=None, k_scale=None, v_scale=None, stream=None):
    """dsa_decode_chained: dsa_decode that loads the tiles holding none of each request's newest
    new_tokens tokens while the preceding kernel in the stream (the layer's prologue) runs."""
    G = q.shape[1] // task_map.num_kv_heads
    if partial_o is None:
        partial_o, partial_lse = partial_buffers(task_map.max_descs, G, q.device)
    args = _attn_args(q, k_pages, v_pages, block_table, seq_lens, task_map.num_kv_heads, sm_scale, q_scale, k_scale,
                      v_scale)
    rc = _lib.dsa_decode_chained(int(new_tokens), *args, ctypes.byref(task_map.struct), _ptr(partial_o),
                                 _ptr(partial_lse), _stream(stream))
    _check(rc, "dsa_decode_chained")
    return partial_o, partial_lse


def decode_fused(q, k_pages, v_pages, block_table, seq_lens, task_map: TaskMap, sm_scale: float, out=None,
                 out_lse=None, out_dtype=torch.bfloat16, partial_o=None, partial_lse=None, unit_counters=None,
                 q_scale=None, k_scale=None, v_scale=None, stream=None):
    """dsa_decode_fused: decode and combine in one persistent launch.  unit_counters
    ([B*Hkv] int32, zero) defaults to a buffer kept on the task map."""
    B, hq, _ = q.shape
    G = hq // task_map.num_kv_heads
    if partial_o is None:
        partial_o, partial_lse = partial_buffers(task_map.max_descs, G, q.device)
    if unit_counters is None:
        unit_counters = task_map.unit_counters()
    if out is None:
        out = torch.empty(B, hq, HEAD_DIM, dtype=out_dtype, device=q.device)
    args = _attn_args(q, k_pages, v_pages, block_table, seq_lens, task_map.num_kv_heads, sm_scale,
                      q_scale, k_scale, v_scale)
    rc = _lib.dsa_decode_fused(*args, ctypes.byref(task_map.struct), _ptr(partial_o), _ptr(partial_lse),
                               _ptr(unit_counters), _ptr(out), _dtype_code(out), _ptr(out_lse), _stream(stream))
    _check(rc, "dsa_decode_fused")
    return out


def combine(task_map: TaskMap, partial_o, partial_lse, num_q_heads: int, out=None, out_lse=None,
            out_dtype=torch.bfloat16, stream=None):
    """dsa_combine: merge each unit's partials into out [B, Hq, 128] (and out_lse [B, Hq])."""
    batch = task_map.batch
    if out is None:
        out = torch.empty(batch, num_q_heads, HEAD_DIM, dtype=out_dtype, device=partial_o.device)
    rc = _lib.dsa_combine(ctypes.byref(task_map.struct), _ptr(partial_o), _ptr(partial_lse), batch, num_q_heads,
                          task_map.num_kv_heads, HEAD_DIM, _ptr(out), _dtype_code(out), _ptr(out_lse),
                          _stream(stream))
    _check(rc, "dsa_combine")
    return out


def decode_multi(q_len: int, q, k_pages, v_pages, block_table, seq_lens, task_map: TaskMap, sm_scale: float,
                 partial_o=None, partial_lse=None, q_scale=None, k_scale=None, v_scale=None, stream=None,
                 kv_layout="HND", cta_times=None):
    """dsa_decode_multi: q [B, q_len, Hq, 128]; partials hold q_len * G rows per slot, two
    slots per descriptor when q_len > 1 (dsa_decode_ex for NHD pages or per-CTA timestamps,
    cta_times uint64-sized [num_ctas, 2])."""
    R = q_len * (q.shape[-2] // task_map.num_kv_heads)
    if partial_o is None:
        spd = int(_lib.dsa_multi_slots_per_desc(q_len, q.shape[-2] // task_map.num_kv_heads))
        partial_o, partial_lse = partial_buffers(task_map.max_descs * spd, R, q.device)
    args = _attn_args(q, k_pages, v_pages, block_table, seq_lens, task_map.num_kv_heads, sm_scale,
                      q_scale, k_scale, v_scale, kv_layout)
    if kv_layout == "HND" and cta_times is None:
        rc = _lib.dsa_decode_multi(q_len, *args, ctypes.byref(task_map.struct), _ptr(partial_o),
                                   _ptr(partial_lse), _stream(stream))
    else:
        rc = _lib.dsa_decode_ex(q_len, KV_LAYOUTS[kv_layout], *args, ctypes.byref(task_map.struct),
                                _ptr(partial_o), _ptr(partial_lse), _ptr(cta_times), _stream(stream))
    _check(rc, "dsa_decode_multi")
    return partial_o, partial_lse


def combine_multi(q_len: int, task_map: TaskMap, partial_o, partial_lse, num_q_heads: int, out=None, out_lse=None,
                  out_dtype=torch.bfloat16, stream=None):
    """dsa_combine_multi: out [B, q_len, Hq, 128] (and out_lse [B, q_len, Hq])."""
    batch = task_map.batch
    if out is None:
        out = torch.empty(batch, q_len, num_q_heads, HEAD_DIM, dtype=out_dtype, device=partial_o.device)
    rc = _lib.dsa_combine_multi(q_len, ctypes.byref(task_map.struct), _ptr(partial_o), _ptr(partial_lse), batch,
                                num_q_heads, task_map.num_kv_heads, HEAD_DIM, _ptr(out), _dtype_code(out),
                                _ptr(out_lse), _stream(stream))
    _check(rc, "dsa_combine_multi")
    return out


def attention_multi(inp: dict, num_ctas: int, min_tiles_per_split: int = 4, out_dtype=torch.bfloat16,
                    task_map: TaskMap | None = None, stream=None):
    """One multi-token verify step (inp["q"] [B, q_len, Hq, 128]): plan, decode_multi,
    combine_multi.  Returns (out, out_lse, task_map, partial_o, partial_lse)."""
    q_len = int(inp["q_len"])
    tm = plan(inp["seq_lens"], inp["num_kv_heads"], num_ctas, min_tiles_per_split, task_map=task_map,
              stream=stream)
    po, pl = decode_multi(q_len, inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"], inp["seq_lens"], tm,
                          inp["sm_scale"], q_scale=inp.get("q_scale"), k_scale=inp.get("k_scale"),
                          v_scale=inp.get("v_scale"), stream=stream, kv_layout=inp.get("kv_layout", "HND"))
    B = inp["seq_lens"].shape[0]
    out_lse = torch.empty(B, q_len, inp["num_q_heads"], dtype=torch.float32, device=po.device)
    out = combine_multi(q_len, tm, po, pl, inp["num_q_heads"], out_lse=out_lse, out_dtype=out_dtype, stream=stream)
    return out, out_lse, tm, po, pl


def static_num_splits(mode: int, param: int, max_seq_len: int) -> int:
    return int(_lib.dsa_static_num_splits(mode, param, max_seq_len))


def static_splitkv(mode: int, param: int, max_seq_len: int, q, k_pages, v_pages, block_table, seq_lens,
                   num_kv_heads: int, sm_scale: float, partial_o=None, partial_lse=None, status=None,
                   q_scale=None, k_scale=None, v_scale=None, stream=None, cta_times=None):
    """dsa_static_splitkv: the fixed-grid comparison (mode 0: param splits; mode 1: param-token chunks)."""
    S = static_num_splits(mode, param, max_seq_len)
    if S < 1:
        raise DSAError(ERR_INVALID_ARG, "dsa_static_num_splits")
    batch, hq, _ = q.shape
    G = hq // num_kv_heads
    if partial_o is None:
        partial_o, partial_lse = partial_buffers(batch * num_kv_heads * S, G, q.device)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=q.device)
    args = _attn_args(q, k_pages, v_pages, block_table, seq_lens, num_kv_heads, sm_scale, q_scale, k_scale,
                      v_scale)
    rc = _lib.dsa_static_splitkv(mode, param, max_seq_len, *args, _ptr(partial_o), _ptr(partial_lse),
                                 _ptr(status), _ptr(cta_times), _stream(stream))
    _check(rc, "dsa_static_splitkv")
    return partial_o, partial_lse, S, status


def static_combine(num_splits: int, partial_o, partial_lse, batch: int, num_q_heads: int, num_kv_heads: int,
                   out=None, out_lse=None, out_dtype=torch.bfloat16, stream=None):
    if out is None:
        out = torch.empty(batch, num_q_heads, HEAD_DIM, dtype=out_dtype, device=partial_o.device)
    rc = _lib.dsa_static_combine(num_splits, _ptr(partial_o), _ptr(partial_lse), batch, num_q_heads,
                                 num_kv_heads, HEAD_DIM, _ptr(out), _dtype_code(out), _ptr(out_lse),
                                 _stream(stream))
    _check(rc, "dsa_static_combine")
    return out


def prologue(qkv, num_q_heads: int, num_kv_heads: int, slot_mapping, k_pages, v_pages, k_scale=None,
             v_scale=None, positions=None, cos_sin=None, rotary_dim: int | None = None, rope_style: str = "neox",
             q_norm_weight=None, k_norm_weight=None, eps: float = 1e-6, hadamard: bool = False,
             q_dtype=torch.bfloat16, q_out=None, q_scale=None, status=None, stream=None, kv_layout="HND"):
    """dsa_prologue: QK-Norm -> RoPE -> [Hadamard] -> Q out (bf16, or E4M3 + per-(token, head)
    scales) and K/V written into the paged cache at slot_mapping (pages [num_pages, Hkv, P, 128]
    for kv_layout "HND", [num_pages, P, Hkv, 128] for "NHD").  Returns (q_out, q_scale)."""
    n = int(qkv.shape[0])
    fp8_q = q_dtype in (torch.uint8, torch.float8_e4m3fn, "e4m3")
    if q_out is None:
        q_out = torch.empty(n, num_q_heads, HEAD_DIM, dtype=torch.uint8 if fp8_q else torch.bfloat16,
                            device=qkv.device)
    if fp8_q and q_scale is None:
        q_scale = torch.empty(n, num_q_heads, dtype=torch.float32, device=qkv.device)
    rot = (0 if cos_sin is None else int(cos_sin.shape[1])) if rotary_dim is None else rotary_dim
    max_pos = 0 if cos_sin is None else int(cos_sin.shape[0])
    style = {"neox": ROPE_NEOX, "interleaved": ROPE_INTERLEAVED}[rope_style]
    rc = _lib.dsa_prologue(_ptr(qkv), n, num_q_heads, num_kv_heads, HEAD_DIM, _ptr(positions), _ptr(cos_sin),
                           max_pos, rot, style, _ptr(q_norm_weight), _ptr(k_norm_weight), float(eps),
                           int(bool(hadamard)), _ptr(slot_mapping), _ptr(q_out), _dtype_code(q_out),
                           _ptr(q_scale), _ptr(k_pages), _ptr(v_pages), _dtype_code(k_pages), _ptr(k_scale),
                           _ptr(v_scale), int(k_pages.shape[0]), int(k_pages.shape[1 if kv_layout == "NHD" else 2]),
                           KV_LAYOUTS[kv_layout], _ptr(status), _stream(stream))
    _check(rc, "dsa_prologue")
    return q_out, q_scale


def get_status(task_map: TaskMap) -> int:
    """Device status word of the step (synchronises the device)."""
    v = ctypes.c_int32()
    rc = _lib.dsa_get_status(ctypes.byref(task_map.struct), ctypes.byref(v))
    if rc not in (OK, ERR_DEVICE_INPUT):
        raise DSAError(rc, "dsa_get_status")
    return v.value


def read_status(status: torch.Tensor) -> int:
    v = ctypes.c_int32()
    rc = _lib.dsa_read_status(_ptr(status), ctypes.byref(v))
    if rc not in (OK, ERR_DEVICE_INPUT):
        raise DSAError(rc, "dsa_read_status")
    return v.value


def selftest_wait_timeout(limit_ns: int = 10_000_000, stream=None) -> int:
    """Runs dsa_selftest_wait_timeout and returns the device status word it produced."""
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    _check(_lib.dsa_selftest_wait_timeout(_ptr(status), int(limit_ns), _stream(stream)),
           "dsa_selftest_wait_timeout")
    return read_status(status)


def status_string(code: int) -> str:
    return _lib.dsa_status_string(code).decode()


def attention_fused(inp: dict, num_ctas: int, min_tiles_per_split: int = 4, out_dtype=torch.bfloat16,
                    task_map: TaskMap | None = None, stream=None):
    """One decode step with the combine fused into the persistent kernel: plan, decode_fused.
    Returns (out, out_lse, task_map)."""
    tm = plan(inp["seq_lens"], inp["num_kv_heads"], num_ctas, min_tiles_per_split, task_map=task_map,
              stream=stream)
    B = inp["seq_lens"].shape[0]
    out_lse = torch.empty(B, inp["num_q_heads"], dtype=torch.float32, device=inp["q"].device)
    out = decode_fused(inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"], inp["seq_lens"], tm,
                       inp["sm_scale"], out_lse=out_lse, out_dtype=out_dtype, q_scale=inp.get("q_scale"),
                       k_scale=inp.get("k_scale"), v_scale=inp.get("v_scale"), stream=stream)
    return out, out_lse, tm


def attention(inp: dict, num_ctas: int, min_tiles_per_split: int = 4, out_dtype=torch.bfloat16,
              task_map: TaskMap | None = None, stream=None):
    """One decode step over a workload dict (workloads.make_inputs): plan, decode, combine.
    Returns (out, out_lse, task_map, partial_o, partial_lse)."""
    tm = plan(inp["seq_lens"], inp["num_kv_heads"], num_ctas, min_tiles_per_split, task_map=task_map,
              stream=stream)
    po, pl = decode(inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"], inp["seq_lens"], tm,
                    inp["sm_scale"], q_scale=inp.get("q_scale"), k_scale=inp.get("k_scale"),
                    v_scale=inp.get("v_scale"), stream=stream, kv_layout=inp.get("kv_layout", "HND"))
    B = inp["seq_lens"].shape[0]
    out_lse = torch.empty(B, inp["num_q_heads"], dtype=torch.float32, device=po.device)
    out = combine(tm, po, pl, inp["num_q_heads"], out_lse=out_lse, out_dtype=out_dtype, stream=stream)
    return out, out_lse, tm, po, pl


def decode_step_noalloc(inp: dict, num_ctas: int, out, out_lse=None, status=None, min_tiles_per_split: int = 4,
                        stream=None):
    """dsa_decode_step_noalloc: plan, decode and combine with the library's own fixed device
    scratch (for callers that cannot allocate device memory); writes out / out_lse / status."""
    args = _attn_args(inp["q"], inp["k_pages"], inp["v_pages"], inp["block_table"], inp["seq_lens"],
                      inp["num_kv_heads"], inp["sm_scale"], inp.get("q_scale"), inp.get("k_scale"),
                      inp.get("v_scale"))
    rc = _lib.dsa_decode_step_noalloc(*args, num_ctas, min_tiles_per_split, _ptr(out), _dtype_code(out),
                                      _ptr(out_lse), _ptr(status), _stream(stream))
    _check(rc, "dsa_decode_step_noalloc")
    return out
