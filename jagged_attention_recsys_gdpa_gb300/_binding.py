"""ctypes binding of libjattn (argument marshalling only).

Every computation runs in the CUDA library; this module only converts torch
tensors to raw pointers and sizes, passes the current CUDA stream, and turns
non-zero return codes into exceptions. The library must exist: there is no
fallback path.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

SOFTMAX, SILU, GELU_TANH, GELU_POLY = 0, 1, 2, 3
MASK_NONE, MASK_CAUSAL, MASK_WINDOW, MASK_BLOCK = 0, 1, 2, 4

EXPORTED = (
    "jattn_workspace_size",
    "jattn_fwd",
    "jattn_fwd_noalloc",
    "jattn_bwd",
    "jattn_bwd_rope",
    "jattn_bwd_rope_workspace_size",
    "jattn_rope",
    "jattn_mxfp8_scale_rows",
    "jattn_mxfp8_quantize",
    "jattn_fwd_mxfp8",
    "jattn_bwd_mxfp8",
    "jattn_schedule",
    "jattn_partition",
    "jattn_max_tiles",
    "jattn_get_status",
    "jattn_error_string",
    "jattn_last_error",
    "jattn_profile_events",
    "jattn_debug_set",
)


class Params(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int64),
        ("total_q", ctypes.c_int64),
        ("total_kv", ctypes.c_int64),
        ("H", ctypes.c_int),
        ("D", ctypes.c_int),
        ("act", ctypes.c_int),
        ("mask", ctypes.c_int),
        ("window", ctypes.c_int),
        ("scale", ctypes.c_float),
        ("norm_by_lkv", ctypes.c_int),
    ]


class JattnError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        detail = ""
        if code in (2, 8):
            detail = " [" + load().jattn_last_error().decode() + "]"
        super().__init__(f"{where}: {error_string(code)} (code {code}){detail}")


_lib = None


def library_path() -> str:
    return _build.LIB


def load(path: str | None = None):
    """Load libjattn.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"libjattn.so not found at {path}; build it with "
            "`python -m jagged_attention_recsys_gdpa_gb300.build` (no CPU fallback exists)"
        )
    lib = ctypes.CDLL(path)
    P = ctypes.POINTER(Params)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.jattn_workspace_size.argtypes = [P, ctypes.POINTER(ctypes.c_size_t)]
    lib.jattn_workspace_size.restype = i32
    lib.jattn_fwd.argtypes = [P] + [vp] * 7 + [vp, ctypes.c_size_t, vp]
    lib.jattn_fwd.restype = i32
    lib.jattn_fwd_noalloc.argtypes = [P] + [vp] * 8 + [vp]
    lib.jattn_fwd_noalloc.restype = i32
    lib.jattn_bwd.argtypes = [P] + [vp] * 11 + [vp, ctypes.c_size_t, vp]
    lib.jattn_bwd.restype = i32
    lib.jattn_bwd_rope.argtypes = [P] + [vp] * 10 + [i64] + [vp] * 3 + [vp, ctypes.c_size_t, vp]
    lib.jattn_bwd_rope.restype = i32
    lib.jattn_rope.argtypes = [P, vp, vp, i32, i32, vp, vp, vp, vp, i64, vp, ctypes.c_size_t, vp]
    lib.jattn_rope.restype = i32
    lib.jattn_mxfp8_scale_rows.argtypes = [i64, i64]
    lib.jattn_mxfp8_scale_rows.restype = i64
    lib.jattn_mxfp8_quantize.argtypes = [i64, i64, i32, i32] + [vp] * 5 + [vp, ctypes.c_size_t, vp]
    lib.jattn_mxfp8_quantize.restype = i32
    lib.jattn_fwd_mxfp8.argtypes = [P] + [vp] * 12 + [vp, ctypes.c_size_t, vp]
    lib.jattn_fwd_mxfp8.restype = i32
    lib.jattn_bwd_mxfp8.argtypes = [P] + [vp] * 17 + [vp, ctypes.c_size_t, vp]
    lib.jattn_bwd_mxfp8.restype = i32
    lib.jattn_bwd_rope_workspace_size.argtypes = [P, i64, ctypes.POINTER(ctypes.c_size_t)]
    lib.jattn_bwd_rope_workspace_size.restype = i32
    lib.jattn_schedule.argtypes = [P, vp, vp, i32, i32, i32, vp, i64, vp, vp, ctypes.c_size_t, vp]
    lib.jattn_schedule.restype = i32
    lib.jattn_partition.argtypes = [i64, vp, vp, i32, i32, i32, vp, vp]
    lib.jattn_partition.restype = i32
    lib.jattn_max_tiles.argtypes = [P, i32, i32]
    lib.jattn_max_tiles.restype = i64
    lib.jattn_get_status.argtypes = [vp, vp, ctypes.POINTER(ctypes.c_int)]
    lib.jattn_get_status.restype = i32
    lib.jattn_error_string.argtypes = [i32]
    lib.jattn_error_string.restype = ctypes.c_char_p
    lib.jattn_last_error.argtypes = []
    lib.jattn_last_error.restype = ctypes.c_char_p
    lib.jattn_profile_events.argtypes = [ctypes.POINTER(vp)]
    lib.jattn_profile_events.restype = None
    lib.jattn_debug_set.argtypes = [i32, ctypes.c_uint64]
    lib.jattn_debug_set.restype = None
    _lib = lib
    return lib


def error_string(code: int) -> str:
    return load().jattn_error_string(int(code)).decode()


def check(code: int, where: str):
    if code != 0:
        raise JattnError(code, where)


def params(B, total_q, total_kv, H, D, act, mask, window, scale, norm_by_lkv) -> Params:
    return Params(int(B), int(total_q), int(total_kv), int(H), int(D), int(act), int(mask), int(window),
                  float(scale or 0.0), int(bool(norm_by_lkv)))


def workspace_size(p: Params) -> int:
    n = ctypes.c_size_t(0)
    check(load().jattn_workspace_size(ctypes.byref(p), ctypes.byref(n)), "jattn_workspace_size")
    return int(n.value)


def bwd_rope_workspace_size(p: Params, rope_rows: int) -> int:
    n = ctypes.c_size_t(0)
    check(load().jattn_bwd_rope_workspace_size(ctypes.byref(p), int(rope_rows), ctypes.byref(n)),
          "jattn_bwd_rope_workspace_size")
    return int(n.value)


def ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def fwd(p: Params, q_off, kv_off, q, k, v, o, lse, ws, ws_bytes: int, stream: int):
    check(load().jattn_fwd(ctypes.byref(p), ptr(q_off), ptr(kv_off), ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse),
                           ws, ws_bytes, stream), "jattn_fwd")


def fwd_noalloc(p: Params, q_off, kv_off, q, k, v, o, lse, device_status, stream: int):
    """Forward without a workspace (scratch held by the library); see jattn_fwd_noalloc."""
    check(load().jattn_fwd_noalloc(ctypes.byref(p), ptr(q_off), ptr(kv_off), ptr(q), ptr(k), ptr(v), ptr(o),
                                   ptr(lse), ptr(device_status), stream), "jattn_fwd_noalloc")


def bwd(p: Params, q_off, kv_off, q, k, v, o, lse, do, dq, dk, dv, ws, ws_bytes: int, stream: int):
    check(load().jattn_bwd(ctypes.byref(p), ptr(q_off), ptr(kv_off), ptr(q), ptr(k), ptr(v), ptr(o), ptr(lse),
                           ptr(do), ptr(dq), ptr(dk), ptr(dv), ws, ws_bytes, stream), "jattn_bwd")


def bwd_rope(p: Params, q_off, kv_off, q, k, v, o, lse, do, rope_cos, rope_sin, dq, dk, dv, ws, ws_bytes: int,
             stream: int):
    """jattn_bwd_rope: q and k are the rotated inputs; dq and dk come back rotated by R^T."""
    check(load().jattn_bwd_rope(ctypes.byref(p), ptr(q_off), ptr(kv_off), ptr(q), ptr(k), ptr(v), ptr(o),
                                ptr(lse), ptr(do), ptr(rope_cos), ptr(rope_sin), int(rope_cos.shape[0]), ptr(dq),
                                ptr(dk), ptr(dv), ws, ws_bytes, stream), "jattn_bwd_rope")


def mxfp8_scale_rows(B: int, total: int) -> int:
    return int(load().jattn_mxfp8_scale_rows(int(B), int(total)))


def mxfp8_quantize(B: int, total: int, H: int, D: int, off, x, codes, scales, block_start, ws, ws_bytes: int,
                   stream: int):
    check(load().jattn_mxfp8_quantize(int(B), int(total), int(H), int(D), ptr(off), ptr(x), ptr(codes), ptr(scales),
                                      ptr(block_start), ws, ws_bytes, stream), "jattn_mxfp8_quantize")


def fwd_mxfp8(p: Params, q_off, kv_off, q, q_scales, q_bs, k, k_scales, v, v_scales, kv_bs, o, lse, ws,
              ws_bytes: int, stream: int):
    check(load().jattn_fwd_mxfp8(ctypes.byref(p), ptr(q_off), ptr(kv_off), ptr(q), ptr(q_scales), ptr(q_bs), ptr(k),
                                 ptr(k_scales), ptr(v), ptr(v_scales), ptr(kv_bs), ptr(o), ptr(lse), ws, ws_bytes,
                                 stream), "jattn_fwd_mxfp8")


def bwd_mxfp8(p: Params, q_off, kv_off, q, q_scales, q_bs, k, k_scales, v, v_scales, kv_bs, o, lse, dout,
              dout_scales, dq, dk, dv, ws, ws_bytes: int, stream: int):
    check(load().jattn_bwd_mxfp8(ctypes.byref(p), ptr(q_off), ptr(kv_off), ptr(q), ptr(q_scales), ptr(q_bs), ptr(k),
                                 ptr(k_scales), ptr(v), ptr(v_scales), ptr(kv_bs), ptr(o), ptr(lse), ptr(dout),
                                 ptr(dout_scales), ptr(dq), ptr(dk), ptr(dv), ws, ws_bytes, stream),
          "jattn_bwd_mxfp8")


def rope(p: Params, q_off, kv_off, keys: bool, inverse: bool, x, y, rope_cos, rope_sin, ws, ws_bytes: int,
         stream: int):
    """jattn_rope: y = R(pos) x (or R(pos)^T x) on query (keys=False) or key rows."""
    check(load().jattn_rope(ctypes.byref(p), ptr(q_off), ptr(kv_off), int(bool(keys)), int(bool(inverse)), ptr(x),
                            ptr(y), ptr(rope_cos), ptr(rope_sin), int(rope_cos.shape[0]), ws, ws_bytes, stream),
          "jattn_rope")


def schedule(p: Params, q_off, kv_off, row_tile, col_tile, transposed, tiles, max_tiles, n_tiles, ws, ws_bytes,
             stream):
    check(load().jattn_schedule(ctypes.byref(p), ptr(q_off), ptr(kv_off), int(row_tile), int(col_tile),
                                int(bool(transposed)), ptr(tiles), int(max_tiles), ptr(n_tiles), ws, ws_bytes,
                                stream), "jattn_schedule")


def partition(q_off, kv_off, mask: int, window: int, n_ranks: int, rank_of, rank_pairs):
    """Host arrays (numpy): q_off, kv_off int64 [B+1]; rank_of int32 [B], rank_pairs int64 [n_ranks] out."""
    B = len(q_off) - 1
    check(load().jattn_partition(B, q_off.ctypes.data, kv_off.ctypes.data, int(mask), int(window), int(n_ranks),
                                 rank_of.ctypes.data, rank_pairs.ctypes.data), "jattn_partition")


def max_tiles(p: Params, row_tile: int, transposed: bool) -> int:
    return int(load().jattn_max_tiles(ctypes.byref(p), int(row_tile), int(bool(transposed))))


def get_status(ws, stream) -> int:
    s = ctypes.c_int(0)
    check(load().jattn_get_status(ws, stream, ctypes.byref(s)), "jattn_get_status")
    return int(s.value)


def debug_set(flags: int, timeout_ns: int):
    load().jattn_debug_set(int(flags), int(timeout_ns))


def profile_events(events):
    """Record the six given torch.cuda.Event objects around the main kernels (None: off)."""
    if events is None:
        load().jattn_profile_events(None)
        return
    arr = (ctypes.c_void_p * 6)(*[e.cuda_event for e in events])
    load().jattn_profile_events(arr)
