"""Plain CPU oracle for jagged generalized dot-product attention.

TEST INFRASTRUCTURE ONLY. Nothing in the product path may import this
package: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg
of ``bench.py`` use it. It shares no code with the CUDA library.

* ``fwd`` / ``bwd`` wrap the double-precision C oracle in ``jattn_oracle.c``,
  which writes out the definition of jagged attention with a softmax or a
  pointwise (SiLU / tanh-GELU) activation ("GEM Training" post, sections
  "Jagged Sequence Flash Attention" and "Generalized Dot-Product Attention").
* ``schedule`` is a plain-Python statement of the jagged tile schedule of the
  same post's GDPA section ("precompute valid tiles, skip empty ones, balance
  them across SMs"): every (sequence, row tile) with the range of column
  tiles its mask allows, ordered longest-first with ties in (sequence, tile)
  order.
* ``count_pairs`` counts allowed (query, key) pairs by visiting every pair.
* ``partition`` is a plain-Python statement of the data-parallel split of a
  batch over ranks: cost of a sequence = its allowed pairs (visited one by
  one), sequences taken in order of decreasing cost (ties by index), each
  given to the rank with the least cost so far (ties by rank) -- the
  sort-then-balance rule of the GEM training summary's "Base Batch
  Shuffling" takeaway applied to attention cost.
* ``rope`` rotates jagged query or key rows by the rotary embedding (the
  RoFormer pairing (2m, 2m+1), angles from the caller's cos / sin tables),
  in double: the forward side of the rotary backward fused into the
  attention epilogue ("GEM Training" post, section "BlockAttention"). The
  gradient of attention on rotated rows w.r.t. the unrotated ones is this
  rotation's transpose applied to ``bwd``'s dQ and dK.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libjattn_oracle.so")
_SRC = os.path.join(_HERE, "jattn_oracle.c")

SOFTMAX, SILU, GELU, GELU_POLY = 0, 1, 2, 3  # GELU_POLY: tanh-GELU here (see the C header)
MASK_NONE, MASK_CAUSAL, MASK_WINDOW, MASK_BLOCK = 0, 1, 2, 4


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP) into ``oracle/_build``."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
        )
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Params(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int64),
        ("H", ctypes.c_int),
        ("D", ctypes.c_int),
        ("act", ctypes.c_int),
        ("mask", ctypes.c_int),
        ("window", ctypes.c_int64),
        ("scale", ctypes.c_double),
        ("norm_by_lkv", ctypes.c_int),
    ]


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        ptr = ctypes.c_void_p
        lib.oracle_fwd.argtypes = [ctypes.POINTER(_Params)] + [ptr] * 7
        lib.oracle_fwd.restype = ctypes.c_int
        lib.oracle_bwd.argtypes = [ctypes.POINTER(_Params)] + [ptr] * 10
        lib.oracle_bwd.restype = ctypes.c_int
        lib.oracle_count_pairs.argtypes = [ctypes.c_int64, ptr, ptr, ctypes.c_int, ctypes.c_int64]
        lib.oracle_count_pairs.restype = ctypes.c_int64
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact decode of bf16 bit patterns: the 16 bits are the top half of an fp32."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _dbl(x) -> np.ndarray:
    """Inputs as contiguous float64: torch bf16 / uint16 bit patterns are decoded
    exactly, float64 arrays pass through (used by finite-difference checks)."""
    if isinstance(x, np.ndarray):
        if x.dtype == np.uint16:
            return np.ascontiguousarray(bf16_bits_to_f64(x))
        assert x.dtype == np.float64
        return np.ascontiguousarray(x)
    import torch

    if x.dtype == torch.float64:
        return np.ascontiguousarray(x.detach().cpu().numpy())
    assert x.dtype == torch.bfloat16
    bits = x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
    return np.ascontiguousarray(bf16_bits_to_f64(bits))


def _off(x) -> np.ndarray:
    if not isinstance(x, np.ndarray):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(x, dtype=np.int64)


def _params(B, H, D, act, mask, window, scale, norm_by_lkv):
    if scale is None:
        scale = 1.0 / np.sqrt(D)
    return _Params(int(B), int(H), int(D), int(act), int(mask), int(window), float(scale), int(bool(norm_by_lkv)))


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def fwd(q_off, kv_off, q, k, v, *, H, D, act=SOFTMAX, mask=MASK_NONE, window=0, scale=None, norm_by_lkv=False):
    """Oracle forward. Returns (o [total_q,H,D] float64, lse [total_q,H] float64)."""
    q_off, kv_off = _off(q_off), _off(kv_off)
    q, k, v = _dbl(q), _dbl(k), _dbl(v)
    B = len(q_off) - 1
    tq = int(q_off[-1])
    o = np.zeros((tq, H, D), dtype=np.float64)
    lse = np.zeros((tq, H), dtype=np.float64)
    P = _params(B, H, D, act, mask, window, scale, norm_by_lkv)
    _load().oracle_fwd(ctypes.byref(P), _p(q_off), _p(kv_off), _p(q), _p(k), _p(v), _p(o), _p(lse))
    return o, lse


def bwd(q_off, kv_off, q, k, v, do, *, H, D, act=SOFTMAX, mask=MASK_NONE, window=0, scale=None, norm_by_lkv=False,
        o=None):
    """Oracle backward. Returns (dq, dk, dv) as float64 arrays.

    ``o``: None, or the stored forward output [total_q,H,D] that softmax's
    D_i = <dO_i, o_i> is formed from, as FlashAttention's backward does (None:
    the output recomputed here in double, which gives the exact gradient)."""
    q_off, kv_off = _off(q_off), _off(kv_off)
    q, k, v, do = _dbl(q), _dbl(k), _dbl(v), _dbl(do)
    o = None if o is None else _dbl(o)
    B = len(q_off) - 1
    tq, tk = int(q_off[-1]), int(kv_off[-1])
    dq = np.zeros((tq, H, D), dtype=np.float64)
    dk = np.zeros((tk, H, D), dtype=np.float64)
    dv = np.zeros((tk, H, D), dtype=np.float64)
    P = _params(B, H, D, act, mask, window, scale, norm_by_lkv)
    o_ptr = None if o is None else _p(o)
    _load().oracle_bwd(ctypes.byref(P), _p(q_off), _p(kv_off), _p(q), _p(k), _p(v), _p(do), o_ptr, _p(dq), _p(dk),
                       _p(dv))
    return dq, dk, dv


def rope(x, q_off, kv_off, cos, sin, *, keys=False, inverse=False) -> np.ndarray:
    """Rotary embedding of jagged rows x [total, H, D] (queries, or keys with
    ``keys``), in double: pair m = (2m, 2m+1) of every head turns by the angle
    at the row's position, y_2m = x_2m cos - x_2m+1 sin, y_2m+1 = x_2m sin +
    x_2m+1 cos (``inverse``: the transpose, i.e. sin negated). cos / sin:
    [rows, D/2] tables of that angle. Positions: the queries and keys of a
    sequence end at the same position and the longer side starts at 0, so
    query row i sits at i + max(delta, 0) and key row j at j + max(-delta, 0),
    delta = Lkv - Lq."""
    q_off, kv_off = _off(q_off), _off(kv_off)
    x = _dbl(x)
    cos = np.asarray(cos, dtype=np.float64)
    sin = np.asarray(sin, dtype=np.float64) * (-1.0 if inverse else 1.0)
    own, other = (kv_off, q_off) if keys else (q_off, kv_off)
    y = np.empty_like(x)
    for b in range(len(own) - 1):
        n_own, n_other = int(own[b + 1] - own[b]), int(other[b + 1] - other[b])
        delta = (n_own - n_other) if keys else (n_other - n_own)  # Lkv - Lq
        shift = max(-delta, 0) if keys else max(delta, 0)
        pos = np.arange(n_own) + shift
        c = cos[pos][:, None, :]
        s = sin[pos][:, None, :]
        rows = slice(int(own[b]), int(own[b + 1]))
        even, odd = x[rows, :, 0::2], x[rows, :, 1::2]
        y[rows, :, 0::2] = even * c - odd * s
        y[rows, :, 1::2] = even * s + odd * c
    return y


def count_pairs(q_off, kv_off, mask=MASK_NONE, window=0) -> int:
    """Allowed (i, j) pairs over all sequences for one head, by brute force."""
    q_off, kv_off = _off(q_off), _off(kv_off)
    return int(_load().oracle_count_pairs(len(q_off) - 1, _p(q_off), _p(kv_off), int(mask), int(window)))


def num_threads() -> int:
    return int(_load().oracle_num_threads())


# ---------------------------------------------------------------------------
# Tile schedule twin
# ---------------------------------------------------------------------------

def _row_intervals(rows: np.ndarray, delta: int, ncols: int, mask: int, window: int, transposed: bool):
    """Half-open interval of visible columns for each row index.

    Not transposed: rows are queries i, columns keys j, allowed when
    j <= i + delta (causal), i + delta - j < window (window) and
    j // window == (i + delta) // window (block).
    Transposed: rows are keys j, columns queries i, same relation solved for i.
    """
    lo = np.zeros_like(rows)
    hi = np.full_like(rows, ncols)
    causal = bool(mask & (MASK_CAUSAL | MASK_WINDOW))
    win = bool(mask & MASK_WINDOW)
    blk = bool(mask & MASK_BLOCK)
    if not transposed:
        if causal:
            hi = np.minimum(hi, rows + delta + 1)
        if win:
            lo = np.maximum(lo, rows + delta - window + 1)
        if blk:
            start = np.floor_divide(rows + delta, window) * window
            lo = np.maximum(lo, start)
            hi = np.minimum(hi, start + window)
    else:
        if causal:
            lo = np.maximum(lo, rows - delta)
        if win:
            hi = np.minimum(hi, rows - delta + window)
        if blk:
            start = np.floor_divide(rows, window) * window
            lo = np.maximum(lo, start - delta)
            hi = np.minimum(hi, start + window - delta)
    return lo, hi


def schedule(q_off, kv_off, *, mask=MASK_NONE, window=0, BM=128, BN=128, transposed=False, cost_cap=1023):
    """Longest-first tile list: int32 [T, 4] rows of (b, row_tile, col_tile_lo, col_tile_hi).

    Rows are query tiles of BM rows (key tiles when ``transposed``); the
    column range covers every column tile of BN that holds at least one
    allowed pair with a row of the tile (empty -> 0, 0). Order: cost =
    col_tile_hi - col_tile_lo, capped at ``cost_cap``, descending; ties by
    (b, row_tile) ascending. Sequences with no rows contribute no tile.
    """
    q_off, kv_off = _off(q_off), _off(kv_off)
    B = len(q_off) - 1
    out = []
    for b in range(B):
        lq = int(q_off[b + 1] - q_off[b])
        lkv = int(kv_off[b + 1] - kv_off[b])
        delta = lkv - lq
        nrows, ncols = (lkv, lq) if transposed else (lq, lkv)
        ntiles = -(-nrows // BM)
        for t in range(ntiles):
            rows = np.arange(t * BM, min((t + 1) * BM, nrows), dtype=np.int64)
            lo, hi = _row_intervals(rows, delta, ncols, mask, window, transposed)
            ok = hi > lo
            if ok.any():
                c_lo = int(lo[ok].min()) // BN
                c_hi = -(-int(hi[ok].max()) // BN)
            else:
                c_lo = c_hi = 0
            out.append((b, t, c_lo, c_hi))
    if not out:
        return np.zeros((0, 4), dtype=np.int32)
    arr = np.array(out, dtype=np.int64)
    cost = np.minimum(arr[:, 3] - arr[:, 2], cost_cap)
    order = np.lexsort((np.arange(len(arr)), -cost))
    return arr[order].astype(np.int32)


def partition(q_off, kv_off, n_ranks: int, mask=MASK_NONE, window=0):
    """(rank of each sequence, total allowed pairs of each rank) as Python lists."""
    q_off, kv_off = _off(q_off), _off(kv_off)
    B = len(q_off) - 1
    cost = []
    for b in range(B):
        qo = np.array([0, q_off[b + 1] - q_off[b]], dtype=np.int64)
        ko = np.array([0, kv_off[b + 1] - kv_off[b]], dtype=np.int64)
        cost.append(count_pairs(qo, ko, mask, window))
    order = sorted(range(B), key=lambda b: (-cost[b], b))
    load = [0] * n_ranks
    rank_of = [0] * B
    for b in order:
        r = min(range(n_ranks), key=lambda i: (load[i], i))
        rank_of[b] = r
        load[r] += cost[b]
    return rank_of, load
