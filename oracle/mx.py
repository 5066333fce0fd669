"""MXFP8 quantization of jagged tensors, in plain numpy (TEST INFRASTRUCTURE
ONLY: only tests/, the smoke check and the benchmark's CPU legs may use it;
it shares no code with the CUDA library).

What it computes ("GEM Training" post, section "Low Precision Flash
Attention": MXFP8 block-scaled operands, FP8 data kept at the unpadded jagged
positions with compact scale factors, and [32, 32] square blocks with one
scale each so that a tensor quantized once serves both its orientations):

* elements are FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 mantissa
  bits; subnormals below 2^-6; largest finite 448; no infinities; code
  S.1111.111 is NaN), rounded to nearest, ties to even, and saturated to
  +-448 (the "satfinite" rule);
* every block of 32 sequence-local rows x 32 head columns (per head; the
  last row block of a sequence is ragged) shares one power-of-two scale
  X = 2^(E - 127) stored as its 8-bit exponent E (E8M0), chosen as the
  Microscaling format defines it: E - 127 = floor(log2(amax)) - 8, where 8
  is the exponent of E4M3's largest power of two and amax the block's largest
  magnitude; E is clamped to >= 0, and an all-zero block gets E = 0;
* element code = E4M3(x / X).

Row block g of sequence b, row block r, is g = block_start[b] + r with
block_start the exclusive prefix sum of ceil(L_b / 32); scales are laid out
[row blocks, H, D/32].

``attention_fwd`` / ``attention_bwd`` state softmax attention on MXFP8
operands (P quantized in the softmax with the scale its row maximum fixes,
dS quantized with [32, 32] blocks); ``attention_fwd`` is the reference of the
block-scaled forward kernel (jattn_fwd_mxfp8), ``attention_bwd`` of a
backward that is not built.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_EMAX = 8  # exponent of the largest power of two E4M3 holds


def e4m3_decode(codes) -> np.ndarray:
    """Value of each E4M3 code (uint8), from the bit fields."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0**-6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    out = sign * mag
    return np.where((e == 15) & (m == 7), np.nan, out)


_POS_CODES = np.arange(0x7F, dtype=np.uint8)  # 0x00 .. 0x7E: every non-negative finite code
_POS_VALUES = e4m3_decode(_POS_CODES)  # increasing in the code


def e4m3_encode(x) -> np.ndarray:
    """E4M3 code of each value: nearest representable magnitude (ties to the
    even code, i.e. even mantissa), saturated to 448, sign kept (negative
    values that round to zero give 0x80); NaN gives 0x7F."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(_POS_VALUES, a, side="left"), 0, len(_POS_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    d_hi = _POS_VALUES[hi] - a
    d_lo = a - _POS_VALUES[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo]).astype(np.uint8)
    code = np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def scale_exponent(amax: float) -> int:
    """E8M0 exponent E of a block whose largest magnitude is amax."""
    if amax == 0.0:
        return 0
    _, e = np.frexp(amax)  # amax = f * 2^e with f in [0.5, 1): floor(log2(amax)) = e - 1
    return int(max(0, min(254, (int(e) - 1) - E4M3_EMAX + 127)))


def quantize_block(x2d) -> tuple[np.ndarray, int]:
    """One block (any shape): its codes and its scale exponent E."""
    x2d = np.asarray(x2d, dtype=np.float64)
    E = scale_exponent(float(np.max(np.abs(x2d))) if x2d.size else 0.0)
    return e4m3_encode(x2d / np.exp2(E - 127.0)), E


def block_starts(off) -> np.ndarray:
    """Exclusive prefix sum [B+1] of ceil(L_b / 32)."""
    off = np.asarray(off, dtype=np.int64)
    n = (off[1:] - off[:-1] + 31) // 32
    out = np.zeros(len(n) + 1, dtype=np.int64)
    np.cumsum(n, out=out[1:])
    return out


def _values(x) -> np.ndarray:
    if isinstance(x, np.ndarray):
        return np.asarray(x, dtype=np.float64)
    import torch

    return x.detach().to(torch.float64).cpu().numpy()


def quantize(x, off):
    """Jagged [total, H, D] values -> (codes uint8 [total, H, D], scale
    exponents uint8 [row blocks, H, D/32], block_start int64 [B+1])."""
    x = _values(x)
    off = np.asarray(off if isinstance(off, np.ndarray) else off.cpu().numpy(), dtype=np.int64)
    total, H, D = x.shape
    bs = block_starts(off)
    codes = np.zeros((total, H, D), dtype=np.uint8)
    scales = np.zeros((int(bs[-1]), H, D // 32), dtype=np.uint8)
    for b in range(len(off) - 1):
        for r in range((int(off[b + 1] - off[b]) + 31) // 32):
            r0 = int(off[b]) + 32 * r
            r1 = min(r0 + 32, int(off[b + 1]))
            for h in range(H):
                for c in range(D // 32):
                    q, E = quantize_block(x[r0:r1, h, 32 * c:32 * c + 32])
                    codes[r0:r1, h, 32 * c:32 * c + 32] = q
                    scales[bs[b] + r, h, c] = E
    return codes, scales, bs


def dequantize(codes, scales, off) -> np.ndarray:
    """Values the codes and scales stand for, [total, H, D] float64."""
    codes = np.asarray(codes, dtype=np.uint8)
    off = np.asarray(off, dtype=np.int64)
    bs = block_starts(off)
    out = e4m3_decode(codes)
    for b in range(len(off) - 1):
        for r in range((int(off[b + 1] - off[b]) + 31) // 32):
            r0 = int(off[b]) + 32 * r
            r1 = min(r0 + 32, int(off[b + 1]))
            X = np.exp2(scales[bs[b] + r].astype(np.float64) - 127.0)  # [H, D/32]
            out[r0:r1] *= np.repeat(X, 32, axis=1)[None]
    return out


# ---------------------------------------------------------------- MXFP8 attention
# Softmax attention on MXFP8 operands, written from the same section: Q, K, V
# (and dO in the backward) arrive as MXFP8 codes with [32, 32] block scales;
# the products run on their exact values; the softmax output P is quantized
# to E4M3 with the scale that the row maximum fixes (P <= 1 with equality at
# the maximum, so X = 2^(0 - 8) for every row: no further reduction), and the
# backward's dS is quantized with [32, 32] blocks over (query, key) tiles of
# each sequence. The normaliser l and D_i stay in high precision. Masks are
# those of the C oracle (causal, causal + window, block, causal + block).

P_SCALE_EXP = 127 - E4M3_EMAX  # E of X = 2^-8


def _allowed(lq: int, lkv: int, mask: int, window: int) -> np.ndarray:
    i = np.arange(lq)[:, None]
    j = np.arange(lkv)[None, :]
    d = lkv - lq
    ok = np.ones((lq, lkv), dtype=bool)
    if mask & 3:
        ok &= j <= i + d
    if mask & 2:
        ok &= i + d - j < window
    if mask & 4:
        ok &= np.floor_divide(j, window) == np.floor_divide(i + d, window)
    return ok


def quantize_p(p: np.ndarray) -> np.ndarray:
    """P in [0, 1] to its E4M3 value with X = 2^-8."""
    X = np.exp2(P_SCALE_EXP - 127.0)
    return e4m3_decode(e4m3_encode(p / X)) * X


def quantize_square(a: np.ndarray) -> np.ndarray:
    """A 2-D array through [32, 32]-block MXFP8 (blocks from the origin,
    ragged at the ends), back to values."""
    out = np.empty_like(a)
    for r0 in range(0, a.shape[0], 32):
        for c0 in range(0, a.shape[1], 32):
            q, E = quantize_block(a[r0:r0 + 32, c0:c0 + 32])
            out[r0:r0 + 32, c0:c0 + 32] = e4m3_decode(q) * np.exp2(E - 127.0)
    return out


def attention_fwd(qd, kd, vd, q_off, kv_off, *, mask=0, window=0, scale=None, quant_p=True):
    """Forward on dequantized operands qd / kd / vd [total, H, D] (float64,
    e.g. from dequantize). Returns (o, lse); quant_p=False keeps P exact."""
    q_off = np.asarray(q_off, dtype=np.int64)
    kv_off = np.asarray(kv_off, dtype=np.int64)
    H, D = qd.shape[1], qd.shape[2]
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    o = np.zeros_like(qd)
    lse = np.full(qd.shape[:2], -np.inf)
    for b in range(len(q_off) - 1):
        lq, lkv = int(q_off[b + 1] - q_off[b]), int(kv_off[b + 1] - kv_off[b])
        if lq == 0 or lkv == 0:
            continue
        ok = _allowed(lq, lkv, mask, window)
        rows = ok.any(axis=1)
        for h in range(H):
            s = scale * qd[q_off[b]:q_off[b + 1], h] @ kd[kv_off[b]:kv_off[b + 1], h].T
            s = np.where(ok, s, -np.inf)
            m = np.where(rows, s.max(axis=1, initial=-np.inf), 0.0)
            p = np.where(ok, np.exp(s - m[:, None]), 0.0)
            l = p.sum(axis=1)
            pq = quantize_p(p) if quant_p else p
            oh = np.zeros((lq, D))
            oh[rows] = (pq @ vd[kv_off[b]:kv_off[b + 1], h])[rows] / l[rows, None]
            o[q_off[b]:q_off[b + 1], h] = oh
            lse[q_off[b]:q_off[b + 1], h] = np.where(rows, m + np.log(np.where(rows, l, 1.0)), -np.inf)
    return o, lse


def attention_bwd(qd, kd, vd, dod, q_off, kv_off, *, mask=0, window=0, scale=None, o=None, quant_p=True,
                  quant_ds=True):
    """Backward on dequantized operands (dod: dequantized dO). D_i = <dO_i,
    o_i> with o the stored forward output (default: this module's forward).
    dV = P~^T dO, dQ = scale dS~ K, dK = scale dS~^T Q with P~ as in the
    forward and dS~ the [32, 32]-block quantization of dS = P (dP - D)."""
    q_off = np.asarray(q_off, dtype=np.int64)
    kv_off = np.asarray(kv_off, dtype=np.int64)
    H, D = qd.shape[1], qd.shape[2]
    scale = 1.0 / np.sqrt(D) if scale is None else scale
    if o is None:
        o, _ = attention_fwd(qd, kd, vd, q_off, kv_off, mask=mask, window=window, scale=scale, quant_p=quant_p)
    dq, dk, dv = np.zeros_like(qd), np.zeros_like(kd), np.zeros_like(vd)
    for b in range(len(q_off) - 1):
        lq, lkv = int(q_off[b + 1] - q_off[b]), int(kv_off[b + 1] - kv_off[b])
        if lq == 0 or lkv == 0:
            continue
        ok = _allowed(lq, lkv, mask, window)
        rows = ok.any(axis=1)
        qs, ks = slice(q_off[b], q_off[b + 1]), slice(kv_off[b], kv_off[b + 1])
        for h in range(H):
            s = np.where(ok, scale * qd[qs, h] @ kd[ks, h].T, -np.inf)
            m = np.where(rows, s.max(axis=1, initial=-np.inf), 0.0)
            e = np.where(ok, np.exp(s - m[:, None]), 0.0)
            l = np.where(rows, e.sum(axis=1), 1.0)
            p = e / l[:, None]  # normalised probabilities
            pq = quantize_p(e) / l[:, None] if quant_p else p
            di = np.einsum("id,id->i", dod[qs, h], o[qs, h])
            dp = dod[qs, h] @ vd[ks, h].T
            ds = np.where(ok, p * (dp - di[:, None]), 0.0)
            dsq = quantize_square(ds) if quant_ds else ds
            dv[ks, h] = pq.T @ dod[qs, h]
            dq[qs, h] = scale * dsq @ kd[ks, h]
            dk[ks, h] = scale * dsq.T @ qd[qs, h]
    return dq, dk, dv
