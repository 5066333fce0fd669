"""Work accounting for jagged attention: allowed (query, key) pairs, effective
FLOPs and algorithmic HBM bytes.

Effective FLOPs count only unpadded, unmasked work, with the usual attention
convention: forward 4*D per allowed pair and head (two products of 2*D),
backward 10*D (five products: the score recompute, dP, dV, dK and dQ).
Activation arithmetic is not counted.
"""
from __future__ import annotations

import numpy as np


def pairs_per_sequence(lq, lkv, mask: int, window: int) -> np.ndarray:
    """Allowed (i, j) pairs of each sequence (one head). mask bits: 1 causal,
    2 window of W keys (implies causal), 4 blocks of W keys."""
    lq = np.asarray(lq, dtype=np.int64)
    lkv = np.asarray(lkv, dtype=np.int64)
    out = np.zeros(len(lq), dtype=np.int64)
    causal = bool(mask & 3)
    win = bool(mask & 2)
    blk = bool(mask & 4)
    for b in range(len(lq)):
        n, m = int(lq[b]), int(lkv[b])
        if n == 0 or m == 0:
            continue
        i = np.arange(n, dtype=np.int64)
        delta = m - n
        hi = np.minimum(m, i + delta + 1) if causal else np.full(n, m, dtype=np.int64)
        lo = np.maximum(0, i + delta - window + 1) if win else np.zeros(n, dtype=np.int64)
        if blk:
            start = np.floor_divide(i + delta, window) * window
            lo = np.maximum(lo, start)
            hi = np.minimum(hi, start + window)
        out[b] = int(np.maximum(hi - lo, 0).sum())
    return out


def effective_flops(pairs: int, H: int, D: int):
    """(forward, backward) effective FLOPs for `pairs` allowed pairs per head."""
    return 4.0 * D * H * pairs, 10.0 * D * H * pairs


def short_query_path(act: int, mask: int, D: int, lq, lkv) -> bool:
    """Whether the library runs a batch on its short-query (pooling) kernels
    in both directions: a pointwise activation, no mask, D = 128, at most 64
    queries per sequence on average (the forward's rule) and every sequence
    with 1 <= Lq <= 64 or no keys (the backward's device-side gate)."""
    lq = np.asarray(lq, dtype=np.int64)
    lkv = np.asarray(lkv, dtype=np.int64)
    if act == 0 or mask != 0 or D != 128 or len(lq) == 0 or int(lq.sum()) > 64 * len(lq):
        return False
    return bool(np.all(((lq >= 1) & (lq <= 64)) | (lkv == 0)))


def short_key_path(act: int, mask: int, D: int, lq, lkv) -> bool:
    """Whether the library runs a batch as cross-attention over short key
    sequences: the short-key forward and the short-key fused backward. A
    pointwise activation, no mask, D = 128, more than 64 queries but at most
    128 keys per sequence on average (the host's rule) and every sequence with
    Lkv <= 128 and keys whenever it has queries (the device-side gate)."""
    lq = np.asarray(lq, dtype=np.int64)
    lkv = np.asarray(lkv, dtype=np.int64)
    if act == 0 or mask != 0 or D != 128 or len(lq) == 0:
        return False
    if int(lq.sum()) <= 64 * len(lq) or int(lkv.sum()) > 128 * len(lq):
        return False
    return bool(np.all((lkv <= 128) & ((lkv >= 1) | (lq == 0))))


def kernel_work(total_q: int, total_kv: int, pairs: int, H: int, D: int, softmax: bool, in_tile: bool = False,
                fused_bwd: bool = False):
    """Algorithmic FLOPs and HBM bytes of each kernel (each byte read or written once).

    forward: reads Q, K, V, writes O (+ LSE)
    dq:      reads Q, K, V, dO (+ LSE), writes dQ; the dQ product (its score
             and dP recompute are not algorithmic work). For softmax it also
             reads O and writes Di = rowsum(dO * O), which the dK/dV pass uses.
             With in-tile statistics (BlockAttention whose blocks divide the
             tile) it reads neither O nor LSE and writes LSE and Di instead.
    dkdv:    reads Q, K, V, dO (+ LSE, Di), writes dK, dV; products S, dP, dV, dK

    fused_bwd (short_query_path or short_key_path): the fused backward, timed
    in the dK/dV slot, reads Q, dO, K, V once and writes dQ, dK, dV, computing
    all five products; the general dQ pass then finds no work.
    """
    e = 2 * H * D  # bytes of one row of a [total, H, D] bf16 tensor
    stats = 4 * H * total_q
    dq_extra = 0
    if softmax:
        dq_extra = 2 * stats if in_tile else e * total_q + 2 * stats
    if fused_bwd:
        return {
            "fwd": {"flops": 4.0 * D * H * pairs, "bytes": e * (2 * total_q + 2 * total_kv)},
            "dkdv": {"flops": 10.0 * D * H * pairs, "bytes": e * (3 * total_q + 4 * total_kv)},
            "dq": {"flops": 0.0, "bytes": 0.0},
        }
    return {
        "fwd": {"flops": 4.0 * D * H * pairs, "bytes": e * (2 * total_q + 2 * total_kv) + (stats if softmax else 0)},
        "dkdv": {"flops": 8.0 * D * H * pairs,
                 "bytes": e * (2 * total_q + 4 * total_kv) + (2 * stats if softmax else 0)},
        "dq": {"flops": 2.0 * D * H * pairs, "bytes": e * (3 * total_q + 2 * total_kv) + dq_extra},
    }
