"""Data-parallel split of one jagged batch over ranks.

Sequences (and heads) are independent problems, so attention shards by
sequence with no exchange inside it. ``split`` assigns every sequence to a
rank through the C library's ``jattn_partition`` (cost = allowed pairs;
longest first onto the least-loaded rank), and ``shard`` turns one rank's
share into what it runs on: its own offsets and the rows of the global
tensors it owns, which also put its outputs back in place.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import _binding as B


@dataclass(frozen=True)
class Shard:
    seqs: np.ndarray     # int64 [B_r]: global indices of this rank's sequences, ascending
    q_off: np.ndarray    # int64 [B_r + 1]: offsets of the rank's query rows
    kv_off: np.ndarray   # int64 [B_r + 1]: offsets of the rank's key/value rows
    q_rows: np.ndarray   # int64 [total_q_r]: global query row of each local query row
    kv_rows: np.ndarray  # int64 [total_kv_r]: global key/value row of each local key/value row


def split(q_off, kv_off, n_ranks: int, mask: int = 0, window: int = 0):
    """(rank_of int32 [B], rank_pairs int64 [n_ranks]) for host int64 offsets."""
    q_off = np.ascontiguousarray(q_off, dtype=np.int64)
    kv_off = np.ascontiguousarray(kv_off, dtype=np.int64)
    if q_off.shape != kv_off.shape or q_off.ndim != 1 or len(q_off) < 2:
        raise ValueError("q_off and kv_off must both be int64 [B+1] with B >= 1")
    rank_of = np.zeros(len(q_off) - 1, dtype=np.int32)
    rank_pairs = np.zeros(max(int(n_ranks), 1), dtype=np.int64)
    B.partition(q_off, kv_off, mask, window, n_ranks, rank_of, rank_pairs)
    return rank_of, rank_pairs


def _rows(off: np.ndarray, seqs: np.ndarray) -> np.ndarray:
    if len(seqs) == 0:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate([np.arange(off[b], off[b + 1], dtype=np.int64) for b in seqs])


def shard(q_off, kv_off, rank_of, rank: int) -> Shard:
    """The sequences of `rank` in batch order, with local offsets and row maps."""
    q_off = np.asarray(q_off, dtype=np.int64)
    kv_off = np.asarray(kv_off, dtype=np.int64)
    seqs = np.flatnonzero(np.asarray(rank_of) == rank).astype(np.int64)
    lq = q_off[seqs + 1] - q_off[seqs]
    lkv = kv_off[seqs + 1] - kv_off[seqs]
    qo = np.zeros(len(seqs) + 1, dtype=np.int64)
    ko = np.zeros(len(seqs) + 1, dtype=np.int64)
    np.cumsum(lq, out=qo[1:])
    np.cumsum(lkv, out=ko[1:])
    return Shard(seqs, qo, ko, _rows(q_off, seqs), _rows(kv_off, seqs))
