"""Seeded synthetic inputs for jagged attention workloads.

This module only draws random lengths and values; it holds none of the
attention arithmetic, and both the CUDA path and the CPU oracle consume what
it produces.

Workloads (the recommendation-model shapes of the "GEM Training" post:
jagged user histories of hundreds to tens of thousands of events, long-query
short-key cross-attention, and short-query pooling attention over long
histories):

* ``tiny``       4 sequences of lengths {3, 17, 64, 130}, H=2, D=64, softmax, causal
* ``jfa``        B=128, lengths lognormal(median 1024, sigma 1) clipped to
                 [64, 16384], H=4, D=128, softmax, causal + window 256
* ``jfa_causal`` the same lengths, causal only (no window)
* ``gdpa_cross`` B=512, Lq lognormal(median 1024, sigma 1) clipped to
                 [128, 8192], Lkv uniform integers in [16, 128], H=8, D=128,
                 values N(0, 0.5^2), SiLU with 1/Lkv normaliser, no mask
* ``gdpa_pma``   B=512, 32 queries per sequence, Lkv lognormal(median 2048,
                 sigma 1) clipped to [100, 20000], H=8, D=128, N(0, 0.5^2),
                 tanh-GELU with 1/Lkv normaliser, no mask
* ``gdpa_pma_poly`` the ``gdpa_pma`` lengths and shapes with GDPA's ALU-only
                 GELU (tanh-GELU's degree-6 Taylor polynomial); query and key
                 rows normalised so that every score has |s| <= 1, the range
                 the polynomial is accurate on
* ``jfa_block``  the ``jfa`` lengths with block attention instead of the
                 window: each query sees only its own 64-key block (the
                 "BlockAttention" step of the same post)
* ``mixed``      B=1024, exactly round(0.3 B) long sequences uniform in
                 [4000, 32000] and the rest short, uniform in [50, 500],
                 shuffled; H=8, D=128, softmax, causal + window 512

Lengths come from ``numpy.random.default_rng(seed)`` (lognormal draws are
rounded with ``np.rint`` then clipped); values come from a
``torch.Generator`` seeded with ``seed`` on the target device, drawn
standard-normal, multiplied by the stated standard deviation and rounded to
bf16 (round-to-nearest-even). Draw order: q, k, v, then dO (always N(0, 1)).
"""
from __future__ import annotations

from dataclasses import dataclass, replace

import numpy as np

SOFTMAX, SILU, GELU, GELU_POLY = 0, 1, 2, 3
MASK_NONE, MASK_CAUSAL, MASK_WINDOW, MASK_BLOCK = 0, 1, 2, 4


@dataclass(frozen=True)
class Workload:
    name: str
    H: int
    D: int
    act: int
    mask: int
    window: int
    norm_by_lkv: bool
    std: float
    self_attn: bool
    # > 0: query and key rows are scaled to L2 norm sqrt(qk_norm * sqrt(D)),
    # as a query/key normalisation layer would leave them, so that with the
    # default scale 1/sqrt(D) every score satisfies |s| <= qk_norm (up to the
    # bf16 rounding of the rows)
    qk_norm: float = 0.0


WORKLOADS = {
    "tiny": Workload("tiny", 2, 64, SOFTMAX, MASK_CAUSAL, 0, False, 1.0, True),
    "jfa": Workload("jfa", 4, 128, SOFTMAX, MASK_CAUSAL | MASK_WINDOW, 256, False, 1.0, True),
    "jfa_causal": Workload("jfa_causal", 4, 128, SOFTMAX, MASK_CAUSAL, 0, False, 1.0, True),
    "jfa_block": Workload("jfa_block", 4, 128, SOFTMAX, MASK_BLOCK, 64, False, 1.0, True),
    "gdpa_cross": Workload("gdpa_cross", 8, 128, SILU, MASK_NONE, 0, True, 0.5, False),
    "gdpa_pma": Workload("gdpa_pma", 8, 128, GELU, MASK_NONE, 0, True, 0.5, False),
    "gdpa_pma_poly": Workload("gdpa_pma_poly", 8, 128, GELU_POLY, MASK_NONE, 0, True, 0.5, False, 1.0),
    "mixed": Workload("mixed", 8, 128, SOFTMAX, MASK_CAUSAL | MASK_WINDOW, 512, False, 1.0, True),
}


def _lognormal_int(rng, median, n, lo, hi):
    x = rng.lognormal(mean=np.log(median), sigma=1.0, size=n)
    return np.clip(np.rint(x), lo, hi).astype(np.int64)


def lengths(name: str, seed: int = 0):
    """Per-sequence (Lq, Lkv) int64 arrays for a named workload."""
    rng = np.random.default_rng(seed)
    if name == "tiny":
        lq = np.array([3, 17, 64, 130], dtype=np.int64)
        return lq, lq.copy()
    if name in ("jfa", "jfa_causal", "jfa_block"):
        lq = _lognormal_int(rng, 1024, 128, 64, 16384)
        return lq, lq.copy()
    if name == "gdpa_cross":
        lq = _lognormal_int(rng, 1024, 512, 128, 8192)
        lkv = rng.integers(16, 129, size=512).astype(np.int64)
        return lq, lkv
    if name in ("gdpa_pma", "gdpa_pma_poly"):
        lkv = _lognormal_int(rng, 2048, 512, 100, 20000)
        lq = np.full(512, 32, dtype=np.int64)
        return lq, lkv
    if name == "mixed":
        B = 1024
        n_long = int(round(0.3 * B))
        short = rng.integers(50, 501, size=B - n_long)
        long_ = rng.integers(4000, 32001, size=n_long)
        lq = rng.permutation(np.concatenate([short, long_])).astype(np.int64)
        return lq, lq.copy()
    raise KeyError(name)


def offsets(lens: np.ndarray) -> np.ndarray:
    """int64 prefix sums [B+1] starting at 0."""
    out = np.zeros(len(lens) + 1, dtype=np.int64)
    np.cumsum(lens, out=out[1:])
    return out


def values(shape, std: float, seed: int, device="cpu", row_norm: float = 0.0):
    """bf16 tensor of N(0, std^2) draws from a seeded torch generator; with
    row_norm > 0 every last-axis row is then scaled to that L2 norm."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if row_norm > 0:
        x.mul_(row_norm / x.norm(dim=-1, keepdim=True).clamp_min(1e-30))
    return x.to(torch.bfloat16)


def make(name_or_workload, seed: int = 0, device="cpu", lens=None, with_grad_out=True):
    """Build a full input set.

    Returns dict with q_off, kv_off (int64 torch tensors on ``device``; one
    shared tensor for self-attention with equal lengths),
    q, k, v, do (bf16 [total, H, D]) and the Workload. ``lens`` overrides the
    sampled (Lq, Lkv) lengths. Each tensor uses its own generator seeded
    from ``seed`` (q: seed, k: seed+1, v: seed+2, dO: seed+3).
    """
    import torch

    w = WORKLOADS[name_or_workload] if isinstance(name_or_workload, str) else name_or_workload
    if lens is None:
        lq, lkv = lengths(w.name, seed)
    else:
        lq, lkv = (np.asarray(lens[0], dtype=np.int64), np.asarray(lens[1], dtype=np.int64))
    qo, ko = offsets(lq), offsets(lkv)
    tq, tk = int(qo[-1]), int(ko[-1])
    qk_row = float(np.sqrt(w.qk_norm * np.sqrt(w.D))) if w.qk_norm > 0 else 0.0
    q_off = torch.from_numpy(qo).to(device)
    # self-attention with equal lengths shares one offsets tensor for both sides
    same = w.self_attn and np.array_equal(lq, lkv)
    out = {
        "workload": w,
        "lq": lq,
        "lkv": lkv,
        "q_off": q_off,
        "kv_off": q_off if same else torch.from_numpy(ko).to(device),
        "q": values((tq, w.H, w.D), w.std, seed, device, qk_row),
        "k": values((tk, w.H, w.D), w.std, seed + 1, device, qk_row),
        "v": values((tk, w.H, w.D), w.std, seed + 2, device),
    }
    if with_grad_out:
        out["do"] = values((tq, w.H, w.D), 1.0, seed + 3, device)
    return out


def with_params(w: Workload, **kw) -> Workload:
    return replace(w, **kw)
