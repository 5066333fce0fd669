"""Padded dense attention in torch fp64 on the CPU (tests only).

An independent route to the same numbers as the oracle: sequences are padded
into [B, H, Lmax, D] blocks, scores come from one batched matmul, masks are
boolean matrices built from the mask definition, the softmax is torch's own
(or torch's scaled_dot_product_attention), the pointwise activations are
torch.nn.functional.silu / gelu(approximate="tanh"), and gradients come from
torch autograd rather than hand-derived formulas.
"""
from __future__ import annotations

import numpy as np
import torch
import torch.nn.functional as F

SOFTMAX, SILU, GELU, GELU_POLY = 0, 1, 2, 3

# tanh-GELU's Taylor polynomial at 0 through x^6 (activation GELU_POLY): with
# c = sqrt(2/pi), a = 0.044715, the coefficients of x^2, x^4 and x^6
_C, _A = float(np.sqrt(2.0 / np.pi)), 0.044715
POLY_G2 = _C / 2
POLY_G4 = (_C * _A - _C**3 / 3) / 2
POLY_G6 = (2 * _C**5 / 15 - _C**3 * _A) / 2


def gelu_poly(x):
    """The polynomial, for torch tensors or numpy arrays (autograd-friendly)."""
    x2 = x * x
    return 0.5 * x + x2 * (POLY_G2 + x2 * (POLY_G4 + x2 * POLY_G6))


def mask_matrix(lq: int, lkv: int, mask: int, window: int) -> torch.Tensor:
    i = torch.arange(lq).view(-1, 1)
    j = torch.arange(lkv).view(1, -1)
    delta = lkv - lq
    ok = torch.ones(lq, lkv, dtype=torch.bool)
    if mask & 3:
        ok &= j <= i + delta
    if mask & 2:
        ok &= (i + delta - j) < window
    if mask & 4:  # blocks of `window` keys; python // rounds toward -inf
        ok &= (j // window) == ((i + delta) // window)
    return ok


def pad(x: torch.Tensor, off, lmax: int) -> torch.Tensor:
    B = len(off) - 1
    T, H, D = x.shape
    out = torch.zeros(B, H, lmax, D, dtype=x.dtype)
    for b in range(B):
        seg = x[off[b] : off[b + 1]]
        out[b, :, : seg.shape[0]] = seg.permute(1, 0, 2)
    return out


def unpad(x: torch.Tensor, off) -> torch.Tensor:
    B, H, L, D = x.shape
    parts = [x[b, :, : off[b + 1] - off[b]].permute(1, 0, 2) for b in range(B)]
    return torch.cat(parts, 0) if parts else x.new_zeros(0, H, D)


def dense_forward(q, k, v, q_off, kv_off, act, mask, window, scale, norm_by_lkv):
    """Padded dense forward; returns (o [total_q,H,D], lse [total_q,H]) in fp64."""
    q_off = [int(x) for x in q_off]
    kv_off = [int(x) for x in kv_off]
    B = len(q_off) - 1
    lq = [q_off[b + 1] - q_off[b] for b in range(B)]
    lk = [kv_off[b + 1] - kv_off[b] for b in range(B)]
    Lq, Lk = max(lq + [1]), max(lk + [1])
    Qp, Kp, Vp = pad(q, q_off, Lq), pad(k, kv_off, Lk), pad(v, kv_off, Lk)
    M = torch.zeros(B, 1, Lq, Lk, dtype=torch.bool)
    for b in range(B):
        M[b, 0, : lq[b], : lk[b]] = mask_matrix(lq[b], lk[b], mask, window)
    S = scale * torch.matmul(Qp, Kp.transpose(-1, -2))
    if act == SOFTMAX:
        Sm = S.masked_fill(~M, float("-inf"))
        lse = torch.logsumexp(Sm, dim=-1)
        P = torch.softmax(Sm, dim=-1)
        P = torch.nan_to_num(P, nan=0.0)
    else:
        A = F.silu(S) if act == SILU else (gelu_poly(S) if act == GELU_POLY else F.gelu(S, approximate="tanh"))
        c = torch.tensor([1.0 / x if (norm_by_lkv and x > 0) else 1.0 for x in lk], dtype=S.dtype)
        P = A * M * c.view(B, 1, 1, 1)
        lse = torch.zeros(B, q.shape[1], Lq, dtype=S.dtype)
    O = torch.matmul(P, Vp)
    o = unpad(O, q_off)
    lse_u = unpad(lse.unsqueeze(-1), q_off)[..., 0]
    return o, lse_u


def dense_grads(q, k, v, do, q_off, kv_off, act, mask, window, scale, norm_by_lkv):
    """Gradients of sum(o * do) by torch autograd through dense_forward."""
    q = q.detach().clone().requires_grad_(True)
    k = k.detach().clone().requires_grad_(True)
    v = v.detach().clone().requires_grad_(True)
    o, _ = dense_forward(q, k, v, q_off, kv_off, act, mask, window, scale, norm_by_lkv)
    (o * do).sum().backward()
    return q.grad, k.grad, v.grad


def sdpa_per_sequence(q, k, v, q_off, kv_off, mask, window, scale):
    """Softmax attention via torch.nn.functional.scaled_dot_product_attention,
    one sequence at a time with an explicit boolean mask. Rows with no
    visible key come back as NaN from the library and are returned as NaN."""
    outs = []
    B = len(q_off) - 1
    for b in range(B):
        qs = q[q_off[b] : q_off[b + 1]].permute(1, 0, 2)
        ks = k[kv_off[b] : kv_off[b + 1]].permute(1, 0, 2)
        vs = v[kv_off[b] : kv_off[b + 1]].permute(1, 0, 2)
        if qs.shape[1] == 0:
            continue
        if ks.shape[1] == 0:
            outs.append(torch.full((qs.shape[1], qs.shape[0], qs.shape[2]), float("nan"), dtype=q.dtype))
            continue
        m = mask_matrix(qs.shape[1], ks.shape[1], mask, window)
        o = F.scaled_dot_product_attention(qs.unsqueeze(0), ks.unsqueeze(0), vs.unsqueeze(0), attn_mask=m, scale=scale)
        outs.append(o[0].permute(1, 0, 2))
    if not outs:
        return q.new_zeros(0, q.shape[1], q.shape[2])
    return torch.cat(outs, 0)


def to_f64(x) -> torch.Tensor:
    if isinstance(x, np.ndarray):
        return torch.from_numpy(x)
    return x.detach().to(torch.float64).cpu()


def rope_tables(rows, D, base=10000.0):
    """RoFormer angles pos * base^(-2m/D) as cos / sin tables [rows, D/2] (and the angles)."""
    theta = base ** (-2.0 * np.arange(D // 2) / D)
    ang = np.arange(rows)[:, None] * theta[None, :]
    return np.cos(ang), np.sin(ang), ang
