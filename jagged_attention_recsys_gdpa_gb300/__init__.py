"""Jagged generalized dot-product attention for one GB300 (sm_103a).

Public API (thin wrappers over the C-ABI library ``libjattn``; every step of
the computation runs in its CUDA kernels):

* ``attention(q, k, v, q_off, kv_off, act=..., causal=..., window=..., scale=...,
  norm_by_lkv=..., block=..., rope=...)``: autograd-enabled jagged attention
  returning O.
* ``forward(...)`` -> (O, LSE) and ``backward(...)`` -> (dQ, dK, dV): the raw passes.
* ``rope(x, q_off, kv_off, (cos, sin), keys=..., inverse=...)``: rotary
  embedding of query or key rows; ``backward(..., rope=(cos, sin))`` and
  ``attention(..., rope=(cos, sin))`` rotate dQ and dK back inside the
  backward kernels' epilogues.
* ``mxfp8_quantize(x, off)``: FP8 E4M3 codes plus one E8M0 scale per 32 x 32
  block of a jagged tensor; ``forward_mxfp8(qm, km, vm, q_off, kv_off, ...)``:
  the softmax forward on such operands (block-scaled FP8 tensor-core products).
* ``schedule(...)``: the device-built longest-first tile list.

Activations (``act``): "softmax", "silu", "gelu" (tanh form) or "gelu_poly"
(its degree-6 Taylor polynomial on the FMA pipe, for |scores| <= 1).
Masks: ``causal``; ``window`` = W > 0 (sliding window of W keys ending at the
query's own position, implies causal); ``block`` = W > 0 (each query sees only
the keys of its own W-wide block, optionally causal inside it; not combined
with ``window``).

Tensors: q [total_q, H, D], k / v [total_kv, H, D] in bf16 on a CUDA device;
q_off / kv_off int64 [B+1] prefix sums on the same device. D is 64 or 128.
"""
from __future__ import annotations

import torch

from . import _binding as B

SOFTMAX, SILU, GELU_TANH, GELU_POLY = B.SOFTMAX, B.SILU, B.GELU_TANH, B.GELU_POLY
MASK_NONE, MASK_CAUSAL, MASK_WINDOW, MASK_BLOCK = B.MASK_NONE, B.MASK_CAUSAL, B.MASK_WINDOW, B.MASK_BLOCK
JattnError = B.JattnError

_ACTS = {"softmax": SOFTMAX, "silu": SILU, "gelu": GELU_TANH, "gelu_tanh": GELU_TANH, "gelu_poly": GELU_POLY}

_ws_cache: dict = {}


def _act(a) -> int:
    return _ACTS[a] if isinstance(a, str) else int(a)


def _mask(causal: bool, window: int, block: int = 0) -> int:
    if block and block > 0:
        if window and window > 0:
            raise ValueError("block and window masks do not combine")
        return MASK_BLOCK | (MASK_CAUSAL if causal else 0)
    if window and window > 0:
        return MASK_CAUSAL | MASK_WINDOW
    return MASK_CAUSAL if causal else MASK_NONE


def _width(window: int, block: int) -> int:
    """The width the library reads from params.window: the block size or the window."""
    return int(block) if block and block > 0 else (int(window) if window and window > 0 else 0)


def _check(q, k, v, q_off, kv_off):
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16 or not t.is_cuda or t.dim() != 3 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA bf16 tensor [total, H, D]")
    for name, t in (("q_off", q_off), ("kv_off", kv_off)):
        if t.dtype != torch.int64 or not t.is_cuda or t.dim() != 1:
            raise ValueError(f"{name} must be a CUDA int64 tensor [B+1]")
    if q_off.numel() != kv_off.numel() or q_off.numel() < 2:
        raise ValueError("q_off and kv_off must both have B+1 >= 2 entries")
    if k.shape != v.shape or q.shape[1:] != k.shape[1:]:
        raise ValueError("q, k, v must share H and D; k and v must have the same shape")


def make_params(q, k, q_off, act, mask, width, scale, norm_by_lkv) -> B.Params:
    return B.params(q_off.numel() - 1, q.shape[0], k.shape[0], q.shape[1], q.shape[2], act, mask,
                    width if mask & (MASK_WINDOW | MASK_BLOCK) else 0, scale, norm_by_lkv)


def workspace(p: B.Params, device, need: int | None = None) -> torch.Tensor:
    """Cached zero-initialised workspace of at least the size ``p`` needs
    (or ``need`` bytes). One per device: calls through this module that run
    at the same time on different streams of one device would share its
    status word and schedules, so issue them from one stream (or call the
    C ABI with a workspace per stream)."""
    need = B.workspace_size(p) if need is None else need
    dev = torch.device(device)
    key = dev.index if dev.index is not None else torch.cuda.current_device()
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < need:
        grown = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
        if ws is not None:
            # keep an error status that an earlier call left and nobody has read yet
            grown[:256].copy_(ws[:256])
        ws = grown
        _ws_cache[key] = ws
    return ws


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def forward(q, k, v, q_off, kv_off, act="softmax", causal=False, window=0, scale=None, norm_by_lkv=False,
            out=None, lse=None, block=0):
    """Forward pass. Returns (O [total_q,H,D] bf16, LSE [total_q,H] fp32 or None)."""
    _check(q, k, v, q_off, kv_off)
    a = _act(act)
    p = make_params(q, k, q_off, a, _mask(causal, window, block), _width(window, block), scale, norm_by_lkv)
    o = out if out is not None else torch.empty_like(q)
    if a == SOFTMAX and lse is None:
        lse = torch.empty(q.shape[0], q.shape[1], dtype=torch.float32, device=q.device)
    ws = workspace(p, q.device)
    B.fwd(p, q_off, kv_off, q, k, v, o, lse if a == SOFTMAX else None, ws.data_ptr(), ws.numel(),
          _stream(q.device))
    return o, (lse if a == SOFTMAX else None)


def _rope_tables(rope, D, device):
    cos, sin = rope
    for t in (cos, sin):
        if t.dtype != torch.float32 or t.dim() != 2 or t.shape[1] != D // 2 or t.device != torch.device(device):
            raise ValueError("rope tables must be fp32 [rows, D/2] on the tensors' device")
    if cos.shape != sin.shape:
        raise ValueError("rope cos and sin tables differ in shape")
    return cos.contiguous(), sin.contiguous()


def rope(x, q_off, kv_off, tables, keys=False, inverse=False, out=None):
    """Rotary embedding of jagged query rows (or key rows with ``keys``):
    y = R(pos) x, or R(pos)^T x with ``inverse``. ``tables`` = (cos, sin) fp32
    [rows, D/2]; positions as in jattn.h (both sides of a sequence end at the
    same position, the longer one starts at 0)."""
    if q_off.numel() != kv_off.numel() or q_off.numel() < 2:
        raise ValueError("q_off and kv_off must both have B+1 >= 2 entries")
    H, D = x.shape[1], x.shape[2]
    cos, sin = _rope_tables(tables, D, x.device)
    x = x.contiguous()
    y = out if out is not None else torch.empty_like(x)
    # the pass reads only this side's total from the params
    tq, tk = (0, x.shape[0]) if keys else (x.shape[0], 0)
    p = B.params(q_off.numel() - 1, tq, tk, H, D, SOFTMAX, 0, 0, 0.0, False)
    ws = workspace(p, x.device)
    B.rope(p, q_off, kv_off, keys, inverse, x, y, cos, sin, ws.data_ptr(), ws.numel(), _stream(x.device))
    return y


def mxfp8_quantize(x, off):
    """MXFP8 quantization of jagged bf16 rows x [total, H, D] (offsets ``off``):
    returns (codes uint8 [total, H, D], scale exponents uint8 [rows, H, D/32],
    block_start int32 [B+1]); row block r of sequence b is scale row
    block_start[b] + r. See jattn_mxfp8_quantize."""
    if x.dtype != torch.bfloat16 or x.dim() != 3 or off.dtype != torch.int64 or off.numel() < 2:
        raise ValueError("x must be bf16 [total, H, D] and off int64 [B+1]")
    x = x.contiguous()
    total, H, D = x.shape
    nb = off.numel() - 1
    codes = torch.empty((total, H, D), dtype=torch.uint8, device=x.device)
    scales = torch.zeros((B.mxfp8_scale_rows(nb, total), H, D // 32), dtype=torch.uint8, device=x.device)
    block_start = torch.empty(nb + 1, dtype=torch.int32, device=x.device)
    p = B.params(nb, total, total, H, D, SOFTMAX, 0, 0, 0.0, False)
    ws = workspace(p, x.device, max(B.workspace_size(p), 512))
    B.mxfp8_quantize(nb, total, H, D, off, x, codes, scales, block_start, ws.data_ptr(), ws.numel(),
                     _stream(x.device))
    return codes, scales, block_start


def forward_mxfp8(qm, km, vm, q_off, kv_off, causal=False, window=0, block=0, scale=None, out=None, lse=None):
    """Softmax attention forward on MXFP8 operands: qm, km, vm are the
    (codes, scales, block_start) triples mxfp8_quantize returns (km and vm
    quantized with kv_off). D must be 128. Returns (O bf16, LSE fp32)."""
    (qc, qs, qbs), (kc, ks, kbs), (vc, vs, _) = qm, km, vm
    total_q, H, D = qc.shape
    p = B.params(q_off.numel() - 1, total_q, kc.shape[0], H, D, SOFTMAX, _mask(causal, window, block),
                 _width(window, block), scale, False)
    o = out if out is not None else torch.empty((total_q, H, D), dtype=torch.bfloat16, device=qc.device)
    lse = lse if lse is not None else torch.empty((total_q, H), dtype=torch.float32, device=qc.device)
    ws = workspace(p, qc.device)
    B.fwd_mxfp8(p, q_off, kv_off, qc, qs, qbs, kc, ks, vc, vs, kbs, o, lse, ws.data_ptr(), ws.numel(),
                _stream(qc.device))
    return o, lse


def backward_mxfp8(qm, km, vm, o, lse, dom, q_off, kv_off, causal=False, window=0, block=0, scale=None, dq=None,
                   dk=None, dv=None):
    """Softmax attention backward on MXFP8 operands: qm, km, vm, dom are
    mxfp8_quantize triples (dom quantized with q_off), o and lse the
    forward's outputs. D must be 128. Returns (dQ, dK, dV) bf16."""
    (qc, qs, qbs), (kc, ks, kbs), (vc, vs, _), (dc, ds, _) = qm, km, vm, dom
    total_q, H, D = qc.shape
    total_kv = kc.shape[0]
    p = B.params(q_off.numel() - 1, total_q, total_kv, H, D, SOFTMAX, _mask(causal, window, block),
                 _width(window, block), scale, False)
    dev = qc.device
    dq = dq if dq is not None else torch.empty((total_q, H, D), dtype=torch.bfloat16, device=dev)
    dk = dk if dk is not None else torch.empty((total_kv, H, D), dtype=torch.bfloat16, device=dev)
    dv = dv if dv is not None else torch.empty((total_kv, H, D), dtype=torch.bfloat16, device=dev)
    ws = workspace(p, dev)
    B.bwd_mxfp8(p, q_off, kv_off, qc, qs, qbs, kc, ks, vc, vs, kbs, o, lse, dc, ds, dq, dk, dv, ws.data_ptr(),
                ws.numel(), _stream(dev))
    return dq, dk, dv


def backward(q, k, v, o, lse, do, q_off, kv_off, act="softmax", causal=False, window=0, scale=None,
             norm_by_lkv=False, dq=None, dk=None, dv=None, block=0, rope=None):
    """Backward pass. Returns (dQ, dK, dV) bf16. With ``rope`` = (cos, sin)
    tables, q and k are the rotated rows the forward read and dQ, dK are
    returned for the unrotated ones (rotated back in the kernels' epilogues)."""
    _check(q, k, v, q_off, kv_off)
    a = _act(act)
    p = make_params(q, k, q_off, a, _mask(causal, window, block), _width(window, block), scale, norm_by_lkv)
    dq = dq if dq is not None else torch.empty_like(q)
    dk = dk if dk is not None else torch.empty_like(k)
    dv = dv if dv is not None else torch.empty_like(v)
    do = do.contiguous()
    if rope is not None:
        cos, sin = _rope_tables(rope, q.shape[2], q.device)
        ws = workspace(p, q.device, B.bwd_rope_workspace_size(p, cos.shape[0]))
        B.bwd_rope(p, q_off, kv_off, q, k, v, o if a == SOFTMAX else None, lse if a == SOFTMAX else None, do, cos,
                   sin, dq, dk, dv, ws.data_ptr(), ws.numel(), _stream(q.device))
        return dq, dk, dv
    ws = workspace(p, q.device)
    B.bwd(p, q_off, kv_off, q, k, v, o if a == SOFTMAX else None, lse if a == SOFTMAX else None, do, dq, dk,
          dv, ws.data_ptr(), ws.numel(), _stream(q.device))
    return dq, dk, dv


class _JaggedAttention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, q_off, kv_off, act, causal, window, scale, norm_by_lkv, block, rope_cos, rope_sin):
        rope_t = None
        if rope_cos is not None:  # attention on R q and R k; the backward rotates dQ, dK back
            rope_t = (rope_cos, rope_sin)
            q = rope(q, q_off, kv_off, rope_t, keys=False)
            k = rope(k, q_off, kv_off, rope_t, keys=True)
        o, lse = forward(q, k, v, q_off, kv_off, act, causal, window, scale, norm_by_lkv, block=block)
        ctx.save_for_backward(q, k, v, o, lse if lse is not None else o.new_empty(0), q_off, kv_off)
        ctx.cfg = (act, causal, window, scale, norm_by_lkv, block, rope_t)
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, lse, q_off, kv_off = ctx.saved_tensors
        act, causal, window, scale, norm_by_lkv, block, rope_t = ctx.cfg
        dq, dk, dv = backward(q, k, v, o, lse if lse.numel() else None, do, q_off, kv_off, act, causal, window,
                              scale, norm_by_lkv, block=block, rope=rope_t)
        return dq, dk, dv, None, None, None, None, None, None, None, None, None, None


def attention(q, k, v, q_off, kv_off, act="softmax", causal=False, window=0, scale=None, norm_by_lkv=False,
              block=0, rope=None):
    """Jagged attention with autograd: O = act(scale Q K^T masked) V per sequence.
    With ``rope`` = (cos, sin) tables, queries and keys are rotated first
    (jattn_rope) and the backward rotates their gradients back in its
    epilogues (jattn_bwd_rope)."""
    rc, rs = rope if rope is not None else (None, None)
    return _JaggedAttention.apply(q, k, v, q_off, kv_off, act, causal, window, scale, norm_by_lkv, block, rc, rs)


def schedule(q_off, kv_off, H, D=128, causal=False, window=0, row_tile=128, col_tile=128, transposed=False,
             total_q=None, total_kv=None, block=0):
    """The longest-first tile list the kernels consume: int32 [n, 4] (b, row tile, col lo, col hi)."""
    tq = int(total_q) if total_q is not None else int(q_off[-1].item())
    tk = int(total_kv) if total_kv is not None else int(kv_off[-1].item())
    p = B.params(q_off.numel() - 1, tq, tk, H, D, SOFTMAX, _mask(causal, window, block), _width(window, block), 0.0,
                 False)
    mt = B.max_tiles(p, row_tile, transposed)
    tiles = torch.zeros(mt, 4, dtype=torch.int32, device=q_off.device)
    n = torch.zeros(1, dtype=torch.int32, device=q_off.device)
    ws = workspace(p, q_off.device)
    B.schedule(p, q_off, kv_off, row_tile, col_tile, transposed, tiles, mt, n, ws.data_ptr(), ws.numel(),
               _stream(q_off.device))
    return tiles[: int(n.item())]


def device_status(device=None) -> int:
    """Read and clear the device status word of the cached workspace (syncs)."""
    dev = torch.device(device) if device is not None else torch.device("cuda", torch.cuda.current_device())
    key = dev.index if dev.index is not None else torch.cuda.current_device()
    ws = _ws_cache.get(key)
    if ws is None:
        return 0
    return B.get_status(ws.data_ptr(), _stream(dev))
