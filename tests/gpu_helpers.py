"""Shared helpers for the GPU parity tests: run the CUDA path and the oracle on
the same bf16 inputs and compare element by element."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from jagged_attention_recsys_gdpa_gb300 import inputs

# bf16 inputs, fp32 accumulation: |got - ref| <= ATOL + RTOL * |ref|
ATOL = 1e-2
RTOL = 1e-2

ACT_NAME = {0: "softmax", 1: "silu", 2: "gelu", 3: "gelu_poly"}


def gpu_run(inp, w, backward=True, stored=None):
    """Forward (+ backward) through the public API on the tensors' device.
    stored: None (the backward reads this forward's O and LSE) or (o, lse)
    device tensors for the backward to read instead."""
    import jagged_attention_recsys_gdpa_gb300 as J

    causal = bool(w.mask & 1)
    window = w.window if w.mask & 2 else 0
    block = w.window if w.mask & 4 else 0
    o, lse = J.forward(inp["q"], inp["k"], inp["v"], inp["q_off"], inp["kv_off"], act=w.act, causal=causal,
                       window=window, block=block, norm_by_lkv=w.norm_by_lkv)
    out = {"o": o, "lse": lse}
    if backward:
        if stored is not None:
            o, lse = stored
        dq, dk, dv = J.backward(inp["q"], inp["k"], inp["v"], o, lse, inp["do"], inp["q_off"], inp["kv_off"],
                                act=w.act, causal=causal, window=window, block=block, norm_by_lkv=w.norm_by_lkv)
        out.update(dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    return out


def oracle_run(inp, w, backward=True, o_stored=None):
    kw = dict(H=w.H, D=w.D, act=w.act, mask=w.mask | (1 if w.mask & 2 else 0), window=w.window,
              norm_by_lkv=w.norm_by_lkv)
    o, lse = oracle.fwd(inp["q_off"], inp["kv_off"], inp["q"], inp["k"], inp["v"], **kw)
    out = {"o": o, "lse": lse}
    if backward:
        dq, dk, dv = oracle.bwd(inp["q_off"], inp["kv_off"], inp["q"], inp["k"], inp["v"], inp["do"], o=o_stored,
                                **kw)
        out.update(dq=dq, dk=dk, dv=dv)
    return out


def to64(t) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def assert_close(got, ref, name):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values from the GPU"
    err = np.abs(got - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    if bad.any():
        idx = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(
            f"{name}: {int(bad.sum())} of {bad.size} elements out of tolerance; worst at {idx}: "
            f"got {got[idx]:.6g} ref {ref[idx]:.6g}"
        )


def compare(g, r, w, backward=True, rows_q=None, rows_kv=None):
    """Compare GPU outputs g (torch) with oracle outputs r (numpy) on the given row subsets."""
    sel_q = slice(None) if rows_q is None else rows_q
    sel_kv = slice(None) if rows_kv is None else rows_kv
    assert_close(to64(g["o"])[sel_q], r["o"], "O")
    if w.act == 0:
        lg = g["lse"].detach().cpu().numpy().astype(np.float64)[sel_q]
        lr = r["lse"]
        assert np.array_equal(np.isneginf(lg), np.isneginf(lr)), "LSE: -inf rows differ"
        fin = np.isfinite(lr)
        assert_close(lg[fin], lr[fin], "LSE")
    if backward:
        assert_close(to64(g["dq"])[sel_q], r["dq"], "dQ")
        assert_close(to64(g["dk"])[sel_kv], r["dk"], "dK")
        assert_close(to64(g["dv"])[sel_kv], r["dv"], "dV")


def cpu_inputs(w, lq, lkv, seed):
    return inputs.make(w, seed=seed, device="cpu", lens=(lq, lkv))


def to_cuda(inp):
    out = dict(inp)
    for k in ("q_off", "kv_off", "q", "k", "v", "do"):
        if k in inp:
            out[k] = inp[k].cuda()
    if inp.get("kv_off") is inp.get("q_off"):  # self-attention: keep one offsets tensor
        out["kv_off"] = out["q_off"]
    return out


def subset(inp, seqs):
    """CPU copy of the given sequences (rows and offsets) of a (GPU) input set,
    plus the row index arrays of those sequences in the full batch."""
    qo = inp["q_off"].cpu().numpy()
    ko = inp["kv_off"].cpu().numpy()
    rq = np.concatenate([np.arange(qo[b], qo[b + 1]) for b in seqs]).astype(np.int64)
    rk = np.concatenate([np.arange(ko[b], ko[b + 1]) for b in seqs]).astype(np.int64)
    lq = np.array([qo[b + 1] - qo[b] for b in seqs], dtype=np.int64)
    lk = np.array([ko[b + 1] - ko[b] for b in seqs], dtype=np.int64)
    tq, tk = torch.from_numpy(rq).to(inp["q"].device), torch.from_numpy(rk).to(inp["q"].device)
    sub = {
        "q_off": torch.from_numpy(inputs.offsets(lq)),
        "kv_off": torch.from_numpy(inputs.offsets(lk)),
        "q": inp["q"].index_select(0, tq).cpu(),
        "k": inp["k"].index_select(0, tk).cpu(),
        "v": inp["v"].index_select(0, tk).cpu(),
    }
    if "do" in inp:
        sub["do"] = inp["do"].index_select(0, tq).cpu()
    return sub, rq, rk


def backward_o(cpu, w, o_ref):
    """The output that softmax's D_i = <dO_i, O_i> is formed from, row by row,
    the way the backward kernels form it: a 128-row query tile whose allowed
    keys all lie in one 128-row key tile gets D_i = sum_j P_ij dP_ij in fp32,
    which equals D_i of the exact O; every other tile reads the stored O.
    Returns (the stored O as bf16 for the GPU, the per-row O for the oracle)."""
    o_st = torch.from_numpy(o_ref).to(torch.bfloat16)
    hyb = o_st.double().numpy()
    if w.act == 0:
        mask = w.mask | (1 if w.mask & 2 else 0)
        qo = cpu["q_off"].numpy()
        for b, t, lo, hi in oracle.schedule(cpu["q_off"], cpu["kv_off"], mask=mask, window=w.window):
            if hi - lo == 1:
                r0 = int(qo[b]) + 128 * int(t)
                r1 = min(r0 + 128, int(qo[b + 1]))
                hyb[r0:r1] = o_ref[r0:r1]
    return o_st, hyb


def run_both_stored(cpu, w, backward=True):
    """GPU and oracle runs whose backward passes both read the same stored
    forward output: the oracle's O rounded to bf16 and its LSE in fp32, as a
    correct forward would have stored them (the oracle forms D_i from it where
    the kernels do, see backward_o). This isolates the backward kernels' own
    arithmetic from the rounding of O, which enters D_i = <dO_i, O_i> (large
    next to dQ for rows that see one or two keys)."""
    r = oracle_run(cpu, w, backward=False)
    o_st, o_rows = backward_o(cpu, w, r["o"])
    lse_st = torch.from_numpy(r["lse"]).to(torch.float32)
    g = gpu_run(to_cuda(cpu), w, backward, stored=(o_st.cuda(), lse_st.cuda()))
    if backward:
        r.update({k: x for k, x in oracle_run(cpu, w, True, o_stored=o_rows).items() if k.startswith("d")})
    return g, r
