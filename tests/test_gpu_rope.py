"""Rotary embedding on the GPU: the jagged rotation pass (jattn_rope) and the
backward whose epilogues rotate dQ and dK back (jattn_bwd_rope), against the
oracle's rotation composed with its backward."""
import numpy as np
import pytest
import torch

import oracle
from jagged_attention_recsys_gdpa_gb300 import inputs
from tests import gpu_helpers as G
from tests.dense_ref import rope_tables

pytestmark = pytest.mark.gpu

SOFTMAX, GELU = 0, 2
NONE, CAUSAL, BLOCK = 0, 1, 4
SELF_LENS = [1, 127, 128, 129, 255, 256, 257, 300, 513, 1000]
CROSS_LQ = [100, 300, 5, 700, 257, 1]
CROSS_LKV = [20, 128, 1, 257, 130, 64]


def _tables(D, rows=1024):
    cos, sin, _ = rope_tables(rows, D)
    return cos, sin, (torch.from_numpy(cos).float().cuda(), torch.from_numpy(sin).float().cuda())


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("lens", [(SELF_LENS, SELF_LENS), (CROSS_LQ, CROSS_LKV)], ids=["self", "cross"])
def test_rope_pass(D, lens):
    import jagged_attention_recsys_gdpa_gb300 as J

    w = inputs.Workload("case", 3, D, SOFTMAX, NONE, 0, False, 1.0, True)
    cpu = G.cpu_inputs(w, *lens, seed=81)
    x = G.to_cuda(cpu)
    cos, sin, t = _tables(D)
    for keys, name in ((False, "q"), (True, "k")):
        for inverse in (False, True):
            y = J.rope(x[name], x["q_off"], x["kv_off"], t, keys=keys, inverse=inverse)
            ref = oracle.rope(cpu[name], cpu["q_off"], cpu["kv_off"], cos, sin, keys=keys, inverse=inverse)
            G.assert_close(G.to64(y), ref, f"rope({name}, inverse={inverse})")
    assert J.device_status() == 0


def _check_bwd_rope(act, mask, window, D, lq, lkv, seed):
    """GPU: forward on q' = R q, k' = R k (the oracle's, rounded to bf16), then
    the rotary backward. Oracle: its backward on the same q', k', then R^T on
    dQ and dK. Softmax's backward reads the oracle's stored O on both sides
    (gpu_helpers.backward_o: where the kernels take D_i from the tile, the
    oracle takes it from the exact O)."""
    import jagged_attention_recsys_gdpa_gb300 as J

    norm = act != SOFTMAX
    w = inputs.Workload("case", 2, D, act, mask, window, norm, 1.0 if act == SOFTMAX else 0.5, True)
    cpu = G.cpu_inputs(w, lq, lkv, seed)
    cos, sin, t = _tables(D)
    rq = _bf16(oracle.rope(cpu["q"], cpu["q_off"], cpu["kv_off"], cos, sin))
    rk = _bf16(oracle.rope(cpu["k"], cpu["q_off"], cpu["kv_off"], cos, sin, keys=True))
    rot = dict(cpu, q=rq, k=rk)
    kw = dict(H=w.H, D=D, act=act, mask=mask, window=window, norm_by_lkv=norm)
    o_ref, lse_ref = oracle.fwd(rot["q_off"], rot["kv_off"], rq, rk, rot["v"], **kw)
    o_st, o_rows = G.backward_o(rot, w, o_ref)
    dq_r, dk_r, dv = oracle.bwd(rot["q_off"], rot["kv_off"], rq, rk, rot["v"], rot["do"],
                                o=o_rows if act == SOFTMAX else None, **kw)
    ref = {"dq": oracle.rope(dq_r, cpu["q_off"], cpu["kv_off"], cos, sin, inverse=True),
           "dk": oracle.rope(dk_r, cpu["q_off"], cpu["kv_off"], cos, sin, keys=True, inverse=True), "dv": dv}
    x = G.to_cuda(rot)
    causal = bool(mask & 1)
    block = window if mask & 4 else 0
    o_g = o_st.cuda()
    lse_g = torch.from_numpy(lse_ref).to(torch.float32).cuda() if act == SOFTMAX else None
    dq, dk, dvg = J.backward(x["q"], x["k"], x["v"], o_g, lse_g, x["do"], x["q_off"], x["kv_off"], act=act,
                             causal=causal, block=block, norm_by_lkv=norm, rope=t)
    torch.cuda.synchronize()
    assert J.device_status() == 0
    G.assert_close(G.to64(dq), ref["dq"], "dQ")
    G.assert_close(G.to64(dk), ref["dk"], "dK")
    G.assert_close(G.to64(dvg), ref["dv"], "dV")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("act,mask,window", [(SOFTMAX, CAUSAL, 0), (GELU, NONE, 0), (SOFTMAX, BLOCK, 64)])
def test_bwd_rope_self(act, mask, window, D):
    """Self-attention lengths: whole 128-row key tiles (the TMA-stored dK
    epilogue at D = 128) and ragged tails (the per-row epilogue)."""
    _check_bwd_rope(act, mask, window, D, SELF_LENS, SELF_LENS, seed=82)


@pytest.mark.parametrize("act", [SOFTMAX, GELU])
def test_bwd_rope_cross(act):
    """Lq != Lkv: query and key positions shift by max(+-delta, 0)."""
    _check_bwd_rope(act, NONE, 0, 128, CROSS_LQ, CROSS_LKV, seed=83)


def test_attention_autograd_with_rope():
    """attention(..., rope=...) end to end (GPU rotation, forward, rotary
    backward) against the exact gradient of attention on rotated rows."""
    import jagged_attention_recsys_gdpa_gb300 as J

    D = 128
    w = inputs.Workload("case", 2, D, GELU, NONE, 0, True, 0.5, True)
    cpu = G.cpu_inputs(w, CROSS_LQ, CROSS_LKV, seed=84)
    cos, sin, t = _tables(D)
    x = G.to_cuda(cpu)
    q = x["q"].clone().requires_grad_(True)
    k = x["k"].clone().requires_grad_(True)
    v = x["v"].clone().requires_grad_(True)
    o = J.attention(q, k, v, x["q_off"], x["kv_off"], act="gelu", norm_by_lkv=True, rope=t)
    o.backward(x["do"])
    torch.cuda.synchronize()
    rq = oracle.rope(cpu["q"], cpu["q_off"], cpu["kv_off"], cos, sin)
    rk = oracle.rope(cpu["k"], cpu["q_off"], cpu["kv_off"], cos, sin, keys=True)
    kw = dict(H=2, D=D, act=GELU, norm_by_lkv=True)
    o_ref, _ = oracle.fwd(cpu["q_off"], cpu["kv_off"], rq, rk, cpu["v"], **kw)
    dq_r, dk_r, dv = oracle.bwd(cpu["q_off"], cpu["kv_off"], rq, rk, cpu["v"], cpu["do"], **kw)
    G.assert_close(G.to64(o), o_ref, "O")
    G.assert_close(G.to64(q.grad), oracle.rope(dq_r, cpu["q_off"], cpu["kv_off"], cos, sin, inverse=True), "dQ")
    G.assert_close(G.to64(k.grad), oracle.rope(dk_r, cpu["q_off"], cpu["kv_off"], cos, sin, keys=True,
                                               inverse=True), "dK")
    G.assert_close(G.to64(v.grad), dv, "dV")


def test_short_tables_report_status():
    """Positions past the tables' rows: no access beyond them, the device
    status reads JATTN_ERR_ROPE, and the next clean call reports OK."""
    import jagged_attention_recsys_gdpa_gb300 as J

    JATTN_ERR_ROPE = 9
    D = 64
    w = inputs.Workload("case", 2, D, SOFTMAX, CAUSAL, 0, False, 1.0, True)
    cpu = G.cpu_inputs(w, [100, 300], [100, 300], seed=85)
    x = G.to_cuda(cpu)
    _, _, t = _tables(D, rows=1024)
    short = (t[0][:200].contiguous(), t[1][:200].contiguous())
    J.device_status()
    J.rope(x["q"], x["q_off"], x["kv_off"], short)
    assert J.device_status() == JATTN_ERR_ROPE
    o, lse = J.forward(x["q"], x["k"], x["v"], x["q_off"], x["kv_off"], causal=True)
    J.backward(x["q"], x["k"], x["v"], o, lse, x["do"], x["q_off"], x["kv_off"], causal=True, rope=short)
    assert J.device_status() == JATTN_ERR_ROPE
    J.backward(x["q"], x["k"], x["v"], o, lse, x["do"], x["q_off"], x["kv_off"], causal=True, rope=t)
    assert J.device_status() == 0


def test_attention_autograd_with_rope_softmax():
    """Softmax, causal: attention(..., rope=...) end to end (GPU rotation, GPU
    forward, GPU rotary backward reading that forward's O and LSE) against the
    exact gradient of attention on rotated rows. Rows that see one or two keys
    lie in each sequence's first query tile, whose keys fit one key tile, so
    their D_i comes from the tile itself and the bf16 rounding of the stored O
    does not reach dQ there."""
    import jagged_attention_recsys_gdpa_gb300 as J

    D = 128
    w = inputs.Workload("case", 2, D, SOFTMAX, CAUSAL, 0, False, 1.0, True)
    cpu = G.cpu_inputs(w, SELF_LENS, SELF_LENS, seed=85)
    cos, sin, t = _tables(D)
    x = G.to_cuda(cpu)
    q = x["q"].clone().requires_grad_(True)
    k = x["k"].clone().requires_grad_(True)
    v = x["v"].clone().requires_grad_(True)
    o = J.attention(q, k, v, x["q_off"], x["kv_off"], causal=True, rope=t)
    o.backward(x["do"])
    torch.cuda.synchronize()
    assert J.device_status() == 0
    rq = oracle.rope(cpu["q"], cpu["q_off"], cpu["kv_off"], cos, sin)
    rk = oracle.rope(cpu["k"], cpu["q_off"], cpu["kv_off"], cos, sin, keys=True)
    kw = dict(H=2, D=D, act=SOFTMAX, mask=CAUSAL, window=0, norm_by_lkv=False)
    o_ref, _ = oracle.fwd(cpu["q_off"], cpu["kv_off"], rq, rk, cpu["v"], **kw)
    dq_r, dk_r, dv = oracle.bwd(cpu["q_off"], cpu["kv_off"], rq, rk, cpu["v"], cpu["do"], **kw)
    G.assert_close(G.to64(o), o_ref, "O")
    G.assert_close(G.to64(q.grad), oracle.rope(dq_r, cpu["q_off"], cpu["kv_off"], cos, sin, inverse=True), "dQ")
    G.assert_close(G.to64(k.grad), oracle.rope(dk_r, cpu["q_off"], cpu["kv_off"], cos, sin, keys=True,
                                               inverse=True), "dK")
    G.assert_close(G.to64(v.grad), dv, "dV")
