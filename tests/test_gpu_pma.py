"""The kernels that put the keys on the MMA's M dimension, for pointwise
attention without a mask at D = 128: the short-query (pooling) forward and
fused backward when sequences average at most 64 queries, and the short-key
forward and fused backward when they average more queries but hold at most
128 keys (and, behind a debug flag, the short-query backward's keys-on-M cross
mode for those shapes).
CUDA path vs the oracle element by element, the gates that hand batches
outside a mode's limits back to the general backward, the rows the stores
touch, and the bounded waits."""
import numpy as np
import pytest
import torch

from jagged_attention_recsys_gdpa_gb300 import inputs
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu

SILU, GELU, POLY = 1, 2, 3
NO_SHORT_Q = 32  # debug flag bit: the general kernels even for pooling shapes
JATTN_ERR_TIMEOUT = 6

# every sequence 1 <= Lq <= 64 (or no keys): the fused backward runs
OPEN_LQ = [32, 1, 64, 33, 31, 5, 64, 17, 3]
OPEN_LKV = [1000, 129, 128, 1, 3000, 0, 257, 700, 0]
# one sequence of 100 queries (two 64-row items in the forward) and one with
# keys but no queries: the forward still takes the short-query kernels, the
# backward the general ones
CLOSED_LQ = [32, 100, 0, 7, 20, 1, 30, 2]
CLOSED_LKV = [500, 300, 129, 1000, 0, 64, 2000, 5]


def _w(act, norm=True, H=3, qk=0.0):
    return inputs.Workload("case", H, 128, act, 0, 0, norm, 0.5, False, qk)


def _check(w, lq, lkv, seed, flags=0):
    from jagged_attention_recsys_gdpa_gb300 import _binding as B

    n = len(lq)  # a shape these kernels take: short queries, or else short keys, on average
    assert sum(lq) <= 64 * n or sum(lkv) <= 128 * n
    cpu = G.cpu_inputs(w, lq, lkv, seed)
    B.debug_set(flags, 0)
    try:
        g = G.gpu_run(G.to_cuda(cpu), w)
    finally:
        B.debug_set(0, 0)
    G.compare(g, G.oracle_run(cpu, w), w)
    return g


@pytest.mark.parametrize("norm", [True, False])
@pytest.mark.parametrize("act", [SILU, GELU])
def test_short_query_matches_oracle(act, norm):
    """Ragged key tiles (1, 127-129 keys), sequences without keys (zero O and
    dQ), 1 to 64 queries per sequence; with and without the 1/Lkv normaliser
    (P and dS as bf16 hi + lo parts without it)."""
    _check(_w(act, norm), OPEN_LQ, OPEN_LKV, seed=80 + act + 2 * norm)


def test_short_query_gelu_poly():
    """The ALU-only GELU on query/key-normalised rows (|s| <= 1)."""
    _check(_w(POLY, qk=1.0), OPEN_LQ, OPEN_LKV, seed=85)


@pytest.mark.parametrize("act", [SILU, GELU])
def test_short_query_pooling_long_keys(act):
    """Pooling lengths: 32 learned queries against up to 20,000 keys."""
    _check(_w(act, H=2), [32, 32, 32, 32, 32], [20000, 5000, 1, 128, 4097], seed=86)


@pytest.mark.parametrize("act", [SILU, GELU])
def test_short_query_gate_closed(act):
    """A sequence of 100 queries and one with keys but no queries: the
    forward's items split the 100 queries in two, and the gate leaves the
    backward (dK = dV = 0 for the keys no query sees) to the general kernels."""
    _check(_w(act), CLOSED_LQ, CLOSED_LKV, seed=87)


@pytest.mark.parametrize("norm", [True, False])
def test_short_query_agrees_with_general_kernels(norm):
    """The same inputs through the short-query and the general kernels: both
    within the tolerance of the oracle, and close to each other."""
    w = _w(GELU, norm)
    a = _check(w, OPEN_LQ, OPEN_LKV, seed=88)
    b = _check(w, OPEN_LQ, OPEN_LKV, seed=88, flags=NO_SHORT_Q)
    for k in ("o", "dq", "dk", "dv"):
        G.assert_close(G.to64(a[k]), G.to64(b[k]), k)


def test_short_query_outputs_only_touch_their_rows():
    """Canary rows around O, dQ, dK and dV stay untouched."""
    import jagged_attention_recsys_gdpa_gb300 as J

    w = _w(GELU)
    cpu = G.cpu_inputs(w, OPEN_LQ, OPEN_LKV, 89)
    x = G.to_cuda(cpu)
    TQ, TK, pad = x["q"].shape[0], x["k"].shape[0], 5
    big = lambda T: torch.full((T + 2 * pad, w.H, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    bo, bq, bk, bv = big(TQ), big(TQ), big(TK), big(TK)
    o, dq, dk, dv = bo[pad : pad + TQ], bq[pad : pad + TQ], bk[pad : pad + TK], bv[pad : pad + TK]
    kw = dict(act=GELU, norm_by_lkv=True)
    J.forward(x["q"], x["k"], x["v"], x["q_off"], x["kv_off"], out=o, **kw)
    J.backward(x["q"], x["k"], x["v"], o, None, x["do"], x["q_off"], x["kv_off"], dq=dq, dk=dk, dv=dv, **kw)
    torch.cuda.synchronize()
    for b, T in ((bo, TQ), (bq, TQ), (bk, TK), (bv, TK)):
        assert torch.all(b[:pad] == 7.0) and torch.all(b[pad + T :] == 7.0)
    G.compare({"o": o, "lse": None, "dq": dq, "dk": dk, "dv": dv}, G.oracle_run(cpu, w), w)


def test_short_query_waits_time_out_then_recover():
    """With the query copies skipped, the short-query forward and backward give
    up their bounded waits, report TIMEOUT and return; clean calls on the same
    context afterwards are correct."""
    import jagged_attention_recsys_gdpa_gb300 as J
    from jagged_attention_recsys_gdpa_gb300 import _binding as B

    w = _w(SILU)
    cpu = G.cpu_inputs(w, OPEN_LQ, OPEN_LKV, 90)
    x = G.to_cuda(cpu)
    kw = dict(act=SILU, norm_by_lkv=True)
    J.device_status()
    try:
        B.debug_set(1, 50_000_000)
        J.forward(x["q"], x["k"], x["v"], x["q_off"], x["kv_off"], **kw)
        assert J.device_status() == JATTN_ERR_TIMEOUT
    finally:
        B.debug_set(0, 0)
    o, _ = J.forward(x["q"], x["k"], x["v"], x["q_off"], x["kv_off"], **kw)
    assert J.device_status() == 0
    try:
        B.debug_set(1, 50_000_000)
        J.backward(x["q"], x["k"], x["v"], o, None, x["do"], x["q_off"], x["kv_off"], **kw)
        assert J.device_status() == JATTN_ERR_TIMEOUT
    finally:
        B.debug_set(0, 0)
    g = G.gpu_run(x, w)
    assert J.device_status() == 0
    G.compare(g, G.oracle_run(cpu, w), w)


# ---------------------------------------------------------------- cross-attention over short key sequences
# every sequence Lkv <= 128 (and keys whenever it has queries): the short-key
# forward and backward; more than 64 queries per sequence on average
CROSS_LQ = [1000, 1, 64, 65, 300, 0, 129, 700, 5]
CROSS_LKV = [16, 128, 1, 127, 100, 40, 64, 128, 3]
FWD_ON_SHORT_Q = 64  # debug flag bit: the short-key shapes' forward on the short-query kernel
KEYS_ON_M_CROSS = 128  # debug flag bit: their backward on the short-query kernel's cross mode


@pytest.mark.parametrize("norm", [True, False])
@pytest.mark.parametrize("act", [SILU, GELU])
def test_short_key_matches_oracle(act, norm):
    """Steps of 1 to 128 queries (ragged last step), 1 to 128 keys, a
    sequence with keys but no queries (zero dK and dV)."""
    _check(_w(act, norm), CROSS_LQ, CROSS_LKV, seed=91 + act + 2 * norm)


def test_short_key_gelu_poly():
    _check(_w(POLY, qk=1.0), CROSS_LQ, CROSS_LKV, seed=95)


@pytest.mark.parametrize("norm", [True, False])
@pytest.mark.parametrize("act", [SILU, GELU])
def test_short_key_long_queries(act, norm):
    """Cross-attention lengths: thousands of queries per 16-128 keys (dK and dV
    accumulate over up to 63 query tiles in TMEM; without the normaliser, P and
    dS enter the products as bf16 hi + lo parts)."""
    _check(_w(act, norm, H=2), [8000, 3000, 129, 5], [128, 16, 100, 1], seed=96)


def test_short_key_warp_and_tile_boundaries():
    """Key counts at the 32-row warp boundaries (a warp whose rows all lie past
    the keys skips the activation) and query counts that fill whole 128-row
    tiles or miss by one."""
    _check(_w(SILU, H=2), [128, 256, 384, 129, 127, 300], [32, 33, 65, 96, 97, 64], seed=106)
    _check(_w(GELU, False, H=2), [128, 256, 384, 129, 127, 300], [32, 33, 65, 96, 97, 64], seed=107)


@pytest.mark.parametrize("norm", [True, False])
def test_short_key_keys_on_m_cross_mode(norm):
    """The short-query backward's cross mode (keys on M, 64-query chunks) on
    the same shapes, behind a debug flag; long and ragged sequences."""
    _check(_w(SILU, norm), CROSS_LQ, CROSS_LKV, seed=104, flags=KEYS_ON_M_CROSS)
    _check(_w(GELU, norm, H=2), [8000, 129, 5], [128, 100, 1], seed=105, flags=KEYS_ON_M_CROSS)


@pytest.mark.parametrize("act", [SILU, GELU])
def test_short_key_gate_closed(act):
    """One sequence with 200 keys and one with queries but no keys: the gate
    leaves the backward to the general kernels (dQ = 0 for the rows that see
    nothing)."""
    _check(_w(act), [300, 500, 20, 7], [100, 200, 0, 50], seed=97)


@pytest.mark.parametrize("norm", [True, False])
def test_short_key_forward_on_short_query_kernel(norm):
    """The short-query forward (items of 64 queries) on cross shapes, behind a
    debug flag; the fused backward as usual."""
    _check(_w(GELU, norm), CROSS_LQ, CROSS_LKV, seed=98, flags=FWD_ON_SHORT_Q)


def test_short_key_agrees_with_general_kernels():
    w = _w(SILU)
    a = _check(w, CROSS_LQ, CROSS_LKV, seed=99)
    b = _check(w, CROSS_LQ, CROSS_LKV, seed=99, flags=NO_SHORT_Q)
    for k in ("o", "dq", "dk", "dv"):
        G.assert_close(G.to64(a[k]), G.to64(b[k]), k)


def test_short_key_outputs_only_touch_their_rows():
    import jagged_attention_recsys_gdpa_gb300 as J

    w = _w(SILU)
    cpu = G.cpu_inputs(w, CROSS_LQ, CROSS_LKV, 100)
    x = G.to_cuda(cpu)
    TQ, TK, pad = x["q"].shape[0], x["k"].shape[0], 5
    big = lambda T: torch.full((T + 2 * pad, w.H, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    bq, bk, bv = big(TQ), big(TK), big(TK)
    dq, dk, dv = bq[pad : pad + TQ], bk[pad : pad + TK], bv[pad : pad + TK]
    kw = dict(act=SILU, norm_by_lkv=True)
    o, _ = J.forward(x["q"], x["k"], x["v"], x["q_off"], x["kv_off"], **kw)
    J.backward(x["q"], x["k"], x["v"], o, None, x["do"], x["q_off"], x["kv_off"], dq=dq, dk=dk, dv=dv, **kw)
    torch.cuda.synchronize()
    for b, T in ((bq, TQ), (bk, TK), (bv, TK)):
        assert torch.all(b[:pad] == 7.0) and torch.all(b[pad + T :] == 7.0)
    G.compare({"o": o, "lse": None, "dq": dq, "dk": dk, "dv": dv}, G.oracle_run(cpu, w), w)


def test_short_key_backward_times_out_then_recovers():
    """With the key copies skipped, the cross-mode backward gives up its bounded
    waits, reports TIMEOUT and returns; a clean call afterwards is correct."""
    import jagged_attention_recsys_gdpa_gb300 as J
    from jagged_attention_recsys_gdpa_gb300 import _binding as B

    w = _w(SILU)
    cpu = G.cpu_inputs(w, CROSS_LQ, CROSS_LKV, 101)
    x = G.to_cuda(cpu)
    kw = dict(act=SILU, norm_by_lkv=True)
    J.device_status()
    o, _ = J.forward(x["q"], x["k"], x["v"], x["q_off"], x["kv_off"], **kw)
    assert J.device_status() == 0
    try:
        B.debug_set(1, 50_000_000)
        J.backward(x["q"], x["k"], x["v"], o, None, x["do"], x["q_off"], x["kv_off"], **kw)
        assert J.device_status() == JATTN_ERR_TIMEOUT
    finally:
        B.debug_set(0, 0)
    g = G.gpu_run(x, w)
    assert J.device_status() == 0
    G.compare(g, G.oracle_run(cpu, w), w)


def test_short_key_forward_times_out_then_recovers():
    """With the key copies skipped, the short-key forward gives up its bounded
    waits, reports TIMEOUT and returns; a clean forward afterwards is correct."""
    import jagged_attention_recsys_gdpa_gb300 as J
    from jagged_attention_recsys_gdpa_gb300 import _binding as B

    w = _w(GELU)
    cpu = G.cpu_inputs(w, CROSS_LQ, CROSS_LKV, 102)
    x = G.to_cuda(cpu)
    kw = dict(act=GELU, norm_by_lkv=True)
    J.device_status()
    try:
        B.debug_set(1, 50_000_000)
        J.forward(x["q"], x["k"], x["v"], x["q_off"], x["kv_off"], **kw)
        assert J.device_status() == JATTN_ERR_TIMEOUT
    finally:
        B.debug_set(0, 0)
    g = G.gpu_run(x, w)
    assert J.device_status() == 0
    G.compare(g, G.oracle_run(cpu, w), w)


def test_short_key_forward_outputs_only_touch_their_rows():
    import jagged_attention_recsys_gdpa_gb300 as J

    w = _w(SILU, norm=False)
    cpu = G.cpu_inputs(w, CROSS_LQ, CROSS_LKV, 103)
    x = G.to_cuda(cpu)
    TQ, pad = x["q"].shape[0], 5
    bo = torch.full((TQ + 2 * pad, w.H, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    o = bo[pad : pad + TQ]
    J.forward(x["q"], x["k"], x["v"], x["q_off"], x["kv_off"], act=SILU, norm_by_lkv=False, out=o)
    torch.cuda.synchronize()
    assert torch.all(bo[:pad] == 7.0) and torch.all(bo[pad + TQ :] == 7.0)
    G.assert_close(G.to64(o), G.oracle_run(cpu, w, backward=False)["o"], "O")
