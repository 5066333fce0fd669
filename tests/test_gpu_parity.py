"""CUDA path vs the CPU oracle on the same seeded bf16 inputs, element by
element, at sizes that span several 128-row tiles with ragged tails."""
import numpy as np
import pytest
import torch

from jagged_attention_recsys_gdpa_gb300 import inputs
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu

SOFTMAX, SILU, GELU = 0, 1, 2
NONE, CAUSAL, WIN = 0, 1, 3
BLOCK, CBLOCK = 4, 5  # block mask; block mask with causal inside the blocks

SELF_LENS = [1, 127, 128, 129, 255, 256, 257, 300, 513, 1000]
CROSS_LQ = [100, 300, 5, 700, 257, 1]
CROSS_LKV = [20, 128, 1, 257, 130, 64]


def _w(act, mask, window, D, H=2, norm=False, std=1.0):
    return inputs.Workload("case", H, D, act, mask, window, norm, std, True)


def _check(w, lq, lkv, seed=0, backward=True, stored=False):
    """stored: the backward reads the oracle's O (bf16) and LSE on both sides
    instead of the GPU forward's O against the exact gradient."""
    cpu = G.cpu_inputs(w, lq, lkv, seed)
    if stored:
        g, r = G.run_both_stored(cpu, w, backward)
    else:
        g = G.gpu_run(G.to_cuda(cpu), w, backward)
        r = G.oracle_run(cpu, w, backward)
    G.compare(g, r, w, backward)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("act", [SOFTMAX, SILU, GELU])
@pytest.mark.parametrize("mask,window", [(NONE, 0), (CAUSAL, 0), (WIN, 1), (WIN, 200)])
def test_self_attention(act, mask, window, D):
    norm = act != SOFTMAX
    _check(_w(act, mask, window, D, norm=norm, std=1.0 if act == SOFTMAX else 0.5), SELF_LENS, SELF_LENS)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("act", [SOFTMAX, SILU, GELU])
@pytest.mark.parametrize("mask", [NONE, CAUSAL])
def test_cross_attention(act, mask, D):
    _check(_w(act, mask, 0, D, norm=act != SOFTMAX), CROSS_LQ, CROSS_LKV, seed=3)


@pytest.mark.parametrize("act", [SOFTMAX, GELU])
def test_pma_short_queries_long_keys(act):
    lq = [32, 32, 32, 32]
    lkv = [100, 1000, 3000, 129]
    _check(_w(act, NONE, 0, 128, H=3, norm=act != SOFTMAX, std=0.5), lq, lkv, seed=5)


def test_tiny_config():
    w = inputs.WORKLOADS["tiny"]
    lq, lkv = inputs.lengths("tiny")
    _check(w, lq, lkv, seed=0)


@pytest.mark.parametrize("act", [SOFTMAX, SILU])
def test_empty_and_degenerate_sequences(act):
    # empty queries, empty keys, a single row, causal with Lq > Lkv (rows that see nothing)
    lq = [0, 5, 130, 1, 0, 200, 3]
    lkv = [4, 0, 130, 1, 0, 60, 9]
    _check(_w(act, CAUSAL, 0, 128, norm=act != SOFTMAX), lq, lkv, seed=7)
    _check(_w(act, NONE, 0, 64, norm=act != SOFTMAX), lq, lkv, seed=8)
    _check(_w(act, WIN, 7, 128, norm=act != SOFTMAX), lq, lkv, seed=9)


def test_window_at_least_length_equals_causal():
    w1 = _w(SOFTMAX, CAUSAL, 0, 128)
    w2 = _w(SOFTMAX, WIN, 5000, 128)
    cpu = G.cpu_inputs(w1, SELF_LENS, SELF_LENS, 11)
    a = G.gpu_run(G.to_cuda(cpu), w1)
    b = G.gpu_run(G.to_cuda(cpu), w2)
    for k in ("o", "lse", "dq", "dk", "dv"):
        assert torch.equal(a[k], b[k]), k


def test_deterministic_repeat():
    w = _w(SOFTMAX, WIN, 100, 128)
    cpu = G.cpu_inputs(w, SELF_LENS, SELF_LENS, 12)
    x = G.to_cuda(cpu)
    a = G.gpu_run(x, w)
    b = G.gpu_run(x, w)
    for k in ("o", "lse", "dq", "dk", "dv"):
        assert torch.equal(a[k], b[k]), k


def test_autograd_function():
    import jagged_attention_recsys_gdpa_gb300 as J

    w = _w(GELU, NONE, 0, 128, norm=True, std=0.5)
    cpu = G.cpu_inputs(w, CROSS_LQ, CROSS_LKV, 13)
    x = G.to_cuda(cpu)
    q = x["q"].clone().requires_grad_(True)
    k = x["k"].clone().requires_grad_(True)
    v = x["v"].clone().requires_grad_(True)
    o = J.attention(q, k, v, x["q_off"], x["kv_off"], act="gelu", norm_by_lkv=True)
    o.backward(x["do"])
    r = G.oracle_run(cpu, w)
    G.assert_close(G.to64(o), r["o"], "O")
    G.assert_close(G.to64(q.grad), r["dq"], "dQ")
    G.assert_close(G.to64(k.grad), r["dk"], "dK")
    G.assert_close(G.to64(v.grad), r["dv"], "dV")


def test_outputs_only_touch_their_rows():
    """Canary rows around the outputs stay untouched (bounds check of every store)."""
    import jagged_attention_recsys_gdpa_gb300 as J

    w = _w(SOFTMAX, CAUSAL, 0, 128)
    cpu = G.cpu_inputs(w, SELF_LENS, SELF_LENS, 14)
    x = G.to_cuda(cpu)
    T = x["q"].shape[0]
    pad = 7
    big = torch.full((T + 2 * pad, 2, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    o = big[pad : pad + T]
    lse_big = torch.full((T + 2 * pad, 2), 5.0, dtype=torch.float32, device="cuda")
    J.forward(x["q"], x["k"], x["v"], x["q_off"], x["kv_off"], causal=True, out=o, lse=lse_big[pad : pad + T])
    torch.cuda.synchronize()
    assert torch.all(big[:pad] == 3.0) and torch.all(big[pad + T :] == 3.0)
    assert torch.all(lse_big[:pad] == 5.0) and torch.all(lse_big[pad + T :] == 5.0)


def test_cuda_graph_replay_matches_eager():
    """Forward + backward captured once in a CUDA graph and replayed on new
    input values give the same bits as eager calls."""
    import jagged_attention_recsys_gdpa_gb300 as J

    w = _w(SOFTMAX, WIN, 100, 128)
    cpu = G.cpu_inputs(w, SELF_LENS, SELF_LENS, 15)
    x = G.to_cuda(cpu)
    o = torch.empty_like(x["q"])
    lse = torch.empty(x["q"].shape[0], 2, dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"])
    kw = dict(causal=True, window=100)

    def step():
        J.forward(x["q"], x["k"], x["v"], x["q_off"], x["kv_off"], out=o, lse=lse, **kw)
        J.backward(x["q"], x["k"], x["v"], o, lse, x["do"], x["q_off"], x["kv_off"], dq=dq, dk=dk, dv=dv, **kw)

    step()
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="thread_local"):
        step()
    for seed in (30, 31):
        fresh = G.to_cuda(G.cpu_inputs(w, SELF_LENS, SELF_LENS, seed))
        for key in ("q", "k", "v", "do"):
            x[key].copy_(fresh[key])
        graph.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (o, lse, dq, dk, dv)]
        step()
        torch.cuda.synchronize()
        for g_t, e_t in zip(got, (o, lse, dq, dk, dv)):
            assert torch.equal(g_t, e_t)
    assert J.device_status() == 0


FWD_SPLIT, FWD_PINGPONG = 2, 4  # debug flag bits that force the forward's warp arrangement


@pytest.mark.parametrize("arrangement", [FWD_SPLIT, FWD_PINGPONG])
@pytest.mark.parametrize(
    "act,mask,window,D,lq,lkv",
    [
        (SOFTMAX, WIN, 200, 128, SELF_LENS, SELF_LENS),
        (SOFTMAX, CAUSAL, 0, 64, SELF_LENS, SELF_LENS),
        (SOFTMAX, CAUSAL, 0, 128, [0, 5, 130, 1, 0, 200, 3], [4, 0, 130, 1, 0, 60, 9]),
        (SOFTMAX, NONE, 0, 128, [32, 32, 32, 7], [100, 1000, 3000, 129]),
        (GELU, NONE, 0, 128, [32, 32, 32, 32], [100, 1000, 3000, 129]),
        (SILU, NONE, 0, 64, CROSS_LQ, CROSS_LKV),
        (SILU, WIN, 7, 128, [0, 5, 130, 1, 0, 200, 3], [4, 0, 130, 1, 0, 60, 9]),
    ],
)
def test_forward_arrangements(arrangement, act, mask, window, D, lq, lkv):
    """Both arrangements of the forward's activation warps (two query tiles in
    ping-pong, or every tile's key columns split over both warpgroups) match the
    oracle on the same inputs, whichever one the shapes would pick."""
    from jagged_attention_recsys_gdpa_gb300 import _binding as B

    w = _w(act, mask, window, D, H=3, norm=act != SOFTMAX, std=1.0 if act == SOFTMAX else 0.5)
    cpu = G.cpu_inputs(w, lq, lkv, seed=21)
    B.debug_set(arrangement, 0)
    try:
        g = G.gpu_run(G.to_cuda(cpu), w, backward=False)
    finally:
        B.debug_set(0, 0)
    G.compare(g, G.oracle_run(cpu, w, backward=False), w, backward=False)


DQ_TWO_RINGS, DQ_ONE_RING = 8, 16  # debug flag bits that force the dQ pass's K / V layout


@pytest.mark.parametrize("layout", [DQ_TWO_RINGS, DQ_ONE_RING])
@pytest.mark.parametrize(
    "act,mask,window,D,lq,lkv",
    [
        (SOFTMAX, CAUSAL, 0, 128, [700, 1, 129, 513, 300], None),
        (SOFTMAX, WIN, 200, 128, SELF_LENS, SELF_LENS),
        (SOFTMAX, CAUSAL, 0, 64, SELF_LENS, SELF_LENS),
        (SOFTMAX, CAUSAL, 0, 128, [0, 5, 130, 1, 0, 200, 3], [4, 0, 130, 1, 0, 60, 9]),
        (GELU, NONE, 0, 128, [32, 32, 32, 7], [100, 1000, 3000, 129]),
        (SILU, NONE, 0, 128, CROSS_LQ, CROSS_LKV),
    ],
)
def test_backward_dq_layouts(layout, act, mask, window, D, lq, lkv):
    """Both layouts of the dQ pass's K / V tiles (two rings with K deeper than
    V, or one ring of K + V stages; the host picks one from the key tiles an
    item holds on average) give the oracle's gradients, whichever the shapes
    would pick."""
    from jagged_attention_recsys_gdpa_gb300 import _binding as B

    lkv = lq if lkv is None else lkv
    w = _w(act, mask, window, D, H=2, norm=act != SOFTMAX, std=1.0 if act == SOFTMAX else 0.5)
    cpu = G.cpu_inputs(w, lq, lkv, seed=23)
    B.debug_set(layout, 0)
    try:
        g, r = G.run_both_stored(cpu, w, backward=True)
    finally:
        B.debug_set(0, 0)
    G.compare(g, r, w, backward=True)


@pytest.mark.parametrize("act", [SOFTMAX, GELU])
def test_outputs_16_byte_aligned_only(act):
    """Output tensors that start 16 bytes past a 32-byte boundary (written
    with 16-byte stores) get the same bits as 32-byte aligned ones (written
    with 32-byte stores)."""
    import jagged_attention_recsys_gdpa_gb300 as J

    w = _w(act, CAUSAL if act == SOFTMAX else NONE, 0, 128, norm=act != SOFTMAX, std=1.0 if act == SOFTMAX else 0.5)
    cpu = G.cpu_inputs(w, SELF_LENS, SELF_LENS, 16)
    x = G.to_cuda(cpu)
    kw = dict(act=G.ACT_NAME[act], causal=bool(w.mask & 1), norm_by_lkv=w.norm_by_lkv)

    def shifted_like(t):
        flat = torch.empty(t.numel() + 8, dtype=t.dtype, device=t.device)  # +8 bf16 = +16 bytes
        v = flat[8:].view(t.shape)
        assert v.data_ptr() % 32 == 16
        return v

    o_ref, lse = J.forward(x["q"], x["k"], x["v"], x["q_off"], x["kv_off"], **kw)
    dq_ref, dk_ref, dv_ref = J.backward(x["q"], x["k"], x["v"], o_ref, lse, x["do"], x["q_off"], x["kv_off"], **kw)
    o = shifted_like(o_ref)
    J.forward(x["q"], x["k"], x["v"], x["q_off"], x["kv_off"], out=o, lse=lse, **kw)
    dq, dk, dv = shifted_like(dq_ref), shifted_like(dk_ref), shifted_like(dv_ref)
    J.backward(x["q"], x["k"], x["v"], o_ref, lse, x["do"], x["q_off"], x["kv_off"], dq=dq, dk=dk, dv=dv, **kw)
    torch.cuda.synchronize()
    for got, ref in ((o, o_ref), (dq, dq_ref), (dk, dk_ref), (dv, dv_ref)):
        assert torch.equal(got, ref)
    G.compare({"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}, G.oracle_run(cpu, w), w)


@pytest.mark.parametrize("D", [128, 64])
def test_backward_outputs_only_touch_their_rows(D):
    """Canary rows around dQ, dK and dV stay untouched: whole-tile stores (TMA
    boxes of 128 rows) and per-row stores write only the tensors' own rows."""
    import jagged_attention_recsys_gdpa_gb300 as J

    w = _w(SOFTMAX, CAUSAL, 0, D)
    lens = [128, 256, 129, 1, 300]
    cpu = G.cpu_inputs(w, lens, lens, 17)
    x = G.to_cuda(cpu)
    T = x["q"].shape[0]
    pad = 5
    o, lse = J.forward(x["q"], x["k"], x["v"], x["q_off"], x["kv_off"], causal=True)
    bigs = [torch.full((T + 2 * pad, 2, D), 7.0, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    dq, dk, dv = (b[pad : pad + T] for b in bigs)
    J.backward(x["q"], x["k"], x["v"], o, lse, x["do"], x["q_off"], x["kv_off"], causal=True, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    for b in bigs:
        assert torch.all(b[:pad] == 7.0) and torch.all(b[pad + T :] == 7.0)
    r = G.oracle_run(cpu, w)
    G.assert_close(G.to64(dq), r["dq"], "dQ")
    G.assert_close(G.to64(dk), r["dk"], "dK")
    G.assert_close(G.to64(dv), r["dv"], "dV")


@pytest.mark.parametrize("act", [SOFTMAX, SILU])
@pytest.mark.parametrize("lq,lkv", [([5, 130, 0], [0, 0, 0]), ([0, 0], [7, 300])])
def test_batch_without_keys_or_queries(act, lq, lkv):
    """A batch with no key rows at all (every output row sees nothing: O = 0,
    LSE = -inf, dQ = 0) or no query rows at all (dK = dV = 0)."""
    w = _w(act, NONE, 0, 128, norm=act != SOFTMAX)
    _check(w, lq, lkv, seed=18)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("act", [SOFTMAX, GELU])
@pytest.mark.parametrize("mask", [BLOCK, CBLOCK])
@pytest.mark.parametrize("W", [1, 16, 37, 64, 128, 200])
def test_block_attention_self(W, mask, act, D):
    """Block masks whose edges fall inside, on and across the 128-row tiles.
    Widths that divide the tile (1, 16, 64, 128) take the BlockAttention path
    of the backward: every query tile meets one key tile, and the softmax
    statistics and D_i come from that tile in fp32, so GPU forward -> GPU
    backward is compared with the exact gradient. Other widths read the
    stored O, whose bf16 rounding moves D_i of rows that see one or two keys
    by more than dQ's tolerance: there the backward is checked on the
    oracle's stored O, the forward against the oracle as everywhere."""
    norm = act != SOFTMAX
    _check(_w(act, mask, W, D, norm=norm, std=1.0 if act == SOFTMAX else 0.5), SELF_LENS, SELF_LENS, seed=31,
           stored=(128 % W != 0))


@pytest.mark.parametrize("mask", [BLOCK, CBLOCK])
def test_block_attention_backward_reads_no_o_or_lse(mask):
    """The BlockAttention backward (self-attention, width dividing the tile)
    takes its statistics from the tile: garbage in place of O and LSE, or
    no LSE from the forward at all, leaves every gradient exact."""
    import jagged_attention_recsys_gdpa_gb300 as J
    from jagged_attention_recsys_gdpa_gb300 import _binding as B

    w = _w(SOFTMAX, mask, 64, 128, H=3)
    cpu = G.cpu_inputs(w, SELF_LENS, SELF_LENS, seed=37)
    x = G.to_cuda(cpu)
    assert x["kv_off"] is x["q_off"]
    r = G.oracle_run(cpu, w)
    causal = bool(mask & 1)
    o, lse = J.forward(x["q"], x["k"], x["v"], x["q_off"], x["kv_off"], causal=causal, block=64)
    # the forward may leave LSE out for block masks
    p = J.make_params(x["q"], x["k"], x["q_off"], SOFTMAX, J._mask(causal, 0, 64), 64, None, False)
    o2 = torch.empty_like(o)
    ws = J.workspace(p, "cuda")
    B.fwd(p, x["q_off"], x["kv_off"], x["q"], x["k"], x["v"], o2, None, ws.data_ptr(), ws.numel(),
          torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert torch.equal(o, o2)
    junk_o = torch.full_like(o, 7.0)
    junk_lse = torch.full_like(lse, -3.0)
    dq, dk, dv = J.backward(x["q"], x["k"], x["v"], junk_o, junk_lse, x["do"], x["q_off"], x["kv_off"],
                            causal=causal, block=64)
    torch.cuda.synchronize()
    assert J.device_status() == 0
    G.compare({"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}, r, w)


@pytest.mark.parametrize("act", [SOFTMAX, SILU])
@pytest.mark.parametrize("mask,W", [(BLOCK, 64), (CBLOCK, 50), (BLOCK, 1)])
def test_block_attention_cross_and_degenerate(act, mask, W):
    """Cross-attention (blocks aligned to the sequence ends, so Lq > Lkv leaves
    queries before the first key block with nothing to see), empty sequences and
    one-key blocks."""
    norm = act != SOFTMAX
    _check(_w(act, mask, W, 128, norm=norm), CROSS_LQ, CROSS_LKV, seed=33, stored=True)
    _check(_w(act, mask, W, 64, norm=norm), [0, 5, 130, 1, 0, 200, 3], [4, 0, 130, 1, 0, 60, 9], seed=34,
           stored=True)


@pytest.mark.parametrize("arrangement", [FWD_SPLIT, FWD_PINGPONG])
def test_block_attention_forward_arrangements(arrangement):
    from jagged_attention_recsys_gdpa_gb300 import _binding as B

    w = _w(SOFTMAX, BLOCK, 96, 128, H=3)
    cpu = G.cpu_inputs(w, SELF_LENS, SELF_LENS, seed=35)
    B.debug_set(arrangement, 0)
    try:
        g = G.gpu_run(G.to_cuda(cpu), w, backward=False)
    finally:
        B.debug_set(0, 0)
    G.compare(g, G.oracle_run(cpu, w, backward=False), w, backward=False)


@pytest.mark.parametrize("act", [SOFTMAX, SILU])
def test_block_at_least_length_equals_unblocked(act):
    """A block wider than every sequence allows what no mask (causal inside the
    blocks: causal) allows, and the kernels take identical paths: bit-equal."""
    for m_blk, m_ref in ((BLOCK, NONE), (CBLOCK, CAUSAL)):
        w1 = _w(act, m_ref, 0, 128, norm=act != SOFTMAX)
        w2 = _w(act, m_blk, 4096, 128, norm=act != SOFTMAX)
        cpu = G.cpu_inputs(w1, SELF_LENS, SELF_LENS, 36)
        a = G.gpu_run(G.to_cuda(cpu), w1)
        b = G.gpu_run(G.to_cuda(cpu), w2)
        for k in ("o", "lse", "dq", "dk", "dv"):
            if a[k] is None:  # no LSE for pointwise activations
                assert b[k] is None, k
                continue
            assert torch.equal(a[k], b[k]), (m_blk, k)


# ---------------------------------------------------------------- GDPA's ALU-only GELU
POLY = 3


def _wp(mask, window, D, H=2, norm=True, qk=1.0):
    return inputs.Workload("case", H, D, POLY, mask, window, norm, 0.5, True, qk)


def _spread_scores(cpu, R, rank=3):
    """Confine query and key rows to a `rank`-dim subspace and scale them so
    that scores fill [-R, R] instead of clustering near 0 (random directions
    in D dims are nearly orthogonal)."""
    D = cpu["q"].shape[-1]
    for key in ("q", "k"):
        x = cpu[key].float()
        x[..., rank:] = 0
        x = x * (float(np.sqrt(R * np.sqrt(D))) / x.norm(dim=-1, keepdim=True).clamp_min(1e-30))
        cpu[key] = x.to(torch.bfloat16)
    return cpu


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("mask,window", [(NONE, 0), (CAUSAL, 0), (BLOCK, 64)])
def test_gelu_poly_self(mask, window, D):
    """Query/key-normalised rows (|s| <= 1): the polynomial GELU matches the
    oracle's tanh-GELU."""
    _check(_wp(mask, window, D), SELF_LENS, SELF_LENS, seed=41)


def test_gelu_poly_cross_and_pma():
    _check(_wp(NONE, 0, 128), CROSS_LQ, CROSS_LKV, seed=42)
    _check(_wp(NONE, 0, 128, H=3), [32, 32, 32, 32], [100, 1000, 3000, 129], seed=43)


def test_gelu_poly_unnormalised_short():
    """The polynomial GELU without the 1/Lkv normaliser on short sequences."""
    _check(_wp(NONE, 0, 128, norm=False), [100, 60, 5, 130, 1], [20, 128, 1, 64, 64], seed=42)


UNNORM_CASES = [
    # pooling: 32 queries over long key sequences (outputs O and dQ sum thousands of terms)
    ([32, 32, 32, 32], [20000, 5000, 130, 1]),
    # cross-attention: long queries over short keys (dK and dV sum thousands of terms)
    ([8000, 3000, 129, 5], [128, 16, 100, 1]),
]


@pytest.mark.parametrize("case", [0, 1])
@pytest.mark.parametrize("act", [SILU, GELU, POLY])
def test_unnormalised_pointwise_long_sequences(act, case):
    """Without the 1/Lkv normaliser, each output sums thousands of unscaled
    terms act(s) v or act'(s) dP: rounding P and dS to bf16 before the second
    products would then miss the element-wise tolerance (an fp64 emulation of
    that one rounding misses it by 3-6x on these lengths). P and dS therefore
    enter those products as bf16 hi + lo parts accumulating into the same fp32
    result; every output is compared with the oracle."""
    lq, lkv = UNNORM_CASES[case]
    if act == POLY:
        w = _wp(NONE, 0, 128, norm=False)
    else:
        w = inputs.Workload("case", 2, 128, act, NONE, 0, False, 0.5, False)
    _check(w, lq, lkv, seed=60 + case)


@pytest.mark.parametrize("arrangement", [FWD_SPLIT, FWD_PINGPONG])
def test_unnormalised_forward_arrangements(arrangement):
    """The lo parts of P sit 32 (column split) or 64 (ping-pong) TMEM columns
    after the hi parts: both arrangements on pooling lengths."""
    from jagged_attention_recsys_gdpa_gb300 import _binding as B

    w = inputs.Workload("case", 3, 128, GELU, NONE, 0, False, 0.5, False)
    cpu = G.cpu_inputs(w, [32, 300, 32, 7], [20000, 3000, 129, 1], seed=64)
    B.debug_set(arrangement, 0)
    try:
        g = G.gpu_run(G.to_cuda(cpu), w, backward=False)
    finally:
        B.debug_set(0, 0)
    G.compare(g, G.oracle_run(cpu, w, backward=False), w, backward=False)


@pytest.mark.parametrize("act", [SILU, GELU])
def test_unnormalised_self_attention_causal(act):
    _check(inputs.Workload("case", 2, 64, act, CAUSAL, 0, False, 0.5, True), SELF_LENS, SELF_LENS, seed=66)


def test_gelu_poly_scores_spread_over_the_range():
    """Scores spread over [-0.9, 0.9], where the polynomial still agrees with
    tanh-GELU within the tolerance (1/Lkv normaliser, as GDPA uses it)."""
    w = _wp(NONE, 0, 128)
    cpu = _spread_scores(G.cpu_inputs(w, CROSS_LQ, CROSS_LKV, seed=44), 0.9)
    G.compare(G.gpu_run(G.to_cuda(cpu), w), G.oracle_run(cpu, w), w)


def test_gelu_poly_is_the_polynomial():
    """With scores out to |s| = 1.5 the polynomial and tanh-GELU part; the
    kernels must follow the polynomial (fp64 padded dense reference of it,
    gradients by autograd), and the case must tell the two apart."""
    from tests import dense_ref as R

    w = _wp(NONE, 0, 128)
    lq, lkv = [100, 5, 260, 1], [20, 128, 130, 64]
    cpu = _spread_scores(G.cpu_inputs(w, lq, lkv, seed=45), 1.5)
    g = G.gpu_run(G.to_cuda(cpu), w)
    args = [R.to_f64(cpu[x]) for x in ("q", "k", "v")]
    offs = (cpu["q_off"].numpy(), cpu["kv_off"].numpy())
    kw = dict(act=POLY, mask=0, window=0, scale=1.0 / np.sqrt(128), norm_by_lkv=True)
    o, _ = R.dense_forward(*args, *offs, **kw)
    dq, dk, dv = R.dense_grads(*args, R.to_f64(cpu["do"]), *offs, **kw)
    ref = {"o": o.numpy(), "dq": dq.numpy(), "dk": dk.numpy(), "dv": dv.numpy()}
    for key, name in (("o", "O"), ("dq", "dQ"), ("dk", "dK"), ("dv", "dV")):
        G.assert_close(G.to64(g[key]), ref[key], name)
    tanh_ref = G.oracle_run(cpu, w)
    err = np.abs(tanh_ref["dk"] - ref["dk"]) - (G.ATOL + G.RTOL * np.abs(ref["dk"]))
    assert err.max() > 0, "case does not separate the polynomial from tanh-GELU"
