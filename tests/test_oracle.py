"""Pins for the CPU oracle (no GPU).

Each check ties the oracle to something other than itself: torch's
scaled_dot_product_attention / logsumexp / silu / gelu and autograd on a
padded dense formulation, finite differences of the oracle's own forward,
closed forms, invariants, and brute-force enumeration for the tile schedule.
"""
import itertools
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from jagged_attention_recsys_gdpa_gb300 import inputs
from tests import dense_ref as R

SOFTMAX, SILU, GELU = 0, 1, 2
NONE, CAUSAL, WINDOW = 0, 1, 3  # WINDOW value as passed: causal | window bits
BLOCK, CBLOCK = 4, 5  # block mask, and block mask with causal inside the blocks


def _batch(lq, lkv, H, D, seed, std=1.0):
    lq = np.asarray(lq, dtype=np.int64)
    lkv = np.asarray(lkv, dtype=np.int64)
    qo, ko = inputs.offsets(lq), inputs.offsets(lkv)
    q = inputs.values((int(qo[-1]), H, D), std, seed)
    k = inputs.values((int(ko[-1]), H, D), std, seed + 1)
    v = inputs.values((int(ko[-1]), H, D), std, seed + 2)
    do = inputs.values((int(qo[-1]), H, D), 1.0, seed + 3)
    return qo, ko, q, k, v, do


SELF_LENS = ([3, 17, 1, 40, 9], [3, 17, 1, 40, 9])
CROSS_LENS = ([5, 12, 7, 1, 20], [9, 4, 30, 6, 2])


@pytest.mark.parametrize("mask,window", [(NONE, 0), (CAUSAL, 0), (WINDOW, 1), (WINDOW, 5), (WINDOW, 64),
                                         (BLOCK, 1), (BLOCK, 4), (BLOCK, 64), (CBLOCK, 4)])
@pytest.mark.parametrize("lens", [SELF_LENS, CROSS_LENS], ids=["self", "cross"])
def test_softmax_matches_torch_sdpa(mask, window, lens):
    H, D = 2, 16
    qo, ko, q, k, v, _ = _batch(*lens, H, D, seed=11)
    scale = 1.0 / math.sqrt(D)
    o, lse = oracle.fwd(qo, ko, q, k, v, H=H, D=D, act=SOFTMAX, mask=mask, window=window, scale=scale)
    ref = R.sdpa_per_sequence(R.to_f64(q), R.to_f64(k), R.to_f64(v), list(qo), list(ko), mask, window, scale)
    ref = ref.numpy()
    # rows with no visible key, from the mask definition (SDPA's own value there varies by version)
    empty_rows = np.concatenate([~R.mask_matrix(int(qo[b + 1] - qo[b]), int(ko[b + 1] - ko[b]), mask, window)
                                 .numpy().any(axis=1) for b in range(len(qo) - 1)])
    empty = np.broadcast_to(empty_rows[:, None], (len(empty_rows), H))
    np.testing.assert_allclose(o[~empty], ref[~empty], rtol=1e-12, atol=1e-12)
    assert np.all(o[empty] == 0.0)
    # log-sum-exp against torch.logsumexp of the masked scores
    _, lse_ref = R.dense_forward(R.to_f64(q), R.to_f64(k), R.to_f64(v), qo, ko, SOFTMAX, mask, window, scale, False)
    lse_ref = lse_ref.numpy()
    assert np.array_equal(np.isneginf(lse), np.isneginf(lse_ref))
    fin = np.isfinite(lse_ref)
    np.testing.assert_allclose(lse[fin], lse_ref[fin], rtol=1e-12, atol=1e-12)
    assert np.array_equal(np.isneginf(lse), empty)


@pytest.mark.parametrize("act", [SILU, GELU])
@pytest.mark.parametrize("mask,window", [(NONE, 0), (CAUSAL, 0), (WINDOW, 4), (BLOCK, 4), (CBLOCK, 3)])
@pytest.mark.parametrize("norm", [False, True])
@pytest.mark.parametrize("lens", [SELF_LENS, CROSS_LENS], ids=["self", "cross"])
def test_pointwise_matches_padded_dense(act, mask, window, norm, lens):
    H, D = 2, 8
    qo, ko, q, k, v, _ = _batch(*lens, H, D, seed=5, std=0.8)
    scale = 0.37
    o, _ = oracle.fwd(qo, ko, q, k, v, H=H, D=D, act=act, mask=mask, window=window, scale=scale, norm_by_lkv=norm)
    ref, _ = R.dense_forward(R.to_f64(q), R.to_f64(k), R.to_f64(v), qo, ko, act, mask, window, scale, norm)
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act", [SOFTMAX, SILU, GELU])
@pytest.mark.parametrize("mask,window", [(NONE, 0), (CAUSAL, 0), (WINDOW, 3), (BLOCK, 4), (CBLOCK, 3)])
@pytest.mark.parametrize("lens", [SELF_LENS, CROSS_LENS], ids=["self", "cross"])
def test_grads_match_torch_autograd(act, mask, window, lens):
    H, D = 2, 8
    qo, ko, q, k, v, do = _batch(*lens, H, D, seed=23, std=0.9)
    scale = 1.0 / math.sqrt(D)
    norm = act != SOFTMAX
    dq, dk, dv = oracle.bwd(qo, ko, q, k, v, do, H=H, D=D, act=act, mask=mask, window=window, scale=scale,
                            norm_by_lkv=norm)
    gq, gk, gv = R.dense_grads(R.to_f64(q), R.to_f64(k), R.to_f64(v), R.to_f64(do), qo, ko, act, mask, window,
                               scale, norm)
    for a, b in ((dq, gq), (dk, gk), (dv, gv)):
        np.testing.assert_allclose(a, b.numpy(), rtol=1e-10, atol=1e-12)


@pytest.mark.parametrize("act", [SOFTMAX, SILU, GELU])
@pytest.mark.parametrize("mask,window", [(NONE, 0), (CAUSAL, 0), (WINDOW, 2), (BLOCK, 2), (CBLOCK, 2)])
def test_grads_finite_differences(act, mask, window):
    """Central differences of L = sum(o * dO) through the oracle's forward."""
    H, D = 1, 4
    rng = np.random.default_rng(3)
    lq, lkv = [4, 0, 3, 5], [6, 2, 3, 0]
    qo, ko = inputs.offsets(np.array(lq)), inputs.offsets(np.array(lkv))
    q = rng.standard_normal((qo[-1], H, D))
    k = rng.standard_normal((ko[-1], H, D))
    v = rng.standard_normal((ko[-1], H, D))
    do = rng.standard_normal((qo[-1], H, D))
    kw = dict(H=H, D=D, act=act, mask=mask, window=window, scale=0.6, norm_by_lkv=True)
    grads = oracle.bwd(qo, ko, q, k, v, do, **kw)

    def loss(qq, kk, vv):
        o, _ = oracle.fwd(qo, ko, qq, kk, vv, **kw)
        return float((o * do).sum())

    eps = 1e-6
    for which, (x, g) in enumerate(zip((q, k, v), grads)):
        for idx in itertools.product(*(range(s) for s in x.shape)):
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = [q, k, v]
            args_m = [q, k, v]
            args_p[which], args_m[which] = xp, xm
            fd = (loss(*args_p) - loss(*args_m)) / (2 * eps)
            assert abs(fd - g[idx]) <= 1e-6 + 1e-6 * abs(fd), (which, idx, fd, g[idx])


def test_closed_forms_softmax():
    H, D = 2, 16
    lens = [5, 1, 33, 8]
    qo, ko, q, k, v, _ = _batch(lens, lens, H, D, seed=2)
    ones = torch.ones_like(v)
    # rows of p sum to one: V = 1 gives O = 1 for every mask
    for mask, w in ((NONE, 0), (CAUSAL, 0), (WINDOW, 3)):
        o, _ = oracle.fwd(qo, ko, q, k, ones, H=H, D=D, act=SOFTMAX, mask=mask, window=w)
        np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-13)
    # window 1: each row sees only its own key -> o_i = v_i, lse_i = s_ii
    o, lse = oracle.fwd(qo, ko, q, k, v, H=H, D=D, act=SOFTMAX, mask=WINDOW, window=1)
    np.testing.assert_array_equal(o, R.to_f64(v).numpy())
    s_ii = (R.to_f64(q) * R.to_f64(k)).sum(-1).numpy() / math.sqrt(D)
    np.testing.assert_allclose(lse, s_ii, rtol=1e-13, atol=1e-13)
    # window >= L equals plain causal
    oc, lc = oracle.fwd(qo, ko, q, k, v, H=H, D=D, act=SOFTMAX, mask=CAUSAL)
    ow, lw = oracle.fwd(qo, ko, q, k, v, H=H, D=D, act=SOFTMAX, mask=WINDOW, window=max(lens))
    np.testing.assert_array_equal(oc, ow)
    np.testing.assert_array_equal(lc, lw)
    # a single key: o = v_0 whatever the query
    qo1, ko1 = inputs.offsets(np.array([4, 7])), inputs.offsets(np.array([1, 1]))
    q1 = inputs.values((11, H, D), 1.0, 9)
    k1 = inputs.values((2, H, D), 1.0, 10)
    v1 = inputs.values((2, H, D), 1.0, 11)
    o1, _ = oracle.fwd(qo1, ko1, q1, k1, v1, H=H, D=D, act=SOFTMAX, mask=NONE)
    vv = R.to_f64(v1).numpy()
    np.testing.assert_array_equal(o1[:4], np.broadcast_to(vv[0], (4, H, D)))
    np.testing.assert_array_equal(o1[4:], np.broadcast_to(vv[1], (7, H, D)))


@pytest.mark.parametrize("act,fn", [(SILU, F.silu), (GELU, lambda t: F.gelu(t, approximate="tanh"))])
def test_activation_values_against_torch(act, fn):
    """D=1, one query and one key with q=x, k=1, v=1, scale=1: o = act(x)."""
    xs = np.linspace(-9.0, 9.0, 73)
    n = len(xs)
    qo = inputs.offsets(np.ones(n, dtype=np.int64))
    q = xs.reshape(n, 1, 1).copy()
    k = np.ones((n, 1, 1))
    v = np.ones((n, 1, 1))
    o, _ = oracle.fwd(qo, qo, q, k, v, H=1, D=1, act=act, mask=NONE, scale=1.0)
    ref = fn(torch.from_numpy(xs)).numpy()
    np.testing.assert_allclose(o[:, 0, 0], ref, rtol=1e-14, atol=1e-15)
    # zero queries give zero scores, act(0) = 0, so O = 0
    H, D = 2, 8
    qo2, ko2, q2, k2, v2, _ = _batch([3, 4], [5, 2], H, D, seed=1)
    o2, _ = oracle.fwd(qo2, ko2, torch.zeros_like(q2), k2, v2, H=H, D=D, act=act, mask=NONE)
    assert np.all(o2 == 0.0)


@pytest.mark.parametrize("act", [SOFTMAX, SILU, GELU])
def test_permutation_equivariance(act):
    H, D = 2, 8
    lq, lkv = np.array([4, 9, 1, 6]), np.array([7, 9, 3, 6])
    qo, ko, q, k, v, do = _batch(lq, lkv, H, D, seed=8)
    kw = dict(H=H, D=D, act=act, mask=NONE, norm_by_lkv=True)
    o, lse = oracle.fwd(qo, ko, q, k, v, **kw)
    dq, dk, dv = oracle.bwd(qo, ko, q, k, v, do, **kw)
    perm = [2, 0, 3, 1]

    def permute(x, off, lens):
        return torch.cat([x[off[b] : off[b + 1]] for b in perm], 0)

    qo2, ko2 = inputs.offsets(lq[perm]), inputs.offsets(lkv[perm])
    P = lambda x, off, lens: permute(torch.as_tensor(x), off, lens)
    o2, lse2 = oracle.fwd(qo2, ko2, P(q, qo, lq), P(k, ko, lkv), P(v, ko, lkv), **kw)
    g2 = oracle.bwd(qo2, ko2, P(q, qo, lq), P(k, ko, lkv), P(v, ko, lkv), P(do, qo, lq), **kw)
    np.testing.assert_array_equal(o2, P(o, qo, lq).numpy())
    np.testing.assert_array_equal(lse2, P(lse, qo, lq).numpy())
    np.testing.assert_array_equal(g2[0], P(dq, qo, lq).numpy())
    np.testing.assert_array_equal(g2[1], P(dk, ko, lkv).numpy())
    np.testing.assert_array_equal(g2[2], P(dv, ko, lkv).numpy())


@pytest.mark.parametrize("act", [SOFTMAX, SILU, GELU])
def test_empty_sequences(act):
    H, D = 2, 8
    lq, lkv = np.array([0, 5, 3, 0, 4]), np.array([3, 0, 6, 0, 4])
    qo, ko, q, k, v, do = _batch(lq, lkv, H, D, seed=4)
    kw = dict(H=H, D=D, act=act, mask=NONE)
    o, lse = oracle.fwd(qo, ko, q, k, v, **kw)
    dq, dk, dv = oracle.bwd(qo, ko, q, k, v, do, **kw)
    rows_no_keys = slice(qo[1], qo[2])  # sequence 1 has queries but no keys
    assert np.all(o[rows_no_keys] == 0.0)
    assert np.all(dq[rows_no_keys] == 0.0)
    if act == SOFTMAX:
        assert np.all(np.isneginf(lse[rows_no_keys]))
    keys_no_queries = slice(ko[0], ko[1])  # sequence 0 has keys but no queries
    assert np.all(dk[keys_no_queries] == 0.0) and np.all(dv[keys_no_queries] == 0.0)
    # the non-empty sequences are unaffected by their empty neighbours
    qo2, ko2 = inputs.offsets(lq[[2, 4]]), inputs.offsets(lkv[[2, 4]])
    sel_q = torch.cat([q[qo[2] : qo[3]], q[qo[4] : qo[5]]])
    sel_k = torch.cat([k[ko[2] : ko[3]], k[ko[4] : ko[5]]])
    sel_v = torch.cat([v[ko[2] : ko[3]], v[ko[4] : ko[5]]])
    o2, _ = oracle.fwd(qo2, ko2, sel_q, sel_k, sel_v, **kw)
    np.testing.assert_array_equal(o2, np.concatenate([o[qo[2] : qo[3]], o[qo[4] : qo[5]]]))


def test_softmax_dv_column_sum():
    """Each softmax row of p sums to one, so sum_j dV_j = sum_i dO_i per (b, h)."""
    H, D = 2, 8
    lens = [6, 13, 2]
    qo, ko, q, k, v, do = _batch(lens, lens, H, D, seed=6)
    for mask, w in ((NONE, 0), (CAUSAL, 0), (WINDOW, 4)):
        _, _, dv = oracle.bwd(qo, ko, q, k, v, do, H=H, D=D, act=SOFTMAX, mask=mask, window=w)
        g = R.to_f64(do).numpy()
        for b in range(len(lens)):
            np.testing.assert_allclose(dv[ko[b] : ko[b + 1]].sum(0), g[qo[b] : qo[b + 1]].sum(0), rtol=1e-12,
                                       atol=1e-12)


def test_count_pairs_closed_forms():
    lens = np.array([1, 7, 30, 129, 0])
    off = inputs.offsets(lens)
    assert oracle.count_pairs(off, off, NONE) == int((lens * lens).sum())
    assert oracle.count_pairs(off, off, CAUSAL) == int((lens * (lens + 1) // 2).sum())
    W = 10
    expect = sum(sum(min(i + 1, W) for i in range(L)) for L in lens)
    assert oracle.count_pairs(off, off, WINDOW, W) == expect
    lq, lk = np.array([3, 5]), np.array([5, 3])
    # bottom-right causal with Lq=3, Lkv=5: row i sees i + 3 keys; Lq=5, Lkv=3: max(0, i - 1)
    assert oracle.count_pairs(inputs.offsets(lq), inputs.offsets(lk), CAUSAL) == (3 + 4 + 5) + (0 + 0 + 1 + 2 + 3)


def _brute_schedule(qo, ko, mask, window, BM, BN, transposed):
    """Every (b, row tile) with the column tiles that hold an allowed pair."""
    tiles = []
    for b in range(len(qo) - 1):
        lq, lk = int(qo[b + 1] - qo[b]), int(ko[b + 1] - ko[b])
        m = R.mask_matrix(lq, lk, mask, window).numpy()
        if transposed:
            m = m.T
        nrows = m.shape[0]
        for t in range(-(-nrows // BM)):
            cols = np.nonzero(m[t * BM : (t + 1) * BM].any(axis=0))[0]
            if len(cols):
                tiles.append((b, t, cols.min() // BN, cols.max() // BN + 1))
            else:
                tiles.append((b, t, 0, 0))
    return tiles


@pytest.mark.parametrize("transposed", [False, True])
@pytest.mark.parametrize("mask,window", [(NONE, 0), (CAUSAL, 0), (WINDOW, 3), (WINDOW, 9), (BLOCK, 3), (BLOCK, 8),
                                         (CBLOCK, 5)])
def test_schedule_twin_brute_force(transposed, mask, window):
    rng = np.random.default_rng(17)
    for trial in range(6):
        B = int(rng.integers(1, 7))
        lq = rng.integers(0, 40, size=B)
        lk = lq.copy() if trial % 2 == 0 else rng.integers(0, 40, size=B)
        qo, ko = inputs.offsets(lq), inputs.offsets(lk)
        BM, BN = (8, 4) if trial < 3 else (4, 8)
        got = oracle.schedule(qo, ko, mask=mask, window=window, BM=BM, BN=BN, transposed=transposed)
        want = _brute_schedule(qo, ko, mask, window, BM, BN, transposed)
        # same multiset of tiles, each (b, row tile) exactly once
        assert sorted(map(tuple, got.tolist())) == sorted(want)
        assert len({(r[0], r[1]) for r in got.tolist()}) == len(got)
        # longest first, ties in (b, row tile) order
        keys = [(-(r[3] - r[2]), r[0], r[1]) for r in got.tolist()]
        assert keys == sorted(keys)


def test_schedule_cost_cap_orders_by_index():
    lens = np.array([40, 300, 64])
    off = inputs.offsets(lens)
    got = oracle.schedule(off, off, mask=NONE, BM=16, BN=4, cost_cap=20)
    costs = np.minimum(got[:, 3] - got[:, 2], 20)
    assert np.all(np.diff(costs) <= 0)
    capped = got[costs == 20]
    assert [tuple(r[:2]) for r in capped.tolist()] == sorted(tuple(r[:2]) for r in capped.tolist())


# ---------------------------------------------------------------- block attention
def _split_into_blocks(lens, W):
    """Lengths of the W-wide blocks every sequence splits into (last one partial)."""
    out = []
    for L in lens:
        out += [min(W, L - s) for s in range(0, L, W)] if L else [0]
    return np.asarray(out, dtype=np.int64)


@pytest.mark.parametrize("act", [SOFTMAX, SILU, GELU])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("W", [1, 3, 8])
def test_block_mask_is_independent_blocks(act, causal, W):
    """Self-attention with a block mask equals attention run on every block as
    its own sequence (unmasked, or causal when the block mask is causal), for
    O, LSE and all gradients; the 1/Lkv normaliser is the full sequence's."""
    H, D = 2, 8
    lens = np.array([3, 17, 1, 0, 40, 9])
    qo = inputs.offsets(lens)
    q = inputs.values((int(qo[-1]), H, D), 0.8, 31)
    k = inputs.values((int(qo[-1]), H, D), 0.8, 32)
    v = inputs.values((int(qo[-1]), H, D), 0.8, 33)
    do = inputs.values((int(qo[-1]), H, D), 1.0, 34)
    kw = dict(H=H, D=D, act=act, scale=0.3)
    o, lse = oracle.fwd(qo, qo, q, k, v, mask=(CBLOCK if causal else BLOCK), window=W, **kw)
    g = oracle.bwd(qo, qo, q, k, v, do, mask=(CBLOCK if causal else BLOCK), window=W, **kw)
    bo = inputs.offsets(_split_into_blocks(lens, W))
    o2, lse2 = oracle.fwd(bo, bo, q, k, v, mask=(CAUSAL if causal else NONE), window=0, **kw)
    g2 = oracle.bwd(bo, bo, q, k, v, do, mask=(CAUSAL if causal else NONE), window=0, **kw)
    np.testing.assert_allclose(o, o2, rtol=1e-13, atol=1e-14)
    if act == SOFTMAX:
        np.testing.assert_allclose(lse, lse2, rtol=1e-13, atol=1e-14)
    for a, b in zip(g, g2):
        np.testing.assert_allclose(a, b, rtol=1e-13, atol=1e-14)


def test_block_mask_closed_forms():
    H, D = 2, 16
    lens = np.array([5, 33, 1, 12])
    qo = inputs.offsets(lens)
    q = inputs.values((int(qo[-1]), H, D), 1.0, 41)
    k = inputs.values((int(qo[-1]), H, D), 1.0, 42)
    v = inputs.values((int(qo[-1]), H, D), 1.0, 43)
    kw = dict(H=H, D=D, act=SOFTMAX, scale=0.25)
    # a block at least as wide as every sequence is no mask (causal inside it: causal)
    for m_blk, m_ref in ((BLOCK, NONE), (CBLOCK, CAUSAL)):
        o, lse = oracle.fwd(qo, qo, q, k, v, mask=m_blk, window=int(lens.max()), **kw)
        o2, lse2 = oracle.fwd(qo, qo, q, k, v, mask=m_ref, window=0, **kw)
        np.testing.assert_array_equal(o, o2)
        np.testing.assert_array_equal(lse, lse2)
    # blocks of one key: every query sees only its own key, so o_i = v_i and lse_i = s_ii
    o, lse = oracle.fwd(qo, qo, q, k, v, mask=BLOCK, window=1, **kw)
    qd, kd, vd = (R.to_f64(t).numpy() for t in (q, k, v))
    np.testing.assert_allclose(o, vd, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(lse, 0.25 * np.einsum("thd,thd->th", qd, kd), rtol=1e-13, atol=1e-14)


def test_block_mask_pair_counts():
    lens = np.array([1, 7, 30, 129, 0, 64])
    off = inputs.offsets(lens)
    for W in (1, 5, 64, 200):
        blocks = _split_into_blocks(lens, W)
        assert oracle.count_pairs(off, off, BLOCK, W) == int((blocks * blocks).sum())
        assert oracle.count_pairs(off, off, CBLOCK, W) == int((blocks * (blocks + 1) // 2).sum())
    # cross-attention, Lq = 3 < Lkv = 8 (delta = 5), blocks of 4: queries sit at key positions 5, 6, 7,
    # all in the block [4, 8), so each sees 4 keys; with causal, 2, 3 and 4
    lq, lk = inputs.offsets(np.array([3])), inputs.offsets(np.array([8]))
    assert oracle.count_pairs(lq, lk, BLOCK, 4) == 12
    assert oracle.count_pairs(lq, lk, CBLOCK, 4) == 2 + 3 + 4


# ---------------------------------------------------------------- stored forward output
@pytest.mark.parametrize("mask,window", [(NONE, 0), (CAUSAL, 0), (CBLOCK, 3)])
@pytest.mark.parametrize("lens", [SELF_LENS, CROSS_LENS], ids=["self", "cross"])
def test_bwd_from_stored_output(mask, window, lens):
    """D_i formed from a stored output O' = O + E: with E = 0 it is the exact
    gradient; otherwise dV is unchanged and dQ_i moves by exactly
    -scale <dO_i, E_i> sum_j p_ij k_j (sum_j p_ij k_j is the forward with V := K)."""
    H, D, scale = 2, 8, 0.4
    qo, ko, q, k, v, do = _batch(*lens, H, D, seed=51)
    kw = dict(H=H, D=D, act=SOFTMAX, mask=mask, window=window, scale=scale)
    o, _ = oracle.fwd(qo, ko, q, k, v, **kw)
    exact = oracle.bwd(qo, ko, q, k, v, do, **kw)
    for a, b in zip(oracle.bwd(qo, ko, q, k, v, do, o=o, **kw), exact):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-13)
    E = np.random.default_rng(5).normal(0.0, 0.01, size=o.shape)
    dq2, _, dv2 = oracle.bwd(qo, ko, q, k, v, do, o=o + E, **kw)
    pk, _ = oracle.fwd(qo, ko, q, k, k, **kw)
    eps = np.einsum("thd,thd->th", R.to_f64(do).numpy(), E)
    np.testing.assert_allclose(dq2, exact[0] - scale * eps[..., None] * pk, rtol=1e-11, atol=1e-13)
    np.testing.assert_array_equal(dv2, exact[2])
    # pointwise activations have no D_i: the stored output is ignored
    kwp = dict(kw, act=SILU)
    for a, b in zip(oracle.bwd(qo, ko, q, k, v, do, o=o + E, **kwp), oracle.bwd(qo, ko, q, k, v, do, **kwp)):
        np.testing.assert_array_equal(a, b)


# ---------------------------------------------------------------- rotary embedding
rope_tables = R.rope_tables


@pytest.mark.parametrize("keys", [False, True])
def test_rope_is_complex_multiplication(keys):
    """Pair m as the complex number x_2m + i x_2m+1 is multiplied by e^(i angle);
    the inverse multiplies by e^(-i angle); positions follow the alignment."""
    H, D = 2, 16
    lq, lk = np.array([5, 0, 9, 3]), np.array([7, 4, 2, 3])
    qo, ko = inputs.offsets(lq), inputs.offsets(lk)
    n = int((ko if keys else qo)[-1])
    x = inputs.values((n, H, D), 1.0, 71)
    cos, sin, ang = rope_tables(16, D)
    xd = R.to_f64(x).numpy()
    for inverse in (False, True):
        y = oracle.rope(x, qo, ko, cos, sin, keys=keys, inverse=inverse)
        own, oth = (lk, lq) if keys else (lq, lk)
        r0 = 0
        for b in range(len(own)):
            delta = (lk[b] - lq[b])
            shift = max(-delta, 0) if keys else max(delta, 0)
            for i in range(own[b]):
                z = xd[r0 + i, :, 0::2] + 1j * xd[r0 + i, :, 1::2]
                w = z * np.exp((-1j if inverse else 1j) * ang[i + shift])[None, :]
                np.testing.assert_allclose(y[r0 + i, :, 0::2], w.real, rtol=1e-13, atol=1e-14)
                np.testing.assert_allclose(y[r0 + i, :, 1::2], w.imag, rtol=1e-13, atol=1e-14)
            r0 += own[b]
        back = oracle.rope(y, qo, ko, cos, sin, keys=keys, inverse=not inverse)
        np.testing.assert_allclose(back, xd, rtol=1e-13, atol=1e-14)


def test_rope_scores_depend_on_relative_position():
    """<R(p) q, R(p') k> depends on p - p' only: moving every position by 5
    (tables read 5 rows later) leaves all scores unchanged."""
    H, D = 1, 8
    lq, lk = np.array([6, 3]), np.array([4, 8])
    qo, ko = inputs.offsets(lq), inputs.offsets(lk)
    q = inputs.values((int(qo[-1]), H, D), 1.0, 72)
    k = inputs.values((int(ko[-1]), H, D), 1.0, 73)
    cos, sin, _ = rope_tables(20, D)
    def scores(c, s):
        rq = oracle.rope(q, qo, ko, c, s)
        rk = oracle.rope(k, qo, ko, c, s, keys=True)
        return [rq[qo[b]:qo[b + 1], 0] @ rk[ko[b]:ko[b + 1], 0].T for b in range(2)]
    for a, b in zip(scores(cos, sin), scores(cos[5:], sin[5:])):
        np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("act,mask", [(SOFTMAX, CAUSAL), (GELU, NONE), (SOFTMAX, BLOCK)])
def test_rope_backward_is_the_transposed_rotation_of_the_gradient(act, mask):
    """Gradients of attention on rotated rows, w.r.t. the unrotated q and k
    (torch fp64 autograd through a padded dense formulation with the rotation
    written in torch), equal R^T applied to the oracle's dQ and dK."""
    H, D, scale = 2, 8, 0.35
    lq, lk = [3, 9, 0, 12], [5, 9, 4, 7]
    qo, ko, q, k, v, do = _batch(lq, lk, H, D, seed=74)
    cos, sin, _ = rope_tables(16, D)
    window = 4 if mask == BLOCK else 0
    kw = dict(H=H, D=D, act=act, mask=mask, window=window, scale=scale)
    rq = oracle.rope(q, qo, ko, cos, sin)
    rk = oracle.rope(k, qo, ko, cos, sin, keys=True)
    dq_r, dk_r, dv = oracle.bwd(qo, ko, rq, rk, v, do, **kw)
    dq = oracle.rope(dq_r, qo, ko, cos, sin, inverse=True)
    dk = oracle.rope(dk_r, qo, ko, cos, sin, keys=True, inverse=True)

    def rot_torch(x, off, oth, keys):
        parts = []
        for b in range(len(off) - 1):
            n, m = off[b + 1] - off[b], oth[b + 1] - oth[b]
            delta = (n - m) if keys else (m - n)
            shift = max(-delta, 0) if keys else max(delta, 0)
            pos = np.arange(n) + shift
            c = torch.from_numpy(cos[pos])[:, None, :]
            s = torch.from_numpy(sin[pos])[:, None, :]
            xs = x[off[b]:off[b + 1]]
            e, o = xs[..., 0::2], xs[..., 1::2]
            parts.append(torch.stack((e * c - o * s, e * s + o * c), dim=-1).reshape(xs.shape))
        return torch.cat(parts, 0)

    tq = R.to_f64(q).requires_grad_(True)
    tk = R.to_f64(k).requires_grad_(True)
    tv = R.to_f64(v).requires_grad_(True)
    o, _ = R.dense_forward(rot_torch(tq, qo, ko, False), rot_torch(tk, ko, qo, True), tv, qo, ko, act, mask, window,
                           scale, False)
    (o * R.to_f64(do)).sum().backward()
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-9, atol=1e-11)
