"""Pins for the MXFP8 quantization oracle (no GPU): the E4M3 element codec
against torch's float8_e4m3fn casts, the block rule against its defining
properties, transpose invariance of the square blocks, and exactness on
values the format represents."""
import numpy as np
import pytest
import torch

from oracle import mx


def test_decode_matches_torch_float8():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = mx.e4m3_decode(codes)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert mx.e4m3_decode(np.uint8(0x7E)) == 448.0 and mx.e4m3_decode(np.uint8(0x01)) == 2.0**-9


def test_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(0)
    vals = mx.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (vals[1:] + vals[:-1]) / 2  # exact ties between neighbours
    x = np.concatenate([
        rng.uniform(-448, 448, 20000),
        rng.normal(0, 1, 20000) * np.exp2(rng.integers(-12, 8, 20000)),
        mids, -mids, vals, -vals, [0.0, -0.0, 2.0**-10, 3 * 2.0**-11],
    ])
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = mx.e4m3_encode(x)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, (x[bad[:5]], got[bad[:5]], ref[bad[:5]])


def test_encode_saturates_and_keeps_nan():
    x = np.array([448.0, 449.0, 500.0, 1e6, -1e30, np.nan])
    assert list(mx.e4m3_encode(x)) == [0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0x7F]


def test_scale_rule():
    # largest element lands in [2^8, 2^9) before rounding; the power of two is exact
    for amax, want in ((1.0, 119), (1.5, 119), (2.0, 120), (255.9, 126), (256.0, 127), (3e-38, 0), (0.0, 0)):
        assert mx.scale_exponent(amax) == want, amax
    rng = np.random.default_rng(1)
    for _ in range(200):
        blk = rng.normal(0, 1, (32, 32)) * np.exp2(rng.integers(-20, 20))
        codes, E = mx.quantize_block(blk)
        a = np.max(np.abs(blk)) / np.exp2(E - 127.0)
        assert 256.0 <= a < 512.0
        top = np.max(np.abs(mx.e4m3_decode(codes)))
        assert 256.0 <= top <= 448.0


def test_error_bound_of_quantize_dequantize():
    """|x - dq(x)| <= 2^-4 |x| for normal codes (3 mantissa bits: half an
    ulp), <= 2^-10 X in the subnormal range, <= 64 X where 448 saturates."""
    rng = np.random.default_rng(2)
    lens = np.array([1, 31, 32, 33, 70, 0, 5])
    off = np.concatenate([[0], np.cumsum(lens)])
    x = rng.normal(0, 1, (int(off[-1]), 2, 64)) * np.exp2(rng.integers(-6, 6, (int(off[-1]), 2, 64)))
    codes, scales, bs = mx.quantize(x, off)
    assert list(bs) == [0, 1, 2, 3, 5, 8, 8, 9]
    dq = mx.dequantize(codes, scales, off)
    for b in range(len(lens)):
        for r in range((lens[b] + 31) // 32):
            rows = slice(off[b] + 32 * r, min(off[b] + 32 * r + 32, off[b + 1]))
            X = np.exp2(scales[bs[b] + r].astype(np.float64) - 127.0)  # [H, D/32]
            Xe = np.repeat(X, 32, axis=1)[None]
            err = np.abs(x[rows] - dq[rows])
            bound = np.maximum(2.0**-4 * np.abs(x[rows]), 2.0**-10 * Xe)
            bound = np.where(np.abs(x[rows]) > 448 * Xe, 64 * Xe, bound)
            assert np.all(err <= bound * (1 + 1e-12))


def test_square_blocks_are_transpose_invariant():
    """One sequence of 96 rows, D = 96 columns, one head: quantizing the
    transpose with the same 32 x 32 blocks gives the transposed codes and
    scales (the property that lets a tensor quantized once serve QK^T and the
    transposed products of the backward)."""
    rng = np.random.default_rng(3)
    x = rng.normal(0, 1, (96, 1, 96)) * np.exp2(rng.integers(-4, 4, (96, 1, 96)))
    off = np.array([0, 96])
    c1, s1, _ = mx.quantize(x, off)
    c2, s2, _ = mx.quantize(np.ascontiguousarray(x[:, 0, :].T[:, None, :]), off)
    assert np.array_equal(c1[:, 0, :].T, c2[:, 0, :])
    assert np.array_equal(s1[:, 0, :].T, s2[:, 0, :])


def test_representable_values_round_trip_exactly():
    """Blocks built from E4M3 codes times a power of two whose largest code
    magnitude is in [256, 448] come back with the same codes and scale."""
    rng = np.random.default_rng(4)
    off = np.array([0, 40, 72])
    codes = rng.integers(0, 0x7F, (72, 1, 32)).astype(np.uint8) | (rng.integers(0, 2, (72, 1, 32)) << 7).astype(np.uint8)
    codes = np.where((codes & 0x7F) == 0x7F, 0x7E, codes).astype(np.uint8)
    bs = mx.block_starts(off)
    E = rng.integers(100, 150, (int(bs[-1]), 1, 1))
    for g, (r0, r1) in enumerate([(0, 32), (32, 40), (40, 72)]):
        codes[r0, 0, 0] = 0x78  # 256: pins the block's scale
    x = mx.e4m3_decode(codes)
    for g, (r0, r1) in enumerate([(0, 32), (32, 40), (40, 72)]):
        x[r0:r1] *= np.exp2(float(E[g, 0, 0]) - 127.0)
    got_codes, got_scales, _ = mx.quantize(x, off)
    assert np.array_equal(got_codes, codes)
    assert np.array_equal(got_scales[:, 0, 0], E[:, 0, 0])


# ---------------------------------------------------------------- MXFP8 attention
import oracle  # noqa: E402


def _mx_inputs(lq, lk, H, D, seed):
    rng = np.random.default_rng(seed)
    qo = np.concatenate([[0], np.cumsum(lq)]).astype(np.int64)
    ko = np.concatenate([[0], np.cumsum(lk)]).astype(np.int64)
    def deq(n, off):
        x = rng.normal(0, 1, (n, H, D))
        c, s, _ = mx.quantize(x, off)
        return mx.dequantize(c, s, off)
    return qo, ko, deq(int(qo[-1]), qo), deq(int(ko[-1]), ko), deq(int(ko[-1]), ko), deq(int(qo[-1]), qo)


@pytest.mark.parametrize("mask,window", [(0, 0), (1, 0), (3, 5), (4, 8), (5, 8)])
def test_mx_attention_without_quantized_intermediates_is_the_oracle(mask, window):
    """With P and dS kept exact, the MXFP8 attention of dequantized operands
    is the C oracle's attention of the same values (forward and backward)."""
    H, D = 2, 64
    qo, ko, q, k, v, do = _mx_inputs([5, 40, 0, 33], [9, 40, 3, 33], H, D, 5)
    kw = dict(mask=mask, window=window, scale=0.125)
    o, lse = mx.attention_fwd(q, k, v, qo, ko, quant_p=False, **kw)
    o_ref, lse_ref = oracle.fwd(qo, ko, q, k, v, H=H, D=D, **kw)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, lse_ref, rtol=1e-12, atol=1e-13)
    g = mx.attention_bwd(q, k, v, do, qo, ko, o=o_ref, quant_p=False, quant_ds=False, **kw)
    g_ref = oracle.bwd(qo, ko, q, k, v, do, H=H, D=D, **kw)
    for a, b in zip(g, g_ref):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12)


def test_mx_attention_quantized_p():
    """P quantized with X = 2^-8: probabilities keep half an E4M3 ulp; a row
    that sees one key (P = 1, exactly representable) returns that value row."""
    p = np.linspace(0, 1, 100001)
    pq = mx.quantize_p(p)
    assert np.all(np.abs(pq - p) <= np.maximum(2.0**-4 * p, 2.0**-18) * (1 + 1e-12))
    assert mx.quantize_p(np.array([1.0]))[0] == 1.0
    qo, ko, q, k, v, _ = _mx_inputs([7], [7], 1, 64, 6)
    o, _ = mx.attention_fwd(q, k, v, qo, ko, mask=1)
    np.testing.assert_array_equal(o[0], v[0])  # causal row 0 sees key 0 only


def test_square_quantization_matches_the_jagged_quantizer():
    """quantize_square (dS blocks) and quantize (operands) agree on one
    sequence, and quantize_square commutes with transposition."""
    rng = np.random.default_rng(7)
    a = rng.normal(0, 1, (70, 96)) * np.exp2(rng.integers(-5, 5, (70, 96)))
    c, s, _ = mx.quantize(a[:, None, :], np.array([0, 70]))
    np.testing.assert_array_equal(mx.quantize_square(a), mx.dequantize(c, s, np.array([0, 70]))[:, 0, :])
    np.testing.assert_array_equal(mx.quantize_square(a.T), mx.quantize_square(a).T)
