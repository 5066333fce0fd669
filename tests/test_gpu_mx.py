"""MXFP8 quantization on the GPU against the oracle's quantizer: codes,
scale exponents and row-block starts bit for bit."""
import numpy as np
import pytest
import torch

from jagged_attention_recsys_gdpa_gb300 import inputs
from oracle import mx
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu


def _check(x_cpu, off_cpu):
    import jagged_attention_recsys_gdpa_gb300 as J

    codes, scales, bs = J.mxfp8_quantize(x_cpu.cuda(), off_cpu.cuda())
    torch.cuda.synchronize()
    assert J.device_status() == 0
    rc, rs, rbs = mx.quantize(x_cpu, off_cpu.numpy())
    assert np.array_equal(bs.cpu().numpy(), rbs)
    got_c = codes.cpu().numpy()
    bad = np.argwhere(got_c != rc)
    assert bad.size == 0, (bad[:5], got_c[tuple(bad[0])], rc[tuple(bad[0])])
    assert np.array_equal(scales.cpu().numpy()[: int(rbs[-1])], rs)


@pytest.mark.parametrize("D", [64, 128])
def test_quantize_matches_oracle(D):
    lens = [1, 31, 32, 33, 300, 0, 129, 7]
    w = inputs.Workload("case", 3, D, 0, 0, 0, False, 1.0, True)
    cpu = G.cpu_inputs(w, lens, lens, seed=91)
    _check(cpu["q"], cpu["q_off"])


def test_quantize_wide_magnitudes_zeros_and_saturation():
    """Blocks scaled over 2^-30 .. 2^30, an all-zero block, negative zeros,
    and values that land in (448 X, 512 X) and saturate."""
    lens = np.array([64, 40])
    off = torch.from_numpy(np.concatenate([[0], np.cumsum(lens)]).astype(np.int64))
    g = torch.Generator().manual_seed(92)
    x = torch.randn(int(off[-1]), 2, 64, generator=g)
    x *= torch.exp2(torch.randint(-30, 31, (int(off[-1]), 2, 1), generator=g).float())
    x[0:32, 0, 0:32] = 0.0
    x[32:64, 1, 32:64] = -0.0
    x[64:96, 0, 0:32] = 0.1 * torch.randn(32, 32, generator=g)
    x[64:70, 0, 0:32] = 500.0  # block max 500: X = 1, so 500 (and 479 -> bf16 480) saturate to 448
    x[64, 0, 1] = 479.0
    _check(x.to(torch.bfloat16), off)


# ---------------------------------------------------------------- MXFP8 attention forward
def _mx_inputs(w, lq, lkv, seed):
    """Seeded bf16 inputs, quantized by the ORACLE's quantizer (the GPU's is
    bit-exact with it, tested above): codes, scales and block starts for both
    sides, as host numpy arrays and as device tensors."""
    cpu = G.cpu_inputs(w, lq, lkv, seed)
    qo, ko = cpu["q_off"].numpy(), cpu["kv_off"].numpy()
    host = {n: mx.quantize(cpu[n], qo if n == "q" else ko) for n in ("q", "k", "v")}
    dev = {n: (torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda(), torch.from_numpy(bs.astype(np.int32)).cuda())
           for n, (c, s, bs) in host.items()}
    return cpu, host, dev


def _mx_bound(host, cpu, w, o_ref):
    """Per-element bound |o - o_ref| <= sum_j (2^-3 e_ij + 2^-16) |v_jd| / l_i
    + 2^-8 |o_ref| + 1e-3: the kernel quantizes P per 32-key block against the
    block's own maximum (under a running row maximum), the oracle against the
    final row maximum, so each P~ may differ by one E4M3 rounding step (2^-4
    relative each way; below E4M3's normal range at most 2^-17 absolute on the
    kernel's side and 2^-18 on the oracle's); the rest covers the bf16
    rounding of o and fp32 accumulation.
    e_ij = exp(s_ij - m_i) and l_i = sum_j e_ij from the dequantized operands."""
    qo, ko = cpu["q_off"].numpy(), cpu["kv_off"].numpy()
    qd, kd, vd = (mx.dequantize(*host[n][:2], qo if n == "q" else ko) for n in ("q", "k", "v"))
    bound = 2.0**-8 * np.abs(o_ref) + 1e-3
    scale = 1.0 / np.sqrt(w.D)
    mask = w.mask | (1 if w.mask & 2 else 0)
    for b in range(len(qo) - 1):
        lq, lkv = int(qo[b + 1] - qo[b]), int(ko[b + 1] - ko[b])
        if lq == 0 or lkv == 0:
            continue
        ok = mx._allowed(lq, lkv, mask, w.window)
        for h in range(w.H):
            s = np.where(ok, scale * qd[qo[b]:qo[b + 1], h] @ kd[ko[b]:ko[b + 1], h].T, -np.inf)
            m = np.where(ok.any(1), s.max(1, initial=-np.inf), 0.0)
            e = np.where(ok, np.exp(s - m[:, None]), 0.0)
            l = np.maximum(e.sum(1), 1e-300)
            term = ((2.0**-3 * e + 2.0**-16 * ok) @ np.abs(vd[ko[b]:ko[b + 1], h])) / l[:, None]
            bound[qo[b]:qo[b + 1], h] += term
    return bound


MX_CASES = [
    # (mask, window, lq, lkv, std)
    (1, 0, [1, 127, 128, 129, 300, 513], None, 1.0),
    (3, 200, [1, 127, 128, 129, 300, 513], None, 1.0),
    (0, 0, [100, 300, 5, 1], [20, 700, 129, 300], 1.0),
    (4, 64, [1, 127, 128, 129, 300, 513], None, 1.0),
    (1, 0, [0, 5, 130, 0], [7, 0, 130, 3], 1.0),
    (1, 0, [300, 700], None, 2.0),  # peaky rows: the running maximum moves often
]


@pytest.mark.parametrize("case", range(len(MX_CASES)))
def test_mxfp8_forward_matches_oracle(case):
    """The block-scaled FP8 forward against oracle/mx.py's attention_fwd on the
    operands the codes and scales stand for, under the per-element bound the
    kernel's P quantization allows (see _mx_bound and jattn.h); LSE, which
    uses the unquantized P, within the bf16 tolerance."""
    import jagged_attention_recsys_gdpa_gb300 as J

    mask, window, lq, lkv, std = MX_CASES[case]
    lkv = lq if lkv is None else lkv
    w = inputs.Workload("case", 2, 128, 0, mask, window, False, std, lq == lkv)
    cpu, host, dev = _mx_inputs(w, lq, lkv, seed=95 + case)
    qo, ko = cpu["q_off"].numpy(), cpu["kv_off"].numpy()
    qd, kd, vd = (mx.dequantize(*host[n][:2], qo if n == "q" else ko) for n in ("q", "k", "v"))
    o_ref, lse_ref = mx.attention_fwd(qd, kd, vd, qo, ko, mask=mask | (1 if mask & 2 else 0), window=window)
    o, lse = J.forward_mxfp8(dev["q"], dev["k"], dev["v"], cpu["q_off"].cuda(), cpu["kv_off"].cuda(),
                             causal=bool(mask & 1), window=window if mask & 2 else 0,
                             block=window if mask & 4 else 0)
    torch.cuda.synchronize()
    assert J.device_status() == 0
    got = G.to64(o)
    assert np.all(np.isfinite(got))
    bound = _mx_bound(host, cpu, w, o_ref)
    err = np.abs(got - o_ref)
    bad = err > bound
    assert not bad.any(), (int(bad.sum()), float((err - bound).max()))
    lg = lse.cpu().numpy().astype(np.float64)
    assert np.array_equal(np.isneginf(lg), np.isneginf(lse_ref))
    fin = np.isfinite(lse_ref)
    G.assert_close(lg[fin], lse_ref[fin], "LSE")



# ---------------------------------------------------------------- MXFP8 attention backward
def _mx_bwd_bounds(host, cpu, w, o64, mask):
    """Reference gradients (oracle/mx.py attention_bwd, on the operands the
    codes and scales stand for and the kernel's own forward output o) and
    per-element bounds for the kernel's:
      dV: each P~ within one E4M3 step of the oracle's (2^-3 p + 2^-16 / l,
          as the forward) plus 2^-10 p for the kernel's fp32 P;
      dQ, dK: each dS~ within the oracle's own quantization error |dS~_o - dS|
          plus the worst quantization error the kernel's block can have
          (2^-4 |x| + 2^-10 X + saturation above 448 X, for the oracle's
          block scale X or, where the block maximum lies within 2^-8 of a
          power of two, the neighbouring scale), at |x| + delta, delta the
          kernel's fp32 error on dS (2^-14 relative sums of the products
          behind dP and D, 2^-12 of dS);
    each plus 2^-7 of itself and 2^-8 |ref| + 1e-3 for the bf16 rounding of
    the output."""
    qo, ko = cpu["q_off"].numpy(), cpu["kv_off"].numpy()
    qd, kd, vd, dod = (mx.dequantize(*host[n][:2], qo if n in ("q", "do") else ko) for n in ("q", "k", "v", "do"))
    scale = 1.0 / np.sqrt(w.D)
    refs = mx.attention_bwd(qd, kd, vd, dod, qo, ko, mask=mask, window=w.window, o=o64)
    bq, bk, bv = (np.zeros_like(r) for r in refs)
    for b in range(len(qo) - 1):
        lq, lkv = int(qo[b + 1] - qo[b]), int(ko[b + 1] - ko[b])
        if lq == 0 or lkv == 0:
            continue
        ok = mx._allowed(lq, lkv, mask, w.window)
        qs, ks = slice(qo[b], qo[b + 1]), slice(ko[b], ko[b + 1])
        for h in range(w.H):
            s = np.where(ok, scale * qd[qs, h] @ kd[ks, h].T, -np.inf)
            m = np.where(ok.any(1), s.max(1, initial=-np.inf), 0.0)
            e = np.where(ok, np.exp(s - m[:, None]), 0.0)
            l = np.maximum(e.sum(1), 1e-300)
            p = e / l[:, None]
            di = np.einsum("id,id->i", dod[qs, h], o64[qs, h])
            dp = dod[qs, h] @ vd[ks, h].T
            ds = np.where(ok, p * (dp - di[:, None]), 0.0)
            absdo = np.abs(dod[qs, h])
            delta = p * 2.0**-14 * (absdo @ np.abs(vd[ks, h]).T + (absdo * np.abs(o64[qs, h])).sum(1)[:, None])
            delta += 2.0**-12 * np.abs(ds)
            qerr = np.zeros_like(ds)
            for r0 in range(0, lq, 32):
                for c0 in range(0, lkv, 32):
                    blk = ds[r0:r0 + 32, c0:c0 + 32]
                    x = np.abs(blk) + delta[r0:r0 + 32, c0:c0 + 32]
                    amax = float(np.abs(blk).max())
                    E = mx.scale_exponent(amax)
                    cands = [E]
                    if amax > 0:
                        f = np.floor(np.log2(amax))
                        if amax * (1 - 2.0**-8) < 2.0**f:
                            cands.append(max(E - 1, 0))
                        if amax * (1 + 2.0**-8) >= 2.0**(f + 1):
                            cands.append(E + 1)
                    worst = np.zeros_like(x)
                    for Ec in cands:
                        X = 2.0**(Ec - 127)
                        worst = np.maximum(worst, 2.0**-4 * x + 2.0**-10 * X + np.maximum(0.0, x - 448.0 * X))
                    qerr[r0:r0 + 32, c0:c0 + 32] = worst
            bds = np.abs(mx.quantize_square(ds) - ds) + qerr + delta
            bq[qs, h] = scale * bds @ np.abs(kd[ks, h])
            bk[ks, h] = scale * bds.T @ np.abs(qd[qs, h])
            bp = 2.0**-3 * p + 2.0**-16 * ok / l[:, None] + 2.0**-10 * p
            bv[ks, h] = bp.T @ absdo
    bounds = [(1 + 2.0**-7) * bb + 2.0**-8 * np.abs(r) + 1e-3 for bb, r in zip((bq, bk, bv), refs)]
    return refs, bounds


MX_BWD_CASES = [
    # (mask, window, lq, lkv)
    (1, 0, [1, 95, 96, 97, 128, 129, 300, 513], None),
    (3, 200, [1, 127, 128, 129, 300, 513], None),
    (0, 0, [100, 300, 5, 1], [20, 700, 129, 300]),
    (4, 64, [1, 127, 128, 129, 300, 513], None),
    (1, 0, [0, 5, 130, 0], [7, 0, 130, 3]),
    (5, 32, [200, 64, 1], None),
]


@pytest.mark.parametrize("case", range(len(MX_BWD_CASES)))
def test_mxfp8_backward_matches_oracle(case):
    """The block-scaled FP8 backward (D, dQ and dK/dV passes) against
    oracle/mx.py's attention_bwd on the dequantized operands and the kernel's
    own forward output, under the per-element bounds of _mx_bwd_bounds."""
    import jagged_attention_recsys_gdpa_gb300 as J

    mask, window, lq, lkv = MX_BWD_CASES[case]
    lkv = lq if lkv is None else lkv
    w = inputs.Workload("case", 2, 128, 0, mask, window, False, 1.0, lq == lkv)
    cpu, host, dev = _mx_inputs(w, lq, lkv, seed=120 + case)
    qo = cpu["q_off"].numpy()
    host["do"] = mx.quantize(cpu["do"], qo)
    c, s, bs = host["do"]
    dev["do"] = (torch.from_numpy(c).cuda(), torch.from_numpy(s).cuda(), torch.from_numpy(bs.astype(np.int32)).cuda())
    q_off, kv_off = cpu["q_off"].cuda(), cpu["kv_off"].cuda()
    kw = dict(causal=bool(mask & 1), window=window if mask & 2 else 0, block=window if mask & 4 else 0)
    o, lse = J.forward_mxfp8(dev["q"], dev["k"], dev["v"], q_off, kv_off, **kw)
    dq, dk, dv = J.backward_mxfp8(dev["q"], dev["k"], dev["v"], o, lse, dev["do"], q_off, kv_off, **kw)
    torch.cuda.synchronize()
    assert J.device_status() == 0
    full_mask = mask | (1 if mask & 2 else 0)
    refs, bounds = _mx_bwd_bounds(host, cpu, w, G.to64(o), full_mask)
    for name, got_t, ref, bound in zip(("dQ", "dK", "dV"), (dq, dk, dv), refs, bounds):
        got = G.to64(got_t)
        assert np.all(np.isfinite(got)), name
        err = np.abs(got - ref)
        bad = err > bound
        assert not bad.any(), (name, int(bad.sum()), float((err - bound).max()), np.argwhere(bad)[:3])
