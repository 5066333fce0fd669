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

