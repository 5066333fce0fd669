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
