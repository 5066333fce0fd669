"""GDPA's ALU-only GELU (activation code 3): tanh-GELU's Taylor polynomial at
0 through x^6. CPU checks of the coefficients the header states, of the
accuracy it claims on the bounded score range, and of the host plumbing; the
GPU kernels are checked against the oracle in test_gpu_parity.py."""
import ctypes

import numpy as np
import pytest

import oracle
from jagged_attention_recsys_gdpa_gb300 import inputs
from tests.dense_ref import POLY_G2 as G2, POLY_G4 as G4, POLY_G6 as G6, gelu_poly

C = np.sqrt(2.0 / np.pi)
A = 0.044715


def _gelu(x):
    return 0.5 * x * (1.0 + np.tanh(C * (x + A * x**3)))


def _gelu_grad(x):
    t = np.tanh(C * (x + A * x**3))
    return 0.5 * (1.0 + t) + 0.5 * x * (1.0 - t * t) * C * (1.0 + 3.0 * A * x * x)


def _poly(x):
    return gelu_poly(x)


def _poly_grad(x):
    return 0.5 + 2 * G2 * x + 4 * G4 * x**3 + 6 * G6 * x**5


def test_coefficients_are_the_taylor_series():
    sp = pytest.importorskip("sympy")
    x = sp.symbols("x")
    c = sp.sqrt(2 / sp.pi)
    a = sp.Rational(44715, 10**6)
    series = sp.series(x / 2 * (1 + sp.tanh(c * (x + a * x**3))), x, 0, 8).removeO()
    coeffs = [float(series.coeff(x, n)) for n in range(8)]
    np.testing.assert_allclose(coeffs, [0.0, 0.5, G2, 0.0, G4, 0.0, G6, 0.0], rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("R,f_err,g_err", [(0.75, 1.2e-4, 1.3e-3), (1.0, 1.2e-3, 9e-3)])
def test_accuracy_on_the_bounded_range(R, f_err, g_err):
    x = np.linspace(-R, R, 400001)
    assert np.abs(_poly(x) - _gelu(x)).max() <= f_err
    assert np.abs(_poly_grad(x) - _gelu_grad(x)).max() <= g_err
    # and the polynomial leaves tanh-GELU outside it, as the header warns
    assert abs(_poly(1.5) - _gelu(1.5)) > 2e-2


def test_oracle_treats_it_as_tanh_gelu():
    H, D = 2, 16
    lq, lk = np.array([5, 0, 40]), np.array([9, 3, 40])
    qo, ko = inputs.offsets(lq), inputs.offsets(lk)
    q = inputs.values((int(qo[-1]), H, D), 0.5, 61)
    k = inputs.values((int(ko[-1]), H, D), 0.5, 62)
    v = inputs.values((int(ko[-1]), H, D), 0.5, 63)
    do = inputs.values((int(qo[-1]), H, D), 1.0, 64)
    kw = dict(H=H, D=D, mask=1, norm_by_lkv=True)
    a = oracle.fwd(qo, ko, q, k, v, act=2, **kw)[0], *oracle.bwd(qo, ko, q, k, v, do, act=2, **kw)
    b = oracle.fwd(qo, ko, q, k, v, act=3, **kw)[0], *oracle.bwd(qo, ko, q, k, v, do, act=3, **kw)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_qk_norm_inputs_bound_the_scores():
    w = inputs.WORKLOADS["gdpa_pma_poly"]
    lens = (np.array([32, 32]), np.array([300, 77]))
    x = inputs.make(w, seed=3, device="cpu", lens=lens)
    q = x["q"].double().numpy()
    k = x["k"].double().numpy()
    target = np.sqrt(w.qk_norm * np.sqrt(w.D))
    np.testing.assert_allclose(np.linalg.norm(q, axis=-1), target, rtol=8e-3)
    s = np.einsum("ihd,jhd->hij", q[:32], k[:300]) / np.sqrt(w.D)
    assert np.abs(s).max() <= w.qk_norm * (1 + 2e-2)


def test_host_plumbing():
    import jagged_attention_recsys_gdpa_gb300 as J
    from jagged_attention_recsys_gdpa_gb300 import _binding as B
    from jagged_attention_recsys_gdpa_gb300 import build as build_mod

    assert J._act("gelu_poly") == 3 == B.GELU_POLY
    build_mod.build()
    lib = B.load()
    for act, ok in ((3, True), (4, False)):
        p = B.params(2, 10, 10, 2, 128, act, 0, 0, 0.0, 1)
        size = ctypes.c_size_t(0)
        assert (lib.jattn_workspace_size(ctypes.byref(p), ctypes.byref(size)) == 0) == ok, act
