"""Device-side error reporting: bad offsets and an expired bounded wait set the
status word, no kernel traps, and the context stays usable afterwards."""
import numpy as np
import pytest
import torch

from jagged_attention_recsys_gdpa_gb300 import inputs
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu

JATTN_ERR_OFFSETS, JATTN_ERR_TIMEOUT = 5, 6


def _small():
    w = inputs.Workload("s", 2, 128, 0, 1, 0, False, 1.0, True)
    cpu = G.cpu_inputs(w, [100, 300, 7], [100, 300, 7], 21)
    return w, G.to_cuda(cpu), cpu


def test_bad_offsets_set_status():
    import jagged_attention_recsys_gdpa_gb300 as J

    w, x, _ = _small()
    assert J.device_status() in (0, JATTN_ERR_OFFSETS, JATTN_ERR_TIMEOUT)  # clear anything earlier
    bad = x["q_off"].clone()
    bad[1] = bad[2] + 1  # offsets decrease from entry 1 to entry 2
    J.forward(x["q"], x["k"], x["v"], bad, bad, causal=True)
    assert J.device_status() == JATTN_ERR_OFFSETS
    end = x["q_off"].clone()
    end[-1] -= 1  # last offset disagrees with the tensor's row count
    J.forward(x["q"], x["k"], x["v"], end, end, causal=True)
    assert J.device_status() == JATTN_ERR_OFFSETS
    # a clean call afterwards reports OK and correct values
    g = G.gpu_run(x, w)
    assert J.device_status() == 0
    assert torch.isfinite(g["o"]).all()


def test_expired_wait_reports_timeout_and_context_survives():
    import jagged_attention_recsys_gdpa_gb300 as J
    from jagged_attention_recsys_gdpa_gb300 import _binding as B

    w, x, cpu = _small()
    J.device_status()
    try:
        B.debug_set(1, 50_000_000)  # skip the first copy; waits give up after 50 ms
        J.forward(x["q"], x["k"], x["v"], x["q_off"], x["kv_off"], causal=True)
        assert J.device_status() == JATTN_ERR_TIMEOUT
    finally:
        B.debug_set(0, 0)
    g = G.gpu_run(x, w)
    assert J.device_status() == 0
    r = G.oracle_run(cpu, w)
    G.compare(g, r, w)


@pytest.mark.parametrize("act", [0, 1])
def test_backward_alone_times_out_then_recovers(act):
    """A clean forward, then only the backward with its first copies skipped:
    the dQ and dK/dV kernels themselves must give up, report TIMEOUT and
    return, and the next clean backward on the same context is correct."""
    import jagged_attention_recsys_gdpa_gb300 as J
    from jagged_attention_recsys_gdpa_gb300 import _binding as B

    w = inputs.Workload("s", 2, 128, act, 1, 0, act != 0, 1.0, True)
    cpu = G.cpu_inputs(w, [100, 300, 7], [100, 300, 7], 22)
    x = G.to_cuda(cpu)
    J.device_status()
    o, lse = J.forward(x["q"], x["k"], x["v"], x["q_off"], x["kv_off"], act=act, causal=True,
                       norm_by_lkv=w.norm_by_lkv)
    assert J.device_status() == 0
    try:
        B.debug_set(1, 50_000_000)
        J.backward(x["q"], x["k"], x["v"], o, lse, x["do"], x["q_off"], x["kv_off"], act=act, causal=True,
                   norm_by_lkv=w.norm_by_lkv)
        assert J.device_status() == JATTN_ERR_TIMEOUT
    finally:
        B.debug_set(0, 0)
    dq, dk, dv = J.backward(x["q"], x["k"], x["v"], o, lse, x["do"], x["q_off"], x["kv_off"], act=act,
                            causal=True, norm_by_lkv=w.norm_by_lkv)
    torch.cuda.synchronize()
    assert J.device_status() == 0
    r = G.oracle_run(cpu, w)
    G.compare({"o": o, "lse": lse, "dq": dq, "dk": dk, "dv": dv}, r, w)
