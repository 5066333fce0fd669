"""The allocation-free forward entry point, jattn_fwd_noalloc.

Some callers cannot allocate device memory where they run attention: their
memory belongs to a pool or a host runtime that forbids allocations outside
it, or they run in a serving loop that must never block in the allocator.
jattn_fwd_noalloc serves them by keeping its scratch in an array inside the
library instead of a caller-provided workspace. Its output must match
jattn_fwd's on the same inputs, and a second call must not be disturbed by
what the first left in the shared array.
"""
import pytest
import torch

from jagged_attention_recsys_gdpa_gb300 import inputs
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu


def _call_noalloc(x, w, q_off=None):
    import jagged_attention_recsys_gdpa_gb300 as J
    from jagged_attention_recsys_gdpa_gb300 import _binding as B

    causal = bool(w.mask & 1)
    window = w.window if w.mask & 2 else 0
    q_off = x["q_off"] if q_off is None else q_off
    kv_off = q_off if w.self_attn else x["kv_off"]
    p = J.make_params(x["q"], x["k"], x["q_off"], w.act, J._mask(causal, window), window, None, w.norm_by_lkv)
    o = torch.empty_like(x["q"])
    lse = torch.empty(x["q"].shape[0], w.H, dtype=torch.float32, device="cuda") if w.act == 0 else None
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    B.fwd_noalloc(p, q_off, kv_off, x["q"], x["k"], x["v"], o, lse, status,
                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return o, lse, int(status.item())


CASES = [
    (inputs.Workload("self", 2, 128, 0, 3, 200, False, 1.0, True), [1, 127, 128, 129, 300, 1000], None),
    (inputs.Workload("cross", 3, 64, 2, 0, 0, True, 0.5, False), [5, 300, 700, 32], [20, 1, 257, 2000]),
]


def test_noalloc_forward_matches_workspace_forward():
    """Three calls in a row (case 1, case 2, case 1 again): each must equal
    jattn_fwd on the same inputs bit for bit (same kernels, no atomics), so
    nothing a previous call left in the shared array changes a result."""
    import jagged_attention_recsys_gdpa_gb300 as J

    for call, ci in enumerate([0, 1, 0]):
        w, lq, lkv = CASES[ci]
        x = G.to_cuda(G.cpu_inputs(w, lq, lkv if lkv is not None else lq, 40 + ci))
        causal = bool(w.mask & 1)
        window = w.window if w.mask & 2 else 0
        o_ref, lse_ref = J.forward(x["q"], x["k"], x["v"], x["q_off"], x["kv_off"], act=w.act, causal=causal,
                                   window=window, norm_by_lkv=w.norm_by_lkv)
        o, lse, status = _call_noalloc(x, w)
        assert status == 0, f"call {call + 1}"
        assert torch.equal(o, o_ref), f"O differs from jattn_fwd (call {call + 1})"
        if w.act == 0:
            assert torch.equal(lse, lse_ref), f"LSE differs from jattn_fwd (call {call + 1})"
        # and within the tolerance of the oracle-checked path, element by element
        G.assert_close(G.to64(o), G.to64(o_ref), f"O (call {call + 1})")


def test_noalloc_reports_device_errors_then_recovers():
    """Bad offsets reach the caller's status int through the scratch status
    word; the next clean call clears it and is correct."""
    import jagged_attention_recsys_gdpa_gb300 as J

    w, lq, _ = CASES[0]
    x = G.to_cuda(G.cpu_inputs(w, lq, lq, 45))
    bad = x["q_off"].clone()
    bad[2] = bad[3] + 1  # offsets decrease from entry 2 to entry 3
    _, _, status = _call_noalloc(x, w, q_off=bad)
    assert status == 5  # JATTN_ERR_OFFSETS
    o, lse, status = _call_noalloc(x, w)
    assert status == 0
    o_ref, lse_ref = J.forward(x["q"], x["k"], x["v"], x["q_off"], x["kv_off"], act=w.act, causal=True,
                               window=w.window)
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)
