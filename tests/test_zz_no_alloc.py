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


def _call_noalloc(x, w):
    import jagged_attention_recsys_gdpa_gb300 as J
    from jagged_attention_recsys_gdpa_gb300 import _binding as B

    causal = bool(w.mask & 1)
    window = w.window if w.mask & 2 else 0
    p = J.make_params(x["q"], x["k"], x["q_off"], w.act, J._mask(causal, window), window, None, w.norm_by_lkv)
    o = torch.empty_like(x["q"])
    lse = torch.empty(x["q"].shape[0], w.H, dtype=torch.float32, device="cuda") if w.act == 0 else None
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    B.fwd_noalloc(p, x["q_off"], x["kv_off"], x["q"], x["k"], x["v"], o, lse, status,
                  torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return o, lse, int(status.item())


def test_noalloc_forward_matches_workspace_forward_twice():
    import jagged_attention_recsys_gdpa_gb300 as J

    cases = [
        (inputs.Workload("self", 2, 128, 0, 3, 200, False, 1.0, True), [1, 127, 128, 129, 300, 1000], None),
        (inputs.Workload("cross", 3, 64, 2, 0, 0, True, 0.5, False), [5, 300, 700, 32], [20, 1, 257, 2000]),
    ]
    for seed, (w, lq, lkv) in enumerate(cases):
        x = G.to_cuda(G.cpu_inputs(w, lq, lkv if lkv is not None else lq, 40 + seed))
        causal = bool(w.mask & 1)
        window = w.window if w.mask & 2 else 0
        o_ref, lse_ref = J.forward(x["q"], x["k"], x["v"], x["q_off"], x["kv_off"], act=w.act, causal=causal,
                                   window=window, norm_by_lkv=w.norm_by_lkv)
        o, lse, status = _call_noalloc(x, w)
        assert status == 0
        G.assert_close(G.to64(o), G.to64(o_ref), f"O (call {seed + 1})")
        if w.act == 0:
            fin = torch.isfinite(lse_ref)
            assert torch.equal(torch.isneginf(lse), torch.isneginf(lse_ref))
            G.assert_close(G.to64(lse[fin]), G.to64(lse_ref[fin]), f"LSE (call {seed + 1})")
