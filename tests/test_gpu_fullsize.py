"""Full-size workloads in the launch configuration the benchmark times: the
whole batch runs on the GPU; the oracle recomputes a sample of whole
sequences (the longest, the shortest and two drawn at random), which is
exact because sequences are independent. Every output must be finite."""
import gc

import numpy as np
import pytest
import torch

from jagged_attention_recsys_gdpa_gb300 import inputs
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize(
    "name", ["tiny", "jfa", "jfa_causal", "jfa_block", "gdpa_cross", "gdpa_pma", "gdpa_pma_poly", "mixed"]
)
def test_fullsize_sampled_sequences(name):
    w = inputs.WORKLOADS[name]
    x = inputs.make(name, seed=0, device="cuda")
    cost = x["lq"] * np.maximum(x["lkv"], 1)
    rng = np.random.default_rng(1)
    seqs = sorted({int(np.argmax(cost)), int(np.argmin(x["lq"])), *rng.choice(len(x["lq"]), 2, replace=False).tolist()})
    if name == "tiny":
        seqs = list(range(len(x["lq"])))
    sub, rq, rk = G.subset(x, seqs)
    if w.mask & 4:
        # Block masks: the backward of the whole batch reads, on the sampled
        # sequences' rows, the oracle's O (bf16) and LSE; sequences are
        # independent, so the sample's gradients are those of the oracle's
        # stored output (other rows keep this forward's O).
        g = G.gpu_run(x, w, backward=False)
        rf = G.oracle_run(sub, w, backward=False)
        o_st = torch.from_numpy(rf["o"]).to(torch.bfloat16)
        o2, lse2 = g["o"].clone(), g["lse"].clone()
        iq = torch.as_tensor(rq, device="cuda")
        o2[iq] = o_st.cuda()
        lse2[iq] = torch.from_numpy(rf["lse"]).to(torch.float32).cuda()
        gb = G.gpu_run(x, w, backward=True, stored=(o2, lse2))
        g.update({k: t for k, t in gb.items() if k.startswith("d")})
        r = dict(rf)
        r.update({k: t for k, t in G.oracle_run(sub, w, True, o_stored=o_st).items() if k.startswith("d")})
    else:
        g = G.gpu_run(x, w)
        r = G.oracle_run(sub, w)
    for key in ("o", "dq", "dk", "dv"):
        assert torch.isfinite(g[key]).all(), key
    if w.act == 0:
        assert not torch.isnan(g["lse"]).any()
    G.compare(g, r, w, rows_q=rq, rows_kv=rk)
    del x, g
    gc.collect()
    torch.cuda.empty_cache()
