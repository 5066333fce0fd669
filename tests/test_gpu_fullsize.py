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


@pytest.mark.parametrize("name", ["tiny", "jfa", "jfa_causal", "gdpa_cross", "gdpa_pma", "mixed"])
def test_fullsize_sampled_sequences(name):
    w = inputs.WORKLOADS[name]
    x = inputs.make(name, seed=0, device="cuda")
    g = G.gpu_run(x, w)
    for key in ("o", "dq", "dk", "dv"):
        assert torch.isfinite(g[key]).all(), key
    if w.act == 0:
        assert not torch.isnan(g["lse"]).any()
    cost = x["lq"] * np.maximum(x["lkv"], 1)
    rng = np.random.default_rng(1)
    seqs = sorted({int(np.argmax(cost)), int(np.argmin(x["lq"])), *rng.choice(len(x["lq"]), 2, replace=False).tolist()})
    if name == "tiny":
        seqs = list(range(len(x["lq"])))
    sub, rq, rk = G.subset(x, seqs)
    r = G.oracle_run(sub, w)
    G.compare(g, r, w, rows_q=rq, rows_kv=rk)
    del x, g
    gc.collect()
    torch.cuda.empty_cache()
