"""Full-size workloads in the launch configuration the benchmark times: the
whole batch runs on the GPU and is compared with the oracle, which is exact
sequence by sequence because sequences are independent.

* The four configured workloads (tiny, jfa, gdpa_cross, gdpa_pma) are
  compared on EVERY sequence. The oracle runs over consecutive groups of
  sequences (a bounded number of rows at a time, so its double-precision
  copies stay a few GB) against the matching rows of the GPU outputs.
* The supplementary workloads and the largest one (mixed: 5.8 M rows, about
  4e13 FLOPs for the oracle) are compared on 16 sequences: the four most
  expensive by allowed pairs, the shortest, and eleven drawn at random.

Every output element of the whole batch must also be finite."""
import gc

import numpy as np
import pytest
import torch

from jagged_attention_recsys_gdpa_gb300 import flops, inputs
from tests import gpu_helpers as G

pytestmark = pytest.mark.gpu

WHOLE = ["tiny", "jfa", "gdpa_cross", "gdpa_pma"]
SAMPLED = ["jfa_causal", "jfa_block", "gdpa_pma_poly", "mixed"]
MAX_ROWS = 200_000  # query + key rows per oracle group


def _groups(x, seqs):
    """Consecutive groups of the given sequences with at most MAX_ROWS rows each
    (a longer sequence forms a group of its own)."""
    rows = x["lq"][seqs] + x["lkv"][seqs]
    out, cur, n = [], [], 0
    for b, r in zip(seqs, rows):
        if cur and n + r > MAX_ROWS:
            out.append(cur)
            cur, n = [], 0
        cur.append(int(b))
        n += int(r)
    if cur:
        out.append(cur)
    return out


def _sampled(x, w):
    pairs = flops.pairs_per_sequence(x["lq"], x["lkv"], w.mask, w.window)
    top = [int(b) for b in np.argsort(-pairs, kind="stable")[:4]]
    chosen = set(top) | {int(np.argmin(x["lq"]))}
    rng = np.random.default_rng(1)
    for b in rng.permutation(len(x["lq"])):
        if len(chosen) >= 16:
            break
        chosen.add(int(b))
    return sorted(chosen)


def _check(name, seqs):
    w = inputs.WORKLOADS[name]
    x = inputs.make(name, seed=0, device="cuda")
    if w.mask & 4:
        # BlockAttention (blocks dividing the tile, self-attention): the backward
        # takes its statistics from the tile, so GPU forward -> GPU backward is
        # compared with the exact gradient like every other workload
        assert x["kv_off"] is x["q_off"] and 128 % w.window == 0
    g = G.gpu_run(x, w)
    for key in ("o", "dq", "dk", "dv"):
        assert torch.isfinite(g[key]).all(), key
    if w.act == 0:
        assert not torch.isnan(g["lse"]).any()
    for grp in _groups(x, seqs):
        sub, rq, rk = G.subset(x, grp)
        iq = torch.as_tensor(rq, device="cuda")
        ik = torch.as_tensor(rk, device="cuda")
        part = {k: g[k].index_select(0, iq) for k in ("o", "dq")}
        part.update({k: g[k].index_select(0, ik) for k in ("dk", "dv")})
        part["lse"] = g["lse"].index_select(0, iq) if g["lse"] is not None else None
        G.compare(part, G.oracle_run(sub, w), w)
    del x, g
    gc.collect()
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", WHOLE)
def test_fullsize_whole_batch(name):
    lens = inputs.lengths(name, 0)
    _check(name, list(range(len(lens[0]))))


@pytest.mark.parametrize("name", SAMPLED)
def test_fullsize_sampled_sequences(name):
    w = inputs.WORKLOADS[name]
    lq, lkv = inputs.lengths(name, 0)
    x = {"lq": np.asarray(lq), "lkv": np.asarray(lkv)}
    _check(name, _sampled(x, w))
