"""The data-parallel split of a jagged batch (jattn_partition, host code):
bit-exact against the oracle's plain-Python twin, balanced within one
sequence's cost of the mean, and its shards cover every row exactly once."""
import numpy as np
import pytest

import oracle
from jagged_attention_recsys_gdpa_gb300 import _binding as B
from jagged_attention_recsys_gdpa_gb300 import flops, inputs, partition

MASKS = [(0, 0), (1, 0), (3, 5), (3, 64), (4, 7), (5, 16), (4, 1)]


@pytest.mark.parametrize("n_ranks", [1, 2, 3, 8])
@pytest.mark.parametrize("mask,window", MASKS)
def test_split_matches_twin(mask, window, n_ranks):
    rng = np.random.default_rng(100 + 7 * mask + window + n_ranks)
    for trial in range(4):
        nb = int(rng.integers(1, 40))
        lq = rng.integers(0, 300, size=nb)
        lkv = lq.copy() if trial % 2 == 0 else rng.integers(0, 300, size=nb)
        lq[rng.random(nb) < 0.1] = 0  # empty sequences cost nothing
        lkv[rng.random(nb) < 0.1] = 0
        qo, ko = inputs.offsets(lq), inputs.offsets(lkv)
        rank_of, loads = partition.split(qo, ko, n_ranks, mask, window)
        t_rank, t_loads = oracle.partition(qo, ko, n_ranks, mask, window)
        assert rank_of.tolist() == t_rank, (nb, trial)
        assert loads.tolist() == t_loads


@pytest.mark.parametrize("name", ["jfa", "gdpa_cross", "gdpa_pma", "mixed", "jfa_block"])
@pytest.mark.parametrize("n_ranks", [2, 4, 8])
def test_split_balance_on_the_workloads(name, n_ranks):
    w = inputs.WORKLOADS[name]
    lq, lkv = inputs.lengths(name, 0)
    qo, ko = inputs.offsets(lq), inputs.offsets(lkv)
    rank_of, loads = partition.split(qo, ko, n_ranks, w.mask, w.window)
    cost = flops.pairs_per_sequence(lq, lkv, w.mask, w.window)
    assert loads.sum() == cost.sum()
    for r in range(n_ranks):
        assert loads[r] == cost[rank_of == r].sum()
    # longest-first greedy: the least loaded rank took every sequence placed
    # after the heaviest rank's last one, so max - min <= the largest cost
    assert loads.max() - loads.min() <= cost.max()
    assert loads.max() <= cost.sum() / n_ranks + cost.max()


def test_shards_cover_every_row_once():
    lq, lkv = inputs.lengths("gdpa_cross", 0)
    qo, ko = inputs.offsets(lq), inputs.offsets(lkv)
    rank_of, _ = partition.split(qo, ko, 3)
    seen_q = np.zeros(qo[-1], dtype=np.int64)
    seen_k = np.zeros(ko[-1], dtype=np.int64)
    for r in range(3):
        s = partition.shard(qo, ko, rank_of, r)
        assert np.all(np.diff(s.seqs) > 0)
        assert s.q_off[-1] == len(s.q_rows) and s.kv_off[-1] == len(s.kv_rows)
        for i, b in enumerate(s.seqs):  # local sequence i is global sequence b, row for row
            assert np.array_equal(s.q_rows[s.q_off[i]:s.q_off[i + 1]], np.arange(qo[b], qo[b + 1]))
            assert np.array_equal(s.kv_rows[s.kv_off[i]:s.kv_off[i + 1]], np.arange(ko[b], ko[b + 1]))
        seen_q[s.q_rows] += 1
        seen_k[s.kv_rows] += 1
    assert np.all(seen_q == 1) and np.all(seen_k == 1)


def test_split_rejects_bad_arguments():
    lib = B.load()
    qo = np.array([0, 3, 5], dtype=np.int64)
    out = np.zeros(2, dtype=np.int32)
    loads = np.zeros(4, dtype=np.int64)

    def call(q=qo, k=qo, mask=0, window=0, n=2, B_=2):
        return lib.jattn_partition(B_, q.ctypes.data, k.ctypes.data, mask, window, n, out.ctypes.data,
                                   loads.ctypes.data)

    assert call() == 0
    assert call(n=0) == 1
    assert call(B_=0) == 1
    assert call(mask=2, window=4) == 1          # window without causal
    assert call(mask=3, window=0) == 1          # window needs a width
    assert call(q=np.array([1, 3, 5], dtype=np.int64)) == 1   # first offset not 0
    assert call(k=np.array([0, 5, 3], dtype=np.int64)) == 1   # decreasing
    assert lib.jattn_partition(2, None, qo.ctypes.data, 0, 0, 2, out.ctypes.data, loads.ctypes.data) == 1
