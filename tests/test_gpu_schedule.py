"""The device-built schedule equals the oracle's tile list bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from jagged_attention_recsys_gdpa_gb300 import inputs

pytestmark = pytest.mark.gpu


def _device_schedule(lq, lkv, mask, window, row_tile, col_tile, transposed, H=2):
    import jagged_attention_recsys_gdpa_gb300 as J

    qo = torch.from_numpy(inputs.offsets(np.asarray(lq))).cuda()
    ko = torch.from_numpy(inputs.offsets(np.asarray(lkv))).cuda()
    t = J.schedule(qo, ko, H, causal=bool(mask & 1), window=window if mask & 2 else 0,
                   block=window if mask & 4 else 0, row_tile=row_tile,
                   col_tile=col_tile, transposed=transposed)
    return t.cpu().numpy()


def _twin(lq, lkv, mask, window, row_tile, col_tile, transposed):
    return oracle.schedule(inputs.offsets(np.asarray(lq)), inputs.offsets(np.asarray(lkv)), mask=mask,
                           window=window, BM=row_tile, BN=col_tile, transposed=transposed, cost_cap=1023)


@pytest.mark.parametrize("name", ["tiny", "jfa", "jfa_causal", "jfa_block", "gdpa_cross", "gdpa_pma", "mixed"])
@pytest.mark.parametrize("row_tile,transposed", [(256, False), (128, False), (128, True)])
def test_schedule_matches_twin_on_workloads(name, row_tile, transposed):
    w = inputs.WORKLOADS[name]
    lq, lkv = inputs.lengths(name, 0)
    mask = w.mask | (1 if w.mask & 2 else 0)
    got = _device_schedule(lq, lkv, mask, w.window, row_tile, 128, transposed, w.H)
    want = _twin(lq, lkv, mask, w.window, row_tile, 128, transposed)
    assert got.shape == want.shape
    assert np.array_equal(got, want)


@pytest.mark.parametrize("mask,window", [(0, 0), (1, 0), (3, 1), (3, 37), (4, 1), (4, 37), (5, 64)])
def test_schedule_random_small(mask, window):
    rng = np.random.default_rng(mask * 100 + window)
    for trial in range(10):
        B = int(rng.integers(1, 40))
        lq = rng.integers(0, 700, size=B)
        lkv = lq.copy() if trial % 2 else rng.integers(0, 700, size=B)
        for row_tile, col_tile, tr in ((128, 128, False), (256, 128, False), (128, 128, True), (128, 16, False)):
            got = _device_schedule(lq, lkv, mask, window, row_tile, col_tile, tr)
            want = _twin(lq, lkv, mask, window, row_tile, col_tile, tr)
            assert np.array_equal(got, want), (trial, row_tile, col_tile, tr)


def test_schedule_cost_cap():
    # one sequence with more than 1023 column tiles of 16 keys: costs saturate at 1023
    lq = [300, 20000, 5]
    got = _device_schedule(lq, lq, 0, 0, 128, 16, False)
    want = _twin(lq, lq, 0, 0, 128, 16, False)
    assert np.array_equal(got, want)
    assert (got[:, 3] - got[:, 2]).max() > 1023
