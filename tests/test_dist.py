"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): the barrier,
the max-over-ranks timing reduction, and weak-scaling inputs (same lengths,
different values per rank). No GPU and no data-path collective."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port), JATTN_BENCH_BACKEND="gloo")
    import bench
    from jagged_attention_recsys_gdpa_gb300 import inputs

    ws, r, local = bench.setup_dist()
    assert (ws, r, local) == (world, rank, rank)
    bench.barrier(ws)
    m = bench.max_over_ranks(1.5 + rank, ws, "cpu")
    lens = inputs.lengths("tiny", 0)
    x = inputs.make("tiny", seed=rank, device="cpu", lens=lens)
    out[rank] = (m, int(x["q"].float().abs().sum().item() * 1000), tuple(x["lq"].tolist()))
    import torch.distributed as dist

    dist.destroy_process_group()


def test_two_rank_reduction_and_weak_scaling_inputs():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.5  # max over ranks
    assert res[0][2] == res[1][2]        # same lengths: per-rank work is fixed
    assert res[0][1] != res[1][1]        # values differ per rank
