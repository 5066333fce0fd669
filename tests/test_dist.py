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


def _split_worker(rank, world, port, out):
    """One rank of a data-parallel split: its shard of one jagged batch, the
    oracle on it (CPU stands in for the GPU), outputs gathered to rank 0."""
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import torch.distributed as dist

    import oracle
    from jagged_attention_recsys_gdpa_gb300 import inputs, partition

    dist.init_process_group("gloo")
    w = inputs.Workload("split", 2, 64, 0, 3, 48, False, 1.0, True)
    lq = np.array([3, 200, 17, 0, 90, 64, 129, 5, 300, 1], dtype=np.int64)
    x = inputs.make(w, seed=9, device="cpu", lens=(lq, lq))
    qo, ko = x["q_off"].numpy(), x["kv_off"].numpy()
    rank_of, loads = partition.split(qo, ko, world, w.mask, w.window)
    s = partition.shard(qo, ko, rank_of, rank)
    tq, tk = torch.from_numpy(s.q_rows), torch.from_numpy(s.kv_rows)
    kw = dict(H=w.H, D=w.D, act=w.act, mask=w.mask, window=w.window)
    q, k, v, do = (x["q"].index_select(0, tq), x["k"].index_select(0, tk), x["v"].index_select(0, tk),
                   x["do"].index_select(0, tq))
    o, lse = oracle.fwd(s.q_off, s.kv_off, q, k, v, **kw)
    dq, dk, dv = oracle.bwd(s.q_off, s.kv_off, q, k, v, do, **kw)
    parts = [None] * world
    dist.all_gather_object(parts, (s.q_rows, s.kv_rows, o, lse, dq, dk, dv, int(loads[rank])))
    if rank == 0:
        ref_o, ref_lse = oracle.fwd(qo, ko, x["q"], x["k"], x["v"], **kw)
        ref_dq, ref_dk, ref_dv = oracle.bwd(qo, ko, x["q"], x["k"], x["v"], x["do"], **kw)
        full = {"o": np.full_like(ref_o, np.nan), "lse": np.full_like(ref_lse, np.nan),
                "dq": np.full_like(ref_dq, np.nan), "dk": np.full_like(ref_dk, np.nan),
                "dv": np.full_like(ref_dv, np.nan)}
        for rq, rk, o_, l_, dq_, dk_, dv_, _ in parts:
            full["o"][rq], full["lse"][rq], full["dq"][rq] = o_, l_, dq_
            full["dk"][rk], full["dv"][rk] = dk_, dv_
        ref = {"o": ref_o, "lse": ref_lse, "dq": ref_dq, "dk": ref_dk, "dv": ref_dv}
        out["equal"] = all(np.array_equal(full[n], ref[n]) for n in ref)
        out["loads"] = [p[-1] for p in parts]
        out["pairs"] = oracle.count_pairs(qo, ko, w.mask, w.window)
    dist.destroy_process_group()


def test_two_rank_split_reassembles_the_whole_batch():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_split_worker, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    assert res["equal"]  # every row placed back by the row maps, bit for bit
    assert sum(res["loads"]) == res["pairs"]
    assert max(res["loads"]) - min(res["loads"]) <= 300 * 48  # within the largest sequence's cost
