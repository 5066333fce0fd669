"""Benchmark: jagged attention forward + backward on one GB300 per rank.

One step = one pass of the whole hot path over one batch: device schedule,
forward (O, LSE), and backward (dQ with Di, then dK/dV). The default workload
is the largest self-attention batch: 1024 jagged sequences, 307 long ones
uniform in [4000, 32000] and 717 short ones uniform in [50, 500], H=8, D=128,
softmax, causal + sliding window 512, bf16 (``--workload`` picks another).

Prints one JSON line. value = effective (unpadded, unmasked) TFLOP/s of the
step (forward 4*D*H*pairs + backward 10*D*H*pairs) of the whole global batch
over the slowest rank's time (N > 1: one batch per rank, drawn as one jagged
batch and split over the ranks by allowed pairs). Inputs are already resident in HBM for `value`; `e2e` repeats the
measurement through the public Python API with pinned host buffers and the
host<->device copies inside the timed region. `--impl reference` times the
CPU oracle instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "effective (unpadded) attention TFLOPs fwd/bwd; % of GB300 BF16 tensor peak"
CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


TRAFFIC_TABLE = os.path.join(ROOT, "profiles", "dram_traffic.txt")


def code_hash(path: str) -> str:
    """sha1 (hex) of a C / CUDA source with its comments, trailing blanks and
    empty lines removed, so that a counter row stays attached to a kernel
    whose code has not changed when only its comments have."""
    import hashlib

    with open(path, encoding="utf-8") as fh:
        text = fh.read()
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":  # string or character literal, copied with its escapes
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            while i < n and text[i] != "\n":
                i += 1
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    lines = [ln.rstrip() for ln in "".join(out).split("\n")]
    return hashlib.sha1("\n".join(ln for ln in lines if ln).encode()).hexdigest()


def ncu_traffic(workload: str, kernel: str, algorithmic: float):
    """DRAM bytes (read + write) per launch from the committed ncu table, scaled
    from the captured case to this launch by algorithmic bytes; None when no
    row matches or the kernel's code changed since the capture (prefix of
    code_hash, which ignores comments)."""
    if not os.path.exists(TRAFFIC_TABLE):
        return None
    with open(TRAFFIC_TABLE) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    for r in rows:
        if len(r) < 6 or r[0] != workload or r[1] != kernel:
            continue
        src, sha, dram, alg = r[2], r[3], float(r[4]), float(r[5])
        path = os.path.join(ROOT, "jagged_attention_recsys_gdpa_gb300", "csrc", src)
        if code_hash(path)[:12] != sha:
            return None
        return dram * algorithmic / alg
    return None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    def __init__(self, gpu_index: int):
        self.proc = None
        # raw samples go to JATTN_CLOCKS_DIR (default: the system temp dir); the JSON line carries the summary
        out_dir = os.environ.get("JATTN_CLOCKS_DIR") or tempfile.gettempdir()
        self.path = os.path.join(out_dir, f"clocks_bench_{os.getpid()}.csv")
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax = float(parts[2])
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons), "samples": len(sm)}


def setup_dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist

        dist.init_process_group(backend=os.environ.get("JATTN_BENCH_BACKEND", "nccl"))
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    import torch
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sample_sequences(lq, lkv, pairs, H, D, target_flops, seed=0):
    """Seeded random sequences whose fwd+bwd effective FLOPs reach target_flops."""
    rng = np.random.default_rng(seed)
    order = rng.permutation(len(lq))
    chosen, acc = [], 0.0
    for b in order:
        chosen.append(int(b))
        acc += 14.0 * D * H * float(pairs[b])
        if acc >= target_flops:
            break
    return sorted(chosen), acc


def cpu_oracle_step(x_cpu, w, seqs):
    """One oracle fwd+bwd over the given sequences of a CPU input set; returns seconds."""
    import torch

    import oracle
    from jagged_attention_recsys_gdpa_gb300 import inputs

    qo = x_cpu["q_off"].numpy()
    ko = x_cpu["kv_off"].numpy()
    rq = np.concatenate([np.arange(qo[b], qo[b + 1]) for b in seqs])
    rk = np.concatenate([np.arange(ko[b], ko[b + 1]) for b in seqs])
    lq = np.array([qo[b + 1] - qo[b] for b in seqs])
    lk = np.array([ko[b + 1] - ko[b] for b in seqs])
    sub_qo, sub_ko = inputs.offsets(lq), inputs.offsets(lk)
    tq, tk = torch.from_numpy(rq), torch.from_numpy(rk)
    q, k, v, do = (x_cpu["q"].index_select(0, tq), x_cpu["k"].index_select(0, tk), x_cpu["v"].index_select(0, tk),
                   x_cpu["do"].index_select(0, tq))
    kw = dict(H=w.H, D=w.D, act=w.act, mask=w.mask, window=w.window, norm_by_lkv=w.norm_by_lkv)
    t0 = time.perf_counter()
    oracle.fwd(sub_qo, sub_ko, q, k, v, **kw)
    oracle.bwd(sub_qo, sub_ko, q, k, v, do, **kw)
    return time.perf_counter() - t0


def workload_desc(name, w, batch, of_batch=None):
    """The workload as both arms name it in `config.workload`."""
    act = {0: "softmax", 1: "silu", 2: "gelu", 3: "gelu (degree-6 polynomial)"}[w.act]
    mask = {0: "none", 1: "causal", 3: "causal+window", 4: "block", 5: "causal+block"}[w.mask]
    qk = f", q/k rows normalised to |s| <= {w.qk_norm:g}" if w.qk_norm > 0 else ""
    sub = f" (the {batch} sequences with the most allowed pairs of B={of_batch})" if of_batch else ""
    return (f"{name}: B={batch}, H={w.H}, D={w.D}, {act}, mask={mask}" + (f" {w.window}" if w.mask & 6 else "")
            + qk + sub)


def subset_lengths(lens, w, k):
    """The k sequences with the most allowed pairs (ties: lower index), in batch order."""
    from jagged_attention_recsys_gdpa_gb300 import flops

    lq, lkv = np.asarray(lens[0]), np.asarray(lens[1])
    pairs = flops.pairs_per_sequence(lq, lkv, w.mask, w.window)
    keep = np.sort(np.argsort(-pairs, kind="stable")[:k])
    return lq[keep], lkv[keep]


def run_reference(args, ws, rank):
    """The CPU oracle timed on this host's cores (rank 0 only)."""
    if rank != 0:
        return
    import oracle
    from jagged_attention_recsys_gdpa_gb300 import flops, inputs

    oracle.build()
    w = inputs.WORKLOADS[args.workload]
    # the sample is drawn from the workload's lengths, and only its sequences'
    # inputs are generated (the whole largest batch would take ~50 GB of host
    # memory); the oracle's time depends on the lengths, not on the values
    lq, lkv = inputs.lengths(args.workload, 0)
    pairs = flops.pairs_per_sequence(lq, lkv, w.mask, w.window)
    seqs, eff = sample_sequences(lq, lkv, pairs, w.H, w.D, args.ref_step_flops)
    x = inputs.make(args.workload, seed=0, device="cpu", lens=(lq[seqs], lkv[seqs]))
    local = list(range(len(seqs)))
    for _ in range(args.warmup):
        cpu_oracle_step(x, w, local)
    times = [cpu_oracle_step(x, w, local) for _ in range(args.steps)]
    total = sum(times)
    value = eff * args.steps / total / 1e12
    cores = oracle.num_threads()
    sample = (f"{len(seqs)} of {len(lq)} sequences ({int(pairs[seqs].sum())} allowed pairs per head), "
              f"fwd+bwd in fp64")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded lengths and values)",
        "config": {"workload": workload_desc(args.workload, w, len(lq)), "sample": sample,
                   "device": f"host CPU, {cores} threads (the oracle; rank 0 only)"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="mixed")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true", help="time eager launches instead of a CUDA graph of the step")
    ap.add_argument("--cpu-flops", type=float, default=1.5e11, help="effective FLOPs of the CPU-baseline sample")
    ap.add_argument("--ref-step-flops", type=float, default=2.0e10, help="effective FLOPs per reference step")
    ap.add_argument("--subset", type=int, default=0,
                    help="keep only the K sequences with the most allowed pairs (small cases for ncu captures)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    ws, rank, local = setup_dist()
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return

    import torch

    import jagged_attention_recsys_gdpa_gb300 as J
    from jagged_attention_recsys_gdpa_gb300 import _binding as BND
    from jagged_attention_recsys_gdpa_gb300 import flops, inputs, partition

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    BND.load()
    w = inputs.WORKLOADS[args.workload]
    # Weak scaling by data parallelism: the global batch holds one draw of the
    # workload's lengths per rank (seeds 0 .. N-1), and the split of that one
    # jagged batch by allowed pairs (longest first onto the least-loaded rank)
    # gives every rank about one batch of work; at N = 1 it is the batch itself.
    draws = [inputs.lengths(args.workload, s) for s in range(ws)]
    n_all = len(draws[0][0])
    if args.subset > 0:
        draws = [subset_lengths(d, w, args.subset) for d in draws]
    g_lq = np.concatenate([d[0] for d in draws])
    g_lkv = np.concatenate([d[1] for d in draws])
    rank_of, rank_pairs = partition.split(inputs.offsets(g_lq), inputs.offsets(g_lkv), ws, w.mask, w.window)
    mine = rank_of == rank
    lens = (g_lq[mine], g_lkv[mine])
    x = inputs.make(args.workload, seed=rank, device=dev, lens=lens)
    causal = bool(w.mask & 1)
    window = w.window if w.mask & 2 else 0
    block = w.window if w.mask & 4 else 0
    kw = dict(act=w.act, causal=causal, window=window, block=block, norm_by_lkv=w.norm_by_lkv)
    pairs_b = flops.pairs_per_sequence(x["lq"], x["lkv"], w.mask, w.window)
    pairs = int(pairs_b.sum())
    f_fwd, f_bwd = flops.effective_flops(pairs, w.H, w.D)
    tq, tk = int(x["lq"].sum()), int(x["lkv"].sum())
    # BlockAttention with blocks that divide the tile on self-attention: the
    # backward takes its statistics from the tile (no O or LSE read)
    in_tile = w.act == 0 and bool(w.mask & 4) and 128 % w.window == 0 and x["kv_off"] is x["q_off"]
    # pooling shapes run on the short-query kernels, cross-attention over short
    # key sequences on the short-key forward; both on the fused backward
    short_q = flops.short_query_path(w.act, w.mask, w.D, x["lq"], x["lkv"])
    short_k = flops.short_key_path(w.act, w.mask, w.D, x["lq"], x["lkv"])
    fused = short_q or short_k
    work = flops.kernel_work(tq, tk, pairs, w.H, w.D, w.act == 0, in_tile=in_tile, fused_bwd=fused)
    o = torch.empty_like(x["q"])
    lse = torch.empty(tq, w.H, dtype=torch.float32, device=dev) if w.act == 0 else None
    dq, dk, dv = torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"])
    stream = torch.cuda.current_stream(dev)

    def step():
        J.forward(x["q"], x["k"], x["v"], x["q_off"], x["kv_off"], out=o, lse=lse, **kw)
        J.backward(x["q"], x["k"], x["v"], o, lse, x["do"], x["q_off"], x["kv_off"], dq=dq, dk=dk, dv=dv, **kw)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = J.device_status(dev)
    if st != 0:
        raise RuntimeError(f"device status after warm-up: {BND.error_string(st)}")

    # Per-kernel durations: events recorded by the library around its three
    # main kernels, on the stream they run on, over eager steps.
    n_ev = min(args.steps, 50)
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(n_ev)]
    for evs in kev:
        for e in evs:
            e.record(stream)  # creates the underlying CUDA events
    torch.cuda.synchronize()
    for i in range(n_ev):
        BND.profile_events(kev[i])
        step()
    torch.cuda.synchronize()
    BND.profile_events(None)
    kt = {
        "fwd": sum(e[0].elapsed_time(e[1]) for e in kev) / n_ev,
        "dkdv": sum(e[2].elapsed_time(e[3]) for e in kev) / n_ev,
        "dq": sum(e[4].elapsed_time(e[5]) for e in kev) / n_ev,
    }

    # The step (15 launches: three tile schedules of four kernels, the forward,
    # dQ with Di, dK/dV; 21 with the fused backward, 27 with the short-key forward too) captured once as a CUDA graph and replayed, so launch
    # gaps between its short kernels disappear; eager launches are used if
    # capture is not possible.
    run = step
    execution = "eager"
    if not args.eager:
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, capture_error_mode="thread_local"):
                step()
            graph.replay()
            torch.cuda.synchronize()
            run = graph.replay
            execution = "cuda_graph"
        except Exception as exc:  # noqa: BLE001 - fall back to eager launches
            execution = f"eager (graph capture failed: {type(exc).__name__})"
            torch.cuda.synchronize()
    for _ in range(2):
        run()
    torch.cuda.synchronize()

    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    time.sleep(0.3)
    barrier(ws)
    torch.cuda.synchronize()
    t_start.record(stream)
    for i in range(args.steps):
        run()
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clocks = sampler.stop()
    ms = t_start.elapsed_time(t_end) / args.steps
    ms_max = max_over_ranks(ms, ws, dev)
    st = J.device_status(dev)
    if st != 0:
        raise RuntimeError(f"device status after timing: {BND.error_string(st)}")
    fwd_ms_all = ms  # whole step
    g_fwd, g_bwd = flops.effective_flops(int(rank_pairs.sum()), w.H, w.D)  # the whole global batch
    value = (g_fwd + g_bwd) / (ms_max * 1e-3) / 1e12
    peaks = load_peaks()

    # roofline of the dominant kernel
    dom = max(kt, key=kt.get)
    wk = work[dom]
    t_s = kt[dom] * 1e-3
    t_hbm = wk["bytes"] / (peaks["hbm_gbs"] * 1e9)
    t_tc = wk["flops"] / (peaks["bf16_tflops"] * 1e12)
    if t_hbm >= t_tc:
        roof = {"bound": "hbm", "achieved": wk["bytes"] / t_s / 1e9, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        roof = {"bound": "tensor", "achieved": wk["flops"] / t_s / 1e12, "peak": peaks["bf16_tflops"],
                "unit": "TFLOP/s"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    roof["traffic"] = ncu_traffic(args.workload, dom, wk["bytes"])
    roof["traffic_unit"] = "bytes per launch (ncu dram read + write)"
    roof["algorithmic"] = wk["bytes"] if roof["bound"] == "hbm" else wk["flops"]
    roof["kernel"] = dom
    if fused:
        roof["kernel_name"] = {"fwd": "pma_fwd_kernel" if short_q else "skv_fwd_kernel",
                               "dkdv": ("pma_bwd_kernel" if short_q else "skv_bwd_kernel")
                               + " (fused dQ, dK, dV)"}.get(dom, dom)
    roof["peak_source"] = peaks["source"] + " (burst)"

    # end to end through the public API: pinned host inputs, copies inside the timed region
    host = {k: x[k].cpu().pin_memory() for k in ("q_off", "kv_off", "q", "k", "v", "do")}
    out_host = {"o": torch.empty(o.shape, dtype=o.dtype).pin_memory(),
                "dq": torch.empty(dq.shape, dtype=dq.dtype).pin_memory(),
                "dk": torch.empty(dk.shape, dtype=dk.dtype).pin_memory(),
                "dv": torch.empty(dv.shape, dtype=dv.dtype).pin_memory()}
    if lse is not None:
        out_host["lse"] = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = sum(t.numel() * t.element_size() for t in out_host.values())
    e2e_steps = max(3, min(args.steps, 20))
    # Every step copies its own inputs in (pinned host -> device) and its results
    # out (device -> pinned host) inside the timed region. Steps are pipelined the
    # way a training loop with a prefetching loader runs: step i+1's inputs travel
    # on a copy stream while step i computes and step i-1's results travel back on
    # a third stream (the link is full duplex); device buffers are double-buffered
    # and every dependency is an event, so no step reads data that is not in yet.
    # The device-resident inputs and outputs of the timed loop serve as the first
    # slot, so the largest workload (~12 GB per tensor) fits twice.
    nbuf = 2
    res_out = {"o": o, "dq": dq, "dk": dk, "dv": dv}
    if lse is not None:
        res_out["lse"] = lse
    dev_in = [{k: x[k] for k in host}] + [
        {k: torch.empty(t.shape, dtype=t.dtype, device=dev) for k, t in host.items()} for _ in range(nbuf - 1)]
    dev_out = [res_out] + [
        {k: torch.empty(t.shape, dtype=t.dtype, device=dev) for k, t in out_host.items()} for _ in range(nbuf - 1)]
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    ev_in = [torch.cuda.Event() for _ in range(nbuf)]    # inputs of the slot have landed
    ev_used = [torch.cuda.Event() for _ in range(nbuf)]  # compute is done with the slot's buffers
    ev_out = [torch.cuda.Event() for _ in range(nbuf)]   # the slot's results are back on the host

    def copy_in(i):
        b = i % nbuf
        with torch.cuda.stream(s_in):
            if i >= nbuf:
                s_in.wait_event(ev_used[b])
            for k, t in host.items():
                dev_in[b][k].copy_(t, non_blocking=True)
            ev_in[b].record(s_in)

    def compute(i):
        b = i % nbuf
        stream.wait_event(ev_in[b])
        if i >= nbuf:
            stream.wait_event(ev_out[b])
        d, r = dev_in[b], dev_out[b]
        J.forward(d["q"], d["k"], d["v"], d["q_off"], d["kv_off"], out=r["o"], lse=r.get("lse"), **kw)
        J.backward(d["q"], d["k"], d["v"], r["o"], r.get("lse"), d["do"], d["q_off"], d["kv_off"], dq=r["dq"],
                   dk=r["dk"], dv=r["dv"], **kw)
        ev_used[b].record(stream)

    def copy_out(i):
        b = i % nbuf
        with torch.cuda.stream(s_out):
            s_out.wait_event(ev_used[b])
            for k, t in out_host.items():
                t.copy_(dev_out[b][k], non_blocking=True)
            ev_out[b].record(s_out)

    def e2e_run(n, start_ev=None):
        if start_ev is not None:
            s_in.wait_event(start_ev)
        copy_in(0)
        for i in range(n):
            if i + 1 < n:
                copy_in(i + 1)
            compute(i)
            copy_out(i)
        stream.wait_event(ev_out[(n - 1) % nbuf])

    e2e_run(3)
    torch.cuda.synchronize()
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    e2e_run(e2e_steps, start_ev=e0)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / e2e_steps, ws, dev)
    e2e_value = (g_fwd + g_bwd) / (e2e_ms * 1e-3) / 1e12

    cpu_base = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle

        oracle.build()
        seqs, eff = sample_sequences(x["lq"], x["lkv"], pairs_b, w.H, w.D, args.cpu_flops)
        # only the sampled sequences' rows come to the host
        qo, ko = x["q_off"].cpu().numpy(), x["kv_off"].cpu().numpy()
        rq = torch.from_numpy(np.concatenate([np.arange(qo[b], qo[b + 1]) for b in seqs])).to(dev)
        rk = torch.from_numpy(np.concatenate([np.arange(ko[b], ko[b + 1]) for b in seqs])).to(dev)
        x_cpu = {"q_off": torch.from_numpy(inputs.offsets(np.array([qo[b + 1] - qo[b] for b in seqs]))),
                 "kv_off": torch.from_numpy(inputs.offsets(np.array([ko[b + 1] - ko[b] for b in seqs])))}
        x_cpu.update({k: x[k].index_select(0, rq).cpu() for k in ("q", "do")})
        x_cpu.update({k: x[k].index_select(0, rk).cpu() for k in ("k", "v")})
        secs = cpu_oracle_step(x_cpu, w, list(range(len(seqs))))
        cpu_base = {
            "value": eff / secs / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{len(seqs)} of {len(x['lq'])} sequences, fwd+bwd in fp64, {secs:.1f} s",
        }

    if rank == 0:
        peak_tf = peaks["bf16_tflops"]
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded lengths and values)",
            "config": {
                "workload": workload_desc(args.workload, w, len(x["lq"]), n_all if args.subset > 0 else None),
                "total_q": tq, "total_kv": tk, "pairs_per_head": pairs,
                "l2": f"inputs larger than L2 ({tq * w.H * w.D * 2 / 1e6:.0f} MB per bf16 tensor)",
                "parallelism": (f"data-parallel x{ws}: one jagged batch of {len(g_lq)} sequences split by allowed "
                                f"pairs (longest first onto the least-loaded rank), no collective" if ws > 1
                                else "one GPU"),
                "execution": execution,
            },
            "fwd_tflops": f_fwd / (kt["fwd"] * 1e-3) / 1e12,
            "bwd_tflops": f_bwd / ((kt["dkdv"] + kt["dq"]) * 1e-3) / 1e12,
            "pct_of_bf16_peak": 100.0 * value / peak_tf,
            "kernel_ms": kt,
            "step_overhead_ms": fwd_ms_all - sum(kt.values()),
            "roofline": roof,
            "cpu_baseline": cpu_base,
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
            # per step: three tile schedules of four kernels each, the forward,
            # dQ (which also computes softmax's Di) and dK/dV; the fused
            # backward adds a fourth schedule, the gate and itself (the general
            # dQ and dK/dV passes still launch and find no work), and so does
            # the short-key forward (the general forward finds no work)
            "gpu_launches": (15 + (6 if fused else 0) + (6 if short_k else 0)) * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
