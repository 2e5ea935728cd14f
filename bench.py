"""Benchmark: MoE dispatch + combine on one GB300 (or N replicas).

One step = the whole hot path on one batch: dispatch layout + FP8 dispatch
(one ep_dispatch call: layout kernel, then the fused cast/scatter kernel) and
the BF16 weighted combine (ep_combine), on the low-latency workload
R=32 virtual ranks x 128 tokens, H=7168, E=256 experts, top-8, padded
per-expert buffers.  Inputs are resident in HBM; L2 is flushed between steps
(a write of twice its size, then a read of twice its size, so no dirty line of
the flush is written back inside a timed step), outside the timed events.

Prints one JSON line.  ``--impl reference`` times the CPU oracle instead.
Multi-GPU (torchrun): every rank runs its own replica of the workload; the
time is the max over ranks and the value is all ranks' tokens over it.
"""
from __future__ import annotations

import argparse
import hashlib
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

METRIC = "dispatch+combine µs/call, tokens/s and % HBM roofline (h7168 top-8 FP8, 1×GB300)"
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "roofline_traffic.txt")
COMBINE_SRC = os.path.join(ROOT, "combine_get_dispatch_02_gb300", "csrc", "combine.cu")
DISPATCH_SRC = os.path.join(ROOT, "combine_get_dispatch_02_gb300", "csrc", "dispatch.cu")
EXPERT_SRC = os.path.join(ROOT, "combine_get_dispatch_02_gb300", "csrc", "expert.cu")


def _args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="ll")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--breakdown-reps", type=int, default=200)
    ap.add_argument("--layout", choices=["padded", "packed"], default=None,
                    help="override the workload's receive layout (packed keeps a profiled run small)")
    ap.add_argument("--rank", action="store_true",
                    help="rank-deduplicated transport (each token sent once per destination rank)")
    ap.add_argument("--sweep", action="store_true",
                    help="time the sweep grid (one JSON line per point) instead of the bench step")
    ap.add_argument("--sweep-filter", default="", help="only sweep points whose name contains this")
    ap.add_argument("--sweep-reps", type=int, default=10)
    ap.add_argument("--dtype", choices=["fp8", "bf16"], default=None,
                    help="override the workload's dispatch payload")
    ap.add_argument("--hidden", type=int, default=None,
                    help="override the workload's hidden size (a profiled run of the layout stays small)")
    ap.add_argument("--backward-reps", type=int, default=20,
                    help="reps of the backward pair (BF16 expert-major workloads; 0: skip)")
    ap.add_argument("--autotune", action="store_true",
                    help="time the launch-shape candidates on the workload first (ep_autotune) and use the best")
    ap.add_argument("--split-reps", type=int, default=50,
                    help="reps of each split (send / receive-hook) call (0: skip)")
    ap.add_argument("--round-trip-reps", type=int, default=50,
                    help="reps per chunk size of the dispatch -> identity expert -> combine round trip (0: skip)")
    ap.add_argument("--wire-reps", type=int, default=10,
                    help="with --rank: reps of the rank transport's wire calls (device and host wire; 0: skip)")
    ap.add_argument("--kernels", action="store_true",
                    help="time the dispatch kernels (the rule's, row, warp-item, token) on the workload, "
                         "cached layout and behind the layout kernel, instead of the bench step")
    ap.add_argument("--ceilings", action="store_true",
                    help="time plain torch write-only, read-only and copy kernels over 8 GB (the HBM ceilings "
                         "of each traffic mix) instead of the bench step")
    return ap.parse_args()


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _sha(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def _peaks(path=None):
    """(HBM copy bandwidth in GB/s, "measured" | "fallback").  The measured
    file may hold the number directly or in an object (its burst figure:
    these kernels are timed alone or inside sub-millisecond steps)."""
    p = path or os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            for k in ("hbm_gbs", "hbm_GBps", "hbm"):
                v = d.get(k)
                if isinstance(v, dict):
                    v = next((v[j] for j in ("burst", "value", "gbs") if j in v), None)
                if v is not None and float(v) > 0:
                    return float(v), "measured"
        except (OSError, ValueError, TypeError, AttributeError):
            pass
    return FALLBACK_HBM_GBS, "fallback"


def _traffic(kernel: str, src: str, workload: str):
    """ncu DRAM bytes per launch recorded for this kernel source and workload,
    or None when none was recorded for the current source."""
    if not os.path.exists(TRAFFIC_FILE):
        return None
    h = _sha(src)
    for line in open(TRAFFIC_FILE):
        parts = line.split("#", 1)[0].split()
        if len(parts) == 4 and parts[0] == kernel and parts[1] == workload and parts[2] == h:
            return int(parts[3])
    return None


class Clocks:
    """nvidia-smi sampler running during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.out, stderr=subprocess.DEVNULL)
        except FileNotFoundError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        self.out.seek(0)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.out.read().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        os.unlink(self.out.name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ------------------------------------------------------------------ CPU oracle

def _oracle_sample_step(w, topk_idx, topk_weights, x_rows, ye, tokens):
    """One oracle step on a token sample: the full layout, then FP8 dispatch
    and combine of the sampled tokens (x_rows, ye: their rows)."""
    import oracle
    o = oracle.layout(topk_idx, w.num_experts, w.max_tokens_per_rank, oracle.LAYOUT_PADDED)
    sl = o["slot"][tokens]
    # dispatch rows of the sample into a compact buffer (row j*K + k)
    compact = np.arange(len(tokens) * w.topk, dtype=np.int32).reshape(len(tokens), w.topk)
    compact = np.where(sl >= 0, compact, -1).astype(np.int32)
    oracle.dispatch(x_rows, compact, len(tokens) * w.topk, True)
    oracle.combine(ye.reshape(-1, w.hidden), compact, topk_weights.reshape(w.num_tokens, -1)[tokens])


def _oracle_timed(w, topk_idx, topk_weights, x_rows, ye, tokens, seconds):
    """Oracle steps on one token sample for about `seconds`: (tokens done, s)."""
    n, t0 = 0, time.perf_counter()
    while True:
        _oracle_sample_step(w, topk_idx, topk_weights, x_rows, ye, tokens)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return n * len(tokens), el


def _oracle_worker(job):
    """Process-pool entry (spawned): one core's share of the CPU baseline."""
    return _oracle_timed(*job)


def cpu_baseline(w, seconds: float, sample_tokens: int):
    """The C oracle as it stands on the host's cores: one process per core,
    each timing full steps (layout + FP8 dispatch + combine) on its own token
    sample; and the same on one core."""
    import multiprocessing
    import oracle
    oracle.build()
    from combine_get_dispatch_02_gb300 import workloads as wl
    d = wl.generate(w)
    x2 = d["x_bits"].reshape(w.num_tokens, w.hidden)
    wts = d["topk_weights"].reshape(w.num_tokens, -1)
    ns = min(sample_tokens, w.num_tokens)

    def job(i):
        tokens = (np.arange(ns) + i * ns) % w.num_tokens
        return (w, d["topk_idx"], wts, np.ascontiguousarray(x2[tokens]), wl.expert_outputs(w, tokens), tokens,
                seconds)

    done1, el1 = _oracle_timed(*job(0))
    one = done1 / el1
    cores = os.cpu_count() or 1
    value, used = one, 1
    if cores > 1:
        # spawned, not forked (this process has already used CUDA); an
        # executor, not a Pool, so that a worker that dies raises instead of
        # being replaced for ever; bounded in time
        from concurrent.futures import ProcessPoolExecutor
        ex = ProcessPoolExecutor(max_workers=cores, mp_context=multiprocessing.get_context("spawn"))
        try:
            res = list(ex.map(_oracle_worker, [job(i) for i in range(cores)], timeout=4 * seconds + 120))
            value, used = sum(r[0] for r in res) / max(r[1] for r in res), cores
        except Exception as exc:  # report the one-core number and why
            for proc in list(getattr(ex, "_processes", {}).values()):
                proc.terminate()
            ex.shutdown(wait=False, cancel_futures=True)
            return {"value": one, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                    "sample": f"{ns} of the {w.num_tokens} tokens per step, full layout each step, one core "
                              f"(the all-cores run failed: {type(exc).__name__})"}
        ex.shutdown(wait=True)
    return {"value": value, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": f"each process: steps on {ns} of the {w.num_tokens} tokens (full layout each step, FP8 "
                      f"dispatch + combine of the sample) for ~{seconds:.0f} s; {used} processes, one per core",
            "one_core": {"value": one, "cores": 1}}


def run_reference(args):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    from combine_get_dispatch_02_gb300 import workloads as wl
    w = wl.WORKLOADS[args.workload]
    d = wl.generate(w)
    # bounded sample per step so that warmup + steps finish in about two minutes
    import oracle
    oracle.build()
    x2 = d["x_bits"].reshape(w.num_tokens, w.hidden)
    wts = d["topk_weights"].reshape(w.num_tokens, -1)
    probe_tokens = np.arange(16)
    ye16 = wl.expert_outputs(w, probe_tokens)
    t0 = time.perf_counter()
    _oracle_sample_step(w, d["topk_idx"], wts, x2[probe_tokens], ye16, probe_tokens)
    per_token = max((time.perf_counter() - t0) / 16, 1e-6)
    budget = 120.0 / max(args.steps + args.warmup, 1)
    ntok = int(max(1, min(w.num_tokens, budget / per_token)))
    tokens = np.arange(ntok)
    ye = wl.expert_outputs(w, tokens)
    x_rows = np.ascontiguousarray(x2[tokens])
    for _ in range(args.warmup):
        _oracle_sample_step(w, d["topk_idx"], wts, x_rows, ye, tokens)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_sample_step(w, d["topk_idx"], wts, x_rows, ye, tokens)
    el = time.perf_counter() - t0
    value = args.steps * ntok / el
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": _workload_desc(w), "sample_tokens_per_step": ntok},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": 1, "kind": "oracle",
                         "sample": f"each step: full layout + FP8 dispatch and combine of {ntok} "
                                   f"of {w.num_tokens} tokens, single-threaded C oracle"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _workload_desc(w):
    return (f"{w.name}: R={w.num_ranks} virtual ranks x {w.tokens_per_rank} tokens, H={w.hidden}, "
            f"E={w.num_experts}, top-{w.topk}, {'FP8 e4m3 (per-128 fp32 scales)' if w.use_fp8 else 'BF16'} "
            f"dispatch into {w.layout} receive buffers, BF16 combine")


# ------------------------------------------------------------------ GPU

def replica_throughput(total_ms: float, steps: int, tokens_per_replica: int, world_size: int,
                       device="cpu"):
    """Whole-job throughput of ``world_size`` independent replicas: the
    slowest rank's time decides (max over ranks), every rank's tokens count.
    Returns (ms per step, tokens/s)."""
    if world_size > 1:
        import torch
        import torch.distributed as dist
        t = torch.tensor([total_ms], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    ms_per_step = total_ms / steps
    return ms_per_step, world_size * tokens_per_replica / (ms_per_step / 1e3)


def _algorithmic_bytes(w, M):
    N, K, H = w.num_tokens, w.topk, w.hidden
    pay = 1 if w.use_fp8 else 2
    disp = N * H * 2 + N * K * 8 + M * H * pay + (M * (H // 128) * 4 if w.use_fp8 else 0) \
        + N * K * 4 + M * 4 + w.num_experts * w.num_ranks * 4
    disp_kernel = N * H * 2 + M * H * pay + (M * (H // 128) * 4 if w.use_fp8 else 0) + N * K * 4
    comb = M * H * 2 + N * K * 4 + N * K * 4 + N * H * 2
    return disp, disp_kernel, comb


def _identity_bytes(w, M):
    """Identity expert: read each received row (and its FP8 scales) and the
    entries' slots, write the row as bf16."""
    N, K, H = w.num_tokens, w.topk, w.hidden
    if w.use_fp8:
        return M * (H + (H // 128) * 4) + M * H * 2 + N * K * 4
    return M * H * 2 * 2 + N * K * 4


def run_ours(args):
    import torch
    ws, rank, local = _dist()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    else:
        torch.cuda.set_device(0)
    dev = torch.cuda.current_device()
    from combine_get_dispatch_02_gb300 import Buffer, ep
    from combine_get_dispatch_02_gb300 import build as epbuild
    from combine_get_dispatch_02_gb300 import workloads as wl
    epbuild.build()
    w = wl.WORKLOADS[args.workload]
    if args.layout is not None:
        w = w.with_(layout=args.layout)
    if args.dtype is not None:
        w = w.with_(use_fp8=(args.dtype == "fp8"))
    if args.hidden is not None:
        w = w.with_(hidden=args.hidden)
    d = wl.generate(w)
    N, K, H = w.num_tokens, w.topk, w.hidden

    buf = Buffer(w.num_ranks, w.max_tokens_per_rank, H, w.num_experts, K,
                 low_latency_mode=(w.layout == wl.PADDED))
    to_dev = lambda a: torch.from_numpy(a).cuda()
    x = to_dev(np.ascontiguousarray(d["x_bits"]).view(np.int16)).view(torch.bfloat16)
    idx = to_dev(d["topk_idx"])
    wts = to_dev(d["topk_weights"].reshape(N, K))
    recv, scales = buf.alloc_rank_recv(w.use_fp8) if args.rank else buf.alloc_recv(w.use_fp8)
    cnt = torch.empty(w.num_experts, dtype=torch.int32, device="cuda")
    out = torch.empty(N, H, dtype=torch.bfloat16, device="cuda")
    h = buf.new_handle()
    ctx = buf.ctx
    stream = torch.cuda.current_stream()

    def enqueue(xb, idxb, wb, outb, s, split=False):
        """One step: layout + dispatch, then combine (on stream s).  With
        split=True an event between the dispatch and the combine is returned;
        it costs the step ~4 µs, because the combine then cannot launch early
        behind the dispatch (programmatic dependent launch), so the timed
        steps go without it and a second pass takes the split."""
        if args.rank:
            ep.ep_get_rank_layout(ctx, idxb, wb, w.tokens_per_rank, None, None, None, h.raw, s)
            ep.ep_dispatch(ctx, xb, None, w.tokens_per_rank, w.use_fp8, h.raw, recv, scales, cnt, s)
        else:
            ep.ep_dispatch(ctx, xb, idxb, w.tokens_per_rank, w.use_fp8, h.raw, recv, scales, cnt, s)
        ev = None
        if split:
            ev = torch.cuda.Event(enable_timing=True)
            ev.record(s)
        ep.ep_combine(ctx, y, None if args.rank else wb, h.raw, outb, s)
        return ev

    # expert outputs (combine input) at the rows the layout assigns
    if args.rank:
        ep.ep_get_rank_layout(ctx, idx, wts, w.tokens_per_rank, None, None, None, h.raw)
    else:
        ep.ep_get_dispatch_layout(ctx, idx, w.tokens_per_rank, None, None, None, h.raw)
    slot = h.tensors()["slot"].view(-1).long()
    valid = slot >= 0
    M = int(valid.sum().item())
    y = torch.zeros(buf.rank_rows if args.rank else buf.rows, H, dtype=torch.bfloat16, device="cuda")
    ye = wl.expert_outputs(w)
    y[slot[valid]] = to_dev(ye.reshape(-1, H).view(np.int16)).view(torch.bfloat16)[valid]
    del ye

    # L2 flush between steps: write 2x L2, then read another 2x L2 so that the
    # flush's own dirty lines are written back before the timed region starts
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    nflush = max(2 * l2, 256 << 20)
    flush_w = torch.empty(nflush, dtype=torch.uint8, device="cuda")
    flush_r = torch.ones(nflush // 4, dtype=torch.float32, device="cuda")
    flush_sink = torch.empty(1, dtype=torch.float32, device="cuda")

    def flush_l2():
        flush_w.fill_(1)
        torch.sum(flush_r, dim=0, keepdim=True, out=flush_sink)

    tuning = None
    if args.autotune and args.rank:
        raise SystemExit("--autotune times the expert-major layout; run it without --rank")
    if args.autotune:
        # the bench's BF16 round trip writes the expert output in place
        y_tune = recv if not w.use_fp8 else torch.empty(buf.rows, H, dtype=torch.bfloat16, device="cuda")
        t = ep.ep_autotune(ctx, x, idx, w.tokens_per_rank, wts, w.use_fp8, recv, scales, y_tune, out, reps=20)
        tuning = t.as_dict()
        tuning["candidates_us"] = [f"{k}={v}: {us:.1f}" for k, v, us in ep.ep_get_autotune_log(ctx)]
        del y_tune
        torch.cuda.empty_cache()

    def step(split=False):
        return enqueue(x, idx, wts, out, stream, split)

    for _ in range(args.warmup):
        flush_l2()
        step()
    torch.cuda.synchronize()
    if buf.device_status() != ep.EP_OK:
        raise RuntimeError("device status error during warmup")

    clocks = Clocks(dev)
    clocks.start()
    time.sleep(0.3)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    # the timed region: K steps, events at the step boundaries only.  The GPU
    # first sleeps ~50 ms (outside the events) so that the host queues the
    # steps well ahead of it: a host-side stall cannot then leave the GPU
    # idle inside a timed step.
    torch.cuda._sleep(100_000_000)
    evs = []
    for _ in range(args.steps):
        flush_l2()
        e0 = torch.cuda.Event(enable_timing=True)
        e2 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e2.record(stream)
        evs.append((e0, e2))
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    time.sleep(0.2)
    clk = clocks.stop()
    step_ms = [a.elapsed_time(b) for a, b in evs]
    ms_per_step, value = replica_throughput(sum(step_ms), args.steps, N, ws, device="cuda")
    # the same K steps again with an event between the dispatch and the
    # combine: each kernel's share of a step (for the rooflines)
    torch.cuda._sleep(100_000_000)
    evs = []
    for _ in range(args.steps):
        flush_l2()
        e0 = torch.cuda.Event(enable_timing=True)
        e2 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        e1 = step(split=True)
        e2.record(stream)
        evs.append((e0, e1, e2))
    torch.cuda.synchronize()
    disp_ms = [a.elapsed_time(b) for a, b, _ in evs]
    comb_ms = [b.elapsed_time(c) for _, b, c in evs]
    split_step_ms = [a.elapsed_time(c) for a, _, c in evs]

    # breakdown: each kernel alone (layout alone, dispatch with the cached
    # layout, combine), same L2 flush between launches
    def timed(fn, reps=args.breakdown_reps):
        if reps <= 0:
            return float("nan"), float("nan")
        ts = []
        for _ in range(reps):
            flush_l2()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            ts.append((a, b))
        torch.cuda.synchronize()
        v = [a.elapsed_time(b) * 1e3 for a, b in ts]
        return statistics.median(v), statistics.mean(v)

    lay_us = timed(lambda: ep.ep_get_rank_layout(ctx, idx, wts, w.tokens_per_rank, None, None, None, h.raw, stream)
                   if args.rank else
                   ep.ep_get_dispatch_layout(ctx, idx, w.tokens_per_rank, None, None, None, h.raw, stream))
    disp_us = timed(lambda: ep.ep_dispatch(ctx, x, None, w.tokens_per_rank, w.use_fp8, h.raw, recv, scales,
                                           None, stream))
    comb_us = timed(lambda: ep.ep_combine(ctx, y, None if args.rank else wts, h.raw, out, stream))

    # the same step captured once in a CUDA graph and replayed (no host
    # launch overhead; programmatic dependent launch becomes a graph edge)
    graph_us = None
    try:
        s_cap = torch.cuda.Stream()
        s_cap.wait_stream(stream)
        with torch.cuda.stream(s_cap):
            for _ in range(2):
                enqueue(x, idx, wts, out, s_cap)
        stream.wait_stream(s_cap)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s_cap):
            enqueue(x, idx, wts, out, s_cap)
        graph_us = timed(graph.replay)
    except Exception as exc:  # report, do not hide, a capture failure
        graph_us = (f"capture failed: {exc}", None)

    # the backward pair on the cached layout: grad of combine = BF16 dispatch
    # of the output gradient, grad of dispatch = unweighted combine of the
    # received-row gradients
    backward = None
    if args.backward_reps > 0 and not args.rank and not w.use_fp8:
        gx = torch.empty(N, H, dtype=torch.bfloat16, device="cuda")
        bd = timed(lambda: ep.ep_dispatch(ctx, out, None, w.tokens_per_rank, False, h.raw, recv, None, None,
                                          stream), args.backward_reps)
        bc = timed(lambda: ep.ep_combine(ctx, y, None, h.raw, gx, stream), args.backward_reps)
        backward = {"grad_combine_dispatch_median_us": bd[0], "grad_dispatch_combine_median_us": bc[0],
                    "tokens_per_s": N / ((bd[0] + bc[0]) / 1e6)}
        del gx

    # the round trip with the identity expert between dispatch and combine,
    # pipelined over token chunks (layout included), and the identity
    # expert alone
    round_trip = None
    if args.round_trip_reps > 0 and not args.rank:
        y_rt = recv if not w.use_fp8 else torch.empty(buf.rows, H, dtype=torch.bfloat16, device="cuda")
        # BF16: the expert output is the receive buffer itself (nothing to time)
        ident_us = (timed(lambda: ep.ep_expert_identity(ctx, h.raw, True, recv, scales, y_rt, 0, N, stream))
                    if w.use_fp8 else (float("nan"), float("nan")))
        auto = ep.ep_round_trip_auto_chunk(ctx, w.use_fp8)
        chunks = [0, ep.EP_CHUNK_AUTO] + sorted({c for c in (N // 16, N // 8, N // 4, N // 2) if c > 0} - {auto})
        per_chunk = {}
        for c in chunks:
            per_chunk[str(c)] = timed(lambda: ep.ep_round_trip(ctx, x, idx, w.tokens_per_rank, wts, w.use_fp8,
                                                               h.raw, recv, scales, y_rt, out, c, stream),
                                      reps=args.round_trip_reps)[0]
        best = min(chunks, key=lambda c: per_chunk[str(c)])
        ident_bytes = _identity_bytes(w, M)
        ident_gbs = ident_bytes / (ident_us[0] / 1e6) / 1e9 if ident_us[0] == ident_us[0] else None
        if ident_gbs is None:
            ident_us, ident_bytes = (None, None), None
        round_trip = {
            "chunk_tokens_us_median": per_chunk, "best_chunk_tokens": best,
            "tokens_per_s_best": N / (per_chunk[str(best)] / 1e6),
            "identity_expert_alone_median_us": ident_us[0],
            "identity_expert_roofline": {"bound": "hbm", "achieved": ident_gbs, "algorithmic_bytes": ident_bytes,
                                         "frac": ident_gbs / _peaks()[0] if ident_gbs else None,
                                         "traffic": _traffic("identity", EXPERT_SRC, w.name) if ident_gbs else None},
            "auto_chunk_tokens": auto,
            "note": "chunk 0 = one chunk, -1 = automatic (L2-sized); layout computed in every call",
        }
        del y_rt

    # split dispatch / combine: the send halves and the receive hooks (copy
    # engine) on several SM budgets
    split = None
    if args.split_reps > 0 and not args.rank and (not w.use_fp8 or H % 512 == 0):
        reps = args.split_reps
        fp8 = w.use_fp8
        if fp8:
            send_x = torch.empty(N, H, dtype=torch.float8_e4m3fn, device="cuda")
            send_sc = torch.empty(N, H // 128, dtype=torch.float32, device="cuda")
        else:
            send_x, send_sc = x, None
        send_y = torch.empty(N * K, H, dtype=torch.bfloat16, device="cuda")
        T = w.tokens_per_rank
        send_us = timed(lambda: ep.ep_dispatch_send(ctx, x, idx, T, fp8, h.raw, send_x, send_sc, stream), reps)
        row_b = H * (1 if fp8 else 2) + (H // 32 if fp8 else 0)
        recv_bytes = N * row_b + M * row_b + N * K * 4
        csend_bytes = 2 * M * H * 2 + N * K * 4
        budgets = [b for b in (8, 16, 32, 76) if b < torch.cuda.get_device_properties(dev).multi_processor_count] + [0]
        recv_us, csend_us = {}, {}
        for b in budgets:
            recv_us[str(b)] = timed(lambda: ep.ep_dispatch_recv(ctx, h.raw, fp8, send_x, send_sc, recv, scales, None,
                                                                b, stream), reps)[0]
            csend_us[str(b)] = timed(lambda: ep.ep_combine_send(ctx, h.raw, y, send_y, b, stream), reps)[0]
        crecv_us = timed(lambda: ep.ep_combine_recv(ctx, h.raw, send_y, wts, out, stream), reps)
        gbs = lambda nbytes, us: nbytes / us / 1e3

        # overlap: the receive hook on 32 SMs (second stream) beside a bf16
        # GEMM that stands in for the expert computation (this stream)
        overlap = None
        if torch.cuda.get_device_properties(dev).multi_processor_count > 32:
            ga = torch.randn(4096, 4096, device="cuda").to(torch.bfloat16)
            gb = torch.randn(4096, 4096, device="cuda").to(torch.bfloat16)
            gc = torch.empty(4096, 4096, dtype=torch.bfloat16, device="cuda")
            s2 = torch.cuda.Stream()

            def gemm():
                torch.matmul(ga, gb, out=gc)

            def hook(s):
                ep.ep_dispatch_recv(ctx, h.raw, fp8, send_x, send_sc, recv, scales, None, 32, s)

            def both():
                start = torch.cuda.Event()
                start.record(stream)
                s2.wait_stream(stream)
                hook(s2)
                gemm()
                stream.wait_stream(s2)

            t_gemm = timed(gemm, reps)[0]
            t_hook = timed(lambda: hook(stream), reps)[0]
            t_both = timed(both, reps)[0]
            overlap = {"gemm_4096_bf16_us": t_gemm, "recv_hook_32_sms_us": t_hook, "both_us": t_both,
                       "hidden_fraction_of_hook": (t_gemm + t_hook - t_both) / t_hook}
            del ga, gb, gc
        split = {
            "dispatch_send_median_us": send_us[0],
            "dispatch_recv_hook_median_us_by_sms": recv_us,
            "dispatch_recv_hook_gbs_by_sms": {k: gbs(recv_bytes, v) for k, v in recv_us.items()},
            "combine_send_median_us_by_sms": csend_us,
            "combine_send_gbs_by_sms": {k: gbs(csend_bytes, v) for k, v in csend_us.items()},
            "combine_recv_hook_median_us": crecv_us[0],
            "overlap_with_gemm": overlap,
            "note": "sms 0 = all SMs; dispatch_send includes the layout; the hooks' copy kernels only issue "
                    "cp.async.bulk copies",
        }
        del send_y

    # the rank transport whose receive runs no kernel: send (layout + send
    # rows + cast), then the runs moved by the device wire (driver copies) or
    # the host wire (copy engines through pinned host memory), and each wire
    # beside GEMMs on another stream
    wire = None
    if args.rank and args.wire_reps > 0 and w.num_ranks <= 32:
        wire = _rank_wire(args, w, buf, ctx, x, idx, wts, h, y, out, stream, timed)

    # HBM copy bandwidth of this GPU through torch (context for the fractions)
    cbuf = torch.empty(2 << 30, dtype=torch.uint8, device="cuda")
    cdst = torch.empty_like(cbuf)
    copy_gbs = 2 * cbuf.numel() / (timed(lambda: cdst.copy_(cbuf), reps=10)[0] / 1e6) / 1e9
    del cbuf, cdst
    torch.cuda.empty_cache()

    # end to end through the public API with host buffers
    e2e = None if args.no_e2e else _e2e(args, w, d, x, idx, wts, out, enqueue, stream)
    if buf.device_status() != ep.EP_OK:
        raise RuntimeError("device status error")

    if rank != 0:
        if ws > 1:
            torch.distributed.destroy_process_group()
        return
    _report(args, w, ws, M, N, step_ms, disp_ms, comb_ms, ms_per_step, value, lay_us, disp_us, comb_us,
            e2e, clk, graph_us, copy_gbs, round_trip, split, tuning, split_step_ms, backward, wire)
    if ws > 1:
        torch.distributed.destroy_process_group()


def _rank_wire(args, w, buf, ctx, x, idx, wts, h, y, out, stream, timed):
    """Timings of the rank transport with a kernel-free receive (see
    ep_rank_dispatch_recv): each call alone, and each wire on a second stream
    beside back-to-back 4096^3 bf16 GEMMs on this stream (as many as take
    about as long as the wire), with the fraction of the wire's time hidden."""
    import torch
    from combine_get_dispatch_02_gb300 import ep
    N, K, H, R = w.num_tokens, w.topk, w.hidden, w.num_ranks
    fp8 = w.use_fp8
    reps = args.wire_reps
    rows = ep.ep_rank_send_rows(buf.cfg)
    if fp8:
        send_x = torch.empty(rows, H, dtype=torch.float8_e4m3fn, device="cuda")
        send_sc = torch.empty(rows, H // 128, dtype=torch.float32, device="cuda")
    else:
        send_x, send_sc = torch.empty(rows, H, dtype=torch.bfloat16, device="cuda"), None
    send_y = torch.empty(rows, H, dtype=torch.bfloat16, device="cuda")
    row_b = H + H // 32 if fp8 else 2 * H
    stage = torch.empty(rows * max(row_b, 2 * H), dtype=torch.uint8).pin_memory()
    recv, scales = buf.alloc_rank_recv(fp8)
    hw = buf.new_handle()
    T = w.tokens_per_rank
    send_us = timed(lambda: ep.ep_rank_dispatch_send(ctx, x, idx, wts, T, fp8, None, None, hw.raw, send_x, send_sc,
                                                     stream), reps)[0]
    runs, _, _ = ep.ep_rank_runs(hw.raw, R)
    moved = sum(map(sum, runs))
    res = {"send_with_layout_median_us": send_us, "rows_moved": moved, "runs": sum(c > 0 for r in runs for c in r)}
    ga = torch.randn(4096, 4096, device="cuda").to(torch.bfloat16)
    gb = torch.randn(4096, 4096, device="cuda").to(torch.bfloat16)
    gc = torch.empty(4096, 4096, dtype=torch.bfloat16, device="cuda")
    s2 = torch.cuda.Stream()
    t_one = timed(lambda: torch.matmul(ga, gb, out=gc), reps)[0]
    for name, wire_id in (("device", ep.EP_WIRE_DEVICE), ("host", ep.EP_WIRE_HOST)):
        st = stage if wire_id == ep.EP_WIRE_HOST else None

        def recv_hook(s, wire_id=wire_id, st=st):
            ep.ep_rank_dispatch_recv(ctx, hw.raw, fp8, send_x, send_sc, recv, scales, None, wire_id, st, s)

        def csend(s, wire_id=wire_id, st=st):
            ep.ep_rank_combine_send(ctx, hw.raw, y_w, send_y, wire_id, st, s)

        # expert outputs in the receive layout: the bf16 receive rows themselves (timing only)
        y_w = recv if not fp8 else torch.zeros(buf.rank_rows, H, dtype=torch.bfloat16, device="cuda")
        t_recv = timed(lambda: recv_hook(stream), reps)[0]
        t_csend = timed(lambda: csend(stream), reps)[0]
        n_gemm = max(1, int(round(t_recv / t_one)))

        def gemms():
            for _ in range(n_gemm):
                torch.matmul(ga, gb, out=gc)

        def both():
            ev = torch.cuda.Event()
            ev.record(stream)
            s2.wait_event(ev)
            gemms()
            recv_hook(s2)
            stream.wait_stream(s2)

        t_g = timed(gemms, reps)[0]
        t_b = timed(both, reps)[0]
        moved_b = moved * row_b
        res[name] = {"dispatch_recv_median_us": t_recv, "dispatch_recv_gbs": moved_b / t_recv / 1e3,
                     "combine_send_median_us": t_csend, "combine_send_gbs": moved * 2 * H / t_csend / 1e3,
                     "beside_gemms": {"gemms": n_gemm, "gemms_us": t_g, "recv_us": t_recv, "both_us": t_b,
                                      "hidden_fraction_of_recv": (t_g + t_recv - t_b) / t_recv}}
        del y_w
    res["combine_recv_median_us"] = timed(lambda: ep.ep_rank_combine_recv(ctx, hw.raw, send_y, out, stream), reps)[0]
    res["note"] = ("receive = one copy per (source rank, destination rank) run issued from the host, no kernel of "
                   "this library; device wire: same-device cudaMemcpyAsync (the driver runs these on SMs); host "
                   "wire: device->pinned host->device on the copy engines (no SM); GB/s count each moved byte once")
    del ga, gb, gc, send_x, send_sc, send_y, stage
    return res


def _e2e(args, w, d, x, idx, wts, out, enqueue, stream):
    """End to end through the public calls with host buffers: every step
    copies its inputs (x, topk_idx, topk_weights) from pinned host memory,
    runs ep_dispatch + ep_combine and copies the combined tokens back.
    Steps are pipelined over three streams (host-to-device copies, compute,
    device-to-host copies) with two sets of device buffers, so one step's
    copies overlap its neighbours' compute; the timed region (wall clock,
    synchronised on both sides) still contains every step's copies.  The
    same loop run serially on one stream is reported beside it."""
    import torch
    N, K, H = w.num_tokens, w.topk, w.hidden
    ws = _dist()[0]
    xh = torch.from_numpy(np.ascontiguousarray(d["x_bits"]).view(np.int16)).view(torch.bfloat16).pin_memory()
    idxh = torch.from_numpy(d["topk_idx"]).pin_memory()
    wh = torch.from_numpy(d["topk_weights"].reshape(N, K)).pin_memory()
    outh = [torch.empty(N, H, dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    xs = [x, torch.empty_like(x)]
    idxs = [idx, torch.empty_like(idx)]
    wss = [wts, torch.empty_like(wts)]
    outs = [out, torch.empty_like(out)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_comp + ev_out:
        e.record(stream)

    def run(steps, pipelined):
        for i in range(steps):
            b = i % 2 if pipelined else 0
            cin = s_in if pipelined else stream
            cout = s_out if pipelined else stream
            cin.wait_event(ev_comp[b])
            with torch.cuda.stream(cin):
                xs[b].copy_(xh, non_blocking=True)
                idxs[b].copy_(idxh, non_blocking=True)
                wss[b].copy_(wh, non_blocking=True)
            ev_in[b].record(cin)
            stream.wait_event(ev_in[b])
            stream.wait_event(ev_out[b])
            enqueue(xs[b], idxs[b], wss[b], outs[b], stream)
            ev_comp[b].record(stream)
            cout.wait_event(ev_comp[b])
            with torch.cuda.stream(cout):
                outh[b].copy_(outs[b], non_blocking=True)
            ev_out[b].record(cout)

    # each mode timed in three segments of e2e_steps steps; the median segment
    # is reported (the host link is shared with the machine's other GPUs, and
    # a single wall-clock segment can catch another job's burst)
    res = {}
    for pipelined in (False, True):
        run(3, pipelined)
        torch.cuda.synchronize()
        seg = []
        for _ in range(3):
            t0 = time.perf_counter()
            run(args.e2e_steps, pipelined)
            torch.cuda.synchronize()
            seg.append((time.perf_counter() - t0) / args.e2e_steps * 1e3)
        res[pipelined] = statistics.median(seg)
    h2d = xh.numel() * 2 + idxh.numel() * 8 + wh.numel() * 4
    d2h = outh[0].numel() * 2

    # the host link alone: the step's H2D and D2H copies, each timed by itself
    def link_gbs(fn, nbytes, reps=10):  # median of three timings of `reps` copies
        fn()
        torch.cuda.synchronize()
        r = []
        for _ in range(3):
            t0 = time.perf_counter()
            for _ in range(reps):
                fn()
            torch.cuda.synchronize()
            r.append(nbytes * reps / (time.perf_counter() - t0) / 1e9)
        return statistics.median(r)

    h2d_gbs = link_gbs(lambda: xs[0].copy_(xh, non_blocking=True), xh.numel() * 2)
    d2h_gbs = link_gbs(lambda: outh[0].copy_(outs[0], non_blocking=True), d2h)

    # both directions at once (the pipelined steps need this): one copy each way
    # per rep, on two streams
    def both():
        with torch.cuda.stream(s_in):
            xs[1].copy_(xh, non_blocking=True)
        with torch.cuda.stream(s_out):
            outh[1].copy_(outs[1], non_blocking=True)
    bidir_gbs = link_gbs(both, xh.numel() * 2 + d2h)
    return {"value": N / (res[True] / 1e3) * ws, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": res[True], "ms_per_step_serial": res[False],
            "pipelining": "H2D / compute / D2H on three streams, two buffer sets",
            "host_link_gbs": {"h2d": h2d_gbs, "d2h": d2h_gbs, "both_directions_at_once": bidir_gbs},
            "host_link_bound_ms_per_step": (h2d + d2h) / bidir_gbs / 1e6}


def _report(args, w, ws, M, N, step_ms, disp_ms, comb_ms, ms_per_step, value, lay_us, disp_us, comb_us,
            e2e, clk, graph_us=None, copy_gbs=None, round_trip=None, split=None, tuning=None,
            split_step_ms=None, backward=None, wire=None):
    peak, peak_kind = _peaks()
    disp_bytes, disp_kernel_bytes, comb_bytes = _algorithmic_bytes(w, M)
    comb_avg_s = statistics.mean(comb_ms) / 1e3
    comb_gbs = comb_bytes / comb_avg_s / 1e9
    traffic = _traffic("combine", COMBINE_SRC, w.name)
    disp_gbs = disp_kernel_bytes / (disp_us[1] / 1e6) / 1e9 if disp_us[1] == disp_us[1] else None
    nan_none = lambda v: None if v != v else v
    lay_us, disp_us, comb_us = [tuple(nan_none(v) for v in t) for t in (lay_us, disp_us, comb_us)]

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "payload": {"dispatch": "e4m3 + f32 scales" if w.use_fp8 else "bf16", "combine": "bf16"},
        "data": "synthetic",
        "config": {"workload": _workload_desc(w) + ("; rank-deduplicated transport" if args.rank else ""),
                   "tokens_per_step": N, "rows_received": M,
                   "launch_shapes": tuning if tuning is not None else "built-in rules",
                   "l2": "flushed between steps (write of 2x L2, then read of 2x L2; outside the timed events)",
                   "parallelism": f"{ws} replica(s), one per GPU" if ws > 1 else "1 GPU, 32 virtual EP ranks"},
        "us_per_call": {
            "step": statistics.mean(step_ms) * 1e3,
            "step_with_split_event": statistics.mean(split_step_ms) * 1e3 if split_step_ms else None,
            "dispatch_with_layout": statistics.mean(disp_ms) * 1e3,
            "combine": statistics.mean(comb_ms) * 1e3,
            "layout_alone_median": lay_us[0],
            "dispatch_cached_layout_median": disp_us[0],
            "combine_alone_median": comb_us[0],
            "step_cuda_graph_replay_median": graph_us[0] if graph_us else None,
        },
        "tokens_per_s": {  # N / t per op (in-step means) and for the step
            "step": value,
            "dispatch_with_layout": ws * N / (statistics.mean(disp_ms) / 1e3),
            "combine": ws * N / (statistics.mean(comb_ms) / 1e3),
            "dispatch_cached_layout": N / (disp_us[0] / 1e6) if disp_us[0] else None,
            "step_cuda_graph_replay": N / (graph_us[0] / 1e6) if graph_us and isinstance(graph_us[0], float) else None,
        },
        "hbm_copy_gbs_torch_here": copy_gbs,
        "roofline": {"bound": "hbm", "kernel": "combine", "achieved": comb_gbs, "peak": peak,
                     "unit": "GB/s", "frac": comb_gbs / peak, "traffic": traffic,
                     "algorithmic_bytes": comb_bytes, "peak_source": f"{peak_kind} HBM copy bandwidth",
                     "duration": "mean combine time inside a step (event after the dispatch to the step's "
                                 "end, second pass of the K steps; includes the combine's launch)"},
        "roofline_dispatch": {"bound": "hbm", "kernel": "dispatch (cached layout)", "achieved": disp_gbs,
                              "peak": peak, "unit": "GB/s", "frac": disp_gbs / peak if disp_gbs else None,
                              "traffic": _traffic("dispatch", DISPATCH_SRC, w.name),
                              "algorithmic_bytes": disp_kernel_bytes},
        "roofline_step": {"bound": "hbm", "achieved": (disp_bytes + comb_bytes) / (ms_per_step / 1e3) / 1e9,
                          "peak": peak, "unit": "GB/s",
                          "frac": (disp_bytes + comb_bytes) / (ms_per_step / 1e3) / 1e9 / peak,
                          "algorithmic_bytes": disp_bytes + comb_bytes,
                          "note": "the whole step (layout + dispatch + combine) over its mean time: no kernel's "
                                  "writes are still in L2 when it ends"},
        "e2e": e2e,
        "round_trip": round_trip,
        "split": split,
        "rank_wire": wire,
        "backward": backward,
        "gpu_launches": 3 * args.steps,
        "clocks": clk,
        "host_cores": os.cpu_count(),
    }
    if not args.no_cpu_baseline and ws == 1:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds, 128)
    print(json.dumps(line), flush=True)


def run_sweep(args):
    """Sweep grid (tokens per rank x R x H x E x K x {BF16, FP8}): per point the
    median µs of layout + dispatch, dispatch with the cached layout and
    combine, with the fraction of the HBM roofline.  Inputs are drawn on the
    device from a seeded torch generator (timing only; parity is covered by
    the tests)."""
    import torch
    from combine_get_dispatch_02_gb300 import Buffer, ep
    from combine_get_dispatch_02_gb300 import build as epbuild
    from combine_get_dispatch_02_gb300 import workloads as wl
    epbuild.build()
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    peak, peak_kind = _peaks()
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush_w = torch.empty(2 * l2, dtype=torch.uint8, device="cuda")
    flush_r = torch.ones(2 * l2 // 4, dtype=torch.float32, device="cuda")
    sink = torch.empty(1, device="cuda")

    def timed(fn):
        ts = []
        for i in range(args.sweep_reps + 2):
            flush_w.fill_(1)
            torch.sum(flush_r, dim=0, keepdim=True, out=sink)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            if i >= 2:
                ts.append((a, b))
        torch.cuda.synchronize()
        return statistics.median([a.elapsed_time(b) * 1e3 for a, b in ts])

    for w in wl.sweep_points():
        if args.sweep_filter not in w.name:
            continue
        N, K, H, E = w.num_tokens, w.topk, w.hidden, w.num_experts
        gen = torch.Generator(device="cuda").manual_seed(w.seed)
        x = torch.randn(N, H, device="cuda", generator=gen).to(torch.bfloat16)
        logits = torch.randn(N, E, device="cuda", generator=gen)
        top = torch.topk(logits, K, dim=1)
        idx = top.indices.to(torch.int64).contiguous()
        wts = torch.softmax(top.values, dim=1).contiguous()
        buf = Buffer(w.num_ranks, w.max_tokens_per_rank, H, E, K, low_latency_mode=(w.layout == wl.PADDED))
        recv, scales = buf.alloc_recv(w.use_fp8)
        y = torch.empty(buf.rows, H, dtype=torch.bfloat16, device="cuda")
        out = torch.empty(N, H, dtype=torch.bfloat16, device="cuda")
        h = buf.new_handle()
        ctx = buf.ctx
        idx3 = idx.view(w.num_ranks, w.tokens_per_rank, K)
        fresh = timed(lambda: ep.ep_dispatch(ctx, x, idx3, w.tokens_per_rank, w.use_fp8, h.raw, recv,
                                             scales, None, stream))
        cached = timed(lambda: ep.ep_dispatch(ctx, x, None, w.tokens_per_rank, w.use_fp8, h.raw, recv,
                                              scales, None, stream))
        comb = timed(lambda: ep.ep_combine(ctx, y, wts, h.raw, out, stream))
        if buf.device_status() != ep.EP_OK:
            raise RuntimeError(f"device status error at {w.name}")
        M = N * K
        _, disp_bytes, comb_bytes = _algorithmic_bytes(w, M)
        line = {"point": w.name, "layout": w.layout, "tokens": N, "rows": M,
                "us": {"layout_and_dispatch": fresh, "dispatch_cached_layout": cached, "combine": comb},
                "hbm_frac": {"dispatch_cached_layout": disp_bytes / (cached / 1e6) / 1e9 / peak,
                             "combine": comb_bytes / (comb / 1e6) / 1e9 / peak},
                "tokens_per_s": {"dispatch_and_combine": N / ((fresh + comb) / 1e6)},
                "peak_gbs": peak, "peak_source": peak_kind}
        print(json.dumps(line), flush=True)
        del buf, recv, scales, y, out, h, x, logits, idx, wts
        torch.cuda.empty_cache()


def run_kernels(args):
    """The dispatch of the workload with each kernel (ep_tuning.dispatch_kernel
    0 = the rule's choice, 1 = row, 2 = warp-item, 3 = token): median µs of
    20 runs on the cached layout and behind the layout kernel (with --rank:
    the rank layout), L2 flushed before each, and the cached time's fraction
    of the HBM peak."""
    import torch
    from combine_get_dispatch_02_gb300 import Buffer, ep
    from combine_get_dispatch_02_gb300 import build as epbuild
    from combine_get_dispatch_02_gb300 import workloads as wl
    epbuild.build()
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    peak, peak_kind = _peaks()
    w = wl.WORKLOADS[args.workload]
    if args.layout is not None:
        w = w.with_(layout=args.layout)
    if args.dtype is not None:
        w = w.with_(use_fp8=(args.dtype == "fp8"))
    if args.hidden is not None:
        w = w.with_(hidden=args.hidden)
    d = wl.generate(w)
    N, K, H = w.num_tokens, w.topk, w.hidden
    x = torch.from_numpy(np.ascontiguousarray(d["x_bits"]).view(np.int16)).cuda().view(torch.bfloat16)
    idx = torch.from_numpy(d["topk_idx"]).cuda()
    wts = torch.from_numpy(d["topk_weights"].reshape(N, K)).cuda()
    buf = Buffer(w.num_ranks, w.max_tokens_per_rank, H, w.num_experts, K, low_latency_mode=(w.layout == wl.PADDED))
    recv, scales = buf.alloc_rank_recv(w.use_fp8) if args.rank else buf.alloc_recv(w.use_fp8)
    h = buf.new_handle()
    ctx = buf.ctx
    T = w.tokens_per_rank

    def with_layout():
        if args.rank:  # the rank layout, then the dispatch on it
            ep.ep_get_rank_layout(ctx, idx, wts, T, None, None, None, h.raw, stream)
            ep.ep_dispatch(ctx, x, None, T, w.use_fp8, h.raw, recv, scales, None, stream)
        else:
            ep.ep_dispatch(ctx, x, idx, T, w.use_fp8, h.raw, recv, scales, None, stream)

    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    flush_w = torch.empty(2 * l2, dtype=torch.uint8, device="cuda")
    flush_r = torch.ones(2 * l2 // 4, dtype=torch.float32, device="cuda")
    sink = torch.empty(1, device="cuda")

    def timed(fn, reps=20):
        ts = []
        for i in range(reps + 3):
            flush_w.fill_(1)
            torch.sum(flush_r, dim=0, keepdim=True, out=sink)
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record(stream)
            fn()
            b.record(stream)
            if i >= 3:
                ts.append((a, b))
        torch.cuda.synchronize()
        return statistics.median([a.elapsed_time(b) * 1e3 for a, b in ts])

    with_layout()
    M = int((h.tensors()["slot"] >= 0).sum().item())
    _, disp_bytes, _ = _algorithmic_bytes(w, M)
    res = {}
    for kern, per, name in ((0, 0, "rule"), (1, 0, "row"), (2, 0, "warp_item"), (3, 0, "token")):
        t = ep.ep_get_tuning(ctx)
        t.dispatch_kernel = kern
        t.dispatch_ctas_per_sm = per
        ep.ep_set_tuning(ctx, t)
        cached = timed(lambda: ep.ep_dispatch(ctx, x, None, T, w.use_fp8, h.raw, recv, scales, None, stream))
        fresh = timed(with_layout)
        res[name] = {"cached_us": round(cached, 1), "with_layout_us": round(fresh, 1),
                     "cached_frac": round(disp_bytes / (cached / 1e6) / 1e9 / peak, 3)}
    if buf.device_status() != ep.EP_OK:
        raise RuntimeError("device status error")
    print(json.dumps({"workload": _workload_desc(w) + (", rank-deduplicated" if args.rank else ""),
                      "rows": M, "dispatch_bytes": disp_bytes,
                      "peak_gbs": peak, "peak_source": peak_kind, "kernels": res}), flush=True)


def run_ceilings(args):
    """HBM bandwidth of plain torch kernels by traffic mix: a fill (writes
    only), a sum (reads only) and a copy (half each), each over 8 GB, medians
    of 20 runs.  The dispatch's traffic is mostly writes (K rows written per
    row read), the combine's mostly reads: these say which ceiling each one
    meets."""
    import torch
    torch.cuda.set_device(0)
    stream = torch.cuda.current_stream()
    peak, peak_kind = _peaks()
    n = 8 << 30
    a = torch.empty(n, dtype=torch.uint8, device="cuda")
    b = torch.empty(n // 2, dtype=torch.uint8, device="cuda")
    f = a.view(torch.float32)
    sink = torch.empty(1, device="cuda")

    def timed(fn, reps=20):
        ts = []
        for i in range(reps + 3):
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            if i >= 3:
                ts.append((e0, e1))
        torch.cuda.synchronize()
        return statistics.median([x.elapsed_time(y) * 1e-3 for x, y in ts])

    f.fill_(1.0)
    res = {
        # fp32 elements: torch's fill then stores 16 bytes per thread and vector
        "write_only_gbs": n / timed(lambda: f.fill_(2.0)) / 1e9,
        "read_only_gbs": n / timed(lambda: torch.sum(f, dim=0, keepdim=True, out=sink)) / 1e9,
        "copy_gbs": n / timed(lambda: b.copy_(a[: n // 2])) / 1e9,
    }
    out = {"ceilings": {k: round(v, 1) for k, v in res.items()}, "bytes_each": n,
           "peak_gbs": peak, "peak_kind": peak_kind}
    out["ceilings_frac_of_peak"] = {k: round(v / peak, 3) for k, v in res.items()}
    print(json.dumps(out), flush=True)


def main():
    args = _args()
    if args.ceilings:
        run_ceilings(args)
        return
    if args.kernels:
        run_kernels(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
