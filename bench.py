#!/usr/bin/env python3
"""Benchmark of the device-resident MoE dispatch + combine data plane.

One step = one pass of the whole path on one batch: splits (histogram + scan),
pack + exchange into the destination windows, and the top-k combine, replayed
from one CUDA graph, with the inputs already resident in HBM.  The L2 is
flushed between timed steps by reading a 512 MiB buffer, outside the step's
events (a read leaves only clean lines behind, so no write-back of the flush
lands inside the next step).

Beside the step figure the line carries the two halves timed apart with the
same flush before each (``split_flush``: in a MoE layer the expert FFN runs
between dispatch and combine, so the combine cannot find the pack's rows in
L2), and, for workloads whose receive arena fits in L2, the step with a warm
L2 (``l2_warm``).  ``--layers L`` captures L independent dispatch+combine
pairs (each with its own buffers) back to back in one graph, as a decode step
over L MoE layers would, and reports the time per pair without the cost of
launching a graph for every call.

Prints ONE JSON line (rank 0).  ``value`` is dispatch+combine algorithmic
bytes / step time in GB/s, summed over all GPUs; tokens/s and microseconds per
call ride along.  ``--impl reference`` times the CPU oracle instead (rank 0
only), on a bounded sample of the same workload.

Multi-GPU (torchrun): each rank runs an independent replica of the workload
on its own GPU (the R ranks of the method are emulated inside one GPU), so
scaling is weak and there is no data-path collective; a barrier brackets the
timed region and the time is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "dispatch+combine HBM GB/s (% of GB300 peak), tokens/s and µs per call at 1 GPU"
DEFAULT_WORKLOAD = 5
FLUSH_BYTES = 512 << 20
L2_BYTES = 126 << 20  # GB300's L2, if the device properties do not say
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", type=int, default=DEFAULT_WORKLOAD, choices=sorted(W.WORKLOADS))
    ap.add_argument("--mode", choices=["dynamic", "padded"], default="dynamic",
                    help="padded: the worst-case baseline (every pair sends T*k rows)")
    ap.add_argument("--recv-order", choices=["source", "expert"], default="source",
                    help="rows inside each window: source segments (AllToAllv convention) or grouped by local expert")
    ap.add_argument("--router", action="store_true",
                    help="start each step from per-token logits: the router kernel, then the splits kernel")
    ap.add_argument("--router-fused", action="store_true",
                    help="with --router: the router inside the splits kernel (a2av_route_splits, fused flag)")
    ap.add_argument("--active-frac", type=float, default=1.0,
                    help="tokens taking part per rank, as a fraction of T (read from device memory)")
    ap.add_argument("--tokens", type=int, default=0,
                    help="run the workload with this many tokens per rank (small cases for profiling)")
    ap.add_argument("--hidden", type=int, default=0,
                    help="run the workload with this row width H (small cases for profiling the router)")
    ap.add_argument("--flags", type=int, default=0,
                    help="a2av_config_t.flags (1 LSU pack, 2 tiled splits, 4 TMA combine, 8 fused router, "
                         "16 warp-per-token router)")
    ap.add_argument("--pack-ctas-per-sm", type=int, default=0)
    ap.add_argument("--pack-stage-bytes", type=int, default=0)
    ap.add_argument("--pack-store-lag", type=int, default=0)
    ap.add_argument("--combine-ctas-per-sm", type=int, default=0)
    ap.add_argument("--combine-stage-bytes", type=int, default=0)
    ap.add_argument("--combine-unroll", type=int, default=0)
    ap.add_argument("--kernel-steps", type=int, default=300, help="steps of the per-kernel timing pass")
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-seconds", type=float, default=20.0, help="CPU baseline sample budget (both settings)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--l2", choices=["flush", "warm"], default="flush",
                    help="flush L2 before every step (default) or replay back to back with a warm L2 "
                         "(context for workloads that fit in L2; not the reported default)")
    ap.add_argument("--reference-seconds", type=float, default=90.0, help="reference arm: total budget")
    ap.add_argument("--layers", type=int, default=0,
                    help="capture this many independent dispatch+combine pairs (own buffers each) in one graph "
                         "and report the time per pair (decode over several MoE layers)")
    ap.add_argument("--chain", action="store_true",
                    help="with --layers: each layer's x is the previous layer's out (written just before, "
                         "so hot in L2, as a decode step's layer input is)")
    ap.add_argument("--cpu-threads", type=int, default=0,
                    help="threads of the CPU baseline's per-rank setting (0 = min(R, usable cores))")
    return ap.parse_args(argv)


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(x: float) -> float:
    """Max of a per-rank float over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else torch.device("cpu")
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job(per_rank_bytes: int, per_rank_tokens: int, ms_max: float, world: int) -> dict:
    """Whole-job throughput of N independent replicas timed by the slowest rank."""
    sec = ms_max * 1e-3
    return {"gbs": per_rank_bytes * world / sec / 1e9, "tokens_per_s": per_rank_tokens * world / sec,
            "us_per_call": ms_max * 1e3}


def read_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


# The sources each timed kernel is built from (its .cu file, the internal
# header, the C ABI header).
KERNEL_SOURCES = {
    "splits": ["csrc/splits.cu"],
    "pack": ["csrc/pack.cu"],
    "combine": ["csrc/combine.cu"],
    "route": ["csrc/router.cu"],
}


_C_TOKENS = re.compile(r'"(?:\\.|[^"\\\n])*"|\'(?:\\.|[^\'\\\n])*\'|/\*.*?\*/|//[^\n]*', re.S)


def _code_only(text: str) -> str:
    """C/CUDA source with comments removed and whitespace runs collapsed
    (string and character literals kept), so that a comment edit does not
    count as a change of the kernel."""
    t = _C_TOKENS.sub(lambda m: m.group(0) if m.group(0)[0] in "\"'" else " ", text)
    return re.sub(r"\s+", " ", t).strip()


def kernel_source_hash(kernel: str) -> str:
    """Hash of the code a kernel is built from: its .cu file, the internal
    header and the public header, comments and whitespace excluded."""
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "combine_device_resident_gb300")
    for rel in KERNEL_SOURCES[kernel] + ["csrc/a2av_internal.cuh"]:
        h.update(rel.encode())
        h.update(_code_only(open(os.path.join(pkg, rel)).read()).encode())
    h.update(_code_only(open(os.path.join(ROOT, "include", "a2av.h")).read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the kernel's current sources and on this workload (else None)."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        d = json.load(open(p))
    except Exception:
        return None
    if kernel not in KERNEL_SOURCES:
        return None
    for ent in d.get("records", []):
        if (ent.get("kernel") == kernel and ent.get("workload") == workload
                and ent.get("source_sha") == kernel_source_hash(kernel)):
            return ent.get("dram_bytes_per_launch")
    return None


# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clocks/throttle sampling in the background (timestamps kept)."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, enabled=True):
        self.proc = None
        self.path = None
        if not enabled:
            return
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0: float, t1: float):
        if self.proc is None or not self.path:
            return None
        import datetime

        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
            except ValueError:
                continue
            rows.append((ts, parts))
        os.unlink(self.path)
        inside = [p for ts, p in rows if t0 - 0.06 <= ts <= t1 + 0.06] or [p for _, p in rows]
        if not inside:
            return None

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(p[2]) for p in inside if num(p[2]) is not None]
        mx = [num(p[3]) for p in inside if num(p[3]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for p in inside for n, v in zip(names, p[6:10]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(inside)}


# ---------------------------------------------------------------------------
def _sample(a, T_s):
    """The first T_s tokens of every rank, as a contiguous array (made
    before the timed region, so no leg pays for the copy)."""
    import numpy as np

    return np.ascontiguousarray(a[:, :T_s])


def oracle_step_threaded(wl: W.Workload, xb, ix, gt, pool, nthr: int):
    """One pass of the unchanged oracle functions with the per-rank work on
    `nthr` threads: the splits (a few integer passes over idx) on the calling
    thread, then each thread dispatches a contiguous range of source ranks
    into the shared arena (disjoint rows), applies the expert stand-in to its
    own assignments and combines its own tokens.  Returns (recv, slot_map,
    out) so that tests can compare it with the one-thread run."""
    import numpy as np

    import oracle

    R, T, k, H = wl.R, wl.T, wl.k, wl.H
    sp = oracle.splits(R, wl.E, ix, wl.window_mode, wl.window_rows)
    recv = np.zeros((oracle.arena_rows(R, T, k, wl.window_mode, wl.window_rows), H), np.uint16)
    sm = np.empty((R, T, k), np.int32)
    bounds = [(R * i // nthr, R * (i + 1) // nthr) for i in range(nthr)]
    bounds = [b for b in bounds if b[0] < b[1]]
    for f in [pool.submit(oracle.dispatch, R, wl.E, xb, ix, sp, wl.window_mode, wl.window_rows, recv=recv,
                          ranks=b, slot_map_out=sm) for b in bounds]:
        f.result()
    y = recv
    if wl.expert == "scale":
        y = recv.copy()
        for f in [pool.submit(oracle.expert_scale, wl.E, recv, ix[s0:s1], sm[s0:s1], y) for s0, s1 in bounds]:
            f.result()
    out = np.empty((R * T, H), np.uint16)
    futs = [(s0, s1, pool.submit(oracle.combine, y, gt, sm, np.arange(s0 * T, s1 * T, dtype=np.int64)))
            for s0, s1 in bounds]
    for s0, s1, f in futs:
        out[s0 * T:s1 * T] = f.result()
    return recv, sm, out.reshape(R, T, H)


def cpu_baseline(w: W.Workload, x_host_bits, idx, gate, budget_s: float, threads: int = 0):
    """Time the CPU oracle on a bounded sample of the workload, in two
    settings: (i) as it stands, one thread (oracle.run_all); (ii) one thread
    per emulated rank, capped at the usable cores: the same oracle functions
    on disjoint source-rank ranges (oracle_step_threaded)."""
    import concurrent.futures

    import oracle

    def run(wl, xb, ix, gt):
        t = time.perf_counter()
        oracle.run_all(wl.R, wl.E, xb, ix, gt, wl.window_mode, wl.window_rows, wl.expert, recv_order=wl.recv_order)
        return time.perf_counter() - t

    # probe with a small slice of tokens, then size the sample to the budget
    probe_T = max(1, min(w.T, 64))
    wp = w.scaled(T=probe_T)
    tp = run(wp, _sample(x_host_bits, probe_T), _sample(idx, probe_T), _sample(gate, probe_T))
    per_token = tp / probe_T
    leg_s = budget_s / 4  # each leg: about a quarter for the sample, the rest for reps
    T_s = int(min(w.T, max(probe_T, leg_s / max(per_token, 1e-9))))
    ws = w.scaled(T=T_s)
    xs, ixs, gs = _sample(x_host_bits, T_s), _sample(idx, T_s), _sample(gate, T_s)
    reps, spent = 0, 0.0
    while spent < leg_s or reps == 0:
        spent += run(ws, xs, ixs, gs)
        reps += 1
    value = ws.algorithmic_bytes() * reps / spent / 1e9
    sample = (f"oracle (splits, dispatch, combine) on the first {T_s} of {w.T} tokens per rank "
              f"of every rank, {reps} rep(s), {spent:.1f} s")
    res = {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample,
           "tokens_per_s": round(ws.R * ws.T * reps / spent, 1), "host": host_cpu()}

    # (ii) per-rank threads (source order: the rank ranges of the dispatch)
    usable = len(os.sched_getaffinity(0))
    nthr = min(w.R, usable) if threads <= 0 else min(threads, w.R)
    if w.recv_order != "source" or nthr < 2:
        res.update({"threads": 1, "value_threaded": None})
        return res
    T_t = int(min(w.T, max(probe_T, T_s * nthr)))
    wt = w.scaled(T=T_t)
    xt, ixt, gtt = _sample(x_host_bits, T_t), _sample(idx, T_t), _sample(gate, T_t)
    reps_t, spent_t = 0, 0.0
    with concurrent.futures.ThreadPoolExecutor(max_workers=nthr) as pool:
        oracle_step_threaded(wp, _sample(x_host_bits, probe_T), _sample(idx, probe_T), _sample(gate, probe_T),
                             pool, nthr)
        while spent_t < leg_s or reps_t == 0:
            t = time.perf_counter()
            oracle_step_threaded(wt, xt, ixt, gtt, pool, nthr)
            spent_t += time.perf_counter() - t
            reps_t += 1
    res.update({"threads": nthr, "value_threaded": round(wt.algorithmic_bytes() * reps_t / spent_t / 1e9, 4),
                "tokens_per_s_threaded": round(wt.R * wt.T * reps_t / spent_t, 1),
                "sample_threaded": (f"the same oracle functions, one thread per emulated rank (capped at the "
                                    f"{usable} usable cores: {nthr} threads; splits on one), first {T_t} of "
                                    f"{w.T} tokens per rank, {reps_t} rep(s), {spent_t:.1f} s")})
    return res


def host_cpu() -> dict:
    """The host the CPU figures come from: usable cores and CPU model."""
    model = platform.machine()
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                return {"usable_cores": len(os.sched_getaffinity(0)),
                        "cpu": f"{platform.machine()} {line.split(':', 1)[1].strip()}"}
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        for line in open("/proc/cpuinfo"):
            key = line.split(":")[0].strip().lower()
            if key in ("model name", "cpu part", "hardware"):
                model = f"{platform.machine()} {line.split(':', 1)[1].strip()}"
                break
    except OSError:
        pass
    return {"usable_cores": len(os.sched_getaffinity(0)), "cpu": model}


# ---------------------------------------------------------------------------
def run_reference(args, w: W.Workload):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import numpy as np
    import torch

    import oracle

    rg = W.make_routing_gate(w, 0)
    idx, gate = rg["topk_idx"], rg["gate_w"]
    steps, warm = args.steps, args.warmup
    per_step = args.reference_seconds / max(1, steps + warm)
    # token sample per step, sized from a probe
    probe_T = max(1, min(w.T, 16))
    xs = W.bf16_bits(W.make_x(w.scaled(T=probe_T), 0))
    wp = w.scaled(T=probe_T)
    t = time.perf_counter()
    oracle.run_all(wp.R, wp.E, xs, idx[:, :probe_T], gate[:, :probe_T], wp.window_mode, wp.window_rows, wp.expert,
                   recv_order=wp.recv_order)
    per_token = (time.perf_counter() - t) / probe_T
    T_s = int(max(1, min(w.T, per_step / max(per_token, 1e-9))))
    ws = w.scaled(T=T_s)
    x_s = W.bf16_bits(W.make_x(ws, 0))
    ix, gt = np.ascontiguousarray(idx[:, :T_s]), np.ascontiguousarray(gate[:, :T_s])
    for _ in range(warm):
        oracle.run_all(ws.R, ws.E, x_s, ix, gt, ws.window_mode, ws.window_rows, ws.expert, recv_order=ws.recv_order)
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle.run_all(ws.R, ws.E, x_s, ix, gt, ws.window_mode, ws.window_rows, ws.expert, recv_order=ws.recv_order)
    dt = (time.perf_counter() - t0) / steps
    value = ws.algorithmic_bytes() / dt / 1e9
    sample = f"CPU oracle, one thread, first {T_s} of {w.T} tokens per rank of every rank per step"
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": warm, "ms_per_step": round(dt * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_block(w, args),
        "tokens_per_s": round(ws.R * ws.T / dt, 2), "us_per_call": round(dt * 1e6, 2),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample,
                         "host": host_cpu()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)
    del torch
    return 0


def l2_protocol(args) -> str:
    """How the L2 is handled between timed steps (the same text in both arms,
    so that their ``config`` blocks compare equal)."""
    if args.l2 == "flush":
        return (f"GPU arm: L2 flushed before every step by reading a {FLUSH_BYTES >> 20} MiB buffer; "
                "CPU arm: host memory")
    return "GPU arm: steps back to back with a warm L2; CPU arm: host memory"


def config_block(w: W.Workload, args) -> dict:
    c = {"workload": w.name, "R": w.R, "E": w.E, "T": w.T, "H": w.H, "k": w.k, "routing": w.routing,
         "gate": w.gate, "window": w.window_mode, "recv_order": w.recv_order, "l2": l2_protocol(args),
         "accumulate": "fp32", "parallelism": "replicas"}
    if getattr(args, "layers", 0) > 0:
        c["layers"] = args.layers
        if getattr(args, "chain", False):
            c["chain"] = "x of layer i = out of layer i-1"
    return c


def make_plan(args, w: W.Workload, dev):
    import combine_device_resident_gb300 as A

    return A.Plan(w.R, w.E, w.T, w.H, w.k, w.window_mode, w.window_rows, device=dev,
                  flags=args.flags | (A.FLAG_ROUTE_FUSED if args.router and args.router_fused else 0),
                  pack_ctas_per_sm=args.pack_ctas_per_sm, pack_stage_bytes=args.pack_stage_bytes,
                  pack_store_lag=args.pack_store_lag, combine_ctas_per_sm=args.combine_ctas_per_sm,
                  combine_stage_bytes=args.combine_stage_bytes, combine_unroll=args.combine_unroll,
                  recv_order=w.recv_order)


# ---------------------------------------------------------------------------
def run_layers(args, w: W.Workload, dev, rank: int, world: int, local: int):
    """L independent dispatch+combine pairs captured back to back in one
    graph, each with its own inputs, splits and buffers (routing drawn with
    seed = layer index), replayed after an L2 flush: the per-pair time of a
    decode step over L MoE layers, without a graph launch per call.  Nested
    graphs of the first 1, 2, 3 stages of every layer give the per-stage
    time per layer."""
    import torch

    L = args.layers
    plan = make_plan(args, w, dev)
    flush = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_out = torch.zeros((), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)
    x0 = W.make_x(w, 0, device=dev)
    layers = []
    for i in range(L):
        rg = W.make_routing_gate(w, i)
        recv, slot_map, out = plan.new_buffers()
        layers.append(dict(x=x0.clone(), idx=torch.from_numpy(rg["topk_idx"]).to(dev),
                           gate=torch.from_numpy(rg["gate_w"]).to(dev), sp=plan.new_splits(), recv=recv,
                           slot=slot_map, out=out))
    del x0
    if args.chain:  # layer i reads what layer i-1 wrote, as in a decode step
        for i in range(1, L):
            layers[i]["x"] = layers[i - 1]["out"]

    def stage_fns(b):
        return [lambda s: plan.splits(b["idx"], b["sp"], b["slot"], stream=s),
                lambda s: plan.pack(b["x"], b["idx"], b["sp"], b["recv"], b["slot"], stream=s),
                lambda s: plan.combine(b["recv"], b["gate"], b["slot"], b["out"], stream=s)]

    with torch.cuda.stream(stream):
        for b in layers:
            for fn in stage_fns(b):
                fn(stream)
    torch.cuda.synchronize(dev)
    if plan.read_status() != 0:
        raise RuntimeError("device status set during warm-up")

    def capture(n_stages):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            s_ = torch.cuda.current_stream(dev)
            for b in layers:
                for fn in stage_fns(b)[:n_stages]:
                    fn(s_)
        return g

    launches0 = plan.launches
    graph = capture(3)
    kernels_per_step = plan.launches - launches0
    nested = [capture(1), capture(2), graph]
    g_null = torch.cuda.CUDAGraph()
    null_t = torch.zeros(1, dtype=torch.int32, device=dev)
    with torch.cuda.graph(g_null, stream=stream):
        null_t.add_(1)

    def flush_l2():
        if args.l2 == "flush":
            torch.sum(flush, dim=0, out=flush_out)

    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            for gr in nested:
                flush_l2()
                gr.replay()
    torch.cuda.synchronize(dev)

    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    sampler = ClockSampler(local, enabled=not args.no_clocks)
    time.sleep(0.15 if sampler.proc else 0)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        for i in range(K):
            flush_l2()
            starts[i].record(stream)
            graph.replay()
            ends[i].record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    t_wall1 = time.time()
    sampler.stop()
    step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    ms = max_over_ranks(sum(step_ms) / K)
    if plan.read_status() != 0:
        raise RuntimeError("device status word set during the timed region")

    KK = max(1, min(K, args.kernel_steps))
    timed = nested + [g_null]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(timed))] for _ in range(KK)]
    with torch.cuda.stream(stream):
        for i in range(KK):
            for j, gr in enumerate(timed):
                flush_l2()
                ev[i][2 * j].record(stream)
                gr.replay()
                ev[i][2 * j + 1].record(stream)
    torch.cuda.synchronize(dev)
    t_ms = [sum(ev[i][2 * j].elapsed_time(ev[i][2 * j + 1]) for i in range(KK)) / KK for j in range(len(timed))]
    per_stage = {"splits": 1e3 * (t_ms[0] - t_ms[3]) / L, "pack": 1e3 * (t_ms[1] - t_ms[0]) / L,
                 "combine": 1e3 * (t_ms[2] - t_ms[1]) / L}
    bytes_pair = w.algorithmic_bytes()
    job = whole_job(bytes_pair * L, w.R * w.T * L, ms, world)
    peak, peak_kind = read_peaks()
    clocks = sampler.summary(t_wall0, t_wall1)
    if rank == 0:
        line = {
            "metric": METRIC, "value": round(job["gbs"], 2), "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": round(ms, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_block(w, args), "layers": L,
            "us_per_pair": round(1e3 * ms / L, 3), "tokens_per_s": round(job["tokens_per_s"], 1),
            "pct_of_peak": round(100 * job["gbs"] / world / peak, 2), "peak_gbs": peak, "peak_kind": peak_kind,
            "per_layer_stage_us": {n: round(v, 3) for n, v in per_stage.items()},
            "graph_floor_us": round(1e3 * t_ms[3], 3),
            "timing": (f"one graph of {L} x [splits, pack, combine], each layer with its own buffers"
                       + (", x of each layer the previous layer's out" if args.chain else "") + "; "
                       f"{K} replays; stages from nested graphs of the first 1..3 stages of every layer, "
                       f"{KK} replays each, minus the graph-launch floor for the first"),
            "gpu_launches": int(kernels_per_step * K), "kernels_per_step": int(kernels_per_step),
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    plan.close()
    return 0


# ---------------------------------------------------------------------------
def resolve_workload(args) -> W.Workload:
    """The workload the command names: --workload, scaled by --tokens and
    --hidden (small cases for profiling), in the --recv-order asked for."""
    w = W.WORKLOADS[args.workload]
    if args.tokens or args.hidden:
        w = w.scaled(T=args.tokens or None, H=args.hidden or None)
    if args.recv_order != "source":
        import dataclasses

        w = dataclasses.replace(w, recv_order=args.recv_order)
    return w


def main():
    args = parse_args()
    w = resolve_workload(args)
    if args.impl == "reference":
        return run_reference(args, w)

    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)  # before the process group, so NCCL binds this rank's GPU
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", init_method="env://")
    dev = torch.device("cuda", local)
    if args.layers > 0:
        rc = run_layers(args, w, dev, rank, world, local)
        if world > 1:
            torch.distributed.destroy_process_group()
        return rc

    padded = args.mode == "padded"
    if padded:
        import dataclasses

        w = dataclasses.replace(w, window_mode="padded", window_rows=0)
        need = 2 * w.R * w.R * w.T * w.k * w.H * 2 * (2 if args.e2e_steps else 1)
        free = torch.cuda.mem_get_info(local)[0]
        if need > 0.9 * free:
            raise SystemExit(f"padded mode needs {need / 1e9:.0f} GB for its worst-case buffers, "
                             f"{free / 1e9:.0f} GB free")

    # ---- inputs (seeded, synthetic) ----------------------------------------------
    rg = W.make_routing_gate(w, 0)
    idx_h, gate_h = rg["topk_idx"], rg["gate_w"]
    x = W.make_x(w, 0, device=dev)
    idx = torch.from_numpy(idx_h).to(dev)
    gate = torch.from_numpy(gate_h).to(dev)
    plan = make_plan(args, w, dev)
    recv, slot_map, out = plan.new_buffers()
    sp = plan.new_splits()
    sendbuf = plan.new_send_buffer() if padded else None
    t_active = w.T
    if args.active_frac < 1.0:
        # variable batch: per-rank counts live in device memory, read at run time
        t_active = max(0, min(w.T, int(round(args.active_frac * w.T))))
        num_tokens = torch.full((w.R,), t_active, dtype=torch.int32, device=dev)
        plan.set_active_tokens(num_tokens)
    # L2 flush by READING a buffer larger than L2: it evicts our lines and leaves
    # clean ones behind (a write flush would leave ~L2-size dirty lines whose
    # write-back would land inside the next timed step).
    flush = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    flush_out = torch.zeros((), dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(dev)

    def make_stages(x_, idx_, gate_, sp_, recv_, slot_, out_, send_):
        """The path as (name, launch(stream)) stages, in order."""
        if padded:
            return [("splits", lambda s: plan.splits(idx_, sp_, slot_, stream=s)),
                    ("pack", lambda s: plan.pack_padded(x_, idx_, sp_, send_, slot_, stream=s)),
                    ("exchange", lambda s: plan.exchange_padded(send_, recv_, stream=s)),
                    ("combine", lambda s: plan.combine(recv_, gate_, slot_, out_, stream=s))]
        return [("splits", lambda s: plan.splits(idx_, sp_, slot_, stream=s)),
                ("pack", lambda s: plan.pack(x_, idx_, sp_, recv_, slot_, stream=s)),
                ("combine", lambda s: plan.combine(recv_, gate_, slot_, out_, stream=s))]

    logits = W.make_logits(w, 0, device=dev) if args.router else None

    def with_router(st, idx_, gate_, sp_, slot_, logits_):
        """The router writes idx and gate in place from logits resident in HBM:
        fused into the splits kernel, or as its own kernel before it."""
        if not args.router:
            return st
        if not args.router_fused:
            return [("route", lambda s: plan.route(logits_, idx_, gate_, stream=s))] + st
        return [("route+splits", lambda s: plan.route_splits(logits_, idx_, gate_, sp_, slot_, stream=s))] + st[1:]

    stages = with_router(make_stages(x, idx, gate, sp, recv, slot_map, out, sendbuf), idx, gate, sp, slot_map,
                         logits)

    def capture(stage_list):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            s_ = torch.cuda.current_stream(dev)
            for _, fn in stage_list:
                fn(s_)
        return g

    # warm-up outside capture, then capture the path once
    with torch.cuda.stream(stream):
        for _, fn in stages:
            fn(stream)
    torch.cuda.synchronize(dev)
    if plan.read_status() != 0:
        raise RuntimeError("device status set during warm-up")

    # The timed graph: the kernels back to back (each one after the first is a
    # programmatic dependent of its predecessor).
    launches0 = plan.launches
    graph = capture(stages)
    kernels_per_step = plan.launches - launches0

    # Per-kernel timing: nested graphs holding the first 1, 2, ... stages; the
    # difference of consecutive ones is the time a kernel adds to the step
    # (programmatic-launch overlap included).
    prefixes = [capture(stages[:n]) for n in range(1, len(stages))] + [graph]

    def flush_l2():
        if args.l2 == "flush":
            torch.sum(flush, dim=0, out=flush_out)

    # graph-launch floor: a graph holding one tiny kernel, timed like a step
    g_null = torch.cuda.CUDAGraph()
    null_t = torch.zeros(1, dtype=torch.int32, device=dev)
    with torch.cuda.graph(g_null, stream=stream):
        null_t.add_(1)

    # ---- warm-up -----------------------------------------------------------------
    with torch.cuda.stream(stream):
        for _ in range(max(3, args.warmup)):
            for gr in prefixes:
                flush_l2()
                gr.replay()
    torch.cuda.synchronize(dev)

    # ---- timed region ----------------------------------------------------------------
    K = args.steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    sampler = ClockSampler(local, enabled=not args.no_clocks)
    time.sleep(0.15 if sampler.proc else 0)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        for i in range(K):
            flush_l2()
            starts[i].record(stream)
            graph.replay()
            ends[i].record(stream)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    t_wall1 = time.time()
    sampler.stop()
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    ms = max_over_ranks(sum(step_ms) / K)
    ms_median = max_over_ranks(sorted(step_ms)[K // 2])
    status = plan.read_status()
    if status != 0:
        raise RuntimeError(f"device status word set during the timed region: {status:#x}")

    # ---- per-kernel durations (same stream, same flush) ------------------------------
    # Also the combine on its own (graph [combine]): with the flush before it,
    # its rows come from DRAM, as they would after an expert FFN between the
    # two halves (the split-flush figures).
    g_comb = capture(stages[-1:])
    KK = max(1, min(K, args.kernel_steps))
    timed = prefixes + [g_null, g_comb]
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(timed))] for _ in range(KK)]
    with torch.cuda.stream(stream):
        for i in range(KK):
            for j, gr in enumerate(timed):
                flush_l2()
                ev[i][2 * j].record(stream)
                gr.replay()
                ev[i][2 * j + 1].record(stream)
    torch.cuda.synchronize(dev)
    prefix_ms = [sum(ev[i][2 * j].elapsed_time(ev[i][2 * j + 1]) for i in range(KK)) / KK for j in range(len(timed))]
    comb_alone_ms = prefix_ms.pop()
    names = [n for n, _ in stages]
    mean = {"+".join(names[:j + 1]): prefix_ms[j] for j in range(len(stages))}
    mean["null"] = prefix_ms[-1]
    kt = {names[0]: [prefix_ms[0]]}
    for j in range(1, len(stages)):
        kt[names[j]] = [prefix_ms[j] - prefix_ms[j - 1]]

    # ---- results -------------------------------------------------------------------
    w_act = w.scaled(T=t_active) if t_active != w.T else w  # the bytes and tokens that take part
    bytes_step = w_act.algorithmic_bytes() + (w.R * t_active * w.E * 4 + 8 * w.R * t_active * w.k if args.router
                                              else 0)
    job = whole_job(bytes_step, w.R * t_active, ms, world)
    gbs = job["gbs"]
    peak, peak_kind = read_peaks()
    A_ = w.R * t_active * w.k
    # algorithmic bytes per launch: pack reads x once and writes k copies (+ idx
    # read, slot_map write); combine reads k rows and writes out (+ slot_map and
    # gate reads).  pack + combine = Workload.algorithmic_bytes().  The padded
    # baseline's exchange moves every worst-case segment: R*R*T*k rows read and
    # written.
    kbytes = {
        "route": w.R * t_active * w.E * 4 + 8 * A_,
        "splits": 8 * A_,
        "route+splits": w.R * t_active * w.E * 4 + 8 * A_,  # logits in, idx and gates out (no idx re-read)
        "pack": w.R * t_active * w.H * 2 * (1 + w.k) + 8 * A_,
        "exchange": 2 * w.R * w.R * w.T * w.k * w.H * 2,
        "combine": w.R * t_active * w.H * 2 * (1 + w.k) + 8 * A_,
    }
    kus = {n: 1e3 * sum(v) / len(v) for n, v in kt.items() if v}
    dom = max((n for n in names if n not in ("splits", "route", "route+splits")), key=lambda n: kus.get(n, 0.0))
    ach = kbytes[dom] / (kus[dom] * 1e-6) / 1e9
    # (captured on the plain path: source order, every token, no padding)
    traffic = None if (padded or t_active != w.T or w.recv_order != "source") else ncu_traffic(dom, w.name)
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(ach, 1), "peak": peak, "unit": "GB/s",
                "frac": round(ach / peak, 4), "traffic": traffic, "peak_kind": peak_kind,
                # the DRAM side of the same launch: measured DRAM bytes over the same
                # duration (below frac when rows are served by or left in L2)
                "traffic_frac": (round(traffic / (kus[dom] * 1e-6) / 1e9 / peak, 4) if traffic else None),
                "kernel_us": {n: round(v, 3) for n, v in kus.items()},
                "kernel_gbs": {n: round(kbytes[n] / (kus[n] * 1e-6) / 1e9, 1) for n in kus},
                "timing": (f"marginal: nested graphs of the first 1..{len(stages)} kernels, "
                           f"{KK} steps each, L2 flushed before each replay"),
                "nested_us": {n: round(1e3 * v, 3) for n, v in mean.items()}}

    # ---- the two halves apart, each after its own flush ------------------------------
    # dispatch = every stage but the combine (one graph), combine = its own
    # graph; the sum is what a MoE layer pays when its expert FFN evicts the
    # pack's rows between the halves.  Per kernel: the last dispatch kernel's
    # marginal over the graph before it, and the combine graph minus the
    # graph-launch floor (an empty-work graph timed the same way).
    disp_ms = prefix_ms[len(stages) - 2]
    floor_ms = mean["null"]
    sf_kus = {names[-2]: 1e3 * (disp_ms - (prefix_ms[len(stages) - 3] if len(stages) >= 3 else floor_ms)),
              names[-1]: 1e3 * (comb_alone_ms - floor_ms)}
    sf_gbs = {n: kbytes[n] / (v * 1e-6) / 1e9 for n, v in sf_kus.items() if v > 0}
    split_flush = {
        "dispatch_us": round(1e3 * disp_ms, 3), "combine_us": round(1e3 * comb_alone_ms, 3),
        "total_us": round(1e3 * (disp_ms + comb_alone_ms), 3), "graph_floor_us": round(1e3 * floor_ms, 3),
        "gbs": round(bytes_step / ((disp_ms + comb_alone_ms) * 1e-3) / 1e9, 1),
        "pct_of_peak": round(100 * bytes_step / ((disp_ms + comb_alone_ms) * 1e-3) / 1e9 / peak, 2),
        "kernel_us": {n: round(v, 3) for n, v in sf_kus.items()},
        "kernel_gbs": {n: round(v, 1) for n, v in sf_gbs.items()},
        "kernel_frac": {n: round(v / peak, 4) for n, v in sf_gbs.items()},
        "timing": (f"graphs [{', '.join(names[:-1])}] and [{names[-1]}] replayed {KK} times each, "
                   "L2 flushed before each replay; the sum counts two graph launches"),
    }
    if traffic and dom in sf_kus and sf_kus[dom] > 0:
        split_flush["traffic_frac"] = {dom: round(traffic / (sf_kus[dom] * 1e-6) / 1e9 / peak, 4)}
    if args.l2 == "flush":
        # Write-back charged: rows a half leaves dirty in L2 are written back
        # during the next flush, outside the half's events.  Time [half, then
        # a flush] and subtract a flush of a clean L2: what remains is the
        # half plus the write-back of its dirty lines.
        pre_g = prefixes[len(stages) - 3] if len(stages) >= 3 else g_null
        wb_graphs = [pre_g, prefixes[len(stages) - 2], g_comb, g_null, None]
        ev_wb = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(wb_graphs))] for _ in range(KK)]
        with torch.cuda.stream(stream):
            for i in range(KK):
                for j, gr in enumerate(wb_graphs):
                    flush_l2()
                    ev_wb[i][2 * j].record(stream)
                    if gr is not None:
                        gr.replay()
                    flush_l2()
                    ev_wb[i][2 * j + 1].record(stream)
        torch.cuda.synchronize(dev)
        wb = [sum(ev_wb[i][2 * j].elapsed_time(ev_wb[i][2 * j + 1]) for i in range(KK)) / KK
              for j in range(len(wb_graphs))]
        clean = wb[-1]
        pre_c, disp_c, comb_c, null_c = (v - clean for v in wb[:4])
        wb_kus = {names[-2]: 1e3 * (disp_c - pre_c), names[-1]: 1e3 * (comb_c - null_c)}
        wb_gbs = {n: kbytes[n] / (v * 1e-6) / 1e9 for n, v in wb_kus.items() if v > 0}
        split_flush["writeback_charged"] = {
            "dispatch_us": round(1e3 * disp_c, 3), "combine_us": round(1e3 * comb_c, 3),
            "total_us": round(1e3 * (disp_c + comb_c), 3),
            "pct_of_peak": round(100 * bytes_step / ((disp_c + comb_c) * 1e-3) / 1e9 / peak, 2),
            "kernel_us": {n: round(v, 3) for n, v in wb_kus.items()},
            "kernel_gbs": {n: round(v, 1) for n, v in wb_gbs.items()},
            "kernel_frac": {n: round(v / peak, 4) for n, v in wb_gbs.items()},
            "clean_flush_us": round(1e3 * clean, 3),
            "timing": ("each graph timed together with the flush after it, minus a flush of a clean L2 "
                       "(the dirty lines a half leaves are written back during that flush)"),
        }

    # ---- warm L2, for workloads whose receive arena fits in L2 ---------------------
    l2_warm = None
    arena_bytes = plan.arena_rows * w.H * 2
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or L2_BYTES)
    if args.l2 == "flush" and arena_bytes <= l2_bytes:
        KW = max(10, min(K, 1000))
        ws_, we_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            for _ in range(10):
                graph.replay()
            ws_.record(stream)
            for _ in range(KW):
                graph.replay()
            we_.record(stream)
        torch.cuda.synchronize(dev)
        warm_ms = max_over_ranks(ws_.elapsed_time(we_) / KW)
        l2_warm = {"ms_per_step": round(warm_ms, 5), "us_per_call": round(1e3 * warm_ms, 3),
                   "gbs": round(whole_job(bytes_step, w.R * t_active, warm_ms, world)["gbs"], 1),
                   "pct_of_peak": round(100 * bytes_step / (warm_ms * 1e-3) / 1e9 / peak, 2), "steps": KW,
                   "timing": "graph replayed back to back, no flush (each step pays the previous one's write-back)"}

    # ---- end to end through host buffers ----------------------------------------
    # Inputs come from pinned host memory and the result goes back to pinned
    # host memory every step.  Serial: one step at a time on one stream.
    # Pipelined (the headline): a double-buffered serving loop -- two sets of
    # device buffers, each with its own captured graph; step i+1's inputs
    # stream in while step i computes and step i-1's result streams out (the
    # kernels of all steps stay on one stream and one plan).
    # The step's inputs: x with the routing (idx, gate), or x with the router's
    # logits when the router is on the path.
    def pinned(t):
        h = torch.empty(t.shape, dtype=t.dtype, pin_memory=True)
        h.copy_(t)
        return h

    in_pins = [pinned(x)] + ([pinned(logits)] if args.router else [pinned(idx), pinned(gate)])
    outs_pin = [torch.empty(out.shape, dtype=out.dtype, pin_memory=True) for _ in range(2)]
    h2d = sum(p_.numel() * p_.element_size() for p_ in in_pins)
    d2h = outs_pin[0].numel() * 2
    ins1 = [x] + ([logits] if args.router else [idx, gate])
    serial_ms = []
    with torch.cuda.stream(stream):
        for i in range(min(args.e2e_steps, 10) + 3):
            flush_l2()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            for dst, src in zip(ins1, in_pins):
                dst.copy_(src, non_blocking=True)
            graph.replay()
            outs_pin[0].copy_(out, non_blocking=True)
            b.record(stream)
            b.synchronize()
            if i >= 3:
                serial_ms.append(a.elapsed_time(b))

    # second buffer set and its graph
    x2 = torch.empty_like(x)
    idx2, gate2 = torch.empty_like(idx), torch.empty_like(gate)
    recv2, slot_map2, out2 = plan.new_buffers()
    sp2 = plan.new_splits()
    send2 = plan.new_send_buffer() if padded else None
    logits2 = torch.empty_like(logits) if args.router else None
    ins2 = [x2] + ([logits2] if args.router else [idx2, gate2])
    sets = [(ins1, out, graph)]
    st2 = with_router(make_stages(x2, idx2, gate2, sp2, recv2, slot_map2, out2, send2), idx2, gate2, sp2,
                      slot_map2, logits2)
    g2 = capture(st2)
    sets.append((ins2, out2, g2))
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    n_pipe = args.e2e_steps

    def pipelined(n, compute=True):
        """Time per step of the double-buffered loop; compute=False leaves the
        graph replays out (the same copies, streams and events).  That is
        not a floor: with nothing between them a step's host-to-device and
        device-to-host copies overlap more, and on the GB300 host link they
        then run slower than when the kernels space them out."""
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        t0.record(s_in)
        for i in range(n):
            b = i % 2
            ins, ob, gr = sets[b]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[b])  # step i-2 has finished reading this set
                for dst, src in zip(ins, in_pins):
                    dst.copy_(src, non_blocking=True)
                ev_in[b].record(s_in)
            with torch.cuda.stream(stream):
                stream.wait_event(ev_in[b])
                if i >= 2:
                    stream.wait_event(ev_out[b])  # step i-2's result has left this set
                if compute:
                    gr.replay()
                ev_comp[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[b])
                outs_pin[b].copy_(ob, non_blocking=True)
                ev_out[b].record(s_out)
        s_out.wait_event(ev_out[(n - 1) % 2])
        s_out.wait_stream(s_in)
        s_out.wait_stream(stream)
        t1.record(s_out)
        t1.synchronize()
        return t0.elapsed_time(t1) / n

    pipelined(4)  # warm-up
    pipe_ms = max_over_ranks(pipelined(n_pipe))

    pipelined(2, compute=False)
    copies_ms = max_over_ranks(pipelined(n_pipe, compute=False))
    serial_t = max_over_ranks(sum(serial_ms) / len(serial_ms))
    e2e = {"value": round(whole_job(bytes_step, w.R * t_active, pipe_ms, world)["gbs"], 2), "unit": "GB/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(pipe_ms, 4),
           "steps": n_pipe,
           "path": ("double-buffered loop: pinned host inputs (x and " +
                    ("logits" if args.router else "idx/gate") + ") -> HBM (copy stream), graph replay "
                    "(compute stream), out -> pinned host (copy stream); every step copies its own "
                    "inputs and result"),
           "copies_only_ms_per_step": round(copies_ms, 4),
           "copies_only": "the same loop with the graph replays left out",
           "host_link_gbs": round((h2d + d2h) / (pipe_ms * 1e-3) / 1e9, 1),
           "serial": {"value": round(whole_job(bytes_step, w.R * t_active, serial_t, world)["gbs"], 2),
                      "ms_per_step": round(serial_t, 4), "path": "one step at a time on one stream"}}

    clocks = sampler.summary(t_wall0, t_wall1)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline and not padded and t_active == w.T and not args.router:
        cpu = cpu_baseline(w, W.bf16_bits(x), idx_h, gate_h, args.cpu_seconds, args.cpu_threads)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": K,
            "warmup": max(3, args.warmup), "ms_per_step": round(ms, 5), "ms_median_per_step": round(ms_median, 5),
            "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_block(w, args),
            "mode": args.mode, "active_tokens_per_rank": t_active,
            "router": (("fused" if args.router_fused else "separate") if args.router else False),
            "pct_of_peak": round(100 * gbs / world / peak, 2), "peak_gbs": peak,
            "tokens_per_s": round(job["tokens_per_s"], 1), "us_per_call": round(job["us_per_call"], 3),
            "roofline": roofline, "split_flush": split_flush, "l2_warm": l2_warm, "cpu_baseline": cpu, "e2e": e2e,
            "gpu_launches": int(kernels_per_step * K), "kernels_per_step": int(kernels_per_step),
            "clocks": clocks, "variant": {"flags": args.flags, "pack_ctas_per_sm": args.pack_ctas_per_sm,
                                          "pack_stage_bytes": args.pack_stage_bytes,
                                          "pack_store_lag": args.pack_store_lag,
                                          "combine_ctas_per_sm": args.combine_ctas_per_sm,
                                          "combine_stage_bytes": args.combine_stage_bytes,
                                          "combine_unroll": args.combine_unroll},
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    plan.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
