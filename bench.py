#!/usr/bin/env python
"""Benchmark of the fused block-scaled FP8 MoE path on GB300.

One step = one pass of the hot path over one batch: the routing plan
(moe_plan) and the fused forward (moe_fp8_block_scale_forward: gate/up GEMM +
SwiGLU + requant, down GEMM writing BF16 route contributions, combine onto
out), on the prefill workload E288/H4096/I1024/top-8 at 8192 tokens, inputs
resident in HBM.
L2 is flushed (a write larger than L2) between timed steps, outside the
timed intervals, and each step is timed with CUDA events on its stream.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU oracle on
a bounded token sample of the same workload instead.
"""

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused FP8 MoE ms/call & TFLOPS (E288 H4096 I1024 top8, 1K-8K tok), % roofline"
UNIT = "TFLOP/s"
HEADLINE = "prefill_8192"
# our kernels per step: moe_plan (rank, scan, scatter) + forward (stage, gate/up, down, combine)
LAUNCHES_PER_STEP = 7
PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")


# ---------------------------------------------------------------- algorithmic work

def work(cfg, topk_ids):
    """Algorithmic FLOPs and bytes of one step (valid routes only, touched experts only)."""
    import numpy as np
    ids = np.asarray(topk_ids).astype(np.int64).reshape(-1)
    valid = ids[(ids >= 0) & (ids < cfg.E)]
    Rv = int(valid.size)
    U = int(np.unique(valid).size)
    M, H, I, R = cfg.M, cfg.H, cfg.I, cfg.R
    w13_b = 2 * I * H + 4 * (2 * I // 128) * (H // 128)
    w2_b = H * I + 4 * (H // 128) * (I // 128)
    act_b = M * H + 4 * M * (H // 128)
    inter_b = Rv * (I + 4 * (I // 128))
    up = {"flop": Rv * 4 * H * I, "bytes": U * w13_b + act_b + inter_b}
    down = {"flop": Rv * 2 * H * I, "bytes": U * w2_b + inter_b + 4 * M * H + 4 * R}
    total = {"flop": Rv * 6 * H * I,
             "bytes": U * (w13_b + w2_b) + act_b + 4 * M * H + 8 * R}
    return {"Rv": Rv, "U": U, "up": up, "down": down, "total": total}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "bf16_tflops": float(p["bf16_tflops"]),
                "bf16_tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def kernel_source_hash():
    h = hashlib.sha256()
    for name in ("forward.cu", "common.cuh"):
        with open(os.path.join(ROOT, "fp8_block_scale_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload):
    """DRAM bytes per launch from the committed ncu summary, if it still
    matches the kernel source; else None."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            t = json.load(f)
        rec = t[kernel][workload]
        if rec.get("source_hash") != kernel_source_hash():
            return None
        return float(rec["dram_bytes_per_launch"])
    except Exception:
        return None


# ---------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = str(gpu_index)
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(gpu_index).uuid)
            self.gpu = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            pass
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------- our arm

def time_steps(prob, steps, warmup, flush, with_kernel_events=True):
    """Events for per-step times of plan + forward and (optionally) per-kernel
    times of the forward; runs the warm-up steps."""
    import torch
    from fp8_block_scale_gb300 import _lib as L

    stream = torch.cuda.current_stream()
    args = prob.fwd_args()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    kev = [[torch.cuda.Event(enable_timing=True) for _ in range(L.PROFILE_EVENTS)] for _ in range(steps)]
    for evs in kev:
        for e in evs:
            e.record(stream)          # creates the underlying cudaEvent
    argsets = []
    for i in range(steps):
        a = prob.fwd_args()
        if with_kernel_events:
            L.set_profile_events(a, kev[i])
        argsets.append(a)
    for _ in range(warmup):
        flush.zero_()
        prob.run_plan()
        prob.run_forward(args)
    torch.cuda.synchronize()
    return starts, ends, kev, argsets


def run_timed(prob, steps, starts, ends, argsets, flush, graph=None):
    for i in range(steps):
        flush.zero_()
        starts[i].record()
        if graph is not None:
            graph.replay()
        else:
            prob.run_plan()
            prob.run_forward(argsets[i])
        ends[i].record()


def capture_step(prob):
    """plan + forward captured once as a CUDA graph (the same launches with the
    same arguments; replay removes the host's per-launch cost, which decode-
    sized steps would otherwise wait on)."""
    import torch
    args = prob.fwd_args()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            prob.run_plan()
            prob.run_forward(args)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        prob.run_plan()
        prob.run_forward(args)
    torch.cuda.synchronize()
    g._moe_args = args            # keep the argument struct alive with the graph
    return g


def capture_forward(prob):
    """The forward alone (the plan already built) captured as a CUDA graph:
    the pages' boundary, which leaves the plan out."""
    import torch
    args = prob.fwd_args()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            prob.run_forward(args)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, capture_error_mode="thread_local"):
        prob.run_forward(args)
    torch.cuda.synchronize()
    g._moe_args = args
    return g


def measure(prob, steps, warmup, flush, dist=None, clocks=None):
    """The headline: `steps` timed replays of the step captured as a CUDA
    graph, nothing recorded between the launches (they overlap through
    programmatic dependent launch).  Then the same steps issued eagerly
    through the API, and a pass with events between the kernels for the
    per-kernel breakdown (those events serialise the launches)."""
    import torch
    graph = capture_step(prob)
    starts, ends, _, argsets = time_steps(prob, steps, warmup, flush, with_kernel_events=False)
    for _ in range(warmup):
        flush.zero_()
        graph.replay()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
    t0 = time.perf_counter()
    run_timed(prob, steps, starts, ends, argsets, flush, graph)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    if dist is not None:
        dist.barrier()
    clk = clocks.stop() if clocks else None
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]

    run_timed(prob, steps, starts, ends, argsets, flush)
    torch.cuda.synchronize()
    eager_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]

    # the forward alone, replayed from its own graph (L2 flushed before each)
    fgraph = capture_forward(prob)
    for _ in range(warmup):
        flush.zero_()
        fgraph.replay()
    run_timed(prob, steps, starts, ends, argsets, flush, fgraph)
    torch.cuda.synchronize()
    fwd_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]

    kstarts, kends, kev, kargs = time_steps(prob, steps, 1, flush, with_kernel_events=True)
    run_timed(prob, steps, kstarts, kends, kargs, flush)
    torch.cuda.synchronize()
    mean = lambda i, j: statistics.mean(k[i].elapsed_time(k[j]) for k in kev)
    return {"step_ms": statistics.mean(step_ms), "step_ms_median": statistics.median(step_ms),
            "step_ms_eager": statistics.mean(eager_ms),
            "stage_ms": mean(0, 1), "up_ms": mean(1, 2), "down_ms": mean(2, 3), "combine_ms": mean(3, 4),
            "plan_ms": statistics.mean(s.elapsed_time(k[0]) for s, k in zip(kstarts, kev)),
            "forward_ms": statistics.mean(fwd_ms), "forward_ms_with_kernel_events": mean(0, 4),
            "step_ms_with_kernel_events": statistics.mean(
                s.elapsed_time(e) for s, e in zip(kstarts, kends)),
            "wall_s": wall, "clocks": clk}


def measure_e2e_pipelined(prob, steps, warmup):
    """The end-to-end step as a user streaming batches would run it through
    the same API: two device copies of the step's inputs and output; a copy
    stream uploads step i+1's inputs (pinned host -> device) while the
    compute stream runs step i's plan + forward, and step i's output goes
    back (device -> pinned host) while step i+1 computes.  Every byte of
    every step crosses the host link inside the timed interval."""
    import torch
    from fp8_block_scale_gb300 import _lib as L
    host = {
        "a": prob.a.cpu().pin_memory(), "a_scale": prob.a_scale.cpu().pin_memory(),
        "topk_ids": prob.topk_ids.cpu().pin_memory(), "topk_weights": prob.topk_weights.cpu().pin_memory(),
        "out": prob.out_prior.cpu().pin_memory(),
    }
    outs_h = [torch.empty_like(host["out"]).pin_memory() for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = outs_h[0].numel() * outs_h[0].element_size()
    sets = []
    for b in range(2):
        d = {k: torch.empty_like(getattr(prob, k)) for k in ("a", "a_scale", "topk_ids", "topk_weights", "out")}
        args = L.make_fwd_args(d["a"], d["a_scale"], prob.w13, prob.w13_scale, prob.w2, prob.w2_scale,
                               d["topk_weights"], prob.sorted_ids, prob.expert_ids, prob.ntpp, d["out"],
                               prob.workspace, prob.cfg.top_k, prob.cfg.block_m, prob.cfg.routed_scale, prob.status)
        sets.append((d, args))
    comp = torch.cuda.current_stream()
    copy_in = torch.cuda.Stream()
    copy_out = torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]
    for e in ev_done + ev_out:
        e.record(comp)

    def step(i):
        b = i % 2
        d, args = sets[b]
        with torch.cuda.stream(copy_in):
            copy_in.wait_event(ev_done[b])          # step i-2's forward no longer reads set b
            copy_in.wait_event(ev_out[b])           # and its output has been read back
            for k in ("a", "a_scale", "topk_ids", "topk_weights", "out"):
                d[k].copy_(host[k], non_blocking=True)
            ev_in[b].record(copy_in)
        comp.wait_event(ev_in[b])
        L.moe_plan(d["topk_ids"], prob.cfg.E, prob.cfg.block_m, prob.sorted_ids, prob.expert_ids, prob.ntpp,
                   prob.plan_ws)
        prob.run_forward(args)
        ev_done[b].record(comp)
        with torch.cuda.stream(copy_out):
            copy_out.wait_event(ev_done[b])
            outs_h[b].copy_(d["out"], non_blocking=True)
            ev_out[b].record(copy_out)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(comp)
    for i in range(steps):
        step(warmup + i)
    for b in range(2):
        comp.wait_event(ev_out[b])
    end.record(comp)
    torch.cuda.synchronize()
    return start.elapsed_time(end) / steps, h2d, d2h


def measure_e2e(prob, steps, warmup):
    """Same step through the public API with host buffers: H2D of the step's
    inputs from pinned memory, plan, forward, D2H of the output."""
    import torch
    cfg = prob.cfg
    host = {
        "a": prob.a.cpu().pin_memory(), "a_scale": prob.a_scale.cpu().pin_memory(),
        "topk_ids": prob.topk_ids.cpu().pin_memory(), "topk_weights": prob.topk_weights.cpu().pin_memory(),
        "out": prob.out_prior.cpu().pin_memory(),
    }
    out_h = torch.empty_like(host["out"]).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = out_h.numel() * out_h.element_size()
    args = prob.fwd_args()

    def step():
        prob.a.copy_(host["a"], non_blocking=True)
        prob.a_scale.copy_(host["a_scale"], non_blocking=True)
        prob.topk_ids.copy_(host["topk_ids"], non_blocking=True)
        prob.topk_weights.copy_(host["topk_weights"], non_blocking=True)
        prob.out.copy_(host["out"], non_blocking=True)
        prob.run_plan()
        prob.run_forward(args)
        out_h.copy_(prob.out, non_blocking=True)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    s = torch.cuda.Event(enable_timing=True)
    e = torch.cuda.Event(enable_timing=True)
    s.record()
    for _ in range(steps):
        step()
    e.record()
    torch.cuda.synchronize()
    return s.elapsed_time(e) / steps, h2d, d2h


# ---------------------------------------------------------------- oracle timing (CPU baseline)

def oracle_workers():
    """Host cores this process may run on: the oracle's expert-partitioned
    threads, one BLAS thread each."""
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except (AttributeError, OSError):
        return max(1, os.cpu_count() or 1)


def _oracle_child(npz_path, groups_json, workers="1"):
    """Runs in a fresh process with one BLAS/OpenMP thread per worker: times
    the oracle forward, its experts computed in `workers` threads, on each
    group of (local) token indices, one timing per group."""
    import numpy as np
    from oracle import moe as O
    d = dict(np.load(npz_path))
    rs = float(d.pop("routed_scale"))
    secs = []
    for g in json.loads(groups_json):
        t0 = time.perf_counter()
        O.moe_forward(**d, routed_scale=rs, tokens=g, workers=int(workers))
        secs.append(time.perf_counter() - t0)
    print(json.dumps({"seconds": secs}))


def oracle_sample_seconds(cfg, routing, tokens, groups, workers=1):
    """Oracle inputs for the token sample (built here, untimed), then the oracle
    forward timed per group of sample positions in a child process whose
    `workers` threads each use one BLAS thread."""
    import numpy as np
    from oracle.inputs import oracle_inputs
    inp, _ = oracle_inputs(cfg, routing, tokens)
    fd, path = tempfile.mkstemp(suffix=".npz")
    os.close(fd)
    np.savez(path, routed_scale=np.float32(cfg.routed_scale), **inp)
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1",
               CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-child", path, json.dumps(groups),
                        str(workers)], env=env, capture_output=True, text=True, cwd=ROOT)
    os.unlink(path)
    if r.returncode != 0:
        raise RuntimeError("oracle child failed: " + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])["seconds"]


def sample_tokens(cfg, n, offset=0):
    import numpy as np
    return np.unique((np.linspace(0, cfg.M - 1, n).astype(np.int64) + offset) % cfg.M)


def _expert_groups(cfg, routing, tokens):
    """Distinct experts the tokens' valid routes touch: the oracle computes
    each expert's routes in one thread, so at most this many threads work."""
    import numpy as np
    import torch
    ids = routing.topk_ids.to(torch.int64).numpy()[np.asarray(tokens)]
    return int(np.unique(ids[(ids >= 0) & (ids < cfg.E)]).size)


def _valid_routes(cfg, routing, tokens):
    import torch
    ids = routing.topk_ids.to(torch.int64).numpy()[tokens]
    return int(((ids >= 0) & (ids < cfg.E)).sum())


def cpu_baseline(cfg, routing, n_tokens=4):
    tokens = sample_tokens(cfg, n_tokens)
    # threads beyond the sample's expert count would have nothing to do
    workers = max(1, min(oracle_workers(), _expert_groups(cfg, routing, tokens)))
    secs = sum(oracle_sample_seconds(cfg, routing, tokens, [list(range(len(tokens)))], workers))
    rv = _valid_routes(cfg, routing, tokens)
    flop = rv * 6 * cfg.H * cfg.I
    return {"value": flop / secs / 1e12, "unit": UNIT, "cores": workers, "kind": "oracle",
            "sample": f"{len(tokens)} of {cfg.M} tokens ({rv} routes) of {cfg.name}, oracle forward only, "
                      f"experts over {workers} threads of one BLAS thread each, {secs:.1f} s"}


# ---------------------------------------------------------------- main

def workload_desc(cfg):
    return (f"{cfg.name}: M={cfg.M} H={cfg.H} I={cfg.I} E={cfg.E} top_k={cfg.top_k} block_m={cfg.block_m}, "
            f"{cfg.routing} routing")


def run_reference(args, rank):
    """The reference arm: the CPU oracle, as it stands, on a bounded sample:
    each step is one token (all of its routes) of the workload."""
    import workloads as W
    if rank != 0:
        return
    cfg = W.CONFIGS[args.workload]
    routing = W.make_routing(cfg)
    n = args.warmup + args.steps
    pool = sample_tokens(cfg, min(n, 4))
    groups = [[i % len(pool)] for i in range(n)]
    # one token per step: at most its top_k experts keep threads busy
    workers = max(1, min(oracle_workers(), min(_expert_groups(cfg, routing, pool[g]) for g in groups)))
    secs = oracle_sample_seconds(cfg, routing, pool, groups, workers)[args.warmup:]
    flops = [_valid_routes(cfg, routing, pool[g]) * 6 * cfg.H * cfg.I for g in groups[args.warmup:]]
    value = sum(flops) / sum(secs) / 1e12
    ms = 1e3 * sum(secs) / len(secs)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64/f32 (numpy oracle)", "data": "synthetic",
        "config": {"workload": workload_desc(cfg), "sample": "1 token per step (all its routes)",
                   "l2": "n/a (CPU)"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": workers, "kind": "oracle",
                         "sample": f"1 token of {cfg.M} per step, {args.steps} steps, experts over "
                                   f"{workers} threads of one BLAS thread each"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# A rank that dies between steps must not hold the other ranks (and their
# GPUs) in their next collective for the backends' default timeouts (10 to
# 30 minutes): the process group gives up after this long, far above the
# longest gap between two collectives of a healthy run (problem set-up plus
# the timed steps).
PG_TIMEOUT_S = 300


def init_distributed(backend, timeout_s=PG_TIMEOUT_S):
    """Join the process group of a torchrun launch (env:// rendezvous) with a
    bounded collective timeout; returns the torch.distributed module."""
    import datetime
    import torch.distributed as tdist
    tdist.init_process_group(backend, timeout=datetime.timedelta(seconds=timeout_s))
    return tdist


def max_over_ranks(x, dist, device):
    """The maximum of x over all ranks (x itself when not distributed).  A NaN
    on any rank (a failed measurement) makes the result NaN: a MAX reduction
    alone would drop it."""
    if dist is None:
        return float(x)
    import torch
    x = float(x)
    t = torch.tensor([-math.inf if x != x else x, 1.0 if x != x else 0.0], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float("nan") if t[1].item() > 0 else float(t[0].item())


def job_tflops(flop_per_rank, world, step_ms):
    """Whole-job throughput: the FLOPs all ranks processed (each rank runs its
    own batch of the workload) over the slowest rank's step time."""
    return flop_per_rank * world / (step_ms * 1e-3) / 1e12


def run_ours(args, rank, world, dist):
    import torch
    from fp8_block_scale_gb300 import _lib as L
    import workloads as W
    from fp8_block_scale_gb300.problem import DeviceProblem

    L.load()
    dev = int(os.environ.get("LOCAL_RANK", 0))
    torch.cuda.set_device(dev)
    peaks = load_peaks()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20), dtype=torch.uint8, device="cuda")

    cfg = W.CONFIGS[args.workload]
    prob = DeviceProblem(cfg)
    w = work(cfg, prob.routing.topk_ids.to(torch.int64).numpy())
    res = measure(prob, args.steps, args.warmup, flush, dist, ClockSampler(dev) if rank == 0 else None)

    # max over ranks of the timed interval
    step_ms = max_over_ranks(res["step_ms"], dist, "cuda")
    value = job_tflops(w["total"]["flop"], world, step_ms)

    if args.no_e2e:
        e2e_ms, h2d, d2h, e2e_serial_ms = float("nan"), 0, 0, float("nan")
    else:
        e2e_ms, h2d, d2h = measure_e2e_pipelined(prob, max(4, args.steps // 2), 2)
        e2e_serial_ms, _, _ = measure_e2e(prob, max(3, args.steps // 2), 2)
    e2e_ms = max_over_ranks(e2e_ms, dist, "cuda")
    e2e_serial_ms = max_over_ranks(e2e_serial_ms, dist, "cuda")
    if rank != 0:
        return

    fp8_peak = 2.0 * peaks["bf16_tflops"]          # FP8 dense = 2x BF16 dense (nominal 4.5 / 2.25 PF)
    hbm = peaks["hbm_gbs"]
    # dominant kernel: the gate/up GEMM
    up_s = res["up_ms"] * 1e-3
    t_up_bytes = w["up"]["bytes"] / (hbm * 1e9)
    t_up_flop = w["up"]["flop"] / (fp8_peak * 1e12)
    if t_up_bytes >= t_up_flop:
        achieved = w["up"]["bytes"] / up_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm}
    else:
        achieved = w["up"]["flop"] / up_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": fp8_peak, "unit": "TFLOP/s",
                "frac": achieved / fp8_peak}
    roof["traffic"] = recorded_traffic("moe_gemm_kernel<up>", cfg.name)
    roof["kernel"] = "moe_gemm_kernel<up> (gate/up GEMM + SwiGLU + requant)"
    roof["peak_source"] = (f"{peaks['source']} (hbm_gbs; fp8 = 2 x bf16_tflops {peaks['bf16_tflops']})")
    roof["algorithmic_per_launch"] = {"bytes": w["up"]["bytes"], "flop": w["up"]["flop"]}
    t_roof = max(w["total"]["flop"] / (fp8_peak * 1e12), w["total"]["bytes"] / (hbm * 1e9))

    clocks = res["clocks"] or {}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
        "config": {"workload": workload_desc(cfg),
                   "step": "moe_plan + moe_fp8_block_scale_forward, captured once as a CUDA graph and replayed",
                   "l2": "flushed between steps (2 x L2 write), per-step CUDA events",
                   "parallelism": f"replicas x{world} (tokens independent, no collective)"},
        "roofline": roof,
        "ms_forward": res["forward_ms"], "ms_forward_with_kernel_events": res["forward_ms_with_kernel_events"],
        "ms_plan": res["plan_ms"],
        "ms_kernels": {"stage": res["stage_ms"], "up": res["up_ms"], "down": res["down_ms"],
                       "combine": res["combine_ms"]},
        "ms_step_with_kernel_events": res["step_ms_with_kernel_events"],
        "ms_step_eager": res["step_ms_eager"],
        "tflops_forward": w["total"]["flop"] / (res["forward_ms"] * 1e-3) / 1e12,
        "roofline_step": {"t_flop_us": w["total"]["flop"] / (fp8_peak * 1e12) * 1e6,
                          "t_bytes_us": w["total"]["bytes"] / (hbm * 1e9) * 1e6,
                          "frac_forward": t_roof / (res["forward_ms"] * 1e-3),
                          "frac_step": t_roof / (step_ms * 1e-3)},
        "gpu_launches": LAUNCHES_PER_STEP * args.steps,
        "clocks": {"sm_mhz": clocks.get("sm_mhz"), "sm_max_mhz": clocks.get("sm_max_mhz"),
                   "reasons": clocks.get("reasons", [])},
        "e2e": {"value": job_tflops(w["total"]["flop"], world, e2e_ms), "unit": UNIT,
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "mode": "pinned host buffers; step i+1's upload and step i's read-back overlap compute "
                        "(two device buffer sets, copy streams)",
                "ms_per_step_serial": e2e_serial_ms},
    }
    if not args.no_extra:
        line["sweep"] = extra_sweep(cfg, prob, flush, peaks)
    del prob
    torch.cuda.empty_cache()
    try:
        if args.no_cpu_baseline:
            raise RuntimeError("skipped (--no-cpu-baseline)")
        line["cpu_baseline"] = cpu_baseline(cfg, W.make_routing(cfg), n_tokens=args.oracle_tokens)
    except Exception as ex:  # the baseline must not hide the measurement
        line["cpu_baseline"] = {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": f"failed: {ex}"}
    print(json.dumps(line), flush=True)


def extra_sweep(cfg, prob, flush, peaks):
    """Other token counts of the same weights, and the decode workload."""
    import torch
    import workloads as W
    from fp8_block_scale_gb300.problem import DeviceProblem
    out = {}
    hbm = peaks["hbm_gbs"]
    fp8_peak = 2.0 * peaks["bf16_tflops"]
    for name in ("prefill_1024", "prefill_2048", "prefill_4096"):
        c = W.CONFIGS[name]
        p = DeviceProblem(c, weights_from=prob)
        r = measure(p, 10, 3, flush)
        w = work(c, p.routing.topk_ids.to(torch.int64).numpy())
        t_roof = max(w["total"]["flop"] / (fp8_peak * 1e12), w["total"]["bytes"] / (hbm * 1e9))
        out[name] = {"ms_step": r["step_ms"], "ms_forward": r["forward_ms"], "ms_plan": r["plan_ms"],
                     "ms_step_eager": r["step_ms_eager"],
                     "tflops_step": w["total"]["flop"] / (r["step_ms"] * 1e-3) / 1e12,
                     "frac_roofline_step": t_roof / (r["step_ms"] * 1e-3),
                     "ms_kernels": {"stage": r["stage_ms"], "up": r["up_ms"], "down": r["down_ms"],
                                    "combine": r["combine_ms"]}}
        del p
    # the headline shape with power-of-two block scales on both operands,
    # once with the FP32 promotion and once with the block-scaled MMA
    # (MOE_SCALES_UE8M0) on the same inputs
    from fp8_block_scale_gb300 import _lib as L
    c = W.CONFIGS["prefill_8192"].with_(name="prefill_8192_ue8m0", ue8m0=True, act_ue8m0=True)
    p = DeviceProblem(c)
    w = work(c, p.routing.topk_ids.to(torch.int64).numpy())
    t_roof = max(w["total"]["flop"] / (fp8_peak * 1e12), w["total"]["bytes"] / (hbm * 1e9))
    for label, mode in (("fp32_promotion", L.SCALES_FP32), ("block_scaled_mma", L.SCALES_UE8M0)):
        p.scale_mode = mode
        r = measure(p, 10, 3, flush)
        out[f"prefill_8192_ue8m0_{label}"] = {
            "ms_step": r["step_ms"], "ms_forward": r["forward_ms"],
            "tflops_step": w["total"]["flop"] / (r["step_ms"] * 1e-3) / 1e12,
            "frac_roofline_step": t_roof / (r["step_ms"] * 1e-3),
            "ms_kernels": {"stage": r["stage_ms"], "up": r["up_ms"], "down": r["down_ms"], "combine": r["combine_ms"]}}
    del p
    torch.cuda.empty_cache()
    # the other two workloads at their own sizes and weights
    for name in ("skewed", "large"):
        c = W.CONFIGS[name]
        p = DeviceProblem(c)
        r = measure(p, 10, 3, flush)
        w = work(c, p.routing.topk_ids.to(torch.int64).numpy())
        t_flop = w["total"]["flop"] / (fp8_peak * 1e12)
        t_bytes = w["total"]["bytes"] / (hbm * 1e9)
        out[name] = {"ms_step": r["step_ms"], "ms_forward": r["forward_ms"], "ms_plan": r["plan_ms"],
                     "tflops_forward": w["total"]["flop"] / (r["forward_ms"] * 1e-3) / 1e12,
                     "t_flop_us": t_flop * 1e6, "t_bytes_us": t_bytes * 1e6,
                     "frac_roofline_forward": max(t_flop, t_bytes) / (r["forward_ms"] * 1e-3),
                     "ms_kernels": {"stage": r["stage_ms"], "up": r["up_ms"], "down": r["down_ms"],
                                    "combine": r["combine_ms"]}}
        del p
        torch.cuda.empty_cache()
    base = None
    for name in ("decode_m1", "decode_m8", "decode_m64"):
        c = W.CONFIGS[name]
        p = DeviceProblem(c, weights_from=base)
        base = base or p
        r = measure(p, 20, 5, flush)
        w = work(c, p.routing.topk_ids.to(torch.int64).numpy())
        gbs = w["total"]["bytes"] / (r["forward_ms"] * 1e-3) / 1e9
        gbs_step = w["total"]["bytes"] / (r["step_ms"] * 1e-3) / 1e9
        out[name] = {"ms_step": r["step_ms"], "ms_step_eager": r["step_ms_eager"], "ms_forward": r["forward_ms"],
                     "ms_plan": r["plan_ms"], "gbs_forward": gbs, "frac_hbm_forward": gbs / hbm, "gbs_step": gbs_step,
                     "frac_hbm_step": gbs_step / hbm,
                     "ms_kernels": {"stage": r["stage_ms"], "up": r["up_ms"], "down": r["down_ms"],
                                    "combine": r["combine_ms"]}}
    del base
    for label, (M, E, k) in (("router_m1", (1, 257, 9)), ("router_m8192", (8192, 288, 8))):
        out[label] = measure_router(M, E, k, flush, peaks)
    for label, M in (("route_plan_m1", 1), ("route_plan_m8", 8)):
        out[label] = measure_route_plan(M, 257, 9, 64, flush)
    torch.cuda.empty_cache()
    for M in (1, 1024):
        try:  # the E2M1-K32 path's timing must not hide the rest of the sweep
            out[f"w4a8_e288_m{M}"] = measure_w4a8(M, flush, peaks)
        except Exception as ex:
            out[f"w4a8_e288_m{M}"] = {"error": str(ex)}
        torch.cuda.empty_cache()
    return out


def measure_w4a8(M, flush, peaks, steps=5, warmup=3, path=0):
    """moe_w4a8_forward (E2M1-K32 weights x per-row FP8 activations; path 0:
    the tensor cores, 1: the CUDA cores) at the SM120 page's timing shape
    E288/H4096/I1024/top-8 with plan blocks of 16 rows; the plan is built
    once and L2 is flushed before each timed forward.  FLOP = Rv * 6 * H * I; bytes = the touched
    experts' packed codes and K32 scales (1.875 * H * I each) + activations,
    their row scales and `out` read and written."""
    import torch
    import workloads as W
    from fp8_block_scale_gb300.problem import W4A8Problem
    cfg = W.MoEConfig(f"w4a8_e288_m{M}", M=M, H=4096, I=1024, E=288, top_k=8, block_m=16)
    p = W4A8Problem(cfg)
    p.run_plan()
    args = p.fwd_args(path=path)
    for _ in range(warmup):
        p.run_forward(args)
    times = []
    for _ in range(steps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        p.run_forward(args)
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    ms = statistics.median(times)
    ids = p.routing.topk_ids.to(torch.int64)
    valid = ids[(ids >= 0) & (ids < cfg.E)]
    Rv, U = int(valid.numel()), int(torch.unique(valid).numel())
    flop = Rv * 6 * cfg.H * cfg.I
    nbytes = U * 1.875 * cfg.H * cfg.I + M * (cfg.H + 4) + 4 * M * cfg.H
    return {"M": M, "ms_forward": ms, "tflops": flop / (ms * 1e-3) / 1e12,
            "gbs": nbytes / (ms * 1e-3) / 1e9, "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"],
            "path": ("tensor cores (tcgen05 E2M1 x E4M3 projections; requant, combine kernels and a flag memset)"
                     if path == 0 else "CUDA cores (gate/up, requant, down, combine kernels and a flag memset)")}


def measure_router(M, E, k, flush, peaks, steps=20, warmup=5):
    """moe_route_topk on FP32 logits (seeded normal), L2 flushed before each
    timed call; bytes = logits read + ids and weights written."""
    import torch
    from fp8_block_scale_gb300 import _lib as L
    g = torch.Generator(device="cpu").manual_seed(M * 131 + E)
    logits = torch.randn((M, E), generator=g).cuda()
    ids = torch.empty((M, k), dtype=torch.int32, device="cuda")
    w = torch.empty((M, k), dtype=torch.float32, device="cuda")
    for _ in range(warmup):
        L.moe_route_topk(logits, k, ids, w)
    times = []
    for _ in range(steps):
        flush.zero_()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        L.moe_route_topk(logits, k, ids, w)
        b.record()
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
    ms = statistics.median(times)
    nbytes = M * E * 4 + M * k * 8
    return {"M": M, "E": E, "top_k": k, "ms": ms, "gbs": nbytes / (ms * 1e-3) / 1e9,
            "frac_hbm": nbytes / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"]}


def measure_route_plan(M, E, k, block_m, flush, steps=20, warmup=5):
    """Router + plan for a decode step: moe_route_plan (one launch) against
    moe_route_topk followed by moe_plan (two launches), each timed alone with
    CUDA events, L2 flushed before each timed call."""
    import torch
    from fp8_block_scale_gb300 import _lib as L
    g = torch.Generator(device="cpu").manual_seed(M * 131 + E)
    logits = torch.randn((M, E), generator=g).cuda()
    ids = torch.empty((M, k), dtype=torch.int32, device="cuda")
    w = torch.empty((M, k), dtype=torch.float32, device="cuda")
    cap, bcap = L.moe_plan_capacity(M, k, E, block_m)
    sids = torch.empty(cap, dtype=torch.int32, device="cuda")
    eids = torch.empty(bcap, dtype=torch.int32, device="cuda")
    ntpp = torch.empty(1, dtype=torch.int32, device="cuda")
    ws = torch.empty(max(L.moe_plan_workspace_size(M, k, E), 256), dtype=torch.uint8, device="cuda")

    def fused():
        L.moe_route_plan(logits, k, ids, w, block_m, sids, eids, ntpp)

    def two():
        L.moe_route_topk(logits, k, ids, w)
        L.moe_plan(ids, E, block_m, sids, eids, ntpp, ws)

    res = {"M": M, "E": E, "top_k": k, "block_m": block_m}
    for name, fn in (("ms_fused", fused), ("ms_router_then_plan", two)):
        for _ in range(warmup):
            fn()
        times = []
        for _ in range(steps):
            flush.zero_()
            a = torch.cuda.Event(enable_timing=True)
            b = torch.cuda.Event(enable_timing=True)
            a.record()
            fn()
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        res[name] = statistics.median(times)
    return res


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--no-extra", action="store_true", help="skip the sweep of other token counts")
    ap.add_argument("--oracle-tokens", type=int, default=4)
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing (profiling runs)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer end-to-end timing (profiling runs)")
    ap.add_argument("--oracle-child", nargs=3, default=None, help=argparse.SUPPRESS)
    ap.add_argument("--w4a8", action="store_true",
                    help="time only the E2M1-K32 weight path at 1 and 1024 tokens (one JSON line)")
    ap.add_argument("--w4a8-tokens", default="1,1024", help="with --w4a8: token counts, comma-separated")
    ap.add_argument("--w4a8-paths", default="tc,cuda_cores", help="with --w4a8: tc and/or cuda_cores")
    ap.add_argument("--w4a8-steps", type=int, default=5, help="with --w4a8: timed forwards per configuration")
    ap.add_argument("--w4a8-warmup", type=int, default=3, help="with --w4a8: untimed forwards first")
    args = ap.parse_args()
    if args.oracle_child:
        _oracle_child(*args.oracle_child)
        return
    if args.w4a8:
        import torch
        from fp8_block_scale_gb300 import _lib as L
        L.load()
        peaks = load_peaks()
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        tokens = [int(t) for t in args.w4a8_tokens.split(",")]
        paths = args.w4a8_paths.split(",")
        res = {}
        for path, suffix in ((0, ""), (1, "_cuda_cores")):
            if ("tc" if path == 0 else "cuda_cores") not in paths:
                continue
            for M in tokens:
                res[f"w4a8_e288_m{M}{suffix}"] = measure_w4a8(M, flush, peaks, steps=args.w4a8_steps,
                                                               warmup=args.w4a8_warmup, path=path)
        print(json.dumps(res), flush=True)
        return
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    dist = None
    if world > 1:
        if args.impl == "ours":
            import torch
            torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", 0)))
            dist = init_distributed("nccl")
        else:
            dist = init_distributed("gloo")
    try:
        if args.impl == "reference":
            run_reference(args, rank)
        else:
            run_ours(args, rank, world, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
