"""Benchmark: Q8_0 decode projections of the Llama-3.2-1B stack on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--M 1] [--impl ours|reference]

A step is one decode step of the whole projection stack (16 layers x
{QKV, O, gate/up, down} + LM head) at M rows: activation quantization, the
Q8_0 GEMVs and the fused quantize+GEMVs, captured once into a CUDA graph and
replayed, calls chained with programmatic dependent launch.  The value is
effective GB/s = (packed weight bytes + fp32 input bytes + fp32 output bytes)
per step / time per step; tok/s = M / time per step.  Each step streams
1.32 GB, ten times the 129 MB L2, so no L2 flush is needed between steps.

Under torchrun (N > 1) every rank runs its own replica on its own GPU (the
path has no exchange step); value = bytes of all ranks / max time over ranks.

--impl reference times the oracle (plain C, one host core) on a bounded
sample of the same workload and prints the same line with "impl": "reference".
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

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Q8_0 decode GEMV effective HBM GB/s (% of GB300 peak) and tok/s, M=1–16"
UNIT = "GB/s"
DTYPE = "i8*i8->i32, f32 scale+sum"
FALLBACK_HBM_GBS = 6800.0
# GB300's nominal HBM3e bandwidth (the data-sheet figure, ~8 TB/s): reported
# beside the measured copy peak, which is the roofline's denominator
NOMINAL_HBM_GBS = 7900.0


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def measured_peaks() -> dict:
    """MEASURED_PEAKS.json as a dict ({} when the file is absent)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(p):
        return {}
    with open(p) as f:
        return json.load(f)


def _workload_name(shape, M, layers):
    return "%s q8_0 projection stack (%d layers x qkv/o/gate_up/down + lm_head), decode M=%d" % (
        shape.name, layers, M)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
CLOCK_Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
           "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
           "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="q8clk", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "--query-gpu=" + CLOCK_Q, "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.dev)],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        sm, mx, pw, reasons = [], None, [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx = float(r[2])
                pw.append(float(r[3]))
            except ValueError:
                continue
            for k, name in enumerate(names):
                if r[5 + k].lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": 0}
        # samples under load: power above the idle floor
        thr = min(pw) + 0.3 * (max(pw) - min(pw)) if pw else 0
        loaded = [s for s, p in zip(sm, pw) if p >= thr] or sm
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": mx,
                "reasons": sorted(reasons), "samples": len(sm), "samples_loaded": len(loaded),
                "power_w_max": max(pw) if pw else None}


# ---------------------------------------------------------------------------
# CPU baseline: the oracle, as it stands, on a bounded sample
# ---------------------------------------------------------------------------
def cpu_baseline(shape, M, budget_s=12.0):
    import numpy as np

    import oracle
    import q8_synth
    oracle.build()
    projs = shape.layer_projs()
    data = []
    for p in projs:
        w = q8_synth.normal_np((p.N, p.K), q8_synth.WEIGHT_STD, q8_synth.derive_seed("cpu", p.name))
        W = oracle.quantize(w)
        del w
        x = q8_synth.normal_np((M, p.K), 1.0, q8_synth.derive_seed("cpu-x", p.name))
        data.append((p, W, x))
    per_rep = sum(W.nbytes + x.nbytes + M * p.N * 4 for p, W, x in data)
    reps, t0 = 0, time.perf_counter()
    while True:
        for p, W, x in data:
            oracle.quant_gemm(W, x, p.K)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    gbs = per_rep * reps / el / 1e9
    return {"value": round(gbs, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "layer-0 projections of %s (qkv, o, gate_up, down; %.1f MB of Q8_0 "
                      "weights) at M=%d, oracle quantize + fp64 product, %d repetitions in "
                      "%.1f s on 1 host thread" % (shape.name, per_rep / 1e6, M, reps, el)}


def _cpu_slice_worker(job):
    """One host process of the all-cores baseline: its own slice of the rows of
    each layer-0 projection (seeded per slice), the oracle as it stands,
    repeated for `seconds`; returns (bytes processed, elapsed seconds)."""
    shape_name, M, idx, parts, seconds = job
    import oracle
    import q8_synth
    shape = q8_synth.LLAMA_3B if shape_name == q8_synth.LLAMA_3B.name else q8_synth.LLAMA_1B
    data = []
    for p in shape.layer_projs():
        n = (p.N + parts - 1) // parts
        w = q8_synth.normal_np((n, p.K), q8_synth.WEIGHT_STD, q8_synth.derive_seed("cpu", p.name, idx))
        x = q8_synth.normal_np((M, p.K), 1.0, q8_synth.derive_seed("cpu-x", p.name))
        data.append((p, oracle.quantize(w), x))
        del w
    per_rep = sum(W.nbytes + x.nbytes + M * (W.shape[0]) * 4 for p, W, x in data)
    for p, W, x in data:  # warm
        oracle.quant_gemm(W, x, p.K)
    reps, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds:
        for p, W, x in data:
            oracle.quant_gemm(W, x, p.K)
        reps += 1
    return per_rep * reps, time.perf_counter() - t0


def cpu_baseline_all_cores(shape, M, seconds=10.0):
    """The same oracle work on every host core: one spawned process per core,
    each on its slice of the output rows; aggregate = all bytes / the slowest
    process's time."""
    import multiprocessing as mp
    cores = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
    jobs = [(shape.name, M, i, cores, seconds) for i in range(cores)]
    with mp.get_context("spawn").Pool(cores) as pool:
        res = pool.map(_cpu_slice_worker, jobs)
    total = sum(b for b, _ in res)
    el = max(t for _, t in res)
    return {"value": round(total / el / 1e9, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": "layer-0 projections of %s at M=%d split by output rows over %d host processes "
                      "(one per core), oracle quantize + fp64 product, %.1f s" % (shape.name, M, cores, el)}


# ---------------------------------------------------------------------------
# multi-rank bookkeeping (replicas: no data-path collective)
# ---------------------------------------------------------------------------
def max_over_ranks(ms: float, world: int, device=None) -> float:
    """The slowest rank's time per step (all_reduce MAX); `ms` itself at N=1."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_gbs(bytes_per_step_per_rank: int, world: int, ms_max: float) -> float:
    """Whole-job effective GB/s: the bytes every rank processed / the max time."""
    return bytes_per_step_per_rank * world / (ms_max * 1e-3) / 1e9


# ---------------------------------------------------------------------------
# ours
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch
    import torch.distributed as dist

    import __graft_entry__
    import q8_synth
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    if rank == 0 or world == 1:
        __graft_entry__.build()
    if world > 1:
        dist.barrier()
        __graft_entry__.build()  # no-op once built; loads the library
    import q8_block_quantized_gb300 as q8
    from q8_block_quantized_gb300.stack import Q8Stack

    shape = q8_synth.LLAMA_3B if args.model == "3b" else q8_synth.LLAMA_1B
    st = Q8Stack(shape, M=args.M, mode=args.mode, layers=args.layers, seed=rank, tcgen05=args.tcgen05)
    graph = st.capture()
    stream = torch.cuda.current_stream()
    bytes_step = st.bytes_per_step()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    for _ in range(max(args.warmup, 3)):
        graph.replay()
    barrier()

    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        graph.replay()
    e1.record(stream)
    barrier()
    clocks = sampler.stop() if rank == 0 else None
    ms = e0.elapsed_time(e1) / args.steps
    ms_max = max_over_ranks(ms, world, device="cuda")
    value = aggregate_gbs(bytes_step, world, ms_max)

    # e2e: every step copies its inputs from pinned host memory and its
    # results back to pinned host memory, inside the timed region.  As a
    # server would, the copies overlap the neighbouring steps' compute:
    # inputs and outputs are double-buffered (a second stack on the same
    # weights, its own graph) and a copy stream, after step k - 1's compute,
    # downloads its results and uploads step k + 1's inputs (the buffers
    # step k - 1 used); step k's compute waits for that stream's upload of
    # its own inputs, which also orders step k - 2's download before step
    # k overwrites that output buffer.  (Copies inside each step's graph as
    # a parallel branch, or one stream per direction, measured the same.)
    st2 = Q8Stack(shape, M=args.M, mode=args.mode, layers=args.layers, seed=rank, tcgen05=args.tcgen05,
                  shared_weights=st.weights)
    graph2 = st2.capture()
    bufs = ((st, graph), (st2, graph2))
    x_host = torch.empty(st.x_all.shape, dtype=torch.float32, pin_memory=True)
    x_host.copy_(st.x_all.cpu())
    y_host = [torch.empty(st.y_all.shape, dtype=torch.float32, pin_memory=True) for _ in range(2)]
    cp = torch.cuda.Stream()
    up_done = [torch.cuda.Event() for _ in range(2)]
    comp_done = [torch.cuda.Event() for _ in range(2)]

    def e2e_steps(n):
        with torch.cuda.stream(cp):  # the first two uploads
            for k in range(min(n, 2)):
                bufs[k][0].x_all.copy_(x_host, non_blocking=True)
                up_done[k].record(cp)
        for k in range(n):
            b = k & 1
            sb, gb = bufs[b]
            stream.wait_event(up_done[b])
            gb.replay()
            comp_done[b].record(stream)
            cp.wait_event(comp_done[b])
            with torch.cuda.stream(cp):
                y_host[b].copy_(sb.y_all, non_blocking=True)
                if k + 2 < n:
                    sb.x_all.copy_(x_host, non_blocking=True)
                    up_done[b].record(cp)
        done = torch.cuda.Event()
        done.record(cp)
        stream.wait_event(done)  # the timed region ends after the last download

    e2e_steps(4)
    barrier()
    e0.record(stream)
    cp.wait_event(e0)
    e2e_steps(args.steps)
    e1.record(stream)
    barrier()
    ms_e2e = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, device="cuda")
    e2e_value = aggregate_gbs(bytes_step, world, ms_e2e)
    del graph2, st2

    # the same e2e step through the ABI without graph capture: every call is
    # planned and launched by the host, as a caller without graphs sees it
    def eager_steps(n):
        for _ in range(n):
            st.x_all.copy_(x_host, non_blocking=True)
            st.step()
            y_host[0].copy_(st.y_all, non_blocking=True)
    eager_steps(3)
    barrier()
    n_eager = max(1, min(args.steps, 300))
    h0 = time.perf_counter()
    e0.record(stream)
    eager_steps(n_eager)
    e1.record(stream)
    h1 = time.perf_counter()
    barrier()
    ms_eager = max_over_ranks(e0.elapsed_time(e1) / n_eager, world, device="cuda")
    host_us_per_call = (h1 - h0) * 1e6 / n_eager / max(1, st.launches_per_step())

    roof = roofline(st, q8) if rank == 0 else None
    prod = producers(q8, shape) if (rank == 0 and not args.no_producers) else None
    tc5 = tcgen05_vs_default(q8, st) if (rank == 0 and world == 1 and not args.no_producers) else None
    pre = prefill(q8, st) if (rank == 0 and world == 1 and not args.no_producers) else None
    cfgs = configs_table(q8, st) if (rank == 0 and world == 1 and not args.no_producers) else None
    kv = kv_codec(q8, shape) if (rank == 0 and world == 1 and not args.no_producers) else None
    peak, peak_kind = _peaks()
    if rank == 0:
        cpu = cpu_baseline(shape, args.M) if (world == 1 and not args.no_cpu) else None
        cpu_all = cpu_baseline_all_cores(shape, args.M) if (world == 1 and not args.no_cpu) else None
        line = {
            "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": DTYPE,
            "data": "synthetic: seeded N(0,0.02) weights, N(0,1) activations",
            "config": {
                "workload": _workload_name(shape, args.M, st.n_layers), "M": args.M,
                "layers": st.n_layers, "mode": args.mode, "bytes_per_step": bytes_step,
                "weight_bytes_per_step": st.weight_bytes(),
                "l2": "no flush: each step streams %.2f GB > 129 MB L2" % (bytes_step / 1e9),
                "graph": True, "pdl": True, "parallelism": "replicas" if world > 1 else "single",
                "tcgen05": bool(args.tcgen05),
            },
            "tok_s": round(args.M * world / (ms_max * 1e-3), 1),
            "pct_of_hbm_peak": round(100.0 * value / world / peak, 2),
            "hbm_peak_gbs": peak, "hbm_peak_kind": peak_kind,
            "pct_of_nominal_hbm_peak": round(100.0 * value / world / NOMINAL_HBM_GBS, 2),
            "nominal_hbm_gbs": NOMINAL_HBM_GBS,
            "roofline": roof,
            "producers": prod,
            "tcgen05_vs_default": tc5,
            "prefill": pre,
            "configs": cfgs,
            "kv_codec": kv,
            "cpu_baseline": cpu,
            "cpu_baseline_all_cores": cpu_all,
            "e2e": {"value": round(e2e_value, 2), "unit": UNIT,
                    "h2d_bytes_per_step": st.x_all.numel() * 4,
                    "d2h_bytes_per_step": st.y_all.numel() * 4,
                    "ms_per_step": round(ms_e2e, 5),
                    "eager": {"value": round(aggregate_gbs(bytes_step, world, ms_eager), 2), "unit": UNIT,
                              "ms_per_step": round(ms_eager, 5), "steps": n_eager,
                              "host_us_per_launch": round(host_us_per_call, 3),
                              "note": "same copies, every call launched by the host through the C ABI "
                                      "(no graph; stream-ordered, PDL chained)"}},
            "gpu_launches": st.launches_per_step() * args.steps,
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemv_traffic_llama1b_m1.json")


GEMV_SOURCES = ("q8_device.cuh", "q8_gemv_impl.cuh", "q8_gemv.cu", "q8_gemv_r16.cu", "q8_gemv_r32.cu",
                "q8_gemv_r64.cu", "q8_gemv_r128.cu", "q8_internal.h")


def kernel_sources_sha256():
    """Hash of the sources the GEMV kernels and their launch plans are built
    from: DRAM traffic measured by ncu is reported only for the sources it was
    measured on."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "q8_block_quantized_gb300", "csrc")
    files = [os.path.join(csrc, f) for f in GEMV_SOURCES]
    for fn in files:
        h.update(os.path.basename(fn).encode())
        with open(fn, "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def measured_traffic(key, calls, M, fused):
    """Mean dram__bytes_read + dram__bytes_write per launch of the dominant
    class's calls, from the committed ncu capture; None if that capture was
    taken on other sources, another configuration, or lacks one of the
    shapes."""
    try:
        with open(TRAFFIC_FILE) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("sources_sha256") != kernel_sources_sha256() or d.get("M") != M or \
            d.get("fused") != fused:
        return None
    per = d.get("dram_bytes_per_launch", {})
    vals = []
    for c in calls:
        v = per.get("%s|%dx%d" % (key, c.N, c.K))
        if v is None:
            return None
        vals.append(float(v))
    return int(sum(vals) / len(vals)) if vals else None


def kernel_class(q8, c, M):
    """The GEMV kernel instantiation a call runs: packed tile height, rows per
    pass, fused or not (the names ncu shows as gemv_kernel<R, MT, fused>)."""
    mt = min(16, 1 << (max(M, 1) - 1).bit_length())
    return "gemv_kernel<%d,%d,%d>" % (q8.q8_packed_tile_rows(c.N), mt, 1 if c.kind == "fused" else 0)


def roofline(st, q8, reps=3):
    """Roofline of the dominant kernel.  For every GEMV kernel instantiation
    the step's calls that run it are captured, in step order, into a CUDA
    graph of their own (no programmatic dependent launch, so each launch runs
    alone) and timed with CUDA events on the stream it is replayed on.  Every class
    streams more than 300 MB of distinct weights per replay, more than L2
    holds, so each launch reads its weights from HBM.  The dominant kernel is
    the class with the largest time per step; achieved = its algorithmic
    bytes (packed weights + fp32 input + fp32 output per launch) / its time."""
    import torch
    ws = st.workspace
    classes = {}
    for c in st.calls:
        if c.kind == "quant":
            continue
        classes.setdefault(kernel_class(q8, c, st.M), []).append(c)

    def run(calls):
        for c in calls:
            if c.kind == "gemm":
                q8.q8_gemm(c.W, c.N, c.K, c.A, st.M, c.y, workspace=ws)
            else:
                q8.q8_fused_quant_gemm(c.W, c.N, c.K, c.x, st.M, c.y, workspace=ws)

    rows = []
    for key, calls in classes.items():
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            run(calls)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            run(calls)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        best = None
        cur = torch.cuda.current_stream()  # replay() launches on the current stream
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(cur)
            g.replay()
            b.record(cur)
            b.synchronize()
            ms = a.elapsed_time(b)
            best = ms if best is None else min(best, ms)
        nbytes = sum(c.W.numel() + 4 * c.x.numel() + 4 * c.y.numel() if c.kind == "fused"
                     else c.W.numel() + c.A.numel() + 4 * c.y.numel() for c in calls)
        rows.append((best, key, nbytes, len(calls), calls))
        del g
    rows.sort(key=lambda r: r[0], reverse=True)
    ms, key, nbytes, n, dom_calls = rows[0]
    traffic = measured_traffic(key, dom_calls, st.M, st.mode == "fused")
    peak, kind = _peaks()
    achieved = nbytes / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": key, "achieved": round(achieved, 1), "peak": peak,
            "peak_kind": kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "traffic": traffic, "launches_per_step": n,
            "bytes_per_launch_avg": int(nbytes / n), "us_per_launch_avg": round(ms * 1e3 / n, 3),
            "classes": {k: {"launches": nn, "us": round(t * 1e3, 2), "GB/s": round(b / (t * 1e-3) / 1e9, 1)}
                        for t, k, b, nn, _ in rows}}


def configs_table(q8, st, rounds=30, reps=20, seed=0, with_3b=True):
    """The workloads of the metric beside the headline step, each as its own
    CUDA graph on the same weights (the pages' method: configurations
    interleaved in a seeded random order, the median over rounds):
      - the full stack at M = 1, 4, 8, 16 (config 4): GB/s and tok/s;
      - one decoder layer's projections at M = 1 (config 2), 16 chained
        calls of layer 0 per graph: us per layer;
      - the Llama-3.2-3B-shaped stack at M = 1, 16, 32, 64 (config 5);
      - one 2048 x 2048 GEMV at M = 1 (config 1), 40 chained calls per graph,
        hot (one W, resident in L2) and cold (40 copies of W rotated,
        179 MB > L2): us per call;
      - the LM head 128256 x 2048 at M = 1 and 8 (config 3), 4 chained calls
        per graph: us per call and GB/s.
    Fused calls (quantization inside the GEMV), PDL chaining as in the step."""
    import numpy as np
    import torch

    import q8_synth
    from q8_block_quantized_gb300.stack import Q8Stack

    dev = torch.device("cuda")
    cases = {}  # name -> (graph, calls per replay, bytes per call, rows)
    keep = []

    def capture(fn):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            fn()
        torch.cuda.synchronize()
        return g

    for M in (1, 4, 8, 16):
        s2 = st if M == st.M else Q8Stack(st.shape, M=M, mode="fused", layers=st.n_layers,
                                          shared_weights=st.weights)
        keep.append(s2)
        cases["stack M=%d" % M] = (s2.capture(), 1, s2.bytes_per_step(), M)
    # one decoder layer's projections at M = 1 (qkv, o, gate/up, down), 16
    # chained copies of layer 0 per graph
    lay = Q8Stack(st.shape, M=1, mode="fused", layers=1, shared_weights=st.weights, include_head=False)
    keep.append(lay)

    def layer_run():
        for _ in range(16):
            lay.step()
    cases["layer M=1"] = (capture(layer_run), 16, lay.bytes_per_step(), 1)

    def gemv_case(W, N, K, M, calls=1, copies=1):
        # `calls` chained calls per graph, rotating over `copies` copies of W
        x = q8_synth.activations(M, K, q8_synth.derive_seed("cfg", N, K, M), dev)
        y = torch.empty(M, N, device=dev)
        ws = q8.new_workspace(N, K, M, dev)
        Wc = [W] + [W.clone() for _ in range(copies - 1)]
        Ws = [Wc[i % copies] for i in range(calls)]
        keep.extend([x, y, ws, Ws])

        def run():
            for Wi in Ws:
                q8.q8_fused_quant_gemm(Wi, N, K, x, M, y, workspace=ws, flags=q8.FLAG_PDL)
        return capture(run), len(Ws), W.numel() + 4 * M * K + 4 * M * N

    N1, K1 = 2048, 2048
    W1 = q8.pack_weights_f32(q8_synth.weights(N1, K1, q8_synth.derive_seed("cfg-w1"), dev))
    g, n, by = gemv_case(W1, N1, K1, 1, calls=40, copies=40)
    cases["gemv 2048x2048 M=1 cold"] = (g, n, by, 1)
    g, n, by = gemv_case(W1, N1, K1, 1, calls=40, copies=1)
    cases["gemv 2048x2048 M=1 hot"] = (g, n, by, 1)
    head = st.shape.head()
    Wh = st.weights[(st.n_layers, head.name)]
    for M in (1, 8):
        g, n, by = gemv_case(Wh, head.N, head.K, M, calls=4)
        cases["lm_head M=%d" % M] = (g, n, by, M)

    # the Llama-3.2-3B-shaped stack (28 layers + head) at M = 1, 16, 32, 64
    if with_3b:
        st3 = Q8Stack(q8_synth.LLAMA_3B, M=1, mode="fused")
        keep.append(st3)
        for M in (1, 16, 32, 64):
            s3 = st3 if M == 1 else Q8Stack(q8_synth.LLAMA_3B, M=M, mode="fused", shared_weights=st3.weights)
            keep.append(s3)
            cases["3b stack M=%d" % M] = (s3.capture(), 1, s3.bytes_per_step(), M)

    names = list(cases)
    samples = {k: [] for k in names}
    cur = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for k in names:  # warm-up
        for _ in range(3):
            cases[k][0].replay()
    torch.cuda.synchronize()
    rng = np.random.default_rng(seed)
    for _ in range(rounds):
        for i in rng.permutation(len(names)):
            g, calls = cases[names[i]][0], cases[names[i]][1]
            a.record(cur)
            for _ in range(reps):
                g.replay()
            b.record(cur)
            b.synchronize()
            samples[names[i]].append(a.elapsed_time(b) / (reps * calls))
    out = {"order": "seeded random permutation per round (numpy PCG64, seed %d)" % seed, "rounds": rounds,
           "replays_per_visit": reps, "results": []}
    for k in names:
        ms = float(np.median(samples[k]))
        by, M = cases[k][2], cases[k][3]
        ent = {"case": k, "M": M, "us_median": round(ms * 1e3, 3), "GB/s": round(by / (ms * 1e-3) / 1e9, 1)}
        if "stack" in k:
            ent["tok_s"] = round(M / (ms * 1e-3), 1)
        ent["frac_of_measured_peak"] = round(by / (ms * 1e-3) / 1e9 / _peaks()[0], 4)
        out["results"].append(ent)
    del cases, keep
    torch.cuda.empty_cache()
    return out


def producers(q8, shape, launches=20):
    """The fused producers that emit a GEMV's activation blocks (residual add
    + RMSNorm + quantization, SwiGLU + quantization), measured beside the
    step: at the step's decode shape (one token: K = hidden, F = ffn; a graph
    of `launches` launches chained with PDL, time per launch) and at a row
    count whose data is several times L2 (plain launches; achieved =
    algorithmic bytes / time against the measured HBM peak).  The oracle's
    single-thread time for the decode shape is reported beside them."""
    import numpy as np
    import torch

    import oracle
    import q8_synth
    peak, kind = _peaks()
    K, F = shape.hidden, shape.ffn
    dev = "cuda"

    def timed(fn, pdl):
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            fn(0)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(launches):
                fn(q8.FLAG_PDL if pdl else 0)
        g.replay()
        torch.cuda.synchronize()
        cur = torch.cuda.current_stream()
        best = None
        for _ in range(3):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(cur)
            g.replay()
            b.record(cur)
            b.synchronize()
            best = a.elapsed_time(b) if best is None else min(best, a.elapsed_time(b))
        del g
        return best * 1e3 / launches  # us per launch

    def oracle_us(fn):
        n, t0 = 0, time.perf_counter()
        while time.perf_counter() - t0 < 0.3:
            fn()
            n += 1
        return (time.perf_counter() - t0) * 1e6 / n

    out = {}
    # residual add + RMSNorm + quantization, in place on the residual stream
    gamma = q8_synth.normal_torch((K,), 0.1, 1, dev) + 1.0
    rows = {}
    for label, M in (("decode", 1), ("bulk", 16384)):
        x = q8_synth.normal_torch((M, K), 1.0, 2, dev)
        d = q8_synth.normal_torch((M, K), 0.01, 3, dev)
        blocks = q8.empty_blocks(M, K)
        us = timed(lambda f: q8.q8_residual_rmsnorm_quantize(x, gamma, 1e-5, blocks, delta=d,
                                                              h_out=x, flags=f), label == "decode")
        nbytes = M * K * 4 * 3 + K * 4 + blocks.numel()  # x, delta, h in place, gamma, blocks
        gbs = nbytes / (us * 1e-6) / 1e9
        rows[label] = {"M": M, "K": K, "us": round(us, 3), "bytes": nbytes, "GB/s": round(gbs, 1)}
        if label == "bulk":
            rows[label].update({"peak": peak, "peak_kind": kind, "frac": round(gbs / peak, 4)})
        del x, d, blocks
    xo = q8_synth.normal_np((1, K), 1.0, 4)
    do = q8_synth.normal_np((1, K), 0.01, 5)
    go = (1.0 + q8_synth.normal_np((K,), 0.1, 6)).astype(np.float32)
    rows["oracle_us_decode"] = round(oracle_us(lambda: oracle.residual_rmsnorm_quantize(xo, do, go, 1e-5)), 2)
    out["residual_rmsnorm_quantize"] = rows
    # SwiGLU + quantization
    rows = {}
    for label, M in (("decode", 1), ("bulk", 8192)):
        gu = q8_synth.normal_torch((M, 2 * F), 1.0, 7, dev)
        blocks = q8.empty_blocks(M, F)
        us = timed(lambda f: q8.q8_swiglu_quantize(gu, blocks, flags=f), label == "decode")
        nbytes = M * 2 * F * 4 + blocks.numel()
        gbs = nbytes / (us * 1e-6) / 1e9
        rows[label] = {"M": M, "F": F, "us": round(us, 3), "bytes": nbytes, "GB/s": round(gbs, 1)}
        if label == "bulk":
            rows[label].update({"peak": peak, "peak_kind": kind, "frac": round(gbs / peak, 4)})
        del gu, blocks
    guo = q8_synth.normal_np((1, 2 * F), 1.0, 8)
    rows["oracle_us_decode"] = round(oracle_us(lambda: oracle.swiglu_quantize(guo, F)), 2)
    out["swiglu_quantize"] = rows
    # SwiGLU in the gate/up GEMV's epilogue against the GEMV followed by the
    # separate SwiGLU kernel (one decode row, each chained with PDL)
    if q8.q8_packed_tile_rows(2 * F) in (64, 128):
        gate = q8_synth.normal_torch((F, K), q8_synth.WEIGHT_STD, 9, dev)
        up = q8_synth.normal_torch((F, K), q8_synth.WEIGHT_STD, 10, dev)
        Wgu = q8.pack_weights_f32(q8.interleave_gate_up(gate, up))
        del gate, up
        x1 = q8_synth.normal_torch((1, K), 1.0, 11, dev)
        y1 = torch.empty((1, 2 * F), dtype=torch.float32, device=dev)
        hb = q8.empty_blocks(1, F)
        ws = q8.new_workspace(2 * F, K, 1)
        us_epi = timed(lambda f: q8.q8_fused_quant_gemm_swiglu(Wgu, F, K, x1, 1, hb, flags=f), True)

        def two(f):
            q8.q8_fused_quant_gemm(Wgu, 2 * F, K, x1, 1, y1, workspace=ws, flags=f)
            q8.q8_swiglu_quantize(y1, hb, flags=f)
        us_two = timed(two, True)
        out["swiglu_epilogue"] = {"M": 1, "F": F, "K": K, "us_gemv_with_epilogue": round(us_epi, 3),
                                  "us_gemv_then_swiglu": round(us_two, 3)}
        del Wgu
    torch.cuda.empty_cache()
    return out


def kv_codec(q8, shape, launches=20):
    """The int8 KV cache codec (cache write with a slot map, and the read
    back), at the model's K/V row width D = kv_heads * head_dim: a bulk case
    of 65536 rows (a 4096-token prefill of all 16 layers' K and V: 128 MB of
    fp32 rows, more than L2) with plain launches, and one decode token's
    rows of all layers (2 * layers rows) chained with PDL in a graph.
    Algorithmic bytes: fp32 rows + int8 quants + fp32 scales + int32 slots."""
    import torch

    import q8_synth
    peak, kind = _peaks()
    D = shape.kv_dim
    dev = "cuda"
    out = {"D": D}
    for label, rows, cap in (("bulk", 65536, 65536), ("decode", 2 * shape.layers, 4 * 4096 * 2 * shape.layers)):
        x = q8_synth.normal_torch((rows, D), 1.0, q8_synth.derive_seed("kvb", rows), dev)
        cq = torch.zeros((cap, D), dtype=torch.int8, device=dev)
        cd = torch.zeros((cap, D // 32), dtype=torch.float32, device=dev)
        slots = torch.randperm(cap, device=dev)[:rows].to(torch.int32)
        back = torch.empty_like(x)

        def timed(fn, pdl):
            fn(0)
            torch.cuda.synchronize()
            g = torch.cuda.CUDAGraph()
            s = torch.cuda.Stream()
            s.wait_stream(torch.cuda.current_stream())
            with torch.cuda.graph(g, stream=s):
                for _ in range(launches):
                    fn(q8.FLAG_PDL if pdl else 0)
            g.replay()
            torch.cuda.synchronize()
            cur = torch.cuda.current_stream()
            best = None
            for _ in range(3):
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(cur)
                g.replay()
                b.record(cur)
                b.synchronize()
                best = a.elapsed_time(b) if best is None else min(best, a.elapsed_time(b))
            del g
            return best * 1e3 / launches

        nbytes = rows * D * 4 + rows * D + rows * (D // 32) * 4 + rows * 4
        us_w = timed(lambda f: q8.q8_kv_quantize(x, cq, cd, slots=slots, flags=f), label == "decode")
        us_r = timed(lambda f: q8.q8_kv_dequantize(cq, cd, back, slots=slots, flags=f), label == "decode")
        ent = {"rows": rows, "capacity": cap, "bytes": nbytes,
               "write_us": round(us_w, 3), "read_us": round(us_r, 3),
               "write_GB/s": round(nbytes / (us_w * 1e-6) / 1e9, 1),
               "read_GB/s": round(nbytes / (us_r * 1e-6) / 1e9, 1)}
        if label == "bulk":
            ent.update({"peak": peak, "peak_kind": kind,
                        "write_frac": round(nbytes / (us_w * 1e-6) / 1e9 / peak, 4),
                        "read_frac": round(nbytes / (us_r * 1e-6) / 1e9 / peak, 4)})
        out[label] = ent
        del x, cq, cd, slots, back
    torch.cuda.empty_cache()
    return out


def prefill(q8, st, M=512, steps=3, tile_rows=(128, 512, 2048), decode_passes=True, warmup=2):
    """Prefill over the same projection stack, each case one CUDA graph:
    the prefill tile GEMM (q8_fused_quant_gemm_prefill: quantize, pack, one
    tile GEMM per projection; each 128-row weight tile reused across 128
    activation rows) at `tile_rows` tokens, and for comparison the decode
    GEMV at M rows (q8_fused_quant_gemm: launches of 32 rows, W streamed once
    per launch).  Time per step, tokens/s; for the tile GEMM also the int8
    multiply-accumulate rate (2 ops per MAC) and the fraction of the
    measured dense bf16 tensor peak (fp16 operands run at the same rate)."""
    import torch

    from q8_block_quantized_gb300.stack import Q8Stack

    def timed(s2, n):
        g = s2.capture()
        for _ in range(warmup):
            g.replay()
        torch.cuda.synchronize()
        cur = torch.cuda.current_stream()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        for _ in range(n):
            g.replay()
        b.record(cur)
        b.synchronize()
        del g
        return a.elapsed_time(b) / n

    peaks = measured_peaks()
    res = {"tile_gemm": []}
    for Mt in tile_rows:
        s2 = Q8Stack(st.shape, M=Mt, mode="prefill", layers=st.n_layers, shared_weights=st.weights)
        ms = timed(s2, steps)
        tops = 2 * s2.mac_per_step() / (ms * 1e-3) / 1e12
        ent = {"M": Mt, "ms_per_step": round(ms, 3), "tok_s": round(Mt / (ms * 1e-3), 1),
               "launches_per_step": s2.launches_per_step(), "TOPS": round(tops, 1)}
        if peaks.get("bf16_tflops"):
            ent["tensor_frac_of_measured_bf16"] = round(tops / peaks["bf16_tflops"], 4)
        res["tile_gemm"].append(ent)
        del s2
        torch.cuda.empty_cache()
    if not decode_passes:
        return res
    s2 = Q8Stack(st.shape, M=M, mode="fused", layers=st.n_layers, shared_weights=st.weights)
    ms = timed(s2, steps)
    res["decode_gemv_passes"] = {"M": M, "ms_per_step": round(ms, 3), "tok_s": round(M / (ms * 1e-3), 1),
                                 "launches_per_step": s2.launches_per_step(),
                                 "GB/s": round(s2.bytes_per_step() / (ms * 1e-3) / 1e9, 1)}
    del s2
    torch.cuda.empty_cache()
    return res


def tcgen05_vs_default(q8, st, M=16, steps=100):
    """The step at 16 activation rows with the default kernels and with
    Q8_FLAG_TCGEN05 (tcgen05 block dots on the 128-row tiles: gate/up and the
    LM head), same weights and inputs: time per step of each (CUDA events over
    graph replays) and whether the outputs are bitwise equal."""
    import torch

    from q8_block_quantized_gb300.stack import Q8Stack
    res = {"M": M}
    outs = {}
    for label, flag in (("default", False), ("tcgen05", True)):
        s2 = Q8Stack(st.shape, M=M, mode="fused", layers=st.n_layers, shared_weights=st.weights,
                     tcgen05=flag)
        g = s2.capture()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        cur = torch.cuda.current_stream()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        for _ in range(steps):
            g.replay()
        b.record(cur)
        b.synchronize()
        ms = a.elapsed_time(b) / steps
        res[label] = {"ms_per_step": round(ms, 5),
                      "GB/s": round(s2.bytes_per_step() / (ms * 1e-3) / 1e9, 1)}
        outs[label] = s2.y_all.clone()
        del g, s2
    res["bitwise_equal"] = bool(torch.equal(outs["default"], outs["tcgen05"]))
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
# reference arm: the oracle on the host cores
# ---------------------------------------------------------------------------
def run_reference(args):
    import q8_synth
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    shape = q8_synth.LLAMA_3B if args.model == "3b" else q8_synth.LLAMA_1B
    layers = shape.layers if args.layers is None else args.layers
    # Each step is one bounded sample of the workload: the first R rows of each
    # layer-0 projection, R sized so the K timed steps take about a minute.
    import oracle
    oracle.build()
    full = []
    for p in shape.layer_projs():
        w = q8_synth.normal_np((p.N, p.K), q8_synth.WEIGHT_STD, q8_synth.derive_seed("cpu", p.name))
        full.append((p, oracle.quantize(w), q8_synth.normal_np((args.M, p.K), 1.0, 1)))
        del w
    t0 = time.perf_counter()
    for p, W, x in full:
        oracle.quant_gemm(W, x, p.K)
    t_layer = time.perf_counter() - t0
    frac = min(1.0, (60.0 / max(args.steps, 1)) / t_layer)
    data = []
    for p, W, x in full:
        rows = max(1, int(p.N * frac))
        data.append((p, rows, W[:rows].copy(), x))
    per_step = sum(W.nbytes + x.nbytes + args.M * rows * 4 for p, rows, W, x in data)

    def one():
        for p, rows, W, x in data:
            oracle.quant_gemm(W, x, p.K)
    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    el = time.perf_counter() - t0
    value = per_step * args.steps / el / 1e9
    cpu = {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
           "sample": "each step = the first %.1f%% of the output rows of each layer-0 projection "
                     "(qkv, o, gate_up, down) of %s at M=%d, %.2f MB per step, 1 host thread"
                     % (100 * frac, shape.name, args.M, per_step / 1e6)}
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(el / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "i32 dots, f64 sum",
        "data": "synthetic: seeded N(0,0.02) weights, N(0,1) activations",
        "config": {"workload": _workload_name(shape, args.M, layers), "M": args.M,
                   "sample_bytes_per_step": per_step},
        "cpu_baseline": cpu,
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def run_prefill_only(args):
    """The prefill leg alone (for profiling): the tile GEMM over the stack at
    --prefill-only rows, --warmup untimed and --steps timed graph replays."""
    import torch

    import __graft_entry__
    import q8_synth
    __graft_entry__.build()
    import q8_block_quantized_gb300 as q8
    from q8_block_quantized_gb300.stack import Q8Stack
    shape = q8_synth.LLAMA_1B if args.model == "1b" else q8_synth.LLAMA_3B
    st = Q8Stack(shape, M=1, mode="fused", layers=args.layers)
    res = prefill(q8, st, steps=max(args.steps, 1), tile_rows=(args.prefill_only,), decode_passes=False,
                  warmup=args.warmup)
    res["layers"] = st.n_layers
    print(json.dumps(res))
    torch.cuda.synchronize()


def run_kv_only(args):
    """The int8 KV codec legs alone (for profiling): one JSON line."""
    import torch

    import __graft_entry__
    import q8_synth
    __graft_entry__.build()
    import q8_block_quantized_gb300 as q8
    shape = q8_synth.LLAMA_1B if args.model == "1b" else q8_synth.LLAMA_3B
    print(json.dumps(kv_codec(q8, shape)))
    torch.cuda.synchronize()


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--M", type=int, default=1)
    ap.add_argument("--model", choices=["1b", "3b"], default="1b")
    ap.add_argument("--layers", type=int, default=None)
    ap.add_argument("--mode", choices=["shared", "fused", "unfused"], default="fused")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU-baseline leg")
    ap.add_argument("--no-producers", action="store_true",
                    help="skip the fused-producer and tcgen05-variant measurements")
    ap.add_argument("--tcgen05", action="store_true",
                    help="GEMV calls with Q8_FLAG_TCGEN05 (tcgen05 block dots where they apply)")
    ap.add_argument("--prefill-only", type=int, default=0, metavar="ROWS",
                    help="only time the prefill tile GEMM over the stack at ROWS tokens (one JSON line; "
                         "not the benchmark line)")
    ap.add_argument("--kv-only", action="store_true",
                    help="only time the int8 KV codec (one JSON line; not the benchmark line)")
    args = ap.parse_args()
    if args.kv_only:
        run_kv_only(args)
    elif args.prefill_only:
        run_prefill_only(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
