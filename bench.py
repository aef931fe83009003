#!/usr/bin/env python3
"""Benchmark of the four-direction VisionHOPE memory scan on GB300.

One step = one pass of the whole scan (zero the output, then the scan
kernel: generation, step control, readout with the fused four-route merge,
shared-gain memory update) over one batch of synthetic feature maps already
resident in HBM.  Default workload: the stage-1 map, B=32, 56x56, 96
channels as 3 heads of d=32, row/column aligned chunks of 56, bf16 x.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

N > 1 runs under torchrun, one process per GPU; images are independent, so
every rank scans its own batch (weak scaling, no collective on the data
path; one barrier and one max-reduction of the timings).  ``--impl
reference`` times the fp64 CPU oracle on the host cores instead (rank 0
only).  Rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "4-dir VisionHOPE scan tokens/s on 1 GB300 at 56×56×96; % of roofline"
METRIC_BLOCK = ("VisionHOPE block (Eq. 27: CPE, LN, projections, gated depthwise, exact "
                "operator, FFN) tokens/s on 1 GB300 at 56×56, D=192, D_m=96")
METRIC_BWD = ("4-dir VisionHOPE scan backward (dx, dmemories0) tokens/s on 1 GB300 at "
              "56×56×96; % of roofline")
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# the sources of each kernel whose DRAM traffic profiles/traffic.txt records
KERNEL_SOURCES_TC = ["visual_backbone_gb300/csrc/vh_scan_tc.cu",
                     "visual_backbone_gb300/csrc/vh_tc_ptx.cuh",
                     "visual_backbone_gb300/csrc/vh_common.cuh"]
KERNEL_SOURCES_TC64 = ["visual_backbone_gb300/csrc/vh_scan_tc64.cu",
                       "visual_backbone_gb300/csrc/vh_tc_ptx.cuh",
                       "visual_backbone_gb300/csrc/vh_common.cuh"]
KERNEL_SOURCES_SIMT = ["visual_backbone_gb300/csrc/vh_scan_simt.cu",
                       "visual_backbone_gb300/csrc/vh_common.cuh"]
KERNEL_SOURCES_BWD = ["visual_backbone_gb300/csrc/vh_scan_bwd.cu",
                      "visual_backbone_gb300/csrc/vh_common.cuh"]
FP32_PEAK_TFLOPS = 152 * 128 * 2 * 2.07e9 / 1e12   # SMs x fp32 lanes x 2 flops x max clock


# ---------------------------------------------------------------- helpers

def metric_for(base: str, wl) -> str:
    """The metric string with the measured map in place of the stage-1 shape (the default
    workload's string is unchanged)."""
    return base.replace("56×56×96", f"{wl.H}×{wl.W}×{wl.Cc}")


def algorithmic_cost(wl, ndirs=4):
    """Algorithmic flops and compulsory HBM bytes of one call.

    Flops: 2 x (7d^2 + 20d + (4d^3 + 2d^2)/C_r) multiply-adds per (token,
    route, head): the interaction count of "VisionHOPE", App. C.3 Eq. (56)
    extended to six memories (generation of k, v, q; readout; the shared-gain
    recurrence; O(d) scalars; the chunk-boundary update of four d x d and two
    1 x d memories).  Bytes: x read once, out written once (fp32), memories0."""
    d = wl.d
    xb = 2 if wl.dtype == "bf16" else 4
    flops = 0.0
    for r in range(ndirs):
        cr = wl.chunk if wl.chunk else (wl.W if r < 2 else wl.H)
        macs = 7 * d * d + 20 * d + (4 * d ** 3 + 2 * d * d) / cr
        flops += 2.0 * macs * wl.tokens * wl.nh
    nbytes = wl.tokens * wl.Cc * (xb + 4) + 4 * wl.nh * (4 * d * d + 2 * d) * 4
    return flops, float(nbytes)


def backward_cost(wl, ndirs=4):
    """Algorithmic flops of one backward call: the forward quantities it consumes plus
    their adjoints, 2 x (20d^2 + 24d + (12d^3 + 6d^2)/C_r) per (token, route, head):
    forward 7d^2 + 20d + (4d^3 + 2d^2)/C_r; gain adjoint 5d^2 (P k, the P update,
    <P, G>, G^T u, P^T z); readout adjoint d^2; dx 3d^2 + 2d; the outer products into the
    state adjoint 4d^2 + 2d; at each chunk end S_b^T dS and dS G^T, 2 (4d + 2) d^2."""
    d = wl.d
    flops = 0.0
    for r in range(ndirs):
        cr = wl.chunk if wl.chunk else (wl.W if r < 2 else wl.H)
        macs = 20 * d * d + 24 * d + (12 * d ** 3 + 6 * d * d) / cr
        flops += 2.0 * macs * wl.tokens * wl.nh
    return flops


def block_dims(wl):
    """Block widths for a workload: D_m = the operator's channels, D = 2 D_m (the pages'
    D_m = D / 2, "VisionHOPE" Sec. 3.4), FFN width 4 D."""
    Dm = wl.Cc
    return 2 * Dm, Dm, 8 * Dm


def block_cost(wl):
    """Algorithmic flops of one block call: the GEMMs (Proj_in, the outer query, Proj_out,
    the two FFN layers) plus the operator (algorithmic_cost)."""
    D, Dm, hidden = block_dims(wl)
    gemm = 2.0 * wl.tokens * (D * Dm + Dm * Dm + Dm * D + 2 * D * hidden)
    return gemm + algorithmic_cost(wl)[0], gemm


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
        return pk, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def forward_sources(wl, kernel: str):
    """Sources of the scan kernel a forward call runs: a tensor-core kernel for d = 32 or
    64, bf16, aligned chunks (unless the CUDA-core kernel is forced), else the CUDA-core one."""
    aligned = wl.chunk == 0 or (wl.chunk == wl.W and wl.chunk == wl.H)
    tc = wl.dtype == "bf16" and aligned and wl.Cc % 8 == 0 and kernel != "simt"
    if tc and wl.d == 32:
        return KERNEL_SOURCES_TC
    if tc and wl.d == 64:
        return KERNEL_SOURCES_TC64
    return KERNEL_SOURCES_SIMT


def kernel_source_hash(sources):
    h = hashlib.sha256()
    for rel in sources:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:12]


def recorded_traffic(workload: str, impl: str, sources):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel sources (profiles/traffic.txt: workload impl hash bytes)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    cur = kernel_source_hash(sources)
    for line in open(path):
        parts = line.split()
        if len(parts) >= 4 and not line.startswith("#"):
            if parts[0] == workload and parts[1] == impl and parts[2] == cur:
                return float(parts[3])
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms in the background."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index=None):
        self.samples = []
        self.proc = None
        self.err = None
        self.gpu_index = gpu_index

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
               "-lms", "200"]
        if self.gpu_index is not None:
            cmd += ["-i", str(self.gpu_index)]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError as e:
            self.err = str(e)
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            f = [s.strip() for s in line.split(",")]
            if len(f) >= 9:
                self.samples.append((time.time(), f))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return self

    def summary(self, t0, t1):
        if self.err or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "note": self.err or "no nvidia-smi samples"}
        inside = [f for (t, f) in self.samples if t0 <= t <= t1]
        if len(inside) < 2:   # short timed region: take the samples nearest to it
            near = sorted(self.samples, key=lambda s: min(abs(s[0] - t0), abs(s[0] - t1)))[:3]
            inside = [f for _, f in near]
        def num(s):
            try:
                return float(s)
            except ValueError:
                return None
        sm = [num(f[1]) for f in inside if num(f[1]) is not None]
        smax = [num(f[2]) for f in inside if num(f[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for f in inside for i in range(4) if f[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(inside)}


def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(values, device=None):
    """Element-wise max of per-rank timings (seconds) over the default process
    group; identity when no group is initialised (N = 1)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def job_throughput(tokens_per_rank_step, steps, world, seconds):
    """Whole-job units per second: all ranks' tokens over the slowest rank's time."""
    return world * tokens_per_rank_step * steps / seconds


# --------------------------------------------------------- oracle timing

def pipelined_e2e(dev, steps, upload, compute, download):
    """Seconds for `steps` end-to-end steps, each with its own host->device upload, call
    and device->host readback, double-buffered: the upload, the call and the readback run
    on three streams, ordered by events, so the copies of one step overlap the calls of
    its neighbours.  upload(i, slot, stream) / compute(slot, stream) /
    download(slot, stream) enqueue the work of step i on buffer slot i % 2."""
    import torch
    s_up, s_run, s_down = (torch.cuda.Stream(device=dev) for _ in range(3))
    up = [torch.cuda.Event() for _ in range(2)]
    ran = [torch.cuda.Event() for _ in range(2)]
    down = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        k = i % 2
        if i >= 2:
            s_up.wait_event(ran[k])       # the call of step i - 2 has read slot k's input
        upload(i, k, s_up)
        up[k].record(s_up)
        s_run.wait_event(up[k])
        if i >= 2:
            s_run.wait_event(down[k])     # step i - 2's result in slot k has been read back
        compute(k, s_run)
        ran[k].record(s_run)
        s_down.wait_event(ran[k])
        download(k, s_down)
        down[k].record(s_down)

    for i in range(2):                    # warm the path
        step(i)
    torch.cuda.synchronize(dev)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(s_up)
    for i in range(steps):
        step(i)
    s_up.wait_stream(s_down)
    t1.record(s_up)
    torch.cuda.synchronize(dev)
    return t0.elapsed_time(t1) / 1e3


def time_oracle(wl, images, nthreads, min_seconds=0.0, max_passes=1000, w_query=None, skip=None):
    """Tokens/s of the oracle over `images` images, repeated until `min_seconds`
    of wall time have passed; returns (tokens/s, seconds, passes).  w_query / skip
    (numpy) select the VisionHOPE-exact readout."""
    import oracle
    from visual_backbone_gb300 import synth
    oracle.build()
    inp = synth.make_inputs(wl, batch=images)
    p = oracle.OracleParams(eta_bias=wl.eta_bias, alpha_init=wl.alpha_init, w_query=w_query,
                            skip=skip)
    t0 = time.perf_counter()
    passes = 0
    while True:
        oracle.forward(inp.x64, inp.mem0, wl.H, wl.W, wl.nh, wl.d, chunk_len=wl.chunk, params=p,
                       nthreads=nthreads)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or passes >= max_passes:
            break
    return passes * images * wl.N / dt, dt, passes


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_images(wl, cores=None):
    """Images in one oracle sample: the fewest (at most the batch) whose (image, head)
    scan jobs fill every host core equally, lcm(cores, heads) / heads.  The reference arm
    and cpu_baseline both use it, so they time the same sample and report one rate."""
    cores = cores or cpu_cores()
    return max(1, min(wl.B, math.lcm(cores, wl.nh) // wl.nh))


def time_grad_oracle(wl, images, min_seconds=0.0, max_passes=1000):
    """Tokens/s of the gradient oracle (fp64 autograd of the restated forward) on the
    first `images` images, repeated until `min_seconds` of wall time have passed;
    returns (tokens/s, seconds, torch threads, passes)."""
    import numpy as np
    import torch
    from oracle import vh_grad
    from visual_backbone_gb300 import synth
    inp = synth.make_inputs(wl, batch=images)
    dout = np.random.default_rng(7).standard_normal(inp.x64.shape)
    p = __import__("oracle").OracleParams(eta_bias=wl.eta_bias, alpha_init=wl.alpha_init)
    m64 = inp.mem0.astype(np.float64)
    t0 = time.perf_counter()
    passes = 0
    while True:
        vh_grad.backward(inp.x64, m64, dout, wl.H, wl.W, wl.nh, wl.d, chunk_len=wl.chunk, params=p)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or passes >= max_passes:
            break
    return passes * images * wl.N / dt, dt, torch.get_num_threads(), passes


def time_block_oracle(wl, images, min_seconds=0.0, max_passes=1000):
    """Tokens/s of the block oracle on the first `images` images, repeated until
    `min_seconds` of wall time have passed; returns (tokens/s, seconds, threads,
    passes)."""
    import numpy as np
    import oracle
    from oracle import vh_block as vb
    from visual_backbone_gb300 import synth
    oracle.build()
    D, Dm, _ = block_dims(wl)
    inp = synth.make_block_inputs(images, wl.H, wl.W, D, Dm, wl.d, wl.seed)
    p = oracle.OracleParams(w_query=inp["w_query"].astype(np.float64),
                            skip=inp["skip"].astype(np.float64),
                            dir_scale=inp["dir_scale"].astype(np.float64))
    cores = min(cpu_cores(), images * wl.nh)
    x64, w64 = inp["x"].astype(np.float64), vb.weights_from(inp["weights"])
    m64 = inp["mem0"].astype(np.float64)
    t0 = time.perf_counter()
    passes = 0
    while True:
        vb.block_forward(x64, w64, m64, wl.H, wl.W, inp["nh"], wl.d, p, nthreads=cores)
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= min_seconds or passes >= max_passes:
            break
    return passes * images * wl.N / dt, dt, cores, passes


def run_reference(args, wl):
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    if args.pass_ == "backward":
        return run_reference_backward(args, wl)
    if args.pass_ == "block":
        return run_reference_block(args, wl)
    # forward: the oracle sample of cpu_baseline, one pass per step
    images = args.ref_images or oracle_images(wl)
    cores = min(cpu_cores(), images * wl.nh)
    for _ in range(args.warmup):
        time_oracle(wl, images, cores)
    times = []
    t_start = time.perf_counter()
    for _ in range(args.steps):
        _, dt, _ = time_oracle(wl, images, cores)
        times.append(dt)
    total = sum(times)
    value = args.steps * images * wl.N / total
    sample = (f"{images} image(s) of the {wl.name} workload per step (all 4 routes x "
              f"{wl.nh} heads, {images * wl.N} tokens), fp64 oracle, {cores} threads")
    line = {
        "impl": "reference", "metric": metric_for(METRIC, wl), "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(wl, args),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": time.perf_counter() - t_start,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference_backward(args, wl):
    args.ref_images = args.ref_images or 1
    for _ in range(args.warmup):
        time_grad_oracle(wl, args.ref_images)
    times, cores = [], 1
    t_start = time.perf_counter()
    for _ in range(args.steps):
        _, dt, cores, _ = time_grad_oracle(wl, args.ref_images)
        times.append(dt)
    total = sum(times)
    value = args.steps * args.ref_images * wl.N / total
    sample = (f"{args.ref_images} image(s) of the {wl.name} workload per step, fp64 gradient "
              f"oracle (PyTorch CPU autograd), {cores} threads")
    line = {
        "impl": "reference", "metric": metric_for(METRIC_BWD, wl), "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(wl, args),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": time.perf_counter() - t_start,
    }
    print(json.dumps(line), flush=True)
    return 0


def run_reference_block(args, wl):
    args.ref_images = args.ref_images or oracle_images(wl)
    for _ in range(args.warmup):
        time_block_oracle(wl, args.ref_images)
    times, cores = [], 1
    t_start = time.perf_counter()
    for _ in range(args.steps):
        _, dt, cores, _ = time_block_oracle(wl, args.ref_images)
        times.append(dt)
    total = sum(times)
    value = args.steps * args.ref_images * wl.N / total
    line = {
        "impl": "reference", "metric": METRIC_BLOCK, "value": value, "unit": UNIT, "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(wl, args),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"{args.ref_images} image(s) per step, fp64 block oracle "
                                   f"(numpy + the C scan oracle), {cores} threads"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "wall_s": time.perf_counter() - t_start,
    }
    print(json.dumps(line), flush=True)
    return 0


def workload_config(wl, args):
    return {"workload": f"{wl.name}: B={wl.B} {wl.H}x{wl.W} map, Cc={wl.Cc} as {wl.nh} heads x "
                        f"d={wl.d}, chunk={'row W / col H' if wl.chunk == 0 else wl.chunk}, "
                        f"4 routes, {wl.dtype} x, fp32 state, alpha_init={wl.alpha_init}, "
                        f"eta_bias={wl.eta_bias}",
            "global_batch": wl.B * dist_env()[1], "tokens_per_step_per_gpu": wl.tokens,
            "parallelism": f"dp{dist_env()[1]}: weak scaling, rank r scans images "
                           f"[r*{wl.B}, (r+1)*{wl.B}) of a synthetic batch of "
                           f"{dist_env()[1] * wl.B} (vh.shard_images), no collective",
            "l2": "256 MiB buffer written between timed steps (L2 is 129 MB)",
            "kernel": args.kernel, "readout": args.readout, "pass": args.pass_,
            "memories_out": bool(getattr(args, "memories_out", False)),
            **({"block": "D=%d D_m=%d hidden=%d, 3x3 depthwise, exact operator" % block_dims(wl)}
               if args.pass_ == "block" else {})}


# ------------------------------------------------------------ our arm

def run_ours(args, wl):
    import torch
    import visual_backbone_gb300 as vh
    from visual_backbone_gb300 import _build, synth

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 and not os.path.exists(vh.LIB_PATH):
        _build.build()
    if world > 1:
        torch.distributed.barrier()

    mine = vh.shard_images(wl.B * world, world, rank)  # this rank's images of the job
    inp = synth.make_inputs(wl, batch=len(mine), first_image=mine.start)
    if wl.dtype == "bf16":
        x_host = torch.from_numpy(inp.x_store.view("int16")).view(torch.bfloat16)
    else:
        x_host = torch.from_numpy(inp.x_store)
    x = x_host.to(dev)
    mem0 = torch.from_numpy(inp.mem0).to(dev)
    out = torch.empty((wl.B, wl.H, wl.W, wl.Cc), dtype=torch.float32, device=dev)
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev)  # 256 MiB > L2
    params = vh.ScanParams(eta_bias=wl.eta_bias, alpha_init=wl.alpha_init, impl=args.kernel)
    stream = torch.cuda.Stream(device=dev)
    # VisionHOPE-exact readout (outer query projection + channel-wise skip), random weights
    extra = {}
    if args.readout == "outer":
        g = torch.Generator(device="cpu").manual_seed(1234)
        extra["w_query"] = (torch.randn(wl.Cc, wl.Cc, generator=g) / wl.Cc ** 0.5).to(dev)
        extra["skip"] = torch.randn(4, wl.Cc, generator=g).to(dev)
        extra["workspace"] = torch.empty(6 * wl.B * wl.H * wl.W * wl.Cc, dtype=torch.uint8,
                                         device=dev)

    # the second row of the measurement: the final memories written as well
    if args.memories_out:
        extra["memories_out"] = torch.empty((wl.B, 4, wl.nh, 4 * wl.d * wl.d + 2 * wl.d),
                                            dtype=torch.float32, device=dev)

    def step(ev_start, ev_mid, ev_end):
        flush.zero_()
        ev_start.record(stream)
        out.zero_()
        ev_mid.record(stream)
        vh.scan_forward(x, mem0, wl.d, chunk=wl.chunk, out=out, params=params, stream=stream,
                        accumulate=True, **extra)
        ev_end.record(stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            evs = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            step(*evs)
        torch.cuda.synchronize(dev)
        events = [[torch.cuda.Event(enable_timing=True) for _ in range(3)]
                  for _ in range(args.steps)]
        sampler = ClockSampler(None).start() if rank == 0 else None
        time.sleep(0.3 if sampler else 0.0)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        t0 = time.time()
        for i in range(args.steps):
            step(*events[i])
        torch.cuda.synchronize(dev)
        t1 = time.time()
        if world > 1:
            torch.distributed.barrier()
        if sampler:
            time.sleep(0.3)
            sampler.stop()
    step_ms = [e[0].elapsed_time(e[2]) for e in events]
    kern_ms = [e[1].elapsed_time(e[2]) for e in events]
    total_s = sum(step_ms) / 1e3
    kern_avg_s = sum(kern_ms) / len(kern_ms) / 1e3
    total_s, kern_avg_s = max_over_ranks([total_s, kern_avg_s], device=dev)
    value = job_throughput(wl.tokens, args.steps, world, total_s)

    # end to end through the public API with host buffers (pinned), copies timed: every
    # step uploads x and reads out back, double-buffered against the neighbouring steps
    x_pin = x_host.pin_memory()
    xs = [x, torch.empty_like(x)]
    outs = [out, torch.empty_like(out)]
    out_pins = [torch.empty(out.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    e2e_steps = max(3, min(args.steps, 20))

    def up(i, k, st):
        with torch.cuda.stream(st):
            xs[k].copy_(x_pin, non_blocking=True)

    def run(k, st):
        vh.scan_forward(xs[k], mem0, wl.d, chunk=wl.chunk, out=outs[k], params=params,
                        stream=st, **extra)

    def down(k, st):
        with torch.cuda.stream(st):
            out_pins[k].copy_(outs[k], non_blocking=True)

    e2e_s, = max_over_ranks([pipelined_e2e(dev, e2e_steps, up, run, down)], device=dev)
    e2e_value = job_throughput(wl.tokens, e2e_steps, world, e2e_s)

    if rank == 0:
        flops, nbytes = algorithmic_cost(wl)
        if args.memories_out:
            nbytes += wl.B * 4 * wl.nh * (4 * wl.d * wl.d + 2 * wl.d) * 4
        if args.readout == "outer":
            nbytes += wl.tokens * wl.Cc * 6  # the scan reads the outer queries' three bf16 pieces
        peaks, src = load_peaks()
        achieved = flops / kern_avg_s / 1e12
        peak = float(peaks["bf16_tflops"])
        # (traffic.txt keys the outer-query readout's scan apart: it also reads the queries)
        traffic = recorded_traffic(wl.name, args.kernel + ("+outer" if args.readout == "outer" else ""),
                                   forward_sources(wl, args.kernel))
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": traffic,
                "peak_source": f"bf16 dense burst, {'of measured' if src == 'measured' else 'of fallback'}",
                "flops_per_launch": flops, "kernel_ms": kern_avg_s * 1e3,
                "hbm_compulsory_bytes": nbytes,
                "hbm_achieved_gbs": nbytes / kern_avg_s / 1e9,
                "hbm_frac_of_measured": nbytes / kern_avg_s / 1e9 / float(peaks["hbm_gbs"]),
                "t_roof_ms": 1e3 * max(flops / (peak * 1e12), nbytes / (float(peaks["hbm_gbs"]) * 1e9))}
        roof["frac_of_roofline_time"] = roof["t_roof_ms"] / (kern_avg_s * 1e3)
        # Secondary view: the shared-gain recurrence (2 d^2 multiply-adds per token, route
        # and head) runs on the fp32 FMA pipe, whose nominal peak is 152 SMs x 128 lanes x
        # 2 flops x 2.07 GHz.
        gain_flops = 4.0 * wl.d * wl.d * wl.tokens * wl.nh * 4
        fp32_peak = 152 * 128 * 2 * 2.07e9 / 1e12
        roof["alu_view"] = {"what": "shared-gain recurrence on the fp32 FMA pipe",
                            "flops_per_launch": gain_flops,
                            "achieved": gain_flops / kern_avg_s / 1e12, "peak": fp32_peak,
                            "unit": "TFLOP/s",
                            "frac": gain_flops / kern_avg_s / 1e12 / fp32_peak,
                            "peak_source": "nominal (SM count x fp32 lanes x max clock)"}
        line = {
            "metric": metric_for(METRIC, wl), "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * total_s / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f32",
            "numerics": ("x bf16 (exact); state, gain recurrence, gates and step control "
                         "fp32; tensor-core products on three bf16 pieces per fp32 operand "
                         "(24 significant bits), fp32 accumulate"),
            "data": "synthetic", "config": workload_config(wl, args),
            "roofline": roof,
            "e2e": {"value": e2e_value, "unit": UNIT,
                    "h2d_bytes_per_step": int(x_host.numel() * x_host.element_size()),
                    "d2h_bytes_per_step": int(out.numel() * 4), "steps": e2e_steps,
                    "copies": "every step, double-buffered against neighbouring steps"},
            "gpu_launches": args.steps * (2 if args.readout == "outer" else 1),
            "clocks": sampler.summary(t0, t1) if sampler else None,
        }
        if world == 1 and not args.no_cpu_baseline:
            cpu_images = args.cpu_images or oracle_images(wl)
            cores = min(cpu_cores(), cpu_images * wl.nh)
            v, dt, passes = time_oracle(
                wl, cpu_images, cores, min_seconds=args.cpu_seconds,
                w_query=extra["w_query"].double().cpu().numpy() if extra else None,
                skip=extra["skip"].double().cpu().numpy() if extra else None)
            line["cpu_baseline"] = {
                "value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                "sample": f"{passes} pass(es) over {cpu_images} of {wl.B} images of the "
                          f"workload (all 4 routes x {wl.nh} heads), fp64, {dt:.1f} s wall"}
            # the same oracle on one host thread (one image, about 3 s)
            v1, dt1, passes1 = time_oracle(
                wl, 1, 1, min_seconds=3.0,
                w_query=extra["w_query"].double().cpu().numpy() if extra else None,
                skip=extra["skip"].double().cpu().numpy() if extra else None)
            line["cpu_baseline"]["single_thread"] = {
                "value": v1, "unit": UNIT, "cores": 1,
                "sample": f"{passes1} pass(es) over 1 image, fp64, {dt1:.1f} s wall"}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_backward(args, wl):
    """The backward call (vh_scan_backward): gradients of <dout, out> with respect to x and
    memories0, on the same synthetic inputs; one kernel launch per step."""
    import numpy as np
    import torch
    import visual_backbone_gb300 as vh
    from visual_backbone_gb300 import _build, synth

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 and not os.path.exists(vh.LIB_PATH):
        _build.build()
    if world > 1:
        torch.distributed.barrier()
    mine = vh.shard_images(wl.B * world, world, rank)  # this rank's images of the job
    inp = synth.make_inputs(wl, batch=len(mine), first_image=mine.start)
    if wl.dtype == "bf16":
        x_host = torch.from_numpy(inp.x_store.view("int16")).view(torch.bfloat16)
    else:
        x_host = torch.from_numpy(inp.x_store)
    dout_host = torch.from_numpy(
        np.random.default_rng(11 + rank).standard_normal((wl.B, wl.H, wl.W, wl.Cc)).astype(np.float32))
    x, dout = x_host.to(dev), dout_host.to(dev)
    mem0 = torch.from_numpy(inp.mem0).to(dev)
    dx = torch.empty((wl.B, wl.H, wl.W, wl.Cc), dtype=torch.float32, device=dev)
    dmem0 = torch.empty_like(mem0)
    ws = torch.empty(vh.backward_workspace_size(x, wl.d, chunk=wl.chunk), dtype=torch.uint8,
                     device=dev)
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev)
    params = vh.ScanParams(eta_bias=wl.eta_bias, alpha_init=wl.alpha_init, impl=args.kernel)
    stream = torch.cuda.Stream(device=dev)

    def call():
        vh.scan_backward(x, mem0, wl.d, dout, chunk=wl.chunk, params=params, dx=dx, dmem0=dmem0,
                         workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            call()
        torch.cuda.synchronize(dev)
        events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
                  for _ in range(args.steps)]
        sampler = ClockSampler(None).start() if rank == 0 else None
        time.sleep(0.3 if sampler else 0.0)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        t0 = time.time()
        for i in range(args.steps):
            flush.zero_()
            events[i][0].record(stream)
            call()
            events[i][1].record(stream)
        torch.cuda.synchronize(dev)
        t1 = time.time()
        if world > 1:
            torch.distributed.barrier()
        if sampler:
            time.sleep(0.3)
            sampler.stop()
    step_ms = [e[0].elapsed_time(e[1]) for e in events]
    total_s, = max_over_ranks([sum(step_ms) / 1e3], device=dev)
    avg_s = total_s / args.steps
    value = job_throughput(wl.tokens, args.steps, world, total_s)

    x_pin, dout_pin = x_host.pin_memory(), dout_host.pin_memory()
    xs, douts = [x, torch.empty_like(x)], [dout, torch.empty_like(dout)]
    dxs, dms = [dx, torch.empty_like(dx)], [dmem0, torch.empty_like(dmem0)]
    dx_pins = [torch.empty(dx.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    dm_pins = [torch.empty(dmem0.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    e2e_steps = max(3, min(args.steps, 10))

    def up(i, k, st):
        with torch.cuda.stream(st):
            xs[k].copy_(x_pin, non_blocking=True)
            douts[k].copy_(dout_pin, non_blocking=True)

    def run(k, st):
        vh.scan_backward(xs[k], mem0, wl.d, douts[k], chunk=wl.chunk, params=params, dx=dxs[k],
                         dmem0=dms[k], workspace=ws, stream=st)

    def down(k, st):
        with torch.cuda.stream(st):
            dx_pins[k].copy_(dxs[k], non_blocking=True)
            dm_pins[k].copy_(dms[k], non_blocking=True)

    e2e_s, = max_over_ranks([pipelined_e2e(dev, e2e_steps, up, run, down)], device=dev)
    e2e_value = job_throughput(wl.tokens, e2e_steps, world, e2e_s)

    tc_ckpt = (wl.d == 32 and wl.dtype == "bf16" and wl.chunk == 0 and wl.Cc % 8 == 0
               and args.kernel != "simt")
    if rank == 0:
        flops = backward_cost(wl)
        achieved = flops / avg_s / 1e12
        roof = {"bound": "alu", "achieved": achieved, "peak": FP32_PEAK_TFLOPS,
                "unit": "TFLOP/s", "frac": achieved / FP32_PEAK_TFLOPS,
                "traffic": recorded_traffic(wl.name, "backward", KERNEL_SOURCES_BWD),
                "peak_source": "nominal fp32 FMA peak (152 SMs x 128 lanes x 2 x 2.07 GHz)",
                "flops_per_launch": flops, "kernel_ms": avg_s * 1e3,
                "workspace_bytes": int(ws.numel())}
        line = {
            "metric": metric_for(METRIC_BWD, wl), "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * avg_s,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "numerics": "fp32 on CUDA cores (x bf16 exact); gradients summed with atomics",
            "data": "synthetic", "config": workload_config(wl, args), "roofline": roof,
            "e2e": {"value": e2e_value, "unit": UNIT,
                    "h2d_bytes_per_step": int(x_host.numel() * x_host.element_size()
                                              + dout_host.numel() * 4),
                    "d2h_bytes_per_step": int(dx.numel() * 4 + dmem0.numel() * 4),
                    "steps": e2e_steps,
                    "copies": "every step, double-buffered against neighbouring steps"},
            # the backward kernel, after the tensor-core forward that writes the chunk
            # boundary states where it applies (d = 32, bf16, aligned chunks)
            "gpu_launches": args.steps * (2 if tc_ckpt else 1),
            "clocks": sampler.summary(t0, t1) if sampler else None,
        }
        if world == 1 and not args.no_cpu_baseline:
            v, dt, cores, passes = time_grad_oracle(wl, 1, min_seconds=10.0)
            line["cpu_baseline"] = {
                "value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                "sample": f"{passes} pass(es) over 1 of {wl.B} images (all 4 routes x {wl.nh} "
                          f"heads), fp64 gradient oracle, {dt:.1f} s wall"}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_block(args, wl):
    """One VisionHOPE block per step (vh_block_forward) on the workload's map with
    D = 2 D_m, synthetic weights; fp32 activations in HBM."""
    import numpy as np
    import torch
    import visual_backbone_gb300 as vh
    from visual_backbone_gb300 import _build, synth

    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 and not os.path.exists(vh.LIB_PATH):
        _build.build()
    if world > 1:
        torch.distributed.barrier()
    D, Dm, hidden = block_dims(wl)
    mine = vh.shard_images(wl.B * world, world, rank)  # this rank's images of the job
    inp = synth.make_block_inputs(len(mine), wl.H, wl.W, D, Dm, wl.d, wl.seed, first_image=mine.start)
    x_host = torch.from_numpy(inp["x"])
    x = x_host.to(dev)
    wts = {k: (torch.from_numpy(np.ascontiguousarray(a)).to(dev).to(torch.bfloat16)
               if k in synth.BLOCK_GEMM_WEIGHTS else torch.from_numpy(np.ascontiguousarray(a)).to(dev))
           for k, a in inp["weights"].items()}
    mem0 = torch.from_numpy(inp["mem0"]).to(dev)
    wq, skip, lam = (torch.from_numpy(inp[k]).to(dev) for k in ("w_query", "skip", "dir_scale"))
    out = torch.empty_like(x)
    ws = torch.empty(vh.block_workspace_size(x, wts, wl.d), dtype=torch.uint8, device=dev)
    flush = torch.empty(64 << 20, dtype=torch.float32, device=dev)
    params = vh.ScanParams(eta_bias=wl.eta_bias, alpha_init=wl.alpha_init, impl=args.kernel)
    stream = torch.cuda.Stream(device=dev)

    def call():
        vh.block_forward(x, mem0, wts, wl.d, params=params, w_query=wq, skip=skip,
                         dir_scale=lam, out=out, workspace=ws, stream=stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            call()
        torch.cuda.synchronize(dev)
        events = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
                  for _ in range(args.steps)]
        sampler = ClockSampler(None).start() if rank == 0 else None
        time.sleep(0.3 if sampler else 0.0)
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)
        t0 = time.time()
        for i in range(args.steps):
            flush.zero_()
            events[i][0].record(stream)
            call()
            events[i][1].record(stream)
        torch.cuda.synchronize(dev)
        t1 = time.time()
        if world > 1:
            torch.distributed.barrier()
        if sampler:
            time.sleep(0.3)
            sampler.stop()
    total_s, = max_over_ranks([sum(e[0].elapsed_time(e[1]) for e in events) / 1e3], device=dev)
    avg_s = total_s / args.steps
    value = job_throughput(wl.tokens, args.steps, world, total_s)
    x_pin = x_host.pin_memory()
    xs, outs = [x, torch.empty_like(x)], [out, torch.empty_like(out)]
    out_pins = [torch.empty(out.shape, dtype=torch.float32).pin_memory() for _ in range(2)]
    e2e_steps = max(3, min(args.steps, 20))

    def up(i, k, st):
        with torch.cuda.stream(st):
            xs[k].copy_(x_pin, non_blocking=True)

    def run(k, st):
        vh.block_forward(xs[k], mem0, wts, wl.d, params=params, w_query=wq, skip=skip,
                         dir_scale=lam, out=outs[k], workspace=ws, stream=st)

    def down(k, st):
        with torch.cuda.stream(st):
            out_pins[k].copy_(outs[k], non_blocking=True)

    e2e_s, = max_over_ranks([pipelined_e2e(dev, e2e_steps, up, run, down)], device=dev)
    e2e_value = job_throughput(wl.tokens, e2e_steps, world, e2e_s)
    if rank == 0:
        flops, gemm_flops = block_cost(wl)
        peaks, src = load_peaks()
        peak = float(peaks["bf16_tflops"])
        achieved = flops / avg_s / 1e12
        line = {
            "metric": METRIC_BLOCK, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * avg_s,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "numerics": ("GEMMs bf16 x bf16 -> fp32 accumulate; fp32 residual stream; the "
                         "operator as in the forward line"),
            "data": "synthetic (random weights)", "config": workload_config(wl, args),
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak,
                         "unit": "TFLOP/s", "frac": achieved / peak, "traffic": None,
                         "scope": "whole block call (GEMMs + operator)",
                         "peak_source": f"bf16 dense burst, {'of measured' if src == 'measured' else 'of fallback'}",
                         "flops_per_call": flops, "gemm_flops_per_call": gemm_flops},
            "e2e": {"value": e2e_value, "unit": UNIT,
                    "h2d_bytes_per_step": int(x_host.numel() * 4),
                    "d2h_bytes_per_step": int(out.numel() * 4), "steps": e2e_steps,
                    "copies": "every step, double-buffered against neighbouring steps"},
            # ours per call: CPE, LN1, Proj_in, gated depthwise, query projection, scan,
            # positional depthwise, Proj_out, LN2, FFN1 (+GELU), FFN2
            "gpu_launches": args.steps * 11,
            "clocks": sampler.summary(t0, t1) if sampler else None,
        }
        if world == 1 and not args.no_cpu_baseline:
            imgs = oracle_images(wl)
            v, dt, cores, passes = time_block_oracle(wl, imgs, min_seconds=10.0)
            line["cpu_baseline"] = {
                "value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
                "sample": f"{passes} pass(es) over {imgs} of {wl.B} images, fp64 block oracle, "
                          f"{dt:.1f} s wall"}
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="stage1")
    ap.add_argument("--variant", choices=["plain", "longmem"], default="plain")
    ap.add_argument("--kernel", choices=["auto", "simt", "tc", "tc_wy", "tc_recur", "tc_pipe"],
                    default="auto",
                    help="scan kernel: auto / tc (tensor core, its faster gain form), tc_wy or "
                         "tc_recur (tensor core with the WY or the blocked-recurrence gain, the "
                         "A/B pair at d = 32), tc_pipe (the recurrence with a line's sub-tiles "
                         "pipelined), simt (fp32 CUDA cores)")
    ap.add_argument("--chunk", type=int, default=-1,
                    help="chunk length for every route (the chunk-length ablation); default: "
                         "the workload's (rows / columns); a length that is not the row or "
                         "column length runs on the CUDA-core kernel")
    ap.add_argument("--readout", choices=["memory", "outer"], default="memory",
                    help="memory: six-memory form (q from M^q); outer: VisionHOPE-exact "
                         "readout with an outer query projection and channel-wise skip")
    ap.add_argument("--pass", dest="pass_", choices=["forward", "backward", "block"],
                    default="forward",
                    help="forward: the scan (default); backward: its outer gradients; "
                         "block: the VisionHOPE block around the operator")
    ap.add_argument("--memories-out", action="store_true",
                    help="forward: also write the final memories (the measurement's second row)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-images", type=int, default=0,
                    help="images in the oracle sample behind cpu_baseline (0: the fewest that "
                         "fill every host core equally, as the reference arm)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="minimum wall time of the oracle sample behind cpu_baseline")
    ap.add_argument("--ref-images", type=int, default=0,
                    help="images per step of the reference arm (0: forward and block, the "
                         "cpu_baseline sample; backward, one)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    from visual_backbone_gb300 import synth
    wl = synth.WORKLOADS[args.workload]
    if args.variant == "longmem":
        wl = wl.long_memory()
    if args.chunk >= 0:
        import dataclasses
        wl = dataclasses.replace(wl, chunk=args.chunk)
    if args.gpus != dist_env()[1] and args.impl == "ours":
        ap.error(f"--gpus {args.gpus} needs torchrun with {args.gpus} processes "
                 f"(WORLD_SIZE={dist_env()[1]})")
    if args.impl == "reference":
        return run_reference(args, wl)
    if args.pass_ == "backward":
        return run_backward(args, wl)
    if args.pass_ == "block":
        return run_block(args, wl)
    return run_ours(args, wl)


if __name__ == "__main__":
    sys.exit(main())
