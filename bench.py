"""Benchmark of the fused fp16 GEMM + ReLU hot path on GB300.

One step = one pass of the whole hot path over one batch of synthetic input:
  1. the fused kernel on M = N = K = 4096 (A, B ~ N(0,1)/sqrt(K)): tile
     rasteriser, TMA ring, tcgen05 MMA into TMEM, ReLU/fp16 epilogue, with
     the stream-K schedule for the partial last wave;
  2. the split-K kernel on M = 16, N = K = 8192 (N(0,1)/sqrt(K)), split 8:
     eight K pieces on CTA pairs, summed in fixed order through shared
     memory, then ReLU and fp16 (one kernel).
Metric: GEMM+ReLU TFLOP/s = total 2*M*N*K of the step / step time, the
steps run back to back on rotating copies of the operands (no L2 reuse
between launches).

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
Under torchrun (N > 1) every rank runs the same step on its own GPU
(independent replicas, weak scaling); rank 0 prints one JSON line.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# fp16 and bf16 dense tensor rates are the same on this architecture (2.25
# PFLOP/s nominal each), so the measured bf16 peak is the fp16 denominator.
FP16_PER_BF16 = 1.0
L2_FLUSH_BYTES = 512 << 20       # > 129 MB of L2, written before each cold launch
L2_CLEAN_BYTES = 256 << 20       # then read, so no dirty flush lines remain in L2
INPUT_SETS = 3                   # operand copies each part rotates through

METRIC = "GEMM+ReLU TFLOP/s (fp16 in, fp32 acc)"

# DRAM bytes (read + write) per launch from an ncu capture of the current
# kernels, keyed by (kind, M, N, K); a shape missing here reports null.
DRAM_BYTES_PER_LAUNCH = {
    # profiles/dram_traffic_bench_launches.md, first captured launch of each:
    # pair kernel with stream-K at 4096^3: 75,324,416 B read + 26,401,280 B written
    ("streamk", 4096, 4096, 4096): 101725696,
    # split-K CTA-pair form at 16x8192x8192, split 8: 134,542,592 B read + 101,120 B written
    ("splitk", 16, 8192, 8192): 134643712,
    # GEMV kernel at 1x8192x8192: 134,254,336 B read + 2,791,168 B written
    ("streamk", 1, 8192, 8192): 137045504,
}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ------------------------------------------------------------------ workload

STEP_NAME = ("square4096 fused (M=N=K=4096, N(0,1)/sqrt(K)) + skinny split-K "
             "(M=16, N=K=8192, N(0,1)/sqrt(K), split 8)")


def describe(w):
    dist = {"normal": "N(0,1)", "uniform": "U[-1,1]"}[w.dist] + ("/sqrt(K)" if w.scale_by_sqrt_k else "")
    s = f"{w.name} (M={w.M}, N={w.N}, K={w.K}, {dist}"
    return s + (f", split-K {w.split_k})" if w.split_k > 1 else ")")


def build_parts(args):
    """[(label, workload, kind)], description.  kind: 'streamk' (the fused
    kernel through gemm_relu_streamk, which runs plain data-parallel tiles when
    the schedule has no cut), 'fused' or 'splitk'."""
    from tiled_tensor_core_03_gb300 import inputs
    W = inputs.WORKLOADS
    if args.shape:
        M, N, K = (int(x) for x in args.shape.lower().split("x"))
        w = inputs.Workload("custom", M, N, K, "normal", True, 7, split_k=args.split)
        kind = "splitk" if args.split > 1 else ("fused" if args.no_streamk else "streamk")
        return [("custom", w, kind)], describe(w)
    if args.workload == "step":
        return [("fused_4096", W["square4096"], "streamk"),
                ("splitk_skinny", W["skinny"], "splitk")], STEP_NAME
    w = W[args.workload]
    kind = "splitk" if w.split_k > 1 else ("fused" if args.no_streamk else "streamk")
    return [(w.name, w, kind)], describe(w)


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms in the background."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.t_start = self.t_end = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", str(self.gpu_index)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.reader.join(timeout=5)

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append((t, parts))
        lo = (self.t_start or 0) - 0.15
        hi = (self.t_end or 1e30) + 0.15
        window = [r for r in rows if lo <= r[0] <= hi] or rows[-3:]
        sm = [float(p[2]) for _, p in window if p[2].replace(".", "").isdigit()]
        smax = [float(p[3]) for _, p in window if p[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, p in window for i in range(4)
                          if p[6 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(window)}


# ------------------------------------------------------------------ CPU oracle leg

def oracle_rows_sample(parts, host_inputs, budget_s, threads=None):
    """Time the CPU oracle, as it stands, on a bounded sample of the step:
    whole output rows of each part's problem, taken in proportion to the
    part's share of the step's FLOPs (at least one row of each), computed by
    `threads` host threads (default: every core; the oracle is a C library
    called through ctypes, which releases the GIL, and each row is computed
    independently with its own fixed order) until `budget_s` seconds of wall
    time have passed.  Returns (flops, seconds, threads, {label: (rows, output)})."""
    import oracle
    orc = oracle.Oracle()
    threads = threads or os.cpu_count() or 1
    total = sum(w.flops for _, w, _ in parts)
    next_row = {label: 0 for label, _, _ in parts}
    flops = {label: 0 for label, _, _ in parts}
    rows_out = {label: {} for label, _, _ in parts}
    lock = threading.Lock()
    t0 = time.perf_counter()

    def take():
        with lock:
            if time.perf_counter() - t0 >= budget_s and all(next_row[l] >= 1 for l in next_row):
                return None
            open_parts = [p for p in parts if next_row[p[0]] < p[1].M]
            if not open_parts:
                return None
            # the part furthest behind its share of the step's FLOPs
            label, w, _ = min(open_parts, key=lambda p: flops[p[0]] / (p[1].flops / total))
            r = next_row[label]
            next_row[label] += 1
            flops[label] += 2 * w.N * w.K
            return label, r

    def worker():
        while True:
            job = take()
            if job is None:
                return
            label, r = job
            A, B = host_inputs[label]
            rows_out[label][r] = orc.gemm_relu_f16_rows(A, B, r, 1)

    pool = [threading.Thread(target=worker) for _ in range(threads)]
    for t in pool:
        t.start()
    for t in pool:
        t.join()
    elapsed = time.perf_counter() - t0
    out = {}
    for label in next_row:
        n = next_row[label]
        out[label] = (n, np.concatenate([rows_out[label][r] for r in range(n)]) if n else None)
    return sum(flops.values()), elapsed, threads, out


# ------------------------------------------------------------------ distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value, world, device=None):
    """Max of a float over all ranks (identity when world == 1)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ------------------------------------------------------------------ reference arm

def run_reference(args, world, rank):
    """The reference arm: the CPU oracle as it stands, timed on the host, each
    step a bounded sample (whole output rows) of the same workload."""
    if rank != 0:
        return 0
    import multiprocessing
    from tiled_tensor_core_03_gb300 import inputs
    parts, name = build_parts(args)
    host_inputs = {label: inputs.make_workload(w) for label, w, _ in parts}
    budget = min(2.0, 150.0 / (args.steps + args.warmup))
    for _ in range(args.warmup):
        oracle_rows_sample(parts, host_inputs, budget * 0.25)
    flops, secs, threads = 0, 0.0, 1
    for _ in range(args.steps):
        f, dt, threads, _ = oracle_rows_sample(parts, host_inputs, budget)
        flops += f
        secs += dt
    value = flops / secs / 1e12
    line = {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": name, "parallelism": f"replicas{args.gpus}"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"per step, whole output rows of each problem in proportion "
                                   f"to its FLOP share, about {budget:.2f} s of wall time of the "
                                   f"fp64 C oracle on {threads} threads (one row each at a time); "
                                   f"host has {multiprocessing.cpu_count()} cores"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm

def run_ours(args, world, rank, local):
    import torch
    import tiled_tensor_core_03_gb300 as gr
    from tiled_tensor_core_03_gb300 import _build, inputs

    if _build.needs_build():
        _build.build()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)

    parts, name = build_parts(args)
    if args.kernel != "auto":
        # profiling aid: every GEMM call of this run takes the named kernel
        gr.gemm_relu_debug_force_kernel(KERNEL_CHOICES[args.kernel])
        name += f", kernel forced: {args.kernel}"
    host_inputs = {label: inputs.make_workload(w) for label, w, _ in parts}
    # INPUT_SETS device copies of each part's operands (and outputs): the
    # back-to-back timed loop rotates through them, so a launch never finds
    # its operands in L2 -- they were last touched INPUT_SETS steps earlier,
    # with every other part's traffic in between.
    dev = {}
    for label, w, kind in parts:
        A, B = host_inputs[label]
        sets = []
        for _ in range(INPUT_SETS):
            a = torch.from_numpy(A).to(device)
            b = torch.from_numpy(B).to(device)
            c = torch.empty((w.M, w.N), dtype=torch.float16, device=device)
            ws = (gr.splitk_workspace(w.M, w.N, w.K, w.split_k, device) if kind == "splitk" else
                  gr.streamk_workspace(w.M, w.N, w.K, device) if kind == "streamk" else None)
            sets.append((a, b, c, ws))
        dev[label] = sets
    set_bytes = sum(w.bytes for _, w, _ in parts)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    clean = torch.ones(L2_CLEAN_BYTES, dtype=torch.uint8, device=device)

    def flush_l2():
        # Writing a buffer larger than L2 evicts the operands but leaves L2
        # full of dirty lines, whose write-back would then be charged to the
        # next timed kernel; reading a second large buffer evicts those too,
        # so each timed step starts from a cold, clean L2.
        flush.zero_()
        torch.amax(clean)            # a plain uint8 read: no temporary is written
    stream = torch.cuda.current_stream(device)

    def launch(label, w, kind, r=0):
        a, b, c, ws = dev[label][r]
        if kind == "splitk":
            gr.gemm_relu_splitk(a, b, w.split_k, out=c, workspace=ws, stream=stream)
        elif kind == "streamk":
            gr.gemm_relu_streamk(a, b, out=c, workspace=ws, stream=stream)
        else:
            gr.gemm_relu(a, b, out=c, stream=stream)

    for i in range(args.warmup):
        for p in parts:
            flush_l2()
            launch(*p, r=i % INPUT_SETS)
    torch.cuda.synchronize(device)
    st = gr.status(stream)
    if st != gr.OK:
        raise RuntimeError(f"device status after warm-up: {gr.strerror(st)}")

    # ---- timed region: K steps back to back, each part on the next input set;
    # events only at the two ends (an event recorded between two launches
    # serialises them and would add its own cost to the step)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    e_start = torch.cuda.Event(enable_timing=True)
    e_end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(device)
    sampler.mark("t_start")
    wall0 = time.perf_counter()
    e_start.record(stream)
    for i in range(args.steps):
        for p in parts:
            launch(*p, r=i % INPUT_SETS)
    e_end.record(stream)
    torch.cuda.synchronize(device)
    wall1 = time.perf_counter()
    sampler.mark("t_end")
    barrier(world)
    sampler.stop()
    st = gr.status(stream)
    if st != gr.OK:
        raise RuntimeError(f"device status after timed steps: {gr.strerror(st)}")
    step_ms = max_over_ranks(e_start.elapsed_time(e_end) / args.steps, world, device)
    flops_step = sum(w.flops for _, w, _ in parts)
    value = world * flops_step / (step_ms * 1e-3) / 1e12

    # ---- each part alone: K launches back to back on rotating input sets,
    # events at both ends -> the kernel's average launch duration
    part_ms = {}
    for p in parts:
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        p0.record(stream)
        for i in range(args.steps):
            launch(*p, r=i % INPUT_SETS)
        p1.record(stream)
        torch.cuda.synchronize(device)
        part_ms[p[0]] = [p0.elapsed_time(p1) / args.steps]
    # ---- warm: each part alone, back to back on the same operands (L2 may
    # hold them: the 4096^3 operands fit, the skinny B is about L2's size)
    warm_ms = {}
    for p in parts:
        p0 = torch.cuda.Event(enable_timing=True)
        p1 = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        p0.record(stream)
        for i in range(args.steps):
            launch(*p)
        p1.record(stream)
        torch.cuda.synchronize(device)
        warm_ms[p[0]] = p0.elapsed_time(p1) / args.steps
    st = gr.status(stream)
    if st != gr.OK:
        raise RuntimeError(f"device status after the per-part loops: {gr.strerror(st)}")

    # ---- cold launches: L2 flushed before each, events around each alone
    cold = [[torch.cuda.Event(enable_timing=True) for _ in range(2 * len(parts))]
            for _ in range(args.steps)]
    torch.cuda.synchronize(device)
    for i in range(args.steps):
        for j, p in enumerate(parts):
            flush_l2()                   # outside the events
            cold[i][2 * j].record(stream)
            launch(*p)
            cold[i][2 * j + 1].record(stream)
    torch.cuda.synchronize(device)
    cold_ms = {label: [cold[i][2 * j].elapsed_time(cold[i][2 * j + 1]) for i in range(args.steps)]
               for j, (label, _, _) in enumerate(parts)}
    st = gr.status(stream)
    if st != gr.OK:
        raise RuntimeError(f"device status after cold launches: {gr.strerror(st)}")

    # ---- end to end through the public API, host buffers in pinned memory
    pinned = {}
    for label, w, _ in parts:
        A, B = host_inputs[label]
        pinned[label] = (torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory(),
                         torch.empty((w.M, w.N), dtype=torch.float16).pin_memory())

    # Uploads run on their own stream, the kernels on `stream`, read-backs on
    # a third: each step still moves all of its inputs up and its result down
    # inside the timed region, while the copy engines and the kernels of
    # neighbouring parts overlap.  Step i uses device set i % INPUT_SETS, and
    # its upload waits until that set's previous kernel and read-back are done.
    up_stream = torch.cuda.Stream(device)
    down_stream = torch.cuda.Stream(device)
    set_free = {}

    def e2e_step(i):
        r = i % INPUT_SETS
        for label, w, kind in parts:
            hA, hB, hC = pinned[label]
            a, b, c, _ = dev[label][r]
            if (label, r) in set_free:
                up_stream.wait_event(set_free[(label, r)])
            with torch.cuda.stream(up_stream):
                a.copy_(hA, non_blocking=True)
                b.copy_(hB, non_blocking=True)
            uploaded = torch.cuda.Event()
            uploaded.record(up_stream)
            stream.wait_event(uploaded)
            launch(label, w, kind, r=r)
            computed = torch.cuda.Event()
            computed.record(stream)
            down_stream.wait_event(computed)
            with torch.cuda.stream(down_stream):
                hC.copy_(c, non_blocking=True)
            done = torch.cuda.Event()
            done.record(down_stream)
            set_free[(label, r)] = done

    def e2e_run(n, x0=None, x1=None):
        if x0 is not None:
            x0.record(stream)
            up_stream.wait_event(x0)
        for i in range(n):
            e2e_step(i)
        for ev in set_free.values():          # every read-back inside the region
            stream.wait_event(ev)
        if x1 is not None:
            x1.record(stream)

    e2e_run(args.warmup)
    torch.cuda.synchronize(device)
    barrier(world)
    x0 = torch.cuda.Event(enable_timing=True)
    x1 = torch.cuda.Event(enable_timing=True)
    e2e_run(args.steps, x0, x1)
    torch.cuda.synchronize(device)
    e2e_ms = max_over_ranks(x0.elapsed_time(x1) / args.steps, world, device)
    barrier(world)
    h2d = sum(2 * (w.M * w.K + w.K * w.N) for _, w, _ in parts)
    d2h = sum(2 * w.M * w.N for _, w, _ in parts)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank != 0:
        return 0

    peaks, peaks_src = load_peaks()
    tensor_peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]) * FP16_PER_BF16
    tensor_peak_sustained = peaks.get("bf16_tflops_sustained",
                                      FALLBACK_PEAKS["bf16_tflops_sustained"]) * FP16_PER_BF16
    hbm_peak = peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
    ridge = tensor_peak * 1e12 / (hbm_peak * 1e9)

    def split_form(w):
        one = gr.gemm_relu_f16_splitk_workspace_bytes(w.M, w.N, w.K, w.split_k) == 0
        return ("CTA-pair form: one kernel, pieces summed in shared memory" if one else
                "two-stage form: partial kernel + reduce kernel"), (1 if one else 2)

    def roofline(label, w, kind, times):
        ms = statistics.mean(times[label])
        kernel = (f"gemm_relu_f16_splitk {w.M}x{w.N}x{w.K} split {w.split_k} ({split_form(w)[0]})"
                  if kind == "splitk" else
                  (f"gemm_relu_f16_streamk {w.M}x{w.N}x{w.K} (CTA-pair or single-CTA fused kernel, "
                   f"as the library selects; stream-K schedule when the tiles leave a partial wave)"
                   if kind == "streamk" and w.M > 4 else
                   f"gemm_relu_f16 {w.M}x{w.N}x{w.K} (GEMV kernel, M <= 4)" if w.M <= 4 else
                   f"gemm_relu_f16 {w.M}x{w.N}x{w.K}"))
        if w.flops / w.bytes >= ridge:
            ach = w.flops / (ms * 1e-3) / 1e12
            return {"bound": "tensor", "kernel": kernel, "achieved": ach, "peak": tensor_peak,
                    "unit": "TFLOP/s", "frac": ach / tensor_peak, "ms": ms,
                    "frac_of_sustained": ach / tensor_peak_sustained,
                    "algorithmic_flops": w.flops,
                    "peak_source": f"{peaks_src} bf16_tflops (burst) x {FP16_PER_BF16} (fp16/bf16)",
                    "traffic": DRAM_BYTES_PER_LAUNCH.get((kind, w.M, w.N, w.K))}
        ach = w.bytes / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "kernel": kernel, "achieved": ach, "peak": hbm_peak,
                "unit": "GB/s", "frac": ach / hbm_peak, "ms": ms, "algorithmic_bytes": w.bytes,
                "peak_source": f"{peaks_src} hbm_gbs",
                "traffic": DRAM_BYTES_PER_LAUNCH.get((kind, w.M, w.N, w.K))}

    roofs = {label: roofline(label, w, kind, part_ms) for label, w, kind in parts}
    cold_roofs = {label: roofline(label, w, kind, cold_ms) for label, w, kind in parts}
    dominant = max(parts, key=lambda p: sum(part_ms[p[0]]))[0]
    line = {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f16",
        "data": "synthetic",
        "config": {
            "workload": name,
            "flops_per_step": flops_step,
            "parallelism": f"replicas{world}",
            "l2": (f"inputs larger than L2: every part rotates through {INPUT_SETS} device "
                   f"copies of its operands ({INPUT_SETS} x {set_bytes / 2**20:.0f} MiB per step "
                   f"in all), so each launch's A and B were last touched {INPUT_SETS} steps "
                   f"earlier, behind {(INPUT_SETS - 1) * set_bytes / 2**20:.0f} MiB of other "
                   f"traffic; no flush inside the timed region. cold_launch: flushed before "
                   f"every launch by a {L2_FLUSH_BYTES >> 20} MiB write and a "
                   f"{L2_CLEAN_BYTES >> 20} MiB read of other buffers"),
            "timing": "steps back to back on one stream, each kernel launched with "
                      "programmatic stream serialisation; value and ms_per_step from CUDA "
                      "events at the two ends of the timed region only; parts (and roofline): "
                      "each part alone, K launches back to back on the rotating input sets, "
                      "events at both ends; cold_launch: L2 flushed, events around each "
                      "launch alone (includes the launch latency an idle GPU pays)",
        },
        "roofline": roofs[dominant],
        "parts": {label: {"ms": statistics.mean(part_ms[label]),
                          "tflops": w.flops / (statistics.mean(part_ms[label]) * 1e-3) / 1e12,
                          "gbs": w.bytes / (statistics.mean(part_ms[label]) * 1e-3) / 1e9,
                          "roofline": roofs[label]}
                  for label, w, _ in parts},
        "cold_launch": {label: {"ms": statistics.mean(cold_ms[label]),
                                "tflops": w.flops / (statistics.mean(cold_ms[label]) * 1e-3) / 1e12,
                                "gbs": w.bytes / (statistics.mean(cold_ms[label]) * 1e-3) / 1e9,
                                "frac": cold_roofs[label]["frac"],
                                "bound": cold_roofs[label]["bound"]}
                        for label, w, _ in parts},
        "warm_launch": {label: {"ms": warm_ms[label],
                                "tflops": w.flops / (warm_ms[label] * 1e-3) / 1e12,
                                "gbs": w.bytes / (warm_ms[label] * 1e-3) / 1e9}
                        for label, w, _ in parts},
        "wall_ms_per_step": 1e3 * (wall1 - wall0) / args.steps,
        "e2e": {"value": world * flops_step / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "api": "tiled_tensor_core_03_gb300.gemm_relu_streamk / gemm_relu_splitk from pinned host "
                       "buffers; uploads, kernels and read-backs on three streams, overlapping "
                       "across parts and steps"},
        # this library's kernels in the timed region: the fused kernel once,
        # split-K once (CTA-pair form) or twice (partial + reduce)
        "gpu_launches": sum(split_form(w)[1] if kind == "splitk" else 1
                            for _, w, kind in parts) * args.steps,
        "clocks": sampler.summary(),
    }

    if world == 1 and not args.no_cpu_baseline:
        import multiprocessing
        f, dt, threads, outs = oracle_rows_sample(parts, host_inputs, args.cpu_budget)
        err = 0.0
        for label, (rows, want) in outs.items():
            if rows:
                got = dev[label][0][2][:rows].cpu().numpy().astype(np.float64)
                err = max(err, float(np.abs(got - want.astype(np.float64)).max()))
        desc = ", ".join(f"first {rows} rows of {label}" for label, (rows, _) in outs.items())
        line["cpu_baseline"] = {
            "value": f / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{desc} ({f / 1e9:.2f} GFLOP in {dt:.1f} s of wall time), fp64 C oracle "
                      f"on {threads} threads, one output row each at a time; host has "
                      f"{multiprocessing.cpu_count()} cores",
            "max_abs_err_vs_gpu_on_sample": err,
        }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ attention forward

ATTN_SHAPES = {"attn": (4, 4096, 32, 128, False), "attn_causal": (4, 4096, 32, 128, True)}
# profiles/dram_traffic_bench_launches.md, first captured launch of each attention workload
# (batch, seq, heads, d, causal): DRAM bytes read + written
ATTN_DRAM_BYTES_PER_LAUNCH = {
    (4, 4096, 32, 128, False): 402995712 + 113100800,
    (4, 4096, 32, 128, True): 402901504 + 114983936,
}


ATTN_METRIC = "attention forward TFLOP/s (fp16 in, fp32 acc)"
# --kernel: the library's debug hook that pins the GEMM kernel (0 = its own choice)
KERNEL_CHOICES = {"auto": 0, "one_cta_256": 1, "one_cta_128": 2, "pair": 3, "gemv": 4}


def attn_workload_name(workload, b, s, h, d, causal):
    return (f"{workload} (batch {b}, seq {s}, heads {h}, d {d}, "
            f"{'causal' if causal else 'non-causal'}, bshd fp16, N(0,1))")


def attn_shape(args):
    b, s, h, d, causal = ATTN_SHAPES[args.workload]
    if args.attn_shape:
        b, s, h, d = (int(x) for x in args.attn_shape.split(","))
    return b, s, h, d, causal


def attn_host_inputs(b, s, h, d):
    """Seeded Q, K, V (standard normal, fp16) of the attention workloads."""
    rng = np.random.default_rng(6)
    return [rng.standard_normal((b, s, h, d), dtype=np.float32).astype(np.float16) for _ in range(3)]


def attn_oracle_sample(Q, K, V, causal, budget_s, threads=None):
    """The attention oracle as it stands on whole output rows (batch, head,
    query row), taken in a fixed order by `threads` host threads until
    `budget_s` of wall time has passed.  Returns (flops, seconds, threads,
    {(b, h, row): fp16 row})."""
    import oracle
    orc = oracle.Oracle()
    b, s, h, d = Q.shape
    lock = threading.Lock()
    state = {"next": 0, "flops": 0}
    rows_out = {}
    threads = threads or os.cpu_count() or 1
    t0 = time.perf_counter()

    def worker():
        while True:
            with lock:
                if time.perf_counter() - t0 >= budget_s and state["next"] > 0:
                    return
                idx = state["next"]
                state["next"] += 1
            bb, hh, r = (idx // s) % b, (idx // (s * b)) % h, idx % s
            out = orc.attention_f16_rows(Q, K, V, causal, bb, hh, r, 1)
            with lock:
                state["flops"] += 4 * d * ((r + 1) if causal else s)
                rows_out[(bb, hh, r)] = out
    pool = [threading.Thread(target=worker) for _ in range(threads)]
    for t in pool:
        t.start()
    for t in pool:
        t.join()
    return state["flops"], time.perf_counter() - t0, threads, rows_out


def run_reference_attention(args, world, rank):
    """The reference arm for the attention workloads: the attention oracle as
    it stands, each step a bounded sample of whole output rows."""
    if rank != 0:
        return 0
    import multiprocessing
    b, s, h, d, causal = attn_shape(args)
    Q, K, V = attn_host_inputs(b, s, h, d)
    budget = min(2.0, 150.0 / (args.steps + args.warmup))
    for _ in range(args.warmup):
        attn_oracle_sample(Q, K, V, causal, budget * 0.25)
    flops, secs, threads = 0, 0.0, 1
    for _ in range(args.steps):
        f, dt, threads, _ = attn_oracle_sample(Q, K, V, causal, budget)
        flops += f
        secs += dt
    value = flops / secs / 1e12
    line = {
        "impl": "reference",
        "metric": ATTN_METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": attn_workload_name(args.workload, b, s, h, d, causal),
                   "parallelism": f"replicas{args.gpus}"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": f"per step, whole output rows (batch, head, query row) for "
                                   f"about {budget:.2f} s of wall time of the fp64 C attention "
                                   f"oracle on {threads} threads; host has "
                                   f"{multiprocessing.cpu_count()} cores"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def attn_flops(b, s, h, d, causal):
    """2 d multiply-adds for Q K^T and 2 d for P V per visible (query, key) pair."""
    pairs = s * (s + 1) // 2 if causal else s * s
    return 4 * b * h * d * pairs


def run_attention(args, world, rank, local):
    """Attention forward (flash_attention_f16) on [batch, seq, heads, d] fp16:
    K launches back to back on rotating input copies, events at both ends."""
    import multiprocessing
    import torch
    import tiled_tensor_core_03_gb300 as gr
    from tiled_tensor_core_03_gb300 import _build

    if _build.needs_build():
        _build.build()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    b, s, h, d, causal = attn_shape(args)
    host = attn_host_inputs(b, s, h, d)
    sets = [[torch.from_numpy(x).to(device) for x in host] + [torch.empty((b, s, h, d), dtype=torch.float16, device=device)]
            for _ in range(INPUT_SETS)]
    stream = torch.cuda.current_stream(device)

    def launch(r):
        q, k, v, o = sets[r]
        gr.flash_attention(q, k, v, causal=causal, out=o, stream=stream)

    for i in range(args.warmup):
        launch(i % INPUT_SETS)
    torch.cuda.synchronize(device)
    if gr.status(stream) != gr.OK:
        raise RuntimeError("device status after warm-up")
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(device)
    sampler.mark("t_start")
    e0.record(stream)
    for i in range(args.steps):
        launch(i % INPUT_SETS)
    e1.record(stream)
    torch.cuda.synchronize(device)
    sampler.mark("t_end")
    barrier(world)
    sampler.stop()
    if gr.status(stream) != gr.OK:
        raise RuntimeError("device status after timed steps")
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, device)
    flops = attn_flops(b, s, h, d, causal)
    value = world * flops / (ms * 1e-3) / 1e12
    # cold single launches after an L2 flush
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    clean = torch.ones(L2_CLEAN_BYTES, dtype=torch.uint8, device=device)
    cold = []
    for i in range(max(3, args.steps // 5)):
        flush.zero_()
        torch.amax(clean)
        c0 = torch.cuda.Event(enable_timing=True)
        c1 = torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        launch(0)
        c1.record(stream)
        torch.cuda.synchronize(device)
        cold.append(c0.elapsed_time(c1))
    # end to end: inputs from pinned host memory, the output back
    pinned = [torch.from_numpy(x).pin_memory() for x in host]
    hout = torch.empty((b, s, h, d), dtype=torch.float16).pin_memory()

    # uploads, the kernel and the read-back on three streams (as in the GEMM
    # bench): step i uses device set i % INPUT_SETS once its previous kernel
    # and read-back are done
    up_stream = torch.cuda.Stream(device)
    down_stream = torch.cuda.Stream(device)
    set_free = {}

    def e2e_step(i):
        r = i % INPUT_SETS
        q, k, v, o = sets[r]
        if r in set_free:
            up_stream.wait_event(set_free[r])
        with torch.cuda.stream(up_stream):
            for dst, src in zip((q, k, v), pinned):
                dst.copy_(src, non_blocking=True)
        uploaded = torch.cuda.Event()
        uploaded.record(up_stream)
        stream.wait_event(uploaded)
        gr.flash_attention(q, k, v, causal=causal, out=o, stream=stream)
        computed = torch.cuda.Event()
        computed.record(stream)
        down_stream.wait_event(computed)
        with torch.cuda.stream(down_stream):
            hout.copy_(o, non_blocking=True)
        done = torch.cuda.Event()
        done.record(down_stream)
        set_free[r] = done

    def e2e_run(n, x0=None, x1=None):
        if x0 is not None:
            x0.record(stream)
            up_stream.wait_event(x0)
        for i in range(n):
            e2e_step(i)
        for ev in set_free.values():
            stream.wait_event(ev)
        if x1 is not None:
            x1.record(stream)

    e2e_run(args.warmup)
    torch.cuda.synchronize(device)
    x0 = torch.cuda.Event(enable_timing=True)
    x1 = torch.cuda.Event(enable_timing=True)
    e2e_run(args.steps, x0, x1)
    torch.cuda.synchronize(device)
    e2e_ms = max_over_ranks(x0.elapsed_time(x1) / args.steps, world, device)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank != 0:
        return 0
    peaks, peaks_src = load_peaks()
    peak = peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]) * FP16_PER_BF16
    peak_sus = peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]) * FP16_PER_BF16
    name = attn_workload_name(args.workload, b, s, h, d, causal)
    line = {
        "metric": ATTN_METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": name, "flops_per_step": flops, "parallelism": f"replicas{world}",
                   "l2": f"inputs larger than L2: {INPUT_SETS} rotating copies of Q, K, V "
                         f"({3 * b * s * h * d * 2 / 2**20:.0f} MiB each set)",
                   "timing": "launches back to back, CUDA events at the two ends"},
        "roofline": {"bound": "tensor", "kernel": f"flash_attention_fwd_kernel<{d}>",
                     "achieved": value / world, "peak": peak, "unit": "TFLOP/s",
                     "frac": value / world / peak, "frac_of_sustained": value / world / peak_sus,
                     "ms": ms, "algorithmic_flops": flops,
                     "peak_source": f"{peaks_src} bf16_tflops (burst) x {FP16_PER_BF16} (fp16/bf16)",
                     "traffic": ATTN_DRAM_BYTES_PER_LAUNCH.get((b, s, h, d, bool(causal)))},
        "cold_launch": {"ms": statistics.mean(cold),
                        "tflops": flops / (statistics.mean(cold) * 1e-3) / 1e12},
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": 3 * b * s * h * d * 2,
                "d2h_bytes_per_step": b * s * h * d * 2,
                "api": "tiled_tensor_core_03_gb300.flash_attention from pinned host buffers; uploads, "
                       "kernel and read-back on three streams, overlapping across steps"},
        "gpu_launches": args.steps,
        "clocks": sampler.summary(),
    }
    if world == 1 and not args.no_cpu_baseline:
        Q, K, V = host
        flops_s, dt, threads, rows_out = attn_oracle_sample(Q, K, V, causal, args.cpu_budget)
        state = {"flops": flops_s}
        got = sets[0][3].cpu().numpy()
        err = max(float(np.abs(got[bb, r, hh].astype(np.float64) - o[0].astype(np.float64)).max())
                  for (bb, hh, r), o in rows_out.items())
        line["cpu_baseline"] = {
            "value": state["flops"] / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(rows_out)} output rows of the workload ({state['flops'] / 1e9:.2f} GFLOP "
                      f"in {dt:.1f} s of wall time), fp64 C oracle on {threads} threads; host has "
                      f"{multiprocessing.cpu_count()} cores",
            "max_abs_err_vs_gpu_on_sample": err,
        }
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of wall time for the cpu_baseline sample")
    ap.add_argument("--workload", default="step",
                    choices=["step", "square256", "square1024", "ragged", "square4096", "skinny",
                             "decode1", "attn", "attn_causal"])
    ap.add_argument("--shape", default=None, help="MxNxK: one custom fused (or split) GEMM")
    ap.add_argument("--split", type=int, default=1, help="split-K for --shape")
    ap.add_argument("--attn-shape", default=None,
                    help="batch,seq,heads,d for --workload attn / attn_causal")
    ap.add_argument("--kernel", default="auto", choices=sorted(KERNEL_CHOICES),
                    help="pin the GEMM kernel (a profiling aid; default: the library's choice)")
    ap.add_argument("--no-streamk", action="store_true",
                    help="time the plain data-parallel fused kernel instead of the stream-K call")
    args = ap.parse_args(argv)
    args.warmup = max(3, args.warmup)          # at least 3 untimed warm-up steps
    world, rank, local = dist_env()
    if args.workload in ATTN_SHAPES:
        if args.impl == "reference":
            return run_reference_attention(args, world, rank)
        return run_attention(args, world, rank, local)
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_ours(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
