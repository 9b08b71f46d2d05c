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

The default run also measures, each in its own sub-object of the same JSON
line: the other GEMM workloads (256^3, 1024^3, ragged 1537x1023x777 on the
predicated-load path, and the 1 x 8192 x 8192 decode row on the GEMV path)
and the attention forward (non-causal and causal), each with its roofline,
end-to-end time, CPU-oracle baseline and a parity check against the oracle.

Usage:  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
                        [--workload NAME] [--no-extra]
Under torchrun (N > 1) every rank runs the same step on its own GPU
(independent replicas, weak scaling); rank 0 prints one JSON line.
"""
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

import numpy as np  # noqa: E402

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# fp16 and bf16 dense tensor rates are the same on this architecture (2.25
# PFLOP/s nominal each), so the measured bf16 peak is the fp16 denominator.
FP16_PER_BF16 = 1.0
L2_FLUSH_BYTES = 512 << 20       # > 129 MB of L2, written before each cold launch
L2_CLEAN_BYTES = 256 << 20       # then read, so no dirty flush lines remain in L2
INPUT_SETS = 3                   # operand copies each headline part rotates through
ROTATE_BYTES = 256 << 20         # small workloads rotate through at least this many operand bytes
PART_LOOP_S = 1.0                # per-part loops run at least this long (clock samples)
HOLD_S = 2e-3                    # GPU-side hold before a timed region (the host queues ahead)
COOL_S = 0.5                     # idle before each per-part measurement
SOAK_S = 1.2                     # clock soak of the step

METRIC = "GEMM+ReLU TFLOP/s (fp16 in, fp32 acc)"
ATTN_METRIC = "attention forward TFLOP/s (fp16 in, fp32 acc)"
EXTRA_CONFIGS = ("square256", "square1024", "ragged", "decode1")
# --kernel: the library's debug hook that pins the GEMM kernel (0 = its own choice)
KERNEL_CHOICES = {"auto": 0, "one_cta_256": 1, "one_cta_128": 2, "pair": 3, "gemv": 4}

# ------------------------------------------------------------------ DRAM traffic

KERNEL_SOURCES = ("gemm_relu_api.cu", "gemm_relu_kernels.cuh", "gemm_relu_splitk.cuh",
                  "gemm_relu_2sm.cuh", "gemm_relu_gemv.cuh", "flash_attention.cuh", "sm103.cuh",
                  "gemm_relu_stage.cuh")


def kernel_source_hash():
    """First 16 hex digits of the SHA-256 of the CUDA sources (in a fixed order)."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "tiled_tensor_core_03_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one launch of
# each benchmarked kernel, from one-pass ncu captures on a GB300 of
#   ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum,gpu__time_duration.sum
#       --clock-control none -k regex:"gemm_relu_pair|splitk" -s 6 -c 6 --csv
#       python bench.py --steps 3 --warmup 3 --no-cpu-baseline --no-extra
# and the same with -k regex:gemm_relu (gemv, flash; "gemm_relu|stage_rows")
# -s 3 (6) -c 3 (6) and --workload square256 / square1024 (decode1; attn,
# attn_causal; ragged), each run after the same command had exited 0 without
# ncu, on the sources whose kernel_source_hash() is `source_hash`.  Launches
# inside the CUDA graphs of the small workloads leave C in L2 (write 0 in the
# launch).  The ragged workload's figure is its GEMM launch; the copy kernel
# before it moves another 3,990,955 bytes (A and B read once).  When the
# sources differ, the figures no longer describe the kernels that run and the
# bench reports null with the reason.
TRAFFIC_CAPTURE = {
    "source_hash": "d3deb7525379ddee",
    # mean of three captured launches each (read + write)
    "bytes": {
        ('streamk', 4096, 4096, 4096): 109_389_653,
        ('splitk', 16, 8192, 8192): 134_635_691,
        ('fused', 256, 256, 256): 314_880,
        ('fused', 1024, 1024, 1024): 4_247_125,
        ('fused', 1537, 1023, 777): 4_057_088,
        ('fused', 1, 8192, 8192): 135_278_933,
        ('attn', 4, 4096, 32, 128, False): 514_283_947,
        ('attn', 4, 4096, 32, 128, True): 516_312_491,
    },
}


def traffic_for(key):
    """(bytes per launch or None, note) for a (kind, M, N, K) or attention key."""
    cap = TRAFFIC_CAPTURE
    if cap["source_hash"] is None:
        return None, "no ncu capture of the current kernels"
    cur = kernel_source_hash()
    if cur != cap["source_hash"]:
        return None, (f"kernel sources changed since the capture (captured on {cap['source_hash']}, "
                      f"running {cur})")
    if key not in cap["bytes"]:
        return None, "shape not in the capture"
    return cap["bytes"][key], f"ncu capture on sources {cur}"


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

    def summary(self, t0=None, t1=None):
        """Median SM clock, max clock and throttle reasons of the samples taken
        between t0 and t1 (default: the marked timed region)."""
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        rows = []
        for t, line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            rows.append((t, parts))
        t0 = self.t_start if t0 is None else t0
        t1 = self.t_end if t1 is None else t1
        lo = (t0 or 0) - 0.15
        hi = (t1 or 1e30) + 0.15
        window = [r for r in rows if lo <= r[0] <= hi] or rows[-3:]
        sm = [float(p[2]) for _, p in window if p[2].replace(".", "").isdigit()]
        smax = [float(p[3]) for _, p in window if p[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, p in window for i in range(4)
                          if p[6 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(window)}


# ------------------------------------------------------------------ CPU oracle legs

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


def oracle_gemm_rows(A, B, budget_s, threads):
    """The oracle on whole output rows of one problem, rows taken in order by
    `threads` host threads until every row is done or `budget_s` of wall time
    has passed.  Returns (rows done, fp16 rows, flops, seconds)."""
    import oracle
    orc = oracle.Oracle()
    M, K = A.shape
    N = B.shape[1]
    lock = threading.Lock()
    state = {"next": 0}
    out = {}
    t0 = time.perf_counter()

    def worker():
        while True:
            with lock:
                if state["next"] >= M or (state["next"] > 0 and time.perf_counter() - t0 >= budget_s):
                    return
                r = state["next"]
                state["next"] += 1
            out[r] = orc.gemm_relu_f16_rows(A, B, r, 1)
    pool = [threading.Thread(target=worker) for _ in range(threads)]
    for t in pool:
        t.start()
    for t in pool:
        t.join()
    dt = time.perf_counter() - t0
    n = state["next"]
    return n, np.concatenate([out[r] for r in range(n)]), 2 * n * N * K, dt


def contract_check(got, want):
    """The parity contract (|g - o| <= 1e-2 + 1e-2 |o| per element) on fp16 arrays."""
    g = np.asarray(got, dtype=np.float16).astype(np.float64)
    o = np.asarray(want, dtype=np.float16).astype(np.float64)
    err = np.abs(g - o)
    nz = o != 0
    return {"elements": int(o.size), "max_abs_err": float(err.max()) if err.size else 0.0,
            "max_rel_err": float((err[nz] / np.abs(o[nz])).max()) if nz.any() else 0.0,
            "contract_ok": bool((err <= 1e-2 + 1e-2 * np.abs(o)).all()),
            "tolerance": "atol = rtol = 1e-2 per element"}


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


# ------------------------------------------------------------------ attention workloads

ATTN_SHAPES = {"attn": (4, 4096, 32, 128, False), "attn_causal": (4, 4096, 32, 128, True)}


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


# ------------------------------------------------------------------ GPU timing helpers

class Gpu:
    """Device, launch stream, L2 flush buffers, peaks and the clock sampler."""

    def __init__(self, local):
        import torch
        self.torch = torch
        torch.cuda.set_device(local)
        self.local = local
        self.device = torch.device("cuda", local)
        self.stream = torch.cuda.current_stream(self.device)
        self.flush_buf = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=self.device)
        self.clean_buf = torch.ones(L2_CLEAN_BYTES, dtype=torch.uint8, device=self.device)
        self.peaks, self.peaks_src = load_peaks()
        self.tensor_peak = self.peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]) * FP16_PER_BF16
        self.tensor_peak_sustained = self.peaks.get(
            "bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]) * FP16_PER_BF16
        self.hbm_peak = self.peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"])
        self.ridge = self.tensor_peak * 1e12 / (self.hbm_peak * 1e9)
        self.sampler = ClockSampler(local)

    def flush_l2(self):
        # Writing a buffer larger than L2 evicts the operands but leaves L2
        # full of dirty lines, whose write-back would then be charged to the
        # next timed kernel; reading a second large buffer evicts those too,
        # so the next launch starts from a cold, clean L2.
        self.flush_buf.zero_()
        self.torch.amax(self.clean_buf)  # a plain uint8 read: no temporary is written

    def sync(self):
        self.torch.cuda.synchronize(self.device)

    def events(self):
        E = self.torch.cuda.Event
        return E(enable_timing=True), E(enable_timing=True)

    def hold(self):
        """Keep the launch stream busy for about HOLD_S (a spinning torch
        kernel) so that the launches the host queues next are already waiting
        when the start event is recorded behind it: the timed region then
        measures the GPU, not the host's launch rate after an idle spell."""
        self.torch.cuda._sleep(int(HOLD_S * 2.1e9))

    def time_stream(self, launch, nsets, n):
        """n launches back to back on the launch stream (set i % nsets),
        queued behind a hold; events at both ends.  Returns ms per launch."""
        e0, e1 = self.events()
        self.sync()
        self.hold()
        e0.record(self.stream)
        for i in range(n):
            launch(i % nsets, self.stream)
        e1.record(self.stream)
        self.sync()
        return e0.elapsed_time(e1) / n

    def time_graph(self, launch, nsets, reps):
        """`reps` launches (set i % nsets) captured into one CUDA graph, so the
        host's per-call cost is out of the measurement; the graph is replayed
        three times with events around each replay.  Returns (median ms per
        launch, reps)."""
        torch = self.torch
        s = torch.cuda.Stream(self.device)
        s.wait_stream(self.stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s, capture_error_mode="thread_local"):
            for i in range(reps):
                launch(i % nsets, s)
        with torch.cuda.stream(s):
            g.replay()
        times = []
        for _ in range(3):
            e0, e1 = self.events()
            with torch.cuda.stream(s):
                e0.record(s)
                g.replay()
                e1.record(s)
            self.sync()
            times.append(e0.elapsed_time(e1) / reps)
        self.stream.wait_stream(s)
        self.sync()
        del g
        return statistics.median(times), reps

    def time_cold(self, launch, n):
        """n single launches, each after an L2 flush, events around each."""
        out = []
        for _ in range(n):
            self.flush_l2()
            e0, e1 = self.events()
            e0.record(self.stream)
            launch(0, self.stream)
            e1.record(self.stream)
            self.sync()
            out.append(e0.elapsed_time(e1))
        return out

    def cold_floor_ms(self, n=10):
        """The cold-launch method around a one-element torch kernel: what a
        single launch between two events costs on this GPU before any work."""
        tiny = self.torch.zeros(1, device=self.device)
        return statistics.median(self.time_cold(lambda r, s: tiny.add_(1), n))

    def time_loop(self, launch, nsets, seconds, est_ms):
        """Launches back to back for about `seconds` (at least 20), clocks
        sampled meanwhile.  Returns (ms per launch, launches, clock summary)."""
        n = max(20, int(math.ceil(seconds / max(est_ms * 1e-3, 1e-6))))
        t0 = time.time()
        ms = self.time_stream(launch, nsets, n)
        t1 = time.time()
        clk = self.sampler.summary(t0, t1)
        if clk.get("sm_mhz"):
            clk["ms_x_sm_mhz"] = ms * clk["sm_mhz"]
        return ms, n, clk

    def e2e(self, jobs, steps, warmup, world):
        """End to end through the public API: every step uploads each job's
        inputs from pinned host memory, launches it and reads its result back.
        Uploads run on their own stream, the kernels on the launch stream,
        read-backs on a third, so the copy engines and the kernels of
        neighbouring jobs and steps overlap; step i uses device set
        i % nsets, and its upload waits until that set's previous kernel and
        read-back are done.  jobs: [(name, nsets, uploads(r) -> [(dst, src)],
        launch(r, stream), downloads(r) -> [(dst, src)])].  Returns ms per
        step (max over ranks)."""
        torch = self.torch
        up = torch.cuda.Stream(self.device)
        down = torch.cuda.Stream(self.device)
        set_free = {}

        def step(i):
            for name, nsets, uploads, launch, downloads in jobs:
                r = i % nsets
                if (name, r) in set_free:
                    up.wait_event(set_free[(name, r)])
                with torch.cuda.stream(up):
                    for dst, src in uploads(r):
                        dst.copy_(src, non_blocking=True)
                uploaded = torch.cuda.Event()
                uploaded.record(up)
                self.stream.wait_event(uploaded)
                launch(r, self.stream)
                computed = torch.cuda.Event()
                computed.record(self.stream)
                down.wait_event(computed)
                with torch.cuda.stream(down):
                    for dst, src in downloads(r):
                        dst.copy_(src, non_blocking=True)
                done = torch.cuda.Event()
                done.record(down)
                set_free[(name, r)] = done

        def run(n, x0=None, x1=None):
            if x0 is not None:
                x0.record(self.stream)
                up.wait_event(x0)
            for i in range(n):
                step(i)
            for ev in set_free.values():          # every read-back inside the region
                self.stream.wait_event(ev)
            if x1 is not None:
                x1.record(self.stream)

        run(warmup)
        self.sync()
        barrier(world)
        x0, x1 = self.events()
        run(steps, x0, x1)
        self.sync()
        ms = max_over_ranks(x0.elapsed_time(x1) / steps, world, self.device)
        barrier(world)
        return ms

    def roofline(self, kernel, flops, nbytes, ms, traffic_key=None):
        """Roofline object of one kernel: tensor-bound when its arithmetic
        intensity is above the ridge point, else HBM-bound."""
        traffic, note = traffic_for(traffic_key) if traffic_key is not None else (None, "not captured")
        base = {"kernel": kernel, "ms": ms, "traffic": traffic, "traffic_source": note}
        if flops / nbytes >= self.ridge:
            ach = flops / (ms * 1e-3) / 1e12
            return {"bound": "tensor", "achieved": ach, "peak": self.tensor_peak, "unit": "TFLOP/s",
                    "frac": ach / self.tensor_peak,
                    "frac_of_sustained": ach / self.tensor_peak_sustained,
                    "algorithmic_flops": flops,
                    "peak_source": f"{self.peaks_src} bf16_tflops (burst) x {FP16_PER_BF16} (fp16/bf16)",
                    **base}
        ach = nbytes / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": ach, "peak": self.hbm_peak, "unit": "GB/s",
                "frac": ach / self.hbm_peak, "algorithmic_bytes": nbytes,
                "peak_source": f"{self.peaks_src} hbm_gbs", **base}


def check_status(gr, stream, where):
    st = gr.status(stream)
    if st != gr.OK:
        raise RuntimeError(f"device status {where}: {gr.strerror(st)}")


# ------------------------------------------------------------------ the headline step

def measure_step(gpu, args, world, parts, name):
    """The contract's timed region: K steps (every part once) back to back on
    rotating operand copies; then each part alone (>= 1 s, clocks sampled),
    warm and cold single launches, the end-to-end leg and the CPU baseline."""
    import torch
    import tiled_tensor_core_03_gb300 as gr
    from tiled_tensor_core_03_gb300 import inputs

    device, stream = gpu.device, gpu.stream
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

    def launcher(label, w, kind):
        def launch(r, s):
            a, b, c, ws = dev[label][r]
            if kind == "splitk":
                gr.gemm_relu_splitk(a, b, w.split_k, out=c, workspace=ws, stream=s)
            elif kind == "streamk":
                gr.gemm_relu_streamk(a, b, out=c, workspace=ws, stream=s)
            else:
                gr.gemm_relu(a, b, out=c, stream=s)
        return launch
    launch = {label: launcher(label, w, kind) for label, w, kind in parts}

    for i in range(args.warmup):
        for label, _, _ in parts:
            gpu.flush_l2()
            launch[label](i % INPUT_SETS, stream)
    gpu.sync()
    check_status(gr, stream, "after warm-up")

    # ---- timed region: K steps back to back, each part on the next input set;
    # events only at the two ends (an event recorded between two launches
    # serialises them and would add its own cost to the step)
    sampler = gpu.sampler
    time.sleep(COOL_S)
    e_start, e_end = gpu.events()
    barrier(world)
    gpu.sync()
    gpu.hold()
    sampler.mark("t_start")
    wall0 = time.perf_counter()
    e_start.record(stream)
    for i in range(args.steps):
        for label, _, _ in parts:
            launch[label](i % INPUT_SETS, stream)
    e_end.record(stream)
    gpu.sync()
    wall1 = time.perf_counter()
    sampler.mark("t_end")
    barrier(world)
    check_status(gr, stream, "after timed steps")
    step_ms = max_over_ranks(e_start.elapsed_time(e_end) / args.steps, world, device)
    flops_step = sum(w.flops for _, w, _ in parts)
    value = world * flops_step / (step_ms * 1e-3) / 1e12
    clocks = sampler.summary()

    # ---- each part alone: K launches back to back on the rotating input
    # sets, events at both ends -> the kernel's average launch duration at
    # the clocks of a burst like the timed region (the roofline); then the
    # same for at least PART_LOOP_S with the clocks sampled during the loop,
    # long enough for the power cap to act (reported against the sustained
    # peak)
    part_ms, sustained = {}, {}
    for label, w, kind in parts:
        # each part from the same idle state: right after another part's
        # power-capped loop the clocks take a while to come back up
        time.sleep(COOL_S)
        part_ms[label] = gpu.time_stream(launch[label], INPUT_SETS, args.steps)
        ms, n, clk = gpu.time_loop(launch[label], INPUT_SETS, PART_LOOP_S, part_ms[label])
        sustained[label] = {"ms": ms, "launches": n, "clocks": clk,
                            "tflops": w.flops / (ms * 1e-3) / 1e12,
                            "gbs": w.bytes / (ms * 1e-3) / 1e9}
    # ---- warm: each part alone, back to back on the same operands (L2 may
    # hold them: the 4096^3 operands fit, the skinny B is about L2's size)
    warm_ms = {}
    for label, _, _ in parts:
        time.sleep(COOL_S)
        warm_ms[label] = gpu.time_stream(launch[label], 1, args.steps)
    check_status(gr, stream, "after the per-part loops")
    # ---- cold launches: L2 flushed before each, events around each alone
    cold_ms = {label: gpu.time_cold(launch[label], max(3, min(args.steps, 10)))
               for label, _, _ in parts}
    cold_floor = gpu.cold_floor_ms()
    check_status(gr, stream, "after cold launches")
    # ---- clock soak: the step back to back for SOAK_S, clocks sampled
    t0 = time.time()
    n_soak = max(20, int(SOAK_S / (step_ms * 1e-3)))
    e0, e1 = gpu.events()
    gpu.hold()
    e0.record(stream)
    for i in range(n_soak):
        for label, _, _ in parts:
            launch[label](i % INPUT_SETS, stream)
    e1.record(stream)
    gpu.sync()
    soak = gpu.sampler.summary(t0, time.time())
    soak.update({"steps": n_soak, "ms_per_step": e0.elapsed_time(e1) / n_soak})
    if soak.get("sm_mhz"):
        soak["ms_x_sm_mhz"] = soak["ms_per_step"] * soak["sm_mhz"]

    # ---- end to end through the public API, host buffers in pinned memory
    pinned = {}
    for label, w, _ in parts:
        A, B = host_inputs[label]
        pinned[label] = (torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory(),
                         torch.empty((w.M, w.N), dtype=torch.float16).pin_memory())
    jobs = []
    for label, w, kind in parts:
        hA, hB, hC = pinned[label]
        jobs.append((label, INPUT_SETS,
                     (lambda r, label=label, hA=hA, hB=hB: [(dev[label][r][0], hA), (dev[label][r][1], hB)]),
                     launch[label],
                     (lambda r, label=label, hC=hC: [(hC, dev[label][r][2])])))
    e2e_ms = gpu.e2e(jobs, args.steps, args.warmup, world)
    h2d = sum(2 * (w.M * w.K + w.K * w.N) for _, w, _ in parts)
    d2h = sum(2 * w.M * w.N for _, w, _ in parts)

    def split_form(w):
        one = gr.gemm_relu_f16_splitk_workspace_bytes(w.M, w.N, w.K, w.split_k) == 0
        return ("CTA-pair form: one kernel, pieces summed in shared memory" if one else
                "two-stage form: partial kernel + reduce kernel"), (1 if one else 2)

    def kernel_name(w, kind):
        if kind == "splitk":
            return f"gemm_relu_f16_splitk {w.M}x{w.N}x{w.K} split {w.split_k} ({split_form(w)[0]})"
        if kind == "streamk" and w.M > 4:
            return (f"gemm_relu_f16_streamk {w.M}x{w.N}x{w.K} (CTA-pair or single-CTA fused kernel, "
                    f"as the library selects; stream-K schedule when the tiles leave a partial wave)")
        if w.M <= 4:
            return f"gemm_relu_f16 {w.M}x{w.N}x{w.K} (GEMV kernel, M <= 4)"
        return f"gemm_relu_f16 {w.M}x{w.N}x{w.K}"

    roofs = {label: gpu.roofline(kernel_name(w, kind), w.flops, w.bytes, part_ms[label],
                                 (kind, w.M, w.N, w.K))
             for label, w, kind in parts}
    for label, w, _ in parts:
        sus = sustained[label]
        if roofs[label]["bound"] == "tensor":
            sus["frac_of_sustained_peak"] = sus["tflops"] / gpu.tensor_peak_sustained
        else:
            sus["frac_of_hbm_peak"] = sus["gbs"] / gpu.hbm_peak
    cold_roofs = {label: gpu.roofline(kernel_name(w, kind), w.flops, w.bytes,
                                      statistics.mean(cold_ms[label]))
                  for label, w, kind in parts}
    dominant = max(parts, key=lambda p: part_ms[p[0]])[0]
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
                      "programmatic stream serialisation, queued behind a ~2 ms GPU-side "
                      "hold recorded before the start event (the host's launch latency after "
                      "an idle spell stays out of the region); value and ms_per_step from CUDA "
                      "events at the two ends of the timed region only; parts (and roofline): "
                      "each part alone after 0.5 s idle, K launches back to back on the rotating input sets, "
                      f"events at both ends; parts.sustained: the same for at least "
                      f"{PART_LOOP_S:.0f} s with the clocks sampled (power cap), against the "
                      f"sustained peak; cold_launch: L2 flushed, "
                      "events around each launch alone (includes the launch latency an idle "
                      "GPU pays; floor_ms: the same method around a one-element torch kernel)",
        },
        "roofline": roofs[dominant],
        "parts": {label: {"ms": part_ms[label],
                          "tflops": w.flops / (part_ms[label] * 1e-3) / 1e12,
                          "gbs": w.bytes / (part_ms[label] * 1e-3) / 1e9,
                          "roofline": roofs[label],
                          "sustained": sustained[label]}
                  for label, w, _ in parts},
        "cold_launch": {label: {"ms": statistics.mean(cold_ms[label]),
                                "tflops": w.flops / (statistics.mean(cold_ms[label]) * 1e-3) / 1e12,
                                "gbs": w.bytes / (statistics.mean(cold_ms[label]) * 1e-3) / 1e9,
                                "frac": cold_roofs[label]["frac"],
                                "bound": cold_roofs[label]["bound"],
                                "floor_ms": cold_floor}
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
        "clocks": clocks,
        "clocks_soak": soak,
    }

    if world == 1 and not args.no_cpu_baseline:
        import multiprocessing
        f, dt, threads, outs = oracle_rows_sample(parts, host_inputs, args.cpu_budget)
        checks = {}
        for label, (rows, want) in outs.items():
            if rows:
                got = dev[label][0][2][:rows].cpu().numpy()
                checks[label] = contract_check(got, want)
        desc = ", ".join(f"first {rows} rows of {label}" for label, (rows, _) in outs.items())
        line["cpu_baseline"] = {
            "value": f / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{desc} ({f / 1e9:.2f} GFLOP in {dt:.1f} s of wall time), fp64 C oracle "
                      f"on {threads} threads, one output row each at a time; host has "
                      f"{multiprocessing.cpu_count()} cores",
            "parity_on_sample": checks,
        }
    return line


# ------------------------------------------------------------------ one GEMM workload

def measure_config(gpu, w, steps, warmup, world, cpu_budget, want_cpu=True):
    """One GEMM workload through gemm_relu_streamk (the library's call with a
    workspace: a stream-K schedule where one applies, operands whose rows TMA
    cannot describe copied into aligned rows first, else gemm_relu_f16's
    kernel): device time by CUDA-graph replay over enough rotating operand
    copies that every launch reads operands last touched at least
    ROTATE_BYTES of other operands earlier; plain back-to-back launches (with
    the host's per-call cost), cold launches, the end-to-end leg, the CPU
    oracle on all host cores (and on one core for the two square shapes) and
    a full-output parity check against it."""
    import torch
    import tiled_tensor_core_03_gb300 as gr
    from tiled_tensor_core_03_gb300 import inputs

    device = gpu.device
    A, B = inputs.make_workload(w)
    nsets = max(INPUT_SETS, int(math.ceil(ROTATE_BYTES / w.bytes)))
    a_dev = torch.from_numpy(A).to(device)
    b_dev = torch.from_numpy(B).to(device)
    sets = [(a_dev.clone(), b_dev.clone(), torch.empty((w.M, w.N), dtype=torch.float16, device=device))
            for _ in range(nsets)]
    del a_dev, b_dev
    path = gr.gemm_relu_f16_path(sets[0][0].data_ptr(), sets[0][1].data_ptr(),
                                 sets[0][2].data_ptr(), w.M, w.N, w.K)
    # one workspace: the launches of a stream run one after another
    ws_bytes = gr.gemm_relu_f16_streamk_workspace_bytes(w.M, w.N, w.K)
    ws = gr.streamk_workspace(w.M, w.N, w.K, device)

    def launch(r, s):
        a, b, c = sets[r]
        gr.gemm_relu_streamk(a, b, out=c, workspace=ws, stream=s)

    for i in range(max(3, warmup)):
        launch(i % nsets, gpu.stream)
    gpu.sync()
    check_status(gr, gpu.stream, f"after warm-up of {w.name}")
    reps = max(nsets, 64)
    ms, reps = gpu.time_graph(launch, nsets, reps)
    stream_ms = gpu.time_stream(launch, nsets, max(steps, 20))
    cold = gpu.time_cold(launch, 5)
    check_status(gr, gpu.stream, f"after timing {w.name}")

    hA, hB = torch.from_numpy(A).pin_memory(), torch.from_numpy(B).pin_memory()
    hC = torch.empty((w.M, w.N), dtype=torch.float16).pin_memory()
    e2e_sets = min(nsets, INPUT_SETS)
    e2e_ms = gpu.e2e([(w.name, e2e_sets,
                       lambda r: [(sets[r][0], hA), (sets[r][1], hB)], launch,
                       lambda r: [(hC, sets[r][2])])], max(steps, 20), max(3, warmup), world)
    check_status(gr, gpu.stream, f"after the end-to-end leg of {w.name}")

    launches_per_call = 1
    if path == 1:
        kid = gr.gemm_relu_f16_kernel(sets[0][0].data_ptr(), sets[0][1].data_ptr(),
                                      sets[0][2].data_ptr(), w.M, w.N, w.K)
        kern = gr.KERNEL_NAMES.get(kid, f"kernel {kid}")
        if ws_bytes > 0:
            kern += ", stream-K schedule"
    else:
        kern = ("copy kernel for the operands whose row pitch is not a multiple of 16 B "
                f"({ws_bytes / 2**20:.1f} MiB of workspace), then the single-CTA TMA kernel "
                "with predicated stores of C")
        launches_per_call = 2
    out = {
        "workload": describe(w),
        "kernel": f"gemm_relu_f16_streamk {w.M}x{w.N}x{w.K}: {kern}, as the library selects",
        "path": {1: "tma", 2: "staged (rows not 16-byte aligned)"}.get(path, str(path)),
        "ms": ms, "tflops": w.flops / (ms * 1e-3) / 1e12, "gbs": w.bytes / (ms * 1e-3) / 1e9,
        "roofline": gpu.roofline(f"gemm_relu_f16_streamk {w.M}x{w.N}x{w.K} ({kern})", w.flops,
                                 w.bytes, ms, ("fused", w.M, w.N, w.K)),
        "timing": (f"CUDA graph of {reps} launches rotating {nsets} operand copies "
                   f"({nsets * w.bytes / 2**20:.0f} MiB: inputs larger than L2), replayed 3 times "
                   f"with events around each replay, median; stream_ms: plain launches back to "
                   f"back from Python (includes the host's per-call cost); cold_ms: one launch "
                   f"after an L2 flush, events around it"),
        "stream_ms": stream_ms,
        "cold_ms": statistics.mean(cold),
        "e2e": {"value": world * w.flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": 2 * (w.M * w.K + w.K * w.N),
                "d2h_bytes_per_step": 2 * w.M * w.N,
                "api": "tiled_tensor_core_03_gb300.gemm_relu_streamk from pinned host buffers; "
                       "upload, kernel and read-back on three streams"},
    }
    if want_cpu:
        import multiprocessing
        threads = os.cpu_count() or 1
        rows, want, f, dt = oracle_gemm_rows(A, B, cpu_budget, threads)
        got = sets[0][2].cpu().numpy()
        cb = {"value": f / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
              "sample": (f"{'all' if rows == w.M else 'first'} {rows} of {w.M} output rows "
                         f"({f / 1e9:.3f} GFLOP in {dt:.2f} s of wall time), fp64 C oracle on "
                         f"{threads} threads, one row each at a time; host has "
                         f"{multiprocessing.cpu_count()} cores")}
        if w.name in ("square256", "square1024"):
            r1, _, f1, dt1 = oracle_gemm_rows(A, B, min(cpu_budget, 4.0), 1)
            cb["single_thread"] = {"value": f1 / dt1 / 1e12, "unit": "TFLOP/s", "cores": 1,
                                   "sample": f"first {r1} of {w.M} output rows "
                                             f"({f1 / 1e9:.3f} GFLOP in {dt1:.2f} s), one thread"}
        out["cpu_baseline"] = cb
        out["parity"] = dict(contract_check(got[:rows], want), rows_checked=rows)
    out["gpu_launches"] = reps * launches_per_call
    return out


# ------------------------------------------------------------------ attention forward

def measure_attention(gpu, b, s, h, d, causal, steps, warmup, world, cpu_budget, want_cpu=True):
    """Attention forward (flash_attention_f16) on [batch, seq, heads, d] fp16:
    K launches back to back on rotating input copies, events at both ends;
    cold launches; the end-to-end leg; the oracle on a sample of rows."""
    import torch
    import tiled_tensor_core_03_gb300 as gr

    device, stream = gpu.device, gpu.stream
    host = attn_host_inputs(b, s, h, d)
    sets = [[torch.from_numpy(x).to(device) for x in host] +
            [torch.empty((b, s, h, d), dtype=torch.float16, device=device)]
            for _ in range(INPUT_SETS)]

    def launch(r, st):
        q, k, v, o = sets[r]
        gr.flash_attention(q, k, v, causal=causal, out=o, stream=st)

    for i in range(max(3, warmup)):
        launch(i % INPUT_SETS, stream)
    gpu.sync()
    check_status(gr, stream, "after attention warm-up")
    t0 = time.time()
    ms = gpu.time_stream(launch, INPUT_SETS, steps)
    clk = gpu.sampler.summary(t0, time.time())
    ms = max_over_ranks(ms, world, device)
    cold = gpu.time_cold(launch, max(3, min(steps, 5)))
    check_status(gr, stream, "after attention timing")
    pinned = [torch.from_numpy(x).pin_memory() for x in host]
    hout = torch.empty((b, s, h, d), dtype=torch.float16).pin_memory()
    e2e_ms = gpu.e2e([("attn", INPUT_SETS,
                       lambda r: list(zip(sets[r][:3], pinned)), launch,
                       lambda r: [(hout, sets[r][3])])], steps, max(3, warmup), world)
    flops = attn_flops(b, s, h, d, causal)
    name = attn_workload_name("attn_causal" if causal else "attn", b, s, h, d, causal)
    roof = gpu.roofline(f"flash_attention_fwd_kernel<{d}>", flops, 4 * b * s * h * d * 2, ms,
                        ("attn", b, s, h, d, bool(causal)))
    out = {
        "workload": name, "ms": ms, "tflops": flops / (ms * 1e-3) / 1e12, "roofline": roof,
        "flops": flops,
        "timing": f"{steps} launches back to back on {INPUT_SETS} rotating copies of Q, K, V "
                  f"({3 * b * s * h * d * 2 / 2**20:.0f} MiB each: inputs larger than L2), events "
                  f"at both ends",
        "cold_ms": statistics.mean(cold),
        "e2e": {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                "ms_per_step": e2e_ms, "h2d_bytes_per_step": 3 * b * s * h * d * 2,
                "d2h_bytes_per_step": b * s * h * d * 2,
                "api": "tiled_tensor_core_03_gb300.flash_attention from pinned host buffers; "
                       "uploads, kernel and read-back on three streams"},
        "clocks": clk,
        "gpu_launches": steps,
    }
    if want_cpu:
        import multiprocessing
        Q, K, V = host
        f, dt, threads, rows_out = attn_oracle_sample(Q, K, V, causal, cpu_budget)
        got = sets[0][3].cpu().numpy()
        keys = sorted(rows_out)
        g = np.stack([got[bb, r, hh] for (bb, hh, r) in keys])
        o = np.stack([rows_out[k][0] for k in keys])
        out["cpu_baseline"] = {
            "value": f / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{len(rows_out)} output rows of the workload ({f / 1e9:.2f} GFLOP in "
                      f"{dt:.1f} s of wall time), fp64 C attention oracle on {threads} threads; "
                      f"host has {multiprocessing.cpu_count()} cores"}
        out["parity"] = dict(contract_check(g, o), rows_checked=len(keys))
    return out


# ------------------------------------------------------------------ our arm

def run_ours(args, world, rank, local):
    import tiled_tensor_core_03_gb300 as gr
    from tiled_tensor_core_03_gb300 import _build, inputs

    if _build.needs_build():
        _build.build()
    gpu = Gpu(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=gpu.device)
    if args.kernel != "auto":
        # profiling aid: every GEMM call of this run takes the named kernel
        gr.gemm_relu_debug_force_kernel(KERNEL_CHOICES[args.kernel])
    gpu.sampler.start()
    try:
        if args.workload in EXTRA_CONFIGS and not args.shape:
            line = single_config_line(gpu, args, world, inputs.WORKLOADS[args.workload])
        else:
            parts, name = build_parts(args)
            if args.kernel != "auto":
                name += f", kernel forced: {args.kernel}"
            line = measure_step(gpu, args, world, parts, name)
            if args.workload == "step" and not args.shape and not args.no_extra:
                cpu = world == 1 and not args.no_cpu_baseline
                line["configs"] = {
                    n: measure_config(gpu, inputs.WORKLOADS[n], args.steps, args.warmup, world,
                                      min(args.cpu_budget, 4.0), cpu)
                    for n in EXTRA_CONFIGS}
                line["attention"] = {
                    n: measure_attention(gpu, *ATTN_SHAPES[n], min(args.steps, 20), args.warmup,
                                         world, min(args.cpu_budget, 3.0), cpu)
                    for n in ATTN_SHAPES}
    finally:
        gpu.sampler.stop()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def single_config_line(gpu, args, world, w):
    """`--workload square256 | square1024 | ragged | decode1`: that workload
    alone as the contract's line (value from CUDA-graph replay)."""
    gpu.sampler.mark("t_start")
    cfg = measure_config(gpu, w, args.steps, args.warmup, world, args.cpu_budget,
                         world == 1 and not args.no_cpu_baseline)
    gpu.sampler.mark("t_end")
    ms = max_over_ranks(cfg["ms"], world, gpu.device)
    line = {
        "metric": METRIC, "value": world * w.flops / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": describe(w), "flops_per_step": w.flops,
                   "parallelism": f"replicas{world}", "timing": cfg["timing"],
                   "l2": "inputs larger than L2 (rotating operand copies, see timing)"},
        "roofline": cfg["roofline"], "e2e": cfg["e2e"], "gpu_launches": cfg["gpu_launches"],
        "stream_ms": cfg["stream_ms"], "cold_ms": cfg["cold_ms"],
        "clocks": gpu.sampler.summary(),
    }
    for k in ("cpu_baseline", "parity"):
        if k in cfg:
            line[k] = cfg[k]
    return line


def run_attention(args, world, rank, local):
    """`--workload attn | attn_causal`: the attention forward as the contract's line."""
    from tiled_tensor_core_03_gb300 import _build
    if _build.needs_build():
        _build.build()
    gpu = Gpu(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=gpu.device)
    b, s, h, d, causal = attn_shape(args)
    gpu.sampler.start()
    try:
        gpu.sampler.mark("t_start")
        a = measure_attention(gpu, b, s, h, d, causal, args.steps, args.warmup, world,
                              args.cpu_budget, world == 1 and not args.no_cpu_baseline)
        gpu.sampler.mark("t_end")
    finally:
        gpu.sampler.stop()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    if rank != 0:
        return 0
    line = {
        "metric": ATTN_METRIC, "value": world * a["tflops"], "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": a["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f16",
        "data": "synthetic",
        "config": {"workload": a["workload"], "flops_per_step": a["flops"],
                   "parallelism": f"replicas{world}", "timing": a["timing"],
                   "l2": "inputs larger than L2 (rotating copies, see timing)"},
        "roofline": a["roofline"], "cold_launch": {"ms": a["cold_ms"]}, "e2e": a["e2e"],
        "gpu_launches": a["gpu_launches"], "clocks": a["clocks"],
    }
    for k in ("cpu_baseline", "parity"):
        if k in a:
            line[k] = a[k]
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true",
                    help="the headline step only (no other workloads, no attention)")
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
