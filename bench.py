"""Benchmark of the GB300 fp16 NT GEMM, C[M,N] = A[M,K] . B[N,K]^T.

One step = one GEMM of the workload (default: M = N = K = 8192, operands
uniform on [-1, 1) rounded to fp16, seed 1003) through the C ABI, with A, B
and C resident in HBM.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--no-cpu-baseline] [--no-e2e]

--impl reference times the CPU oracle (double accumulation, fp16 rounding)
on this machine's host cores over a bounded sample of the same workload:
the only reference that exists for this product is that definition.

After the headline step the line also carries a "workloads" object: every
configured product (256^3, 4096^3, 8192^3, 3000 x 5000 x 4096 and
128 x 16384 x 16384) timed back to back through the same entry point, each
rotating over enough copies of its operands that the launches do not find
them in L2.

One GPU per process: the library is meant for single-GPU processes (its
multicast TMA loads read only this GPU's own buffers), so this script
refuses to run as several ranks (WORLD_SIZE > 1) or with --gpus > 1.
"""
import argparse
import hashlib
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

from dense_fp16_gemm_03_gb300 import inputs  # noqa: E402

METRIC = "GEMM TFLOP/s (2MNK/time) at 1 GB300; fraction of dense fp16 tensor peak"
UNIT = "TFLOP/s"
NOMINAL_PEAK_TFLOPS = 2250.0      # dense fp16/bf16 tensor peak quoted for GB300
FALLBACK_BURST_TFLOPS = 1900.0    # bf16 burst, measured earlier on a GB300 (used without MEASURED_PEAKS.json)
FALLBACK_SUSTAINED_TFLOPS = 1700.0  # bf16 sustained, same
FALLBACK_HBM_GBS = 6800.0         # copy bandwidth, same
L2_BYTES = 129 * 10 ** 6
KERNEL_SOURCES = ["dense_fp16_gemm_03_gb300/csrc/gemm_kernel.cuh", "dense_fp16_gemm_03_gb300/csrc/gemm_kernel_wide.cuh",
                  "dense_fp16_gemm_03_gb300/csrc/ptx.cuh", "dense_fp16_gemm_03_gb300/csrc/sched.cuh",
                  "dense_fp16_gemm_03_gb300/csrc/gemm_launch.cuh"]


def kernel_source_hash():
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


def traffic_record(workload_name, plan):
    """DRAM bytes per launch from a committed ncu capture, if it was taken on
    the current kernel sources with the same plan; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_hash") != kernel_source_hash():
        return None
    entry = rec.get("workloads", {}).get(workload_name)
    if entry is None:
        return None
    if any(getattr(plan, k) != v for k, v in entry.get("plan", {}).items()):
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.samples = []
        self.proc = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [x.strip() for x in line.split(",")]))

    def mark_begin(self):
        self.t0 = time.time()

    def mark_end(self):
        self.t1 = time.time()

    def summary(self):
        """Clocks over the marked region (the samples 50 ms before to 150 ms
        after it; all samples so far if none fell inside)."""
        if self.proc is None:
            return None
        time.sleep(0.25)
        samples = list(self.samples)
        inside = [s for (t, s) in samples if self.t0 is not None and self.t0 - 0.05 <= t <= self.t1 + 0.15]
        use = inside if inside else [s for (_, s) in samples]
        if not use:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(s[2]) for s in use if len(s) > 2 and num(s[2]) is not None]
        smax = [num(s[3]) for s in use if len(s) > 3 and num(s[3]) is not None]
        power = [num(s[4]) for s in use if len(s) > 4 and num(s[4]) is not None]
        reasons = sorted({self.REASONS[i] for s in use for i in range(4)
                          if len(s) > 6 + i and s[6 + i].lower() == "active"})
        return {
            "sm_mhz": statistics.median(sm) if sm else None,
            "sm_max_mhz": max(smax) if smax else None,
            "power_w_max": max(power) if power else None,
            "reasons": reasons,
            "samples": len(use),
            "samples_in_timed_region": len(inside),
        }

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()


def cpu_oracle_rate(A, B, target_s=10.0):
    """Time the CPU oracle on the first R rows of C (all N columns, full K),
    R sized for about target_s seconds and at least one row per oracle
    thread.  Returns (tflops, seconds, rows)."""
    import oracle

    M, K = A.shape
    N = B.shape[0]
    rows = min(M, max(1, oracle.num_threads()))
    while True:
        t = time.perf_counter()
        oracle.gemm_nt(A[:rows], B)
        dt = time.perf_counter() - t
        if dt > min(0.5, target_s / 4) or rows >= M:
            break
        rows = min(M, rows * 4)
    want = max(min(M, oracle.num_threads()), min(M, int(rows * target_s / max(dt, 1e-6))))
    if want != rows:
        rows = want
        t = time.perf_counter()
        oracle.gemm_nt(A[:rows], B)
        dt = time.perf_counter() - t
    return 2.0 * rows * N * K / dt / 1e12, dt, rows


def throughput(total_ms, flops_per_step, steps):
    """TFLOP/s of `steps` steps of `flops_per_step` timed as `total_ms` in all."""
    return flops_per_step * steps / (total_ms * 1e-3) / 1e12


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def timing_regime(total_ms, clocks):
    """"sustained" when the timed region ran long enough for the board power
    cap to matter (a second or more of back-to-back launches, or sw_power_cap
    seen by the clock sampler inside it), else "burst"."""
    if total_ms >= 1000.0:
        return "sustained"
    if clocks and "sw_power_cap" in (clocks.get("reasons") or []):
        return "sustained"
    return "burst"


def tensor_roofline(achieved, regime, peaks):
    """Roofline of a contraction: the measured cuBLAS bf16 rate of the same
    regime (burst for a short timed region, sustained for one under the
    power cap) is the denominator; fp16 and bf16 share the nominal tensor
    rate.  Both fractions are reported."""
    burst = sustained = None
    if peaks:
        burst = float(peaks.get("bf16_tflops") or 0.0) or None
        sustained = float(peaks.get("bf16_tflops_sustained") or 0.0) or None
    if regime == "sustained" and sustained:
        peak, note = sustained, "of measured: cuBLAS bf16 sustained (timed region under the power cap); fp16 rate = bf16 rate"
    elif burst:
        peak, note = burst, "of measured: cuBLAS bf16 burst (short timed region); fp16 rate = bf16 rate"
    elif sustained:
        peak, note = sustained, "of measured: cuBLAS bf16 sustained (no burst figure); fp16 rate = bf16 rate"
    elif regime == "sustained":
        peak, note = FALLBACK_SUSTAINED_TFLOPS, "of fallback (bf16 sustained)"
    else:
        peak, note = FALLBACK_BURST_TFLOPS, "of fallback (bf16 burst)"
    return {
        "bound": "tensor", "achieved": achieved, "peak": peak, "unit": UNIT, "frac": achieved / peak,
        "regime": regime, "peak_source": note,
        "burst_peak": burst, "frac_burst": (achieved / burst) if burst else None,
        "sustained_peak": sustained, "frac_sustained": (achieved / sustained) if sustained else None,
        "frac_of_nominal_2250": achieved / NOMINAL_PEAK_TFLOPS,
    }


def run_reference(args, w, world, rank):
    if rank != 0:
        return 0
    import oracle

    A, B = inputs.workload_operands(w)
    threads = oracle.num_threads()
    # each step is a bounded sample of the workload: the first R rows of C
    _, probe_s, rows = cpu_oracle_rate(A, B, target_s=min(10.0, max(0.05, 120.0 / (args.steps + args.warmup))))
    for _ in range(args.warmup):
        oracle.gemm_nt(A[:rows], B)
    t = time.perf_counter()
    for _ in range(args.steps):
        oracle.gemm_nt(A[:rows], B)
    dt = (time.perf_counter() - t) / max(1, args.steps)
    value = 2.0 * rows * w.N * w.K / dt / 1e12
    sample = "first %d of %d rows of C (all %d columns, full K=%d) per step" % (rows, w.M, w.N, w.K)
    line = {
        "impl": "reference",
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w),
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# Pipeline ablation on GB300, rung by rung, after the Hopper tutorial's
# version table ("1. WGMMA" section "Performance"; "4. Pipeline Abstraction
# and Two Consumer Warp Groups" sections "Pipeline Depth" and "Performance"):
# (label, page analogue, variant, raster width, one tile per cluster?)
ABLATION = [
    ("single stage: TMA load, then MMA, then the next load", "V1", 8, 1, True),
    ("two-stage ring, TMA producer warp", "V3", 9, 1, True),
    ("CTA pair (two accumulators share B), three stages", "V4", 10, 1, True),
    ("CTA pair, six stages", "-", 2, 1, True),
    ("persistent: epilogue overlaps the next tile, raster 8", "-", 2, 8, False),
    ("persistent, two pairs share B by multicast", "-", 4, 8, False),
    ("persistent 256 x 512 pair tile, one accumulator filling tensor memory, raster 4", "-", 15, 4, False),
]


def run_ablation(args, w):
    import torch
    from dense_fp16_gemm_03_gb300 import gemm as G

    dev = torch.device("cuda", 0)
    A, B = inputs.workload_operands(w)
    a = torch.from_numpy(A.view(np.int16)).view(torch.float16).to(dev)
    b = torch.from_numpy(B.view(np.int16)).view(torch.float16).to(dev)
    c = torch.empty((w.M, w.N), dtype=torch.float16, device=dev)
    rungs = []
    for label, page, variant, raster, one_tile in ABLATION:
        plan = G.gemm_f16_nt_plan_ex(w.M, w.N, w.K, variant, raster, 0)
        if one_tile:
            plan.grid = int(plan.num_tiles * plan.cluster)
        rungs.append((label, page, variant, raster, one_tile, plan))
    sampler = ClockSampler(0)
    sampler.start()
    for _, _, _, _, _, plan in rungs:
        for _ in range(args.warmup):
            G.gemm_f16_nt_run(plan, a, b, c)
    torch.cuda.synchronize()
    times = {i: [] for i in range(len(rungs))}
    windows = {i: [] for i in range(len(rungs))}
    for _ in range(max(1, args.rounds)):
        for i, (_, _, _, _, _, plan) in enumerate(rungs):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            torch.cuda.synchronize()
            t0 = time.time()
            e0.record()
            for _ in range(args.steps):
                G.gemm_f16_nt_run(plan, a, b, c)
            e1.record()
            torch.cuda.synchronize()
            windows[i].append((t0, time.time()))
            times[i].append(e0.elapsed_time(e1) / args.steps)
    st, code = G.gemm_f16_take_device_error()
    if st != G.GEMM_OK:
        raise RuntimeError("kernel reported error word 0x%x" % code)
    sampler.stop()
    for i, (label, page, variant, raster, one_tile, plan) in enumerate(rungs):
        ms = statistics.median(times[i])
        mhz = [float(smp[2]) for (t, smp) in sampler.samples if len(smp) > 2 and
               any(t0 + 0.05 <= t <= t1 for (t0, t1) in windows[i])]
        mhz_med = statistics.median(mhz) if mhz else None
        tf = w.flops / (ms * 1e-3) / 1e12
        print(json.dumps({"ablation_rung": i + 1, "what": label, "page_analogue": page, "variant": variant,
                          "cta_group": plan.cta_group, "cluster": plan.cluster, "stages": plan.stages,
                          "tile": "%dx%d" % (plan.block_m, plan.block_n), "one_tile_per_cluster": one_tile,
                          "grid": plan.grid, "raster_width": raster, "workload": w.name, "ms": ms, "tflops": tf,
                          "sm_mhz": mhz_med, "tflops_per_ghz": (tf / mhz_med * 1000.0) if mhz_med else None}),
              flush=True)
    return 0


def workload_config(w):
    return {
        "workload": "%s: C[%d,%d] = A[%d,%d] . B[%d,%d]^T fp16, %s operands, seed %d" % (
            w.name, w.M, w.N, w.M, w.K, w.N, w.K, w.dist, w.seed),
        "M": w.M, "N": w.N, "K": w.K, "distribution": w.dist, "seed": w.seed,
        "l2": ("inputs larger than L2: %.0f MiB of A, B and C per step vs %d MB L2" % (
            w.algorithmic_bytes / 2 ** 20, L2_BYTES // 10 ** 6)) if w.algorithmic_bytes > L2_BYTES
        else "working set smaller than L2 (no flush)",
    }


def to_device(x, dev):
    import torch
    return torch.from_numpy(x.view(np.int16)).view(torch.float16).to(dev)


def time_workload(G, w, dev, stream, sampler, launches, warmup, peaks):
    """Time `launches` back-to-back launches of the automatic plan of workload
    `w` through gemm_f16_nt_ws, rotating over enough copies of A, B and C that
    their bytes exceed twice the L2 (so no launch finds its operands there).
    One CUDA event pair on the launching stream brackets the launches."""
    import torch
    A, B = inputs.workload_operands(w)
    a0, b0 = to_device(A, dev), to_device(B, dev)
    sets = max(1, min(1024, -(-2 * L2_BYTES // w.algorithmic_bytes)))
    bufs = [(a0, b0, torch.empty((w.M, w.N), dtype=torch.float16, device=dev))]
    for _ in range(sets - 1):
        bufs.append((a0.clone(), b0.clone(), torch.empty((w.M, w.N), dtype=torch.float16, device=dev)))
    plan = G.gemm_f16_nt_plan(w.M, w.N, w.K)
    ws = G.workspace_for(plan, dev)
    for i in range(warmup):
        a, b, c = bufs[i % sets]
        G.gemm_f16_nt_ws(a, b, c, ws, stream=stream)
    stream.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    t0 = time.time()
    e0.record(stream)
    h0 = time.perf_counter()
    for i in range(launches):
        a, b, c = bufs[i % sets]
        G.gemm_f16_nt_ws(a, b, c, ws, stream=stream)
    host_s = time.perf_counter() - h0
    e1.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    st, code = G.gemm_f16_take_device_error(stream)
    if st != G.GEMM_OK:
        raise RuntimeError("%s: kernel reported error word 0x%x" % (w.name, code))
    ms = e0.elapsed_time(e1) / launches
    # The same launches replayed from a CUDA graph: device time without the per-call host work (the
    # Python binding and the library's planning and tensor-map encoding), which bounds the small,
    # latency-bound products when they are launched one call at a time.
    ms_graph = None
    try:
        n_graph = min(launches, 400)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(n_graph):
                a, b, c = bufs[i % sets]
                G.gemm_f16_nt_ws(a, b, c, ws, stream=stream)
        with torch.cuda.stream(stream):  # a graph replays on the current stream
            graph.replay()
            stream.synchronize()
            g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            g0.record(stream)
            graph.replay()
            g1.record(stream)
        torch.cuda.synchronize(dev)
        ms_graph = g0.elapsed_time(g1) / n_graph
        del graph
    except RuntimeError:
        ms_graph = None
    mhz = [float(s[2]) for (t, s) in list(sampler.samples) if len(s) > 2 and t0 - 0.05 <= t <= t1 + 0.15
           and s[2].replace(".", "", 1).isdigit()]
    reasons = sorted({n for (t, s) in list(sampler.samples) if t0 - 0.05 <= t <= t1 + 0.15
                      for i, n in enumerate(ClockSampler.REASONS) if len(s) > 6 + i and s[6 + i].lower() == "active"})
    # each product is timed alone for a short region (milliseconds): the burst denominator, whatever
    # throttle state the samples around it caught from the work before
    regime = timing_regime(ms * launches, None)
    tflops = w.flops / (ms * 1e-3) / 1e12
    entry = {
        "M": w.M, "N": w.N, "K": w.K, "distribution": w.dist, "seed": w.seed,
        "ms": ms, "tflops": tflops, "launches": launches, "operand_copies": sets,
        "host_us_per_call": host_s / launches * 1e6,
        "ms_graph": ms_graph, "tflops_graph": (w.flops / (ms_graph * 1e-3) / 1e12) if ms_graph else None,
        "sm_mhz": statistics.median(mhz) if mhz else None, "clock_reasons": reasons,
        "plan": {k: getattr(plan, k) for k in ("variant", "block_m", "block_n", "grid", "stream_k", "split_k",
                                               "k_rotate", "raster_width")},
        "roofline": tensor_roofline(tflops, regime, peaks),
        "algorithmic_bytes": w.algorithmic_bytes,
        "algorithmic_gbs": w.algorithmic_bytes / (ms * 1e-3) / 1e9,
    }
    hbm = float(peaks["hbm_gbs"]) if peaks and peaks.get("hbm_gbs") else FALLBACK_HBM_GBS
    if w.flops < 1e9:
        # a few tiles on a few SMs: launch and pipeline latency bound it, not a roofline
        entry["roofline"] = {"bound": "latency", "achieved": tflops, "unit": UNIT, "peak": None, "frac": None,
                             "regime": regime, "tensor": entry["roofline"]}
    elif w.flops / w.algorithmic_bytes < (entry["roofline"]["peak"] * 1e12) / (hbm * 1e9):
        # below the ridge point: HBM bounds the product
        entry["roofline"] = {
            "bound": "hbm", "achieved": entry["algorithmic_gbs"], "peak": hbm, "unit": "GB/s",
            "frac": entry["algorithmic_gbs"] / hbm, "regime": regime,
            "peak_source": "of measured: copy bandwidth" if peaks and peaks.get("hbm_gbs") else "of fallback",
            "tensor": entry["roofline"],
        }
    del bufs
    torch.cuda.empty_cache()
    return entry


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="square_8192", choices=sorted(inputs.BY_NAME))
    ap.add_argument("--shape", default=None, help="MxNxK: time this product instead of a configured workload "
                    "(uniform operands, seed 0; for measurement and profiling)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="skip timing the other configured products")
    ap.add_argument("--workload-launches", type=int, default=400,
                    help="launches per configured product in the workloads object")
    ap.add_argument("--variant", type=int, default=-1, help="force a compiled kernel variant (measurement)")
    ap.add_argument("--raster", type=int, default=0, help="force a raster width (measurement)")
    ap.add_argument("--stream-k", type=int, default=-1,
                    help="force no split (0), a stream-K tail (1) or split-K (2) (measurement)")
    ap.add_argument("--ablation", action="store_true",
                    help="time the pipeline ablation ladder (one JSON line per rung) instead of the bench step")
    ap.add_argument("--rounds", type=int, default=3, help="interleaved rounds of the ablation ladder")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    w = inputs.BY_NAME[args.workload]
    if args.shape:
        m_, n_, k_ = (int(x) for x in args.shape.lower().split("x"))
        w = inputs.Workload("shape_%dx%dx%d" % (m_, n_, k_), m_, n_, k_, "uniform", 0)
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, w, world, rank)
    if world > 1 or args.gpus != 1:
        print("bench.py: this library is for single-GPU processes (it has no multi-GPU path); "
              "run one process on one GPU (WORLD_SIZE=%d, --gpus %d)" % (world, args.gpus), file=sys.stderr)
        return 2
    if args.ablation:
        return run_ablation(args, w)

    import torch
    from dense_fp16_gemm_03_gb300 import gemm as G

    torch.cuda.set_device(0)
    G.lib()
    dev = torch.device("cuda", 0)
    A, B = inputs.workload_operands(w)
    a, b = to_device(A, dev), to_device(B, dev)
    c = torch.empty((w.M, w.N), dtype=torch.float16, device=dev)
    stream = torch.cuda.Stream(device=dev)
    if args.variant >= 0 or args.raster > 0 or args.stream_k >= 0:
        plan = G.gemm_f16_nt_plan_ex(w.M, w.N, w.K, args.variant, args.raster, args.stream_k)
        ws = G.workspace_for(plan, dev)
        step = lambda: G.gemm_f16_nt_run(plan, a, b, c, ws, stream=stream)  # noqa: E731
    else:
        # the automatic plan through the workspace entry point (stream-K tail or split K when they pay)
        plan = G.gemm_f16_nt_plan(w.M, w.N, w.K)
        ws = G.workspace_for(plan, dev)
        step = lambda: G.gemm_f16_nt_ws(a, b, c, ws, stream=stream)  # noqa: E731

    for _ in range(args.warmup):
        step()
    stream.synchronize()
    st, code = G.gemm_f16_take_device_error(stream)
    if st != G.GEMM_OK:
        raise RuntimeError("kernel reported error word 0x%x" % code)

    sampler = ClockSampler(0)
    sampler.start()
    time.sleep(0.3)
    # One event pair around the K steps: events between launches would stand between two kernels
    # in the stream and stop a launch's set-up from overlapping its predecessor's tail.  Each step
    # is exactly one launch of the GEMM kernel (plus the reduction of a split-K plan), back to back,
    # so the average launch duration is the timed region over K (inter-kernel gaps included).
    e_begin, e_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    sampler.mark_begin()
    with torch.cuda.stream(stream):
        e_begin.record(stream)
        for _ in range(args.steps):
            step()
        e_end.record(stream)
    torch.cuda.synchronize(dev)
    sampler.mark_end()
    st, code = G.gemm_f16_take_device_error(stream)
    if st != G.GEMM_OK:
        raise RuntimeError("kernel reported error word 0x%x" % code)
    total_ms = e_begin.elapsed_time(e_end)
    ms_per_step = total_ms / args.steps
    value = throughput(total_ms, w.flops, args.steps)
    clocks = sampler.summary()

    # end to end through the host-buffer entry point: H2D of A and B from
    # pinned memory, the GEMM, D2H of C, every step
    e2e = None
    if not args.no_e2e:
        a_h = torch.from_numpy(A.view(np.int16)).view(torch.float16).pin_memory()
        b_h = torch.from_numpy(B.view(np.int16)).view(torch.float16).pin_memory()
        c_h = torch.empty((w.M, w.N), dtype=torch.float16).pin_memory()
        e_steps = max(3, min(args.steps, 200))
        for _ in range(3):
            G.gemm_f16_nt_host(a_h, b_h, c_h, a, b, c, ws, stream=stream)
        stream.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        e0.record(stream)
        for _ in range(e_steps):
            G.gemm_f16_nt_host(a_h, b_h, c_h, a, b, c, ws, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize(dev)
        e2e = {"value": throughput(e0.elapsed_time(e1), w.flops, e_steps), "unit": UNIT,
               "h2d_bytes_per_step": 2 * (w.M * w.K + w.N * w.K), "d2h_bytes_per_step": 2 * w.M * w.N,
               "steps": e_steps}

    peaks = measured_peaks()
    regime = timing_regime(total_ms, clocks)
    roofline = tensor_roofline(value, regime, peaks)
    roofline.update({
        "traffic": traffic_record(w.name, plan), "algorithmic_bytes": w.algorithmic_bytes,
        "kernel": "gemm_f16_nt_wide_kernel" if plan.block_n > 256 else "gemm_f16_nt_kernel",
    })

    workloads = None
    if not args.no_workloads:
        workloads = {}
        for other in inputs.WORKLOADS:
            if other.name == w.name:
                workloads[other.name] = {"M": w.M, "N": w.N, "K": w.K, "ms": ms_per_step, "tflops": value,
                                         "note": "the headline step above", "roofline": roofline}
                continue
            workloads[other.name] = time_workload(G, other, dev, stream, sampler, args.workload_launches,
                                                  max(20, args.warmup), peaks)
    sampler.stop()

    cpu = None
    if not args.no_cpu_baseline:
        import oracle
        rate, secs, rows = cpu_oracle_rate(A, B, target_s=10.0)
        cpu = {"value": rate, "unit": UNIT, "cores": oracle.num_threads(), "kind": "oracle",
               "sample": "first %d of %d rows of C (all %d columns, full K=%d), %.1f s" % (rows, w.M, w.N, w.K, secs)}
    cfg = workload_config(w)
    cfg["plan"] = {k: v for k, v in plan.as_dict().items() if k in (
        "variant", "cta_group", "block_m", "block_n", "stages", "raster_width", "grid", "stream_k", "dp_tiles",
        "workspace_bytes", "split_k", "k_rotate")}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16", "data": "synthetic", "config": cfg,
        "frac_of_nominal_peak": value / NOMINAL_PEAK_TFLOPS,
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
        "gpu_launches": args.steps * (2 if plan.split_k > 1 else 1),  # a split-K plan adds its reduction
        "workloads": workloads,
    }
    print(json.dumps(line), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
