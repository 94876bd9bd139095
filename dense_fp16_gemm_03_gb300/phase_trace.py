"""Phase timeline of back-to-back launches of small products (measurement tool).

Builds the trace library (``build.build_trace``: the same sources with
GEMM_F16_PHASE_TRACE, whose single-CTA / CTA-pair kernel stamps %globaltimer at
ten phases per CTA), captures ``--launches`` calls of one product in a CUDA
graph with stamps taken for three consecutive launches in the middle, and
replays it.  For each traced launch it prints, per phase, the earliest and the
latest CTA (microseconds from the first traced launch's first entry), and the
hand-over from one launch's last exit to the next launch's release from its
dependency wait.  Beside it, the per-launch time of the product library
(no stamps) replayed the same way, and whether both libraries wrote the same C.

    python -m dense_fp16_gemm_03_gb300.phase_trace 64x64x64,256x256x256
"""
import argparse
import ctypes
import json
import statistics

import torch

from . import build as _build
from . import gemm as G

PHASES = ["entry", "set_up", "dep_wait", "first_full", "mma_done", "acc_ready", "stored", "stores_done",
          "teardown", "exit", "ks_sent", "ks_received"]
COMMON = PHASES[:10]  # phases every traced plan passes (the last two are the K-split exchange's)
SLOTS = 16


def _trace_lib():
    L = ctypes.CDLL(_build.build_trace())
    i64, vp = ctypes.c_int64, ctypes.c_void_p
    L.gemm_f16_nt_ws.restype = ctypes.c_int
    L.gemm_f16_nt_ws.argtypes = [i64, i64, i64, vp, vp, vp, vp, ctypes.c_size_t, vp]
    L.gemm_f16_trace_set.restype = None
    L.gemm_f16_trace_set.argtypes = [vp]
    L.gemm_f16_nt_run.restype = ctypes.c_int
    L.gemm_f16_nt_run.argtypes = [ctypes.POINTER(G.Plan), vp, vp, vp, vp, ctypes.c_size_t, vp]
    return L


def _replay_us(graph, stream, launches, reps=5):
    ts = []
    with torch.cuda.stream(stream):
        for _ in range(reps):
            graph.replay()
            stream.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            graph.replay()
            e1.record(stream)
            stream.synchronize()
            ts.append(e0.elapsed_time(e1) * 1000.0 / launches)
    return statistics.median(ts)


def trace_shape(m, n, k, launches=40, traced_at=20, seed=0, variant=-1):
    T = _trace_lib()
    P = G.lib()
    gen = torch.Generator(device="cuda").manual_seed(seed)
    a = (torch.randint(-8, 9, (m, k), device="cuda", generator=gen).to(torch.float16) / 8)
    b = (torch.randint(-8, 9, (n, k), device="cuda", generator=gen).to(torch.float16) / 8)
    c_trace = torch.empty((m, n), dtype=torch.float16, device="cuda")
    c_prod = torch.empty((m, n), dtype=torch.float16, device="cuda")
    plan = G.gemm_f16_nt_plan(m, n, k) if variant < 0 else G.gemm_f16_nt_plan_ex(m, n, k, variant, 0, 0)
    ws = torch.empty(max(256, int(plan.workspace_bytes)), dtype=torch.uint8, device="cuda")
    bufs = [torch.zeros(plan.grid * SLOTS, dtype=torch.int64, device="cuda") for _ in range(3)]
    stream = torch.cuda.Stream()

    def call_trace():
        st = T.gemm_f16_nt_run(ctypes.byref(plan), a.data_ptr(), b.data_ptr(), c_trace.data_ptr(), ws.data_ptr(),
                               ws.numel(), stream.cuda_stream)
        if st != 0:
            raise G.GemmError(st, "gemm_f16_nt_run (trace build)")

    def call_prod():
        st = P.gemm_f16_nt_run(ctypes.byref(plan), a.data_ptr(), b.data_ptr(), c_prod.data_ptr(), ws.data_ptr(),
                               ws.numel(), stream.cuda_stream)
        if st != 0:
            raise G.GemmError(st, "gemm_f16_nt_run")

    with torch.cuda.stream(stream):
        for _ in range(3):
            call_trace()
            call_prod()
    stream.synchronize()
    g_trace, g_prod = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_trace, stream=stream):
        for i in range(launches):
            if traced_at <= i < traced_at + 3:
                T.gemm_f16_trace_set(bufs[i - traced_at].data_ptr())
            call_trace()
            T.gemm_f16_trace_set(None)
    with torch.cuda.graph(g_prod, stream=stream):
        for _ in range(launches):
            call_prod()
    with torch.cuda.stream(stream):
        for t in bufs:
            t.zero_()
        g_trace.replay()
    stream.synchronize()
    stamps = [t.view(plan.grid, SLOTS).cpu() for t in bufs]
    us_prod = _replay_us(g_prod, stream, launches)
    us_trace = _replay_us(g_trace, stream, launches)
    same_c = bool(torch.equal(c_trace.view(torch.int16), c_prod.view(torch.int16)))
    del g_trace, g_prod

    if not all(bool((s[:, 0] != 0).any()) for s in stamps):
        raise ValueError("no stamps: the plan of %dx%dx%d runs the wide-tile kernel, which is not traced" % (m, n, k))
    t0 = int(stamps[0][:, 0].min())
    out = {"shape": "%dx%dx%d" % (m, n, k), "variant": plan.variant, "grid": plan.grid,
           "block_m": plan.block_m, "block_n": plan.block_n, "k_blocks": plan.k_blocks,
           "us_per_launch": round(us_prod, 3), "us_per_launch_traced": round(us_trace, 3),
           "same_c": same_c, "launches": []}
    monotone = True
    for s in stamps:
        row = {}
        for ph, name in enumerate(PHASES):
            col = s[:, ph]
            hit = col[col != 0]
            if hit.numel() == 0:
                continue
            row[name] = [round((int(hit.min()) - t0) / 1e3, 3), round((int(hit.max()) - t0) / 1e3, 3)]
        # per CTA, the phases it reached come in causal order.  Without a K split: entry .. teardown
        # each after the one before, and exit (thread 32 frees tensor memory after the teardown
        # barrier) after the stores completed, not necessarily after thread 0's teardown stamp.  With
        # one, the epilogue warps arrive on the teardown barrier right after the partner slices are in
        # and only then store C: accumulator ready, slices sent, slices received, stored, stores done
        # in order, and teardown and exit after the slices were received
        for cta in range(plan.grid):
            v = [int(x) for x in s[cta, :len(PHASES)].tolist()]
            if v[10] == 0 and v[11] == 0:
                chain = [x for x in v[:9] if x != 0]
                monotone &= all(x <= y for x, y in zip(chain, chain[1:]))
                if v[9] != 0 and v[7] != 0:
                    monotone &= v[7] <= v[9]
            else:
                chain = [x for x in (v[0], v[1], v[2], v[3], v[4], v[5], v[10], v[11], v[6], v[7]) if x != 0]
                monotone &= all(x <= y for x, y in zip(chain, chain[1:]))
                monotone &= all(v[11] <= x for x in (v[8], v[9]) if x != 0)
        out["launches"].append(row)
    out["phases_in_order"] = monotone
    out["handover_us"] = [round(out["launches"][i + 1]["dep_wait"][0] - out["launches"][i]["exit"][1], 3)
                          for i in range(2)]
    return out


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("shapes", help="comma-separated MxNxK list")
    ap.add_argument("--launches", type=int, default=40)
    ap.add_argument("--variants", default="-1", help="comma-separated variants (-1: the automatic plan)")
    args = ap.parse_args(argv)
    for spec in args.shapes.split(","):
        m, n, k = (int(x) for x in spec.split("x"))
        for v in args.variants.split(","):
            print(json.dumps(trace_shape(m, n, k, launches=args.launches, variant=int(v))), flush=True)


if __name__ == "__main__":
    main()
