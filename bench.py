#!/usr/bin/env python
"""Benchmark: quantized GEMV weight GB/s (and fraction of HBM peak) and tokens/s per layer.

Workload (default): one Llama-7B-shaped decode layer, Q4_0 with f16 scales, batch 1,
bfloat16 activations: wq, wo 4096x4096; wk, wv 1024x4096; w1, w3 11008x4096; w2 4096x11008
(99,680,256 weight bytes).  A step is the seven products y = W x of the layer, issued in
the order the layer's data dependencies allow -- {wq, wk, wv}, {wo}, {w1, w3}, {w2} -- as
four grouped libqmv launches (each may start fetching its weights while the previous one
finishes).  Consecutive steps are captured together in CUDA graphs of up to 500 steps, the
way a model's layers run one after another (a graph launch per layer would add its own
launch gap to every layer).  Weights are seeded synthetic data; distinct copies of the layer
rotate from step to step so that every step streams its weights from HBM (the copies
together are more than 4x the L2 size).

Prints one JSON line.  --impl reference times the CPU oracle (the plain C checker) on a
bounded sample of the same workload instead.  --case ROWS COLS WTYPE SCALE_F16 BATCH times one
product shape alone (the command the profiles under profiles/ run) and prints one JSON line
describing it.

Timing: warm-up steps, then K timed steps between CUDA events on the launching stream,
synchronized on both sides; with several GPUs every rank runs its own replica (nothing is
exchanged) and the slowest rank's time is used.
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

from block_quantized_weight_q4_gb300 import inputs  # noqa: E402

METRIC = "quantized GEMV weight GB/s (fraction of GB300 HBM peak) and tokens/s per layer"
UNIT = "GB/s"
WORKLOAD = "llama7b"
# launches of one layer step, in dependency order: the attention projections read the
# normalized input, wo reads the attention output, w1/w3 the normalized residual, w2 the
# gated product
LAYER_GROUPS = [["wq", "wk", "wv"], ["wo"], ["w1", "w3"], ["w2"]]
FALLBACK_HBM_GBS = 6800.0
STEPS_PER_GRAPH = 500  # layer steps captured in one CUDA graph


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=40000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-other-configs", action="store_true", help="only the headline workload")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="budget of the oracle sample")
    ap.add_argument("--case", type=int, nargs=5, metavar=("ROWS", "COLS", "WTYPE", "SCALE_F16", "BATCH"),
                    help="time one product shape alone (WTYPE 1 = Q8_0, 2 = Q4_0) instead of the workload")
    ap.add_argument("--x-f32", action="store_true", help="--case: float32 activations (default bfloat16)")
    ap.add_argument("--bf16-weights", action="store_true", help="--case: the prefill kernel's bf16-weights variant")
    ap.add_argument("--qx", action="store_true", help="--case: the activation-quantized product (qmv_matvec_qx_grouped)")
    ap.add_argument("--qx-image", action="store_true",
                    help="--case: the activation-quantized product on a quantized image (qmv_quantize_x once, "
                         "then qmv_matvec_qx per call)")
    ap.add_argument("--case-calls", type=int, default=20, help="--case: calls per timed CUDA graph")
    ap.add_argument("--case-copies", type=int, default=4, help="--case: rotating copies of the matrix")
    return ap.parse_args()


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world):
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


FALLBACK_BF16_TFLOPS = 1900.0


def measured_peaks():
    """(HBM GB/s, dense bf16 TFLOP/s burst, source) from the generated peaks file."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return (float(d.get("hbm_gbs", FALLBACK_HBM_GBS)), float(d.get("bf16_tflops", FALLBACK_BF16_TFLOPS)),
                "measured")
    return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, "fallback"


def layer_specs():
    return inputs.WORKLOADS[WORKLOAD].matrices


def layer_bytes(specs):
    return sum(inputs.array_offsets(s.wtype, s.scale_f16, s.rows, s.cols)[1] +
               inputs.array_offsets(s.wtype, s.scale_f16, s.rows, s.cols)[2] for s in specs)


def recorded_traffic(workload):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary, or None
    when the kernel source changed since the capture."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "roofline_traffic.txt")
    if not os.path.exists(path):
        return None
    for line in open(path):
        parts = line.split()
        if len(parts) == 4 and not line.startswith("#") and parts[3] == workload:
            src = os.path.join(ROOT, parts[0])
            if not os.path.exists(src):
                return None
            h = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
            return int(parts[2]) if h == parts[1] else None
    return None


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.path = None
        self.gpu = gpu_index

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        busy = [s for s in sm if mx and s >= 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ CPU oracle sample
def oracle_sample(specs, seconds, all_cores=False):
    """Time the oracle on the first rows of each matrix of the layer.

    Returns a dict: value (GB/s of weight bytes), cores, sample (text), rows, bytes, seconds."""
    import oracle
    oracle.build()
    mats, xs = [], []
    for i, s in enumerate(specs):
        mats.append(inputs.make_matrix(s.wtype, s.scale_f16, s.rows, s.cols, seed=inputs.matrix_seed(WORKLOAD, i)))
        xs.append(inputs.make_x(1, s.cols, True, seed=inputs.x_seed(WORKLOAD, i)))

    def run(nrows):
        nbytes = 0
        t0 = time.perf_counter()
        for m, x, s in zip(mats, xs, specs):
            r = min(nrows, s.rows)
            oracle.matvec_rows(m.W, s.wtype, s.scale_f16, s.rows, s.cols, x, np.arange(r))
            nbytes += r * s.cols * (0.5 if s.wtype == 2 else 1.0) + r * (s.cols // 32) * (2 if s.scale_f16 else 4)
        return time.perf_counter() - t0, int(nbytes)

    def run_threaded(nrows, nthreads):
        # the same oracle on every host core: each thread takes a contiguous share of the sampled
        # rows of every matrix (the oracle's C code runs outside the interpreter lock)
        import concurrent.futures as cf
        jobs, nbytes = [], 0
        for m, x, s in zip(mats, xs, specs):
            r = min(nrows, s.rows)
            nbytes += r * s.cols * (0.5 if s.wtype == 2 else 1.0) + r * (s.cols // 32) * (2 if s.scale_f16 else 4)
            for part in np.array_split(np.arange(r), nthreads):
                if part.size:
                    jobs.append((m, x, s, part))
        t0 = time.perf_counter()
        with cf.ThreadPoolExecutor(max_workers=nthreads) as ex:
            list(ex.map(lambda j: oracle.matvec_rows(j[0].W, j[2].wtype, j[2].scale_f16, j[2].rows, j[2].cols,
                                                     j[1], j[3]), jobs))
        return time.perf_counter() - t0, int(nbytes)

    t1, _ = run(1)  # calibration: one row of every matrix
    nrows = max(1, int(seconds / max(t1, 1e-9)))
    dt, nbytes = run(nrows)
    desc = (f"first {nrows} rows of each of the 7 layer matrices, batch 1, bf16 x "
            f"({nbytes / 1e6:.2f} MB of the layer's {layer_bytes(specs) / 1e6:.2f} MB), single thread")
    out = {"value": nbytes / dt / 1e9, "cores": 1, "sample": desc, "rows": nrows, "bytes": nbytes,
           "seconds": dt, "run": run}
    ncores = os.cpu_count() or 1
    if all_cores and ncores > 1:
        nrt = nrows * ncores
        dtt, nbt = run_threaded(nrt, ncores)
        out["all_cores"] = {"value": nbt / dtt / 1e9, "unit": UNIT, "cores": ncores,
                            "sample": f"first {nrt} rows of each of the 7 layer matrices, batch 1, bf16 x, "
                                      f"{ncores} threads over row ranges"}
    return out


def run_reference(args, world, rank):
    """The oracle as it stands, timed on the host cores; rank 0 only."""
    if rank != 0:
        return
    specs = layer_specs()
    per_step = 90.0 / max(1, args.steps + args.warmup)  # whole run within about 1.5 minutes
    smp = oracle_sample(specs, min(per_step, 2.0))
    times = []
    for step in range(args.warmup + args.steps):
        dt, nbytes = smp["run"](smp["rows"])
        if step >= args.warmup:
            times.append(dt)
    t = sum(times) / len(times)
    v = smp["bytes"] / t / 1e9
    out = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": args.gpus,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": t * 1e3, "higher_is_better": True,
           "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
           "config": {"workload": "llama7b_decode_layer_q4_0_f16_batch1", "sample": smp["sample"]},
           "cpu_baseline": {"value": v, "unit": UNIT, "cores": smp["cores"], "kind": "oracle",
                            "sample": smp["sample"]},
           "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)



# ------------------------------------------------------------------ other workloads
def _graph_time_us(torch, launches, cap, replays=5):
    """Per-launch GPU time of a list of launch closures, replayed as one CUDA graph (warmed up
    on the capture stream, whose first calls create its workspaces)."""
    with torch.cuda.stream(cap):
        for f in launches[:2]:
            f()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        for f in launches:
            f()
    g.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(st)
    for _ in range(replays):
        g.replay()
    b.record(st)
    torch.cuda.synchronize()
    return a.elapsed_time(b) * 1e3 / (replays * len(launches))


def other_workloads(torch, qmv, dev, l2, cap, peak_hbm, peak_tf):
    """The remaining workloads, each timed on its own (weight copies rotate past 4x L2)."""
    res = {}

    def copies_for(W, nbytes, minimum=2):
        n = max(minimum, -(-4 * l2 // nbytes) + 1)
        return [W] + [W.clone() for _ in range(n - 1)]

    def xdev(x):
        if x.dtype == np.uint16:
            return torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16)
        return torch.from_numpy(x).to(dev)

    # Q8_0 256 x 256, f32 scales, f32 x, batch 1, seed 0: a few microseconds of launch latency
    m = inputs.make_matrix(1, 0, 256, 256, seed=0)
    W = torch.from_numpy(m.W).to(dev)
    x = xdev(inputs.make_x(1, 256, False, seed=0))
    y = torch.empty((1, 256), device=dev)
    us = _graph_time_us(torch, [lambda: qmv.matvec(1, 0, 256, 256, W, x, y)] * 64, cap)
    res["q8_256_f32x_b1"] = {"us_per_product": round(us, 3), "weight_gbs": round(m.W.size / us / 1e3, 1),
                             "note": "73,728 weight bytes: bound by launch latency, not HBM"}

    # Q4_0 4096 x 4096, f16 scales, bf16 x, batch 1: a stream of products over rotating copies,
    # plain and with programmatic overlap between consecutive launches
    m = inputs.make_matrix(2, 1, 4096, 4096, seed=0)
    Ws = copies_for(torch.from_numpy(m.W).to(dev), m.W.size)
    x = xdev(inputs.make_x(1, 4096, True, seed=1000))
    y = torch.empty((1, 4096), device=dev)
    n = len(Ws)
    plain = _graph_time_us(torch, [lambda i=i: qmv.matvec(2, 1, 4096, 4096, Ws[i % n], x, y) for i in range(2 * n)], cap)
    ov = _graph_time_us(torch, [lambda i=i: qmv.matvec_grouped(2, 1, [(4096, 4096, Ws[i % n], x, y)], overlap=True)
                                for i in range(2 * n)], cap)
    # Q4_0 65536 x 4096 (151 MB), f16 scales, bf16 x, batch 1: one large launch, rotating copies
    ml = inputs.make_matrix(2, 1, 65536, 4096, seed=0)
    Wl = copies_for(torch.from_numpy(ml.W).to(dev), ml.W.size)
    xl = xdev(inputs.make_x(1, 4096, True, seed=1000))
    yl = torch.empty((1, 65536), device=dev)
    nl = len(Wl)
    us_l = _graph_time_us(torch, [lambda i=i: qmv.matvec(2, 1, 65536, 4096, Wl[i % nl], xl, yl) for i in range(2 * nl)],
                          cap)
    res["q4_65536x4096_f16_b1"] = {"us_per_product": round(us_l, 3), "weight_gbs": round(ml.W.size / us_l / 1e3, 1),
                                   "frac_hbm": round(ml.W.size / us_l / 1e3 / peak_hbm, 4)}
    del Wl, ml
    res["q4_4096_f16_b1"] = {"us_per_product": round(plain, 3), "weight_gbs": round(m.W.size / plain / 1e3, 1),
                             "frac_hbm": round(m.W.size / plain / 1e3 / peak_hbm, 4),
                             "overlapped_us_per_product": round(ov, 3),
                             "overlapped_weight_gbs": round(m.W.size / ov / 1e3, 1),
                             "overlapped_frac_hbm": round(m.W.size / ov / 1e3 / peak_hbm, 4)}
    del Ws

    # mixed q8_mask = 2 model: Q4_0 body of one dim-1024 layer (f32 scales) + Q8_0 classifier
    wl = inputs.WORKLOADS["mixed_qwen"]
    mats, nbytes = [], 0
    for i, spec in enumerate(wl.matrices):
        wt = qmv.matrix_wtype(wl.file_wtype, wl.q8_mask, spec.cls)
        mm = inputs.make_matrix(wt, spec.scale_f16, spec.rows, spec.cols, seed=inputs.matrix_seed("mixed_qwen", i))
        mats.append((spec, wt, torch.from_numpy(mm.W).to(dev)))
        nbytes += mm.W.size
    ncopy = max(2, -(-4 * l2 // nbytes) + 1)
    sets = [[(s, wt, W if c == 0 else W.clone()) for s, wt, W in mats] for c in range(ncopy)]
    body_groups = [["wq", "wk", "wv"], ["wo"], ["w1", "w3"], ["w2"]]
    for batch in wl.batches:
        for xbf16 in (True, False):
            xs = [xdev(inputs.make_x(batch, s.cols, xbf16, seed=inputs.x_seed("mixed_qwen", i)))
                  for i, (s, _, _) in enumerate(mats)]
            ys = [torch.empty((batch, s.rows), device=dev) for s, _, _ in mats]
            idx = {s.name: i for i, (s, _, _) in enumerate(mats)}

            def step(c):
                for grp in body_groups:
                    probs = [(sets[c][idx[n]][0].rows, sets[c][idx[n]][0].cols, sets[c][idx[n]][2], xs[idx[n]],
                              ys[idx[n]]) for n in grp]
                    qmv.matvec_grouped(2, 0, probs, overlap=True)
                s, wt, W = sets[c][idx["wcls"]]
                qmv.matvec_grouped(wt, 0, [(s.rows, s.cols, W, xs[idx["wcls"]], ys[idx["wcls"]])], overlap=True)
            us = _graph_time_us(torch, [lambda c=c: step(c) for c in range(ncopy)] * 2, cap)
            s, wt, W = sets[0][idx["wcls"]]
            cls_us = _graph_time_us(torch, [lambda c=c: qmv.matvec(wt, 0, s.rows, s.cols, sets[c][idx["wcls"]][2],
                                                                   xs[idx["wcls"]], ys[idx["wcls"]])
                                            for c in range(ncopy)] * 2, cap)
            cls_bytes = inputs.array_offsets(wt, 0, s.rows, s.cols)
            cls_bytes = cls_bytes[1] + cls_bytes[2]
            res[f"mixed_qwen_b{batch}_{'bf16' if xbf16 else 'f32'}x"] = {
                "us_per_model_step": round(us, 3), "weight_gbs": round(nbytes / us / 1e3, 1),
                "frac_hbm": round(nbytes / us / 1e3 / peak_hbm, 4), "tokens_per_s": round(batch / (us * 1e-6), 1),
                "classifier_us": round(cls_us, 3), "classifier_gbs": round(cls_bytes / cls_us / 1e3, 1),
                "classifier_frac_hbm": round(cls_bytes / cls_us / 1e3 / peak_hbm, 4)}
    del sets, mats

    # prefill: Q4_0 f16, W 14336 x 4096 and 4096 x 14336, X bf16 of 16, 64, 128 tokens
    for i, spec in enumerate(inputs.WORKLOADS["prefill"].matrices):
        mm = inputs.make_matrix(2, 1, spec.rows, spec.cols, seed=i)
        Ws = copies_for(torch.from_numpy(mm.W).to(dev), mm.W.size)
        n = len(Ws)
        for batch in inputs.WORKLOADS["prefill"].batches:
            x = xdev(inputs.make_x(batch, spec.cols, True, seed=1000 + i))
            y = torch.empty((batch, spec.rows), device=dev)
            us = _graph_time_us(torch, [lambda j=j: qmv.matvec(2, 1, spec.rows, spec.cols, Ws[j % n], x, y)
                                        for j in range(2 * n)], cap)
            # the same products launched with the overlap flag: each call's weight loads start
            # while the previous call finishes (its activations and y still wait for it)
            ov_us = _graph_time_us(torch, [lambda j=j: qmv.matvec_grouped(
                2, 1, [(spec.rows, spec.cols, Ws[j % n], x, y)], overlap=True) for j in range(2 * n)], cap)
            flops = 2.0 * spec.rows * spec.cols * batch
            # batch 16 over 8 MB of weights takes one 16-vector pass of the tensor-memory decode
            # kernel (measured faster there than the prefill kernel)
            kern = "decode_tc (16-vector pass)" if batch <= 16 and mm.W.size >= (8 << 20) else "prefill"
            res[f"prefill_{spec.rows}x{spec.cols}_b{batch}"] = {
                "kernel": kern, "us": round(us, 3), "tflops": round(flops / us / 1e6, 1),
                "frac_bf16_tensor_peak": round(flops / us / 1e6 / peak_tf, 4),
                "weight_gbs": round(mm.W.size / us / 1e3, 1), "frac_hbm": round(mm.W.size / us / 1e3 / peak_hbm, 4),
                "overlapped_us": round(ov_us, 3), "overlapped_tflops": round(flops / ov_us / 1e6, 1),
                "overlapped_frac_bf16_tensor_peak": round(flops / ov_us / 1e6 / peak_tf, 4)}
        del Ws

    # the writer rules on the device: float32 14336 x 4096 (235 MB, past L2) into Q4_0 with
    # f16 scales and Q8_0 with f32 scales; bytes = float32 read + quantized bytes written
    lib = qmv.load_library()
    rows, cols = 14336, 4096
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    src = torch.randn((rows, cols), device=dev, generator=gen, dtype=torch.float32)
    first = torch.empty(1, dtype=torch.int64, device=dev)
    for wt, sf, name in ((2, 1, "q4_0_f16"), (1, 0, "q8_0_f32")):
        nbytes = qmv.weight_bytes(wt, sf, rows, cols)
        W = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        call = lambda wt=wt, sf=sf, W=W: lib.qmv_quantize(wt, sf, rows, cols, src.data_ptr(), W.data_ptr(),
                                                        first.data_ptr(), torch.cuda.current_stream().cuda_stream)
        us = _graph_time_us(torch, [call] * 8, cap)
        moved = 4 * rows * cols + nbytes
        res[f"quantize_{rows}x{cols}_{name}"] = {
            "us": round(us, 3), "gbs": round(moved / us / 1e3, 1), "frac_hbm": round(moved / us / 1e3 / peak_hbm, 4),
            "bytes": moved}
        del W
    # the Q4_0 best-fit writer (13 candidate fits per block): compute-bound, reported in GB/s too
    nbytes = qmv.weight_bytes(2, 1, rows, cols)
    W = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    call = lambda: lib.qmv_quantize_q4_fit(1, rows, cols, src.data_ptr(), W.data_ptr(), first.data_ptr(),
                                           torch.cuda.current_stream().cuda_stream)
    us = _graph_time_us(torch, [call] * 4, cap)
    moved = 4 * rows * cols + nbytes
    res[f"quantize_q4_fit_{rows}x{cols}_f16"] = {
        "us": round(us, 3), "gbs": round(moved / us / 1e3, 1), "frac_hbm": round(moved / us / 1e3 / peak_hbm, 4),
        "bytes": moved}
    del W
    del src

    # GGUF interleaved blocks into the two-array layout: the page's 151,936 x 896 tensors
    # (Q8_0 output.weight, Q4_0 token_embd.weight); bytes = the tensor read + the same written;
    # source / destination pairs rotate past 4x L2
    rows, cols = 151936, 896
    for wt, name in ((1, "q8_0"), (2, "q4_0")):
        gb = qmv.gguf_bytes(wt, rows, cols)
        moved = gb + qmv.weight_bytes(wt, 1, rows, cols)
        npair = max(2, -(-4 * l2 // moved) + 1)
        gs = [torch.randint(0, 256, (gb,), dtype=torch.uint8, device=dev) for _ in range(npair)]
        Wd = [torch.empty(qmv.weight_bytes(wt, 1, rows, cols), dtype=torch.uint8, device=dev) for _ in range(npair)]
        us = _graph_time_us(torch, [lambda wt=wt, i=i: qmv.gguf_to_mlb(wt, rows, cols, gs[i % npair], W=Wd[i % npair])
                                    for i in range(2 * npair)], cap)
        res[f"gguf_to_mlb_{rows}x{cols}_{name}"] = {
            "us": round(us, 3), "gbs": round(moved / us / 1e3, 1), "frac_hbm": round(moved / us / 1e3 / peak_hbm, 4),
            "bytes": moved}
        del gs, Wd

    # the activation-quantized product (activations to Q8_0 blocks by qmv_quantize_x, then exact
    # int8 block dot products by qmv_matvec_qx): Q4_0 65536 x 4096 alone, batch 1 and 8, and
    # the Llama-7B layer step with one quantized activation vector per dependency group
    m = inputs.make_matrix(2, 1, 65536, 4096, seed=0)
    Ws = copies_for(torch.from_numpy(m.W).to(dev), m.W.size)
    n = len(Ws)
    for batch in (1, 8):
        x = xdev(inputs.make_x(batch, 4096, True, seed=1000))
        xq = qmv.quantize_x(x)
        y = torch.empty((batch, 65536), device=dev)
        us = _graph_time_us(torch, [lambda i=i: qmv.matvec_qx(2, 1, 65536, 4096, Ws[i % n], xq, batch, y=y)
                                    for i in range(2 * n)], cap)
        qus = _graph_time_us(torch, [lambda: qmv.quantize_x(x, xq=xq)] * 64, cap)
        # the quantizer inside the call (qmv_matvec_qx_grouped): one launch at one vector, a
        # quantizer launch and the product at 8
        gus = _graph_time_us(torch, [lambda i=i: qmv.matvec_qx_grouped(2, 1, [(65536, 4096, Ws[i % n], x, y)])
                                     for i in range(2 * n)], cap)
        res[f"qx_q4_65536x4096_f16_b{batch}"] = {
            "us_per_product": round(us, 3), "weight_gbs": round(m.W.size / us / 1e3, 1),
            "frac_hbm": round(m.W.size / us / 1e3 / peak_hbm, 4), "quantize_x_us": round(qus, 3),
            "grouped_us_per_product": round(gus, 3), "grouped_weight_gbs": round(m.W.size / gus / 1e3, 1),
            "grouped_frac_hbm": round(m.W.size / gus / 1e3 / peak_hbm, 4),
            "grouped_launches": 1 if batch == 1 else 2}
    del Ws
    specs = layer_specs()
    lb = layer_bytes(specs)
    ncopy = max(2, -(-4 * l2 // lb) + 1)
    mats = [torch.from_numpy(inputs.make_matrix(s.wtype, s.scale_f16, s.rows, s.cols,
                                                seed=inputs.matrix_seed(WORKLOAD, i)).W).to(dev)
            for i, s in enumerate(specs)]
    copies = [[w if c == 0 else w.clone() for w in mats] for c in range(ncopy)]
    names = [s.name for s in specs]
    groups = [[names.index(nm) for nm in grp] for grp in LAYER_GROUPS]
    gx = [xdev(inputs.make_x(1, specs[grp[0]].cols, True, seed=inputs.x_seed(WORKLOAD, grp[0]))) for grp in groups]
    gxq = [qmv.quantize_x(x) for x in gx]
    ys = [torch.empty((1, s.rows), device=dev) for s in specs]

    def qx_step(c):
        for g, grp in enumerate(groups):
            qmv.quantize_x(gx[g], xq=gxq[g])
            for i in grp:
                s = specs[i]
                qmv.matvec_qx(s.wtype, s.scale_f16, s.rows, s.cols, copies[c][i], gxq[g], 1, y=ys[i])

    us = _graph_time_us(torch, [lambda c=c: qx_step(c) for c in range(ncopy)] * 2, cap)
    res["qx_llama7b_layer_unfused_b1"] = {"us_per_step": round(us, 3), "weight_gbs": round(lb / us / 1e3, 1),
                                          "frac_hbm": round(lb / us / 1e3 / peak_hbm, 4),
                                          "launches_per_step": len(groups) + len(specs),
                                          "note": "qmv_quantize_x per group, then qmv_matvec_qx per matrix"}

    def qx_fused_step(c):
        for g, grp in enumerate(groups):
            qmv.matvec_qx_grouped(2, 1, [(specs[i].rows, specs[i].cols, copies[c][i], gx[g], ys[i]) for i in grp],
                                  overlap=True)

    us = _graph_time_us(torch, [lambda c=c: qx_fused_step(c) for c in range(ncopy)] * 2, cap)
    res["qx_llama7b_layer_b1"] = {"us_per_step": round(us, 3), "weight_gbs": round(lb / us / 1e3, 1),
                                  "frac_hbm": round(lb / us / 1e3 / peak_hbm, 4), "launches_per_step": len(groups),
                                  "note": "qmv_matvec_qx_grouped per group: activations quantized inside the "
                                          "product, grouped problems, programmatic overlap"}

    # the layer step with the FFN's SwiGLU in the down projection's activation prep: w1 and w3
    # write gate and up into one buffer, w2 takes SiLU(gate) * up as float32 activations
    xs_b = [xdev(inputs.make_x(1, s.cols, True, seed=inputs.x_seed(WORKLOAD, i))) for i, s in enumerate(specs)]
    i1, i3, i2 = names.index("w1"), names.index("w3"), names.index("w2")
    gu = torch.empty((2, 1, specs[i1].rows), device=dev)
    outs = {i: ys[i] for i in range(len(specs))}
    outs[i1], outs[i3] = gu[0], gu[1]

    def glu_step(c):
        for grp in groups:
            s0 = specs[grp[0]]
            if grp == [i2]:
                qmv.matvec_grouped(s0.wtype, s0.scale_f16, [(s0.rows, s0.cols, copies[c][i2], gu, ys[i2])],
                                   overlap=True, act="silu")
            else:
                qmv.matvec_grouped(s0.wtype, s0.scale_f16,
                                   [(specs[i].rows, specs[i].cols, copies[c][i], xs_b[i], outs[i]) for i in grp],
                                   overlap=True)

    us = _graph_time_us(torch, [lambda c=c: glu_step(c) for c in range(ncopy)] * 2, cap)
    res["llama7b_layer_swiglu_unfused_b1"] = {
        "us_per_step": round(us, 3), "weight_gbs": round(lb / us / 1e3, 1), "frac_hbm": round(lb / us / 1e3 / peak_hbm, 4),
        "launches_per_step": 5,
        "note": "{w1,w3} into float32 gate and up; w2 on SiLU(gate) * up (split kernel + hi/lo bf16 product)"}

    # the same step with the activation as the {w1,w3} launch's epilogue (qmv_matvec_glu writes
    # SiLU(w1 x) * (w3 x) as a bf16 hi/lo pair that w2 reads directly): four launches
    hpair = torch.empty((2, specs[i1].rows), dtype=torch.bfloat16, device=dev)

    def fused_step(c):
        for grp in groups:
            s0 = specs[grp[0]]
            if grp == [i1, i3]:
                qmv.matvec_glu(s0.wtype, s0.scale_f16, s0.rows, s0.cols, copies[c][i1], copies[c][i3], xs_b[i1][0],
                               act="silu", h=hpair, overlap=True)
            elif grp == [i2]:
                qmv.matvec_grouped(s0.wtype, s0.scale_f16, [(s0.rows, s0.cols, copies[c][i2], hpair, ys[i2])],
                                   overlap=True, pair=True)
            else:
                qmv.matvec_grouped(s0.wtype, s0.scale_f16,
                                   [(specs[i].rows, specs[i].cols, copies[c][i], xs_b[i], outs[i]) for i in grp],
                                   overlap=True)

    us_f = _graph_time_us(torch, [lambda c=c: fused_step(c) for c in range(ncopy)] * 2, cap)
    res["llama7b_layer_swiglu_b1"] = {
        "us_per_step": round(us_f, 3), "weight_gbs": round(lb / us_f / 1e3, 1),
        "frac_hbm": round(lb / us_f / 1e3 / peak_hbm, 4), "launches_per_step": 4,
        "note": "SiLU(w1 x) * (w3 x) as the epilogue of the {w1,w3} launch (qmv_matvec_glu), written as the bf16 "
                "hi/lo pair w2 reads (x_dtype QMV_X_BF16_PAIR)"}
    del copies, mats
    return res

# ------------------------------------------------------------------ GPU arm
def run_ours(args, world, rank, local):
    import torch
    import block_quantized_weight_q4_gb300 as qmv
    from block_quantized_weight_q4_gb300.build import build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (no CPU fallback)")
    torch.cuda.set_device(local)
    build()
    qmv.load_library()
    dev = torch.device("cuda", local)
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))

    specs = layer_specs()
    lb = layer_bytes(specs)
    ncopy = max(2, -(-4 * l2 // lb) + 1)

    # seeded synthetic weights (host), uploaded once, then cloned into rotating copies
    Ws = []
    for i, s in enumerate(specs):
        m = inputs.make_matrix(s.wtype, s.scale_f16, s.rows, s.cols, seed=inputs.matrix_seed(WORKLOAD, i))
        Ws.append(torch.from_numpy(m.W).to(dev))
    copies = [[w if c == 0 else w.clone() for w in Ws] for c in range(ncopy)]
    xs_host = [inputs.make_x(1, s.cols, True, seed=inputs.x_seed(WORKLOAD, i)) for i, s in enumerate(specs)]
    xs = [torch.from_numpy(x.view(np.int16)).to(dev).view(torch.bfloat16) for x in xs_host]
    ys = [torch.empty((1, s.rows), dtype=torch.float32, device=dev) for s in specs]

    names = [s.name for s in specs]
    groups = [[names.index(n) for n in grp] for grp in LAYER_GROUPS]

    def step(c):
        for grp in groups:
            qmv.matvec_grouped(specs[grp[0]].wtype, specs[grp[0]].scale_f16,
                               [(specs[i].rows, specs[i].cols, copies[c][i], xs[i], ys[i]) for i in grp],
                               overlap=True)

    # eager warm-up on the capture stream (sets kernel attributes, creates the stream's
    # workspace), then graphs of consecutive steps: `chunk` steps each, and the remainder
    cap = torch.cuda.Stream()
    with torch.cuda.stream(cap):
        for c in range(ncopy):
            step(c)
    torch.cuda.synchronize()

    def capture(nsteps, first):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            for i in range(nsteps):
                step((first + i) % ncopy)
        return g

    chunk = min(args.steps, STEPS_PER_GRAPH)
    g_chunk = capture(chunk, 0)
    rem = args.steps % chunk
    g_rem = capture(rem, (args.steps // chunk) * chunk) if rem else None
    g_warm = capture(min(args.warmup, STEPS_PER_GRAPH), 0)
    for _ in range(-(-args.warmup // STEPS_PER_GRAPH)):
        g_warm.replay()
    # the graphs timed below are replayed once first: a graph's first launch uploads it to the
    # device, a one-time cost that does not belong to the steps
    g_chunk.replay()
    if g_rem is not None:
        g_rem.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # a spin kernel of ~50 us ahead of the start event keeps the GPU busy while the host submits
    # the timed graphs, so that the first timed step does not wait for the submission (a decode
    # loop's steps follow one another on a GPU that never idles); it ends before the start event
    torch.cuda._sleep(100000)
    e0.record(stream)
    for _ in range(args.steps // chunk):
        g_chunk.replay()
    if g_rem is not None:
        g_rem.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    clk = clocks.stop()
    ms = e0.elapsed_time(e1) / args.steps
    ms = max_over_ranks(ms, world)
    status = qmv.last_error()
    if status != 0:
        raise SystemExit(f"device status {status} after the timed region")

    value = lb * world / (ms * 1e-3) / 1e9
    tokens_per_s = 1.0 / (ms * 1e-3)

    # per-launch kernel durations: each of the step's four grouped launches alone, back to back
    # over the rotating copies (with the overlap flag, as in the step), captured in a graph
    def time_graph(launch, reps):
        gm = torch.cuda.CUDAGraph()
        with torch.cuda.graph(gm, stream=cap):
            for r in range(reps):
                launch(r)
        gm.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(5):
            gm.replay()
        b.record(stream)
        torch.cuda.synchronize()
        del gm
        return a.elapsed_time(b) * 1e3 / (5 * reps)

    reps = 4 * ncopy
    per_launch = {}
    launch_us, launch_bytes = [], []
    for grp in groups:
        nb = sum(sum(inputs.array_offsets(specs[i].wtype, specs[i].scale_f16, specs[i].rows, specs[i].cols)[1:])
                 for i in grp)

        def launch(r, grp=grp):
            qmv.matvec_grouped(specs[grp[0]].wtype, specs[grp[0]].scale_f16,
                               [(specs[i].rows, specs[i].cols, copies[r % ncopy][i], xs[i], ys[i]) for i in grp],
                               overlap=True)
        us = time_graph(launch, reps)
        launch_us.append(us)
        launch_bytes.append(nb)
        per_launch["{" + ",".join(names[i] for i in grp) + "}"] = {
            "us": round(us, 3), "gbs": round(nb / (us * 1e-6) / 1e9, 1), "bytes": nb}
    # and each matrix alone (plain calls)
    per_matrix = {}
    for i, s in enumerate(specs):
        nb = sum(inputs.array_offsets(s.wtype, s.scale_f16, s.rows, s.cols)[1:])
        us = time_graph(lambda r, i=i, s=s: qmv.matvec(s.wtype, s.scale_f16, s.rows, s.cols, copies[r % ncopy][i],
                                                       xs[i], ys[i]), reps)
        per_matrix[s.name] = {"us": round(us, 3), "gbs": round(nb / (us * 1e-6) / 1e9, 1)}

    # end to end through the public API: pinned host x in, y back to pinned host
    x_all = np.concatenate([x.reshape(-1) for x in xs_host])
    xh = torch.from_numpy(x_all.view(np.int16)).pin_memory()
    xd = torch.empty_like(xh, device=dev)
    offs = np.cumsum([0] + [s.cols for s in specs])
    yh = torch.empty(sum(s.rows for s in specs), dtype=torch.float32).pin_memory()
    yoffs = np.cumsum([0] + [s.rows for s in specs])
    # one gated compiled step per weight copy (qmv_step_create_gated): a gate kernel that waits
    # until the host opens the run and then copies x from pinned host memory to the device, the
    # four dependency-ordered grouped launches, whose kernels store y straight into the pinned
    # host buffer (mapped into the device's address space: the device -> host transfer of the
    # result, without a copy launch after the last product), and a kernel that reports the run
    # done to the host.  Every step: the host opens the run (its input in place), enqueues the
    # next token's run behind it (which waits at its gate) and waits for this run's y, all in
    # one call (qmv_step_open_wait), as a decode loop must before its next token
    xb = xd.view(torch.bfloat16)
    e2e_steps_objs = [qmv.Step([(specs[grp[0]].wtype, specs[grp[0]].scale_f16,
                                 [(specs[i].rows, specs[i].cols, copies[c][i],
                                   xb[offs[i]:offs[i + 1]].view(1, specs[i].cols),
                                   yh[yoffs[i]:yoffs[i + 1]].view(1, specs[i].rows)) for i in grp], True)
                                for grp in groups], before=[(xd, xh)], gated=True)
                      for c in range(ncopy)]
    e2e_steps = max(10, min(args.steps, 2000))
    stream = torch.cuda.current_stream()
    for it in range(min(e2e_steps, 3 * ncopy)):   # warm-up
        e2e_steps_objs[it % ncopy].run(stream, wait=True)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    e2e_steps_objs[0].run(stream)                   # the first token's run, waiting at its gate
    for it in range(e2e_steps):
        nxt = e2e_steps_objs[(it + 1) % ncopy] if it + 1 < e2e_steps else None
        e2e_steps_objs[it % ncopy].open_wait(nxt, stream)   # open, enqueue the next, wait for y
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    for st in e2e_steps_objs:
        st.close()
    e2e_s = max_over_ranks(e2e_s, world)
    e2e = {"value": lb * world / e2e_s / 1e9, "unit": UNIT, "h2d_bytes_per_step": int(xh.numel() * 2),
           "d2h_bytes_per_step": int(yh.numel() * 4), "ms_per_step": e2e_s * 1e3,
           "d2h": "the products' stores into pinned host memory",
           "loop": "gated compiled steps: each run opened by the host after the previous y, the next run enqueued behind it"}

    peak, peak_tf, peak_src = measured_peaks()
    # the dominant (only) kernel of the step runs its four launches; achieved = algorithmic bytes
    # per launch / mean launch duration, both averaged over the four (each launch timed alone)
    avg_us = sum(launch_us) / len(launch_us)
    achieved = (lb / len(LAYER_GROUPS)) / (avg_us * 1e-6) / 1e9
    roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "traffic": recorded_traffic("llama7b_decode_layer_q4_0_f16_batch1"), "peak_source": peak_src,
                "kernel": "matvec_bdiag_kernel<Q4_0, f16 scales> (one bf16 vector)",
                "bytes_per_launch": round(lb / len(LAYER_GROUPS)),
                "avg_launch_us": round(avg_us, 3),
                "step_us": round(ms * 1e3, 3),
                "timing": "each of the 4 grouped launches timed alone over rotating copies (CUDA events around "
                          "graph replays); the step's value includes the launch boundaries"}

    others = None
    if not args.no_other_configs:
        others = other_workloads(torch, qmv, dev, l2, cap, peak, peak_tf)

    cpu = None
    if rank == 0 and not args.no_cpu_baseline:
        smp = oracle_sample(specs, args.cpu_seconds, all_cores=True)
        cpu = {"value": smp["value"], "unit": UNIT, "cores": smp["cores"], "kind": "oracle", "sample": smp["sample"]}
        if "all_cores" in smp:
            cpu["all_cores"] = smp["all_cores"]

    if rank == 0:
        out = {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
               "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
               "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
               "config": {"workload": "llama7b_decode_layer_q4_0_f16_batch1",
                          "matrices": {s.name: [s.rows, s.cols] for s in specs}, "batch": 1,
                          "x_dtype": "bf16", "weight_bytes_per_step": lb, "parallelism": f"replicas{world}",
                          "l2_defeat": f"{ncopy} rotating weight copies, {ncopy * lb / 1e6:.0f} MB > 4x L2 "
                                       f"({l2 / 1e6:.0f} MB)",
                          "step": "4 grouped libqmv launches: {wq,wk,wv} {wo} {w1,w3} {w2}; consecutive steps "
                                  f"captured together in CUDA graphs of up to {STEPS_PER_GRAPH} steps, each graph "
                                  "replayed once before the timed region; a ~50 us spin kernel ahead of the start "
                                  "event covers the host's submission of the first timed graph"},
               "tokens_per_s_per_layer": round(tokens_per_s * world, 1),
               "per_launch": per_launch, "per_matrix": per_matrix, "other_workloads": others, "e2e": e2e, "roofline": roofline, "cpu_baseline": cpu,
               "clocks": clk, "gpu_launches": len(LAYER_GROUPS) * args.steps}
        print(json.dumps(out), flush=True)


# ------------------------------------------------------------------ one shape (--case)
def run_case(args):
    """One product shape through libqmv: a few eager calls, then back-to-back calls over
    rotating copies captured in a CUDA graph (no host overhead between calls), timed with CUDA
    events.  Seeded synthetic weights (uniform quants, scales ~ U[1e-3, 2e-2]) and N(0, 1)
    activations.  Prints one JSON line."""
    import torch
    import block_quantized_weight_q4_gb300 as qmv
    from block_quantized_weight_q4_gb300.build import build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (no CPU fallback)")
    rows, cols, wt, sf, batch = args.case
    build()
    qmv.load_library()
    m = inputs.make_matrix(wt, sf, rows, cols, seed=1)
    W0 = torch.from_numpy(m.W).cuda()
    ncopy = max(1, args.case_copies)
    Ws = [W0] + [W0.clone() for _ in range(ncopy - 1)]
    x = inputs.make_x(batch, cols, not args.x_f32, seed=2)
    xd = torch.from_numpy(x).cuda() if args.x_f32 else torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    y = torch.empty((batch, rows), device="cuda")

    xq = qmv.quantize_x(xd) if args.qx_image else None

    def call(i):
        if args.qx_image:
            qmv.matvec_qx(wt, sf, rows, cols, Ws[i % ncopy], xq, batch, y)
        elif args.qx:
            qmv.matvec_qx_grouped(wt, sf, [(rows, cols, Ws[i % ncopy], xd, y)])
        else:
            qmv.matvec_grouped(wt, sf, [(rows, cols, Ws[i % ncopy], xd, y)], bf16_weights=args.bf16_weights)

    # eager calls on the stream that is captured below: a stream's first call creates the
    # workspaces its kernels use (never while it is being captured)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for i in range(max(args.warmup, 1)):
            call(i)
    torch.cuda.synchronize()
    out = {"case": {"rows": rows, "cols": cols, "wtype": wt, "scale_f16": sf, "batch": batch,
                    "x_dtype": "f32" if args.x_f32 else "bf16", "bf16_weights": bool(args.bf16_weights),
                    "activation_quantized": "image" if args.qx_image else bool(args.qx),
                    "copies": ncopy}}
    if args.case_calls > 0:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(args.case_calls):
                call(i)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(max(args.steps, 1)):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (max(args.steps, 1) * args.case_calls)
        peak, peak_tf, src = measured_peaks()
        out.update({"us_per_call": round(us, 3), "weight_gbs": round(m.W.size / us / 1e3, 1),
                    "frac_hbm": round(m.W.size / us / 1e3 / peak, 4),
                    "tflops": round(2.0 * rows * cols * batch / us / 1e6, 1),
                    "frac_bf16_tensor_peak": round(2.0 * rows * cols * batch / us / 1e6 / peak_tf, 4),
                    "peak_source": src})
    status = qmv.last_error()
    if status != 0:
        raise SystemExit(f"device status {status}")
    print(json.dumps(out), flush=True)


def main():
    args = parse()
    if args.case:
        run_case(args)
        return
    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
