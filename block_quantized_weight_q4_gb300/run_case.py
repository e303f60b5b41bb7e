"""Run one product shape through libqmv a number of times (for timing and profiling).

    python -m block_quantized_weight_q4_gb300.run_case --rows 11008 --cols 4096 \\
        --wtype 2 --scale-f16 1 --batch 1 --iters 8

Seeded synthetic weights (uniform quants, scales ~ U[1e-3, 2e-2]) and N(0,1) activations;
the products rotate over several copies of the matrix so that consecutive calls read their
weights from HBM.  Prints the mean per-call time measured over back-to-back calls captured
in a CUDA graph (no host overhead between calls).
"""
from __future__ import annotations

import argparse

import numpy as np


def main(argv=None):
    import torch

    import block_quantized_weight_q4_gb300 as qmv
    from block_quantized_weight_q4_gb300 import inputs
    from block_quantized_weight_q4_gb300.build import build

    ap = argparse.ArgumentParser()
    ap.add_argument("--rows", type=int, default=11008)
    ap.add_argument("--cols", type=int, default=4096)
    ap.add_argument("--wtype", type=int, default=2, help="1 = Q8_0, 2 = Q4_0")
    ap.add_argument("--scale-f16", type=int, default=1)
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--x-f32", action="store_true", help="float32 activations (default bfloat16)")
    ap.add_argument("--iters", type=int, default=8, help="eager calls before the timed graph")
    ap.add_argument("--copies", type=int, default=4)
    ap.add_argument("--graph-calls", type=int, default=20)
    a = ap.parse_args(argv)

    build()
    qmv.load_library()
    m = inputs.make_matrix(a.wtype, a.scale_f16, a.rows, a.cols, seed=1)
    W0 = torch.from_numpy(m.W).cuda()
    Ws = [W0] + [W0.clone() for _ in range(a.copies - 1)]
    x = inputs.make_x(a.batch, a.cols, not a.x_f32, seed=2)
    xd = torch.from_numpy(x).cuda() if a.x_f32 else torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    y = torch.empty((a.batch, a.rows), device="cuda")
    # eager calls on the stream that is captured below: a stream's first call creates the
    # workspace its split tiles use (never while it is being captured)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for i in range(a.iters):
            qmv.matvec(a.wtype, a.scale_f16, a.rows, a.cols, Ws[i % a.copies], xd, y)
    torch.cuda.synchronize()
    if a.graph_calls > 0:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for i in range(a.graph_calls):
                qmv.matvec(a.wtype, a.scale_f16, a.rows, a.cols, Ws[i % a.copies], xd, y)
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(5):
            g.replay()
        e1.record()
        torch.cuda.synchronize()
        us = e0.elapsed_time(e1) * 1e3 / (5 * a.graph_calls)
        nb = m.W.size
        print(f"{a.rows}x{a.cols} wtype {a.wtype} scale_f16 {a.scale_f16} batch {a.batch}: {us:.2f} us per call, "
              f"{nb / us / 1e3:.1f} GB/s of weights, {2.0 * a.rows * a.cols * a.batch / us / 1e6:.1f} TFLOP/s")
    status = qmv.last_error()
    if status != 0:
        raise SystemExit(f"device status {status}")


if __name__ == "__main__":
    main()
