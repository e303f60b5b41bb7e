"""The tcgen05 prefill path (bf16 activations, 16..128 vectors per pass) vs the oracle.

The prefill kernel rounds each dequantized weight to bfloat16 before the tensor-core
product, so each term carries a relative error of at most 2^-9.  Over rows of 1024 and
more columns (the prefill workloads have 4096 and 14336) that averages well inside
|y - y_ref| <= 1e-3 * sum |w x|; on short rows it can use a good part of the bar, so
there the check is against the bf16-weight product itself.  Where the bf16 weights are
exact (power-of-two scales) and every partial sum is an exact dyadic number, the product
is bit-exact.  Batches below 16 go to the decode kernels (covered in test_gpu_parity.py).
"""
import numpy as np
import pytest

import oracle
from block_quantized_weight_q4_gb300 import inputs
from helpers import check_product, dev_u8, dev_x

pytestmark = pytest.mark.gpu

TOL = 1e-3
TYPES = [(1, 0), (1, 1), (2, 0), (2, 1)]


@pytest.fixture(scope="module", autouse=True)
def qmv():
    import torch
    from block_quantized_weight_q4_gb300.build import build
    import block_quantized_weight_q4_gb300 as q
    assert torch.cuda.is_available()
    build()
    q.load_library()
    yield q
    assert q.last_error() == 0


def run(q, m, x):
    import torch
    y = q.matvec(m.wtype, m.scale_f16, m.rows, m.cols, dev_u8(m.W), dev_x(x))
    torch.cuda.synchronize()
    return y.cpu().numpy()


def bf16_weight_product(W, wt, sf, rows, cols, x):
    """The product the prefill design computes, evaluated in float64: the oracle's
    dequantized weights rounded to bfloat16 (ties to even), times the activations."""
    deq = oracle.dequant(W, wt, sf, rows, cols)
    wb = (inputs.bf16_codes(deq).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return xf @ wb.T


@pytest.mark.parametrize("wt,sf", TYPES)
@pytest.mark.parametrize("rows,cols", [(128, 1024), (200, 2048), (37, 4096), (300, 1024)])
@pytest.mark.parametrize("batch", [16, 17, 64, 100, 128, 130])
def test_prefill_random(qmv, wt, sf, rows, cols, batch):
    # the 1e-3 bar against the exact oracle; bf16 weights round each term by at most 2^-9,
    # which averages out over rows of 1024 and more columns (the prefill workloads use
    # 4096 and 14336)
    m = inputs.make_matrix(wt, sf, rows, cols, seed=rows + cols + batch)
    x = inputs.make_x(batch, cols, True, seed=batch)
    y_ref, absref = oracle.matvec(m.W, wt, sf, rows, cols, x)
    y = run(qmv, m, x)
    check_product(y, y_ref, absref, TOL, f"prefill {wt},{sf} {rows}x{cols} b{batch}")
    # and the tensor core adds the bf16-weight terms with float32 care: within 2^-16 of
    # sum |w x| of the bf16-weight product
    check_product(y, bf16_weight_product(m.W, wt, sf, rows, cols, x), absref, 2.0 ** -16, "bf16 product")


@pytest.mark.parametrize("wt,sf", TYPES)
@pytest.mark.parametrize("rows,cols", [(128, 256), (33, 512)])
def test_prefill_short_rows_follow_bf16_product(qmv, wt, sf, rows, cols):
    # short rows: the bf16 rounding can use a good part of the 1e-3 bar, so the check here
    # is against the bf16-weight product the design defines
    m = inputs.make_matrix(wt, sf, rows, cols, seed=cols + wt)
    x = inputs.make_x(40, cols, True, seed=2)
    _, absref = oracle.matvec(m.W, wt, sf, rows, cols, x)
    check_product(run(qmv, m, x), bf16_weight_product(m.W, wt, sf, rows, cols, x), absref, 2.0 ** -16,
                  "short rows")


@pytest.mark.parametrize("wt,sf", TYPES)
@pytest.mark.parametrize("batch", [16, 48, 128])
def test_prefill_exact_pow2(qmv, wt, sf, batch):
    # power-of-two scales make every bf16 weight exact (levels have <= 8 bits); integer x in
    # [-4, 4]: all partial sums are exact, so the tensor-core result equals the oracle.
    rows, cols = 160, 768
    rng = np.random.default_rng(batch + wt)
    m = inputs.make_matrix(wt, sf, rows, cols, seed=3)
    codes = inputs.pow2_scales(rng, rows * cols // 32, sf)
    W = inputs.assemble(wt, sf, rows, cols, m.q, codes)
    m2 = inputs.Matrix(wt, sf, rows, cols, W, m.q, codes)
    x = inputs.make_int_x(batch, cols, True, seed=4)
    y_ref, _ = oracle.matvec(W, wt, sf, rows, cols, x)
    assert np.array_equal(run(qmv, m2, x).astype(np.float64), y_ref)


def test_prefill_one_hot_pow2_is_dequant(qmv):
    rows, cols, batch = 129, 512, 32
    rng = np.random.default_rng(8)
    m = inputs.make_matrix(2, 1, rows, cols, seed=8)
    codes = inputs.pow2_scales(rng, rows * cols // 32, 1, -6, 3)
    W = inputs.assemble(2, 1, rows, cols, m.q, codes)
    m2 = inputs.Matrix(2, 1, rows, cols, W, m.q, codes)
    picks = rng.integers(0, cols, batch)
    x = np.zeros((batch, cols), np.float32)
    x[np.arange(batch), picks] = 1.0
    deq = oracle.dequant(W, 2, 1, rows, cols)
    y = run(qmv, m2, inputs.bf16_codes(x))
    assert np.array_equal(y, deq[:, picks].T)


@pytest.mark.parametrize("wt,sf", TYPES)
def test_prefill_one_hot_general_scales_is_bf16_of_dequant(qmv, wt, sf):
    # one-hot activations with the workload's scale distribution (not powers of two): each
    # output is one weight as the tensor core saw it, which must be the bfloat16 (ties to
    # even) of the exact dequantized weight, bit for bit, whichever way the kernel forms it
    rows, cols, batch = 300, 1024, 48
    rng = np.random.default_rng(18 + wt + sf)
    m = inputs.make_matrix(wt, sf, rows, cols, seed=18 + wt + sf)
    picks = rng.integers(0, cols, batch)
    x = np.zeros((batch, cols), np.float32)
    x[np.arange(batch), picks] = 1.0
    deq = oracle.dequant(m.W, wt, sf, rows, cols)
    wb = (inputs.bf16_codes(deq).astype(np.uint32) << 16).view(np.float32)
    y = run(qmv, m, inputs.bf16_codes(x))
    expect = wb[:, picks].T
    assert np.array_equal(y, expect), f"{np.count_nonzero(y != expect)} weights differ"


def test_prefill_zero_rows_exact(qmv):
    rows, cols, batch = 140, 512, 24
    m = inputs.make_matrix(2, 1, rows, cols, seed=9)
    q = m.q.copy().reshape(rows, -1)
    q[::5] = 0x88
    W = inputs.assemble(2, 1, rows, cols, q.reshape(-1), m.d_codes)
    m2 = inputs.Matrix(2, 1, rows, cols, W, q.reshape(-1), m.d_codes)
    x = inputs.make_x(batch, cols, True, seed=9)
    y_ref, absref = oracle.matvec(W, 2, 1, rows, cols, x)
    y = run(qmv, m2, x)
    assert np.all(y[:, ::5] == 0.0)
    check_product(y, y_ref, absref, TOL, "prefill zero rows")


def test_prefill_output_guards(qmv):
    import torch
    rows, cols, batch = 130, 256, 20
    m = inputs.make_matrix(2, 1, rows, cols, seed=10)
    x = dev_x(inputs.make_x(batch, cols, True, seed=10))
    buf = torch.full((batch * rows + 256,), 4321.0, device="cuda")
    y = buf[128:128 + batch * rows].view(batch, rows)
    qmv.matvec(2, 1, rows, cols, dev_u8(m.W), x, y)
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.all(b[:128] == 4321.0) and np.all(b[128 + batch * rows:] == 4321.0)


@pytest.mark.parametrize("wt,sf", [(2, 1), (1, 0)])
def test_prefill_split_tiles_repeat_and_graph_bit_identical(qmv, wt, sf):
    # 3 row tiles of 128 over 56 raw stages: each tile's columns are split between 16 CTAs,
    # whose parts the last of them adds in split order; the counters must be back at zero after
    # every call (repeated calls and graph replays give the same bits)
    import torch
    from helpers import assert_bits_equal
    rows, cols, batch = 300, 14336, 64
    m = inputs.make_matrix(wt, sf, rows, cols, seed=31)
    x = inputs.make_x(batch, cols, True, seed=32)
    y_ref, absref = oracle.matvec(m.W, wt, sf, rows, cols, x)
    W, xd = dev_u8(m.W), dev_x(x)
    s = torch.cuda.Stream()
    y = torch.empty((batch, rows), device="cuda")
    with torch.cuda.stream(s):
        qmv.matvec(wt, sf, rows, cols, W, xd, y)
    torch.cuda.synchronize()
    first = y.cpu().numpy().copy()
    check_product(first, y_ref, absref, TOL, f"prefill split {wt},{sf}")
    for _ in range(3):
        with torch.cuda.stream(s):
            qmv.matvec(wt, sf, rows, cols, W, xd, y)
        torch.cuda.synchronize()
        assert_bits_equal(y.cpu().numpy(), first, "repeated split-tile prefill")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(2):
            qmv.matvec(wt, sf, rows, cols, W, xd, y)
    y.fill_(0.0)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert_bits_equal(y.cpu().numpy(), first, "split-tile prefill graph replay")


def test_prefill_split_tiles_exact_pow2(qmv):
    # exact case over split tiles: power-of-two scales, integer x; any order of the parts'
    # addition gives the oracle's value
    rows, cols, batch = 256, 8192, 32
    rng = np.random.default_rng(33)
    m = inputs.make_matrix(2, 1, rows, cols, seed=34)
    codes = inputs.pow2_scales(rng, rows * cols // 32, 1)
    W = inputs.assemble(2, 1, rows, cols, m.q, codes)
    m2 = inputs.Matrix(2, 1, rows, cols, W, m.q, codes)
    x = inputs.make_int_x(batch, cols, True, seed=35)
    y_ref, _ = oracle.matvec(W, 2, 1, rows, cols, x)
    assert np.array_equal(run(qmv, m2, x).astype(np.float64), y_ref)


@pytest.mark.parametrize("offset,batch", [(1, 48), (2, 40), (4, 40)])
def test_prefill_split_tiles_unaligned_y_and_guards(qmv, offset, batch):
    # split tiles (2 row tiles over 16 raw stages) whose last CTA stores 4 consecutive rows
    # of y at a time: y only 4-byte aligned (offset 1 or 2 floats), or 16-byte aligned with
    # a batch that is not a multiple of 16; nothing outside y is written
    import torch
    rows, cols = 256, 4096
    m = inputs.make_matrix(2, 1, rows, cols, seed=40 + offset)
    x = inputs.make_x(batch, cols, True, seed=41 + offset)
    y_ref, absref = oracle.matvec(m.W, 2, 1, rows, cols, x)
    buf = torch.full((batch * rows + 64,), 4321.0, device="cuda")
    y = buf[offset:offset + batch * rows].view(batch, rows)
    qmv.matvec(2, 1, rows, cols, dev_u8(m.W), dev_x(x), y)
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.all(b[:offset] == 4321.0) and np.all(b[offset + batch * rows:] == 4321.0)
    check_product(b[offset:offset + batch * rows].reshape(batch, rows), y_ref, absref, TOL, f"unaligned y {offset}")


@pytest.mark.parametrize("wt,sf,batch", [(1, 0, 128), (2, 1, 128), (2, 1, 64), (1, 1, 48)])
def test_prefill_full_size_graph_replays_stable(qmv, wt, sf, batch):
    # the prefill workload's 14336 x 4096 matrix, many calls back to back in CUDA graphs (the
    # pipeline's rings run through many phases and the two MMA warps drift against each
    # other): every replay gives the first call's bits, no wait runs out, and sampled rows
    # (every tile's first and last, a ragged set inside) match the oracle
    import torch
    from helpers import assert_bits_equal
    rows, cols = 14336, 4096
    m = inputs.make_matrix(wt, sf, rows, cols, seed=50 + wt + batch)
    x = inputs.make_x(batch, cols, True, seed=51 + batch)
    W, xd = dev_u8(m.W), dev_x(x)
    y = torch.empty((batch, rows), device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        qmv.matvec(wt, sf, rows, cols, W, xd, y)
    torch.cuda.synchronize()
    first = y.cpu().numpy().copy()
    ids = np.unique(np.concatenate([np.arange(0, rows, 128), np.arange(127, rows, 128),
                                    np.random.default_rng(52).integers(0, rows, 64)]))
    y_ref, absref = oracle.matvec_rows(m.W, wt, sf, rows, cols, x, ids)
    check_product(first[:, ids], y_ref, absref, TOL, f"full-size prefill {wt},{sf} b{batch}")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(16):
            qmv.matvec(wt, sf, rows, cols, W, xd, y)
    for _ in range(8):
        y.fill_(0.0)
        g.replay()
        torch.cuda.synchronize()
        assert_bits_equal(y.cpu().numpy(), first, "full-size prefill graph replay")
    assert qmv.last_error() == 0


def test_prefill_overlap_waits_for_the_preceding_kernel(qmv):
    # y1 = W1 x (prefill); x2 = bf16(y1) by a torch kernel; y2 = W2 x2 launched with the
    # overlap flag: its weight loads may start early, but it must read x2 only after the
    # conversion kernel has finished (eager and in a graph, repeated)
    import torch
    from helpers import assert_bits_equal
    batch, rows1, cols1, rows2 = 48, 1024, 2048, 384
    m1 = inputs.make_matrix(2, 1, rows1, cols1, seed=61)
    m2 = inputs.make_matrix(2, 1, rows2, rows1, seed=62)
    x = inputs.make_x(batch, cols1, True, seed=63)
    W1, W2, xd = dev_u8(m1.W), dev_u8(m2.W), dev_x(x)
    y1 = torch.empty((batch, rows1), device="cuda")
    y2 = torch.empty((batch, rows2), device="cuda")
    x2 = torch.empty((batch, rows1), device="cuda", dtype=torch.bfloat16)
    s = torch.cuda.Stream()

    def step():
        qmv.matvec_grouped(2, 1, [(rows1, cols1, W1, xd, y1)], overlap=True)
        x2.copy_(y1)  # float32 -> bfloat16, ties to even
        qmv.matvec_grouped(2, 1, [(rows2, rows1, W2, x2, y2)], overlap=True)

    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    x2_codes = x2.view(torch.int16).cpu().numpy().view(np.uint16)
    y_ref, absref = oracle.matvec(m2.W, 2, 1, rows2, rows1, x2_codes)
    first = y2.cpu().numpy().copy()
    check_product(first, y_ref, absref, TOL, "overlapped chain")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            step()
    for _ in range(4):
        y1.fill_(0.0)
        x2.fill_(0.0)
        y2.fill_(0.0)
        g.replay()
        torch.cuda.synchronize()
        assert_bits_equal(y2.cpu().numpy(), first, "overlapped chain graph replay")
    assert qmv.last_error() == 0
