"""The tcgen05 prefill path (bf16 activations, 16..128 vectors per pass) vs the oracle.

Each dequantized weight w enters the tensor core as two bfloat16 parts, hi = RN_bf16(w) and
lo = RN_bf16(w - hi), with one MMA each: for Q4_0 with f16 scales hi + lo = w exactly, for
the other formats within 2^-17 |w|.  So every product meets |y - y_ref| <= 1e-3 * sum |w x|
against the exact oracle on any input, including short rows and one-hot activations (one
term per output), which the tests below check at every prefill batch.  The opt-in
bf16-weights variant (QMV_FLAG_BF16_WEIGHTS: one rounding of w, up to 2^-9 per term) is
checked against the bf16-weight product it defines.  Where the weights are exact in
bfloat16 (power-of-two scales) and every partial sum is an exact dyadic number, the product
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


def run(q, m, x, bf16_weights=False):
    import torch
    if bf16_weights:
        xd = dev_x(x)
        y = torch.empty((xd.shape[0], m.rows), device="cuda")
        q.matvec_grouped(m.wtype, m.scale_f16, [(m.rows, m.cols, dev_u8(m.W), xd, y)], bf16_weights=True)
    else:
        y = q.matvec(m.wtype, m.scale_f16, m.rows, m.cols, dev_u8(m.W), dev_x(x))
    torch.cuda.synchronize()
    return y.cpu().numpy()


# hi + lo carries each weight to within 2^-17 |w| (exactly for Q4_0 with f16 scales), so the
# kernel stays far inside the 1e-3 bar: within 2^-14 of sum |w x| of the exact product
HILO_TOL = 2.0 ** -14


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
    m = inputs.make_matrix(wt, sf, rows, cols, seed=rows + cols + batch)
    x = inputs.make_x(batch, cols, True, seed=batch)
    y_ref, absref = oracle.matvec(m.W, wt, sf, rows, cols, x)
    y = run(qmv, m, x)
    check_product(y, y_ref, absref, TOL, f"prefill {wt},{sf} {rows}x{cols} b{batch}")
    check_product(y, y_ref, absref, HILO_TOL, f"prefill hi+lo {wt},{sf} {rows}x{cols} b{batch}")


@pytest.mark.parametrize("wt,sf", TYPES)
@pytest.mark.parametrize("rows,cols", [(128, 1024), (37, 4096)])
@pytest.mark.parametrize("batch", [16, 100, 130])
def test_prefill_bf16_weights_follow_bf16_product(qmv, wt, sf, rows, cols, batch):
    # the opt-in variant: the tensor core adds the bf16-weight terms with float32 care, within
    # 2^-16 of sum |w x| of the bf16-weight product, and each term is off the exact one by at
    # most 2^-9 of its magnitude
    m = inputs.make_matrix(wt, sf, rows, cols, seed=rows + cols + batch)
    x = inputs.make_x(batch, cols, True, seed=batch)
    y_ref, absref = oracle.matvec(m.W, wt, sf, rows, cols, x)
    y = run(qmv, m, x, bf16_weights=True)
    check_product(y, bf16_weight_product(m.W, wt, sf, rows, cols, x), absref, 2.0 ** -16, "bf16 product")
    check_product(y, y_ref, absref, 2.0 ** -9 + 2.0 ** -16, "bf16 weights vs exact")


@pytest.mark.parametrize("wt,sf", TYPES)
@pytest.mark.parametrize("rows,cols", [(128, 256), (33, 512)])
def test_prefill_short_rows(qmv, wt, sf, rows, cols):
    # short rows (8 and 16 blocks): the exact oracle at the 1e-3 bar and at the hi + lo bound
    m = inputs.make_matrix(wt, sf, rows, cols, seed=cols + wt)
    x = inputs.make_x(40, cols, True, seed=2)
    y_ref, absref = oracle.matvec(m.W, wt, sf, rows, cols, x)
    y = run(qmv, m, x)
    check_product(y, y_ref, absref, TOL, "short rows")
    check_product(y, y_ref, absref, HILO_TOL, "short rows (hi + lo)")
    # the bf16-weights variant is held to its own definition
    check_product(run(qmv, m, x, bf16_weights=True), bf16_weight_product(m.W, wt, sf, rows, cols, x), absref,
                  2.0 ** -16, "short rows, bf16 weights")


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


PREFILL_BATCHES = [16, 17, 31, 48, 64, 65, 100, 127, 128, 129, 200, 256]


def _one_hot(rng, batch, cols):
    picks = rng.integers(0, cols, batch)
    x = np.zeros((batch, cols), np.float32)
    x[np.arange(batch), picks] = 1.0
    return picks, inputs.bf16_codes(x)


@pytest.mark.parametrize("wt,sf", TYPES)
@pytest.mark.parametrize("batch", PREFILL_BATCHES)
def test_prefill_one_hot_meets_bar(qmv, wt, sf, batch):
    # one-hot activations with the workload's scales (d ~ U[1e-3, 2e-2], not powers of two):
    # each output is a single term w * 1, so the 1e-3 bar applies to one weight alone; the
    # result must be within 2^-17 |w| of the exact dequantized weight (bit for bit for Q4_0
    # with f16 scales, where hi + lo = w exactly), at every prefill batch (one and two passes)
    rows, cols = 300, 1024
    rng = np.random.default_rng(18 + wt + sf + batch)
    m = inputs.make_matrix(wt, sf, rows, cols, seed=18 + wt + sf)
    picks, x = _one_hot(rng, batch, cols)
    y_ref, absref = oracle.matvec(m.W, wt, sf, rows, cols, x)
    y = run(qmv, m, x)
    check_product(y, y_ref, absref, TOL, f"one-hot {wt},{sf} b{batch}")
    deq = oracle.dequant(m.W, wt, sf, rows, cols)
    expect = deq[:, picks].T
    if (wt, sf) == (2, 1):
        assert np.array_equal(y, expect), f"{np.count_nonzero(y != expect)} weights differ"
    else:
        err = np.abs(y.astype(np.float64) - expect)
        assert np.all(err <= 2.0 ** -17 * np.abs(expect)), float(np.max(err / np.maximum(np.abs(expect), 1e-30)))


@pytest.mark.parametrize("wt,sf", TYPES)
@pytest.mark.parametrize("batch", [16, 64, 128])
def test_prefill_dominated_rows_meet_bar(qmv, wt, sf, batch):
    # each vector: one activation of 1 plus activations of 1e-4 elsewhere; each output is then
    # dominated by one weight, where a single bf16 rounding of the weights (2^-9 ~ 1.95e-3)
    # would use up to twice the 1e-3 bar
    rows, cols = 256, 4096
    rng = np.random.default_rng(70 + wt + sf + batch)
    m = inputs.make_matrix(wt, sf, rows, cols, seed=70 + wt + sf)
    picks = rng.integers(0, cols, batch)
    xf = 1e-4 * rng.standard_normal((batch, cols)).astype(np.float32)
    xf[np.arange(batch), picks] = 1.0
    x = inputs.bf16_codes(xf)
    y_ref, absref = oracle.matvec(m.W, wt, sf, rows, cols, x)
    y = run(qmv, m, x)
    check_product(y, y_ref, absref, TOL, f"dominated rows {wt},{sf} b{batch}")
    check_product(y, y_ref, absref, HILO_TOL, f"dominated rows (hi + lo) {wt},{sf} b{batch}")


@pytest.mark.parametrize("wt,sf", TYPES)
def test_prefill_bf16_weights_one_hot_is_bf16_of_dequant(qmv, wt, sf):
    # the bf16-weights variant with one-hot activations: each output is one weight as the
    # tensor core saw it, the bfloat16 (ties to even) of the exact dequantized weight
    rows, cols, batch = 300, 1024, 48
    rng = np.random.default_rng(18 + wt + sf)
    m = inputs.make_matrix(wt, sf, rows, cols, seed=18 + wt + sf)
    picks, x = _one_hot(rng, batch, cols)
    deq = oracle.dequant(m.W, wt, sf, rows, cols)
    wb = (inputs.bf16_codes(deq).astype(np.uint32) << 16).view(np.float32)
    y = run(qmv, m, x, bf16_weights=True)
    expect = wb[:, picks].T
    assert np.array_equal(y, expect), f"{np.count_nonzero(y != expect)} weights differ"


@pytest.mark.parametrize("wt,sf", TYPES)
def test_prefill_special_scales(qmv, wt, sf):
    # every scale is valid input: infinite and NaN scales propagate (hi carries them,
    # lo is zero); zero, negative and f16-subnormal scales (as weights: normal bfloat16 values)
    # and small normal f32 scales meet the bar like any other
    rows, cols, batch = 64, 512, 32
    m = inputs.make_matrix(wt, sf, rows, cols, seed=90 + wt + sf)
    codes = m.d_codes.reshape(rows, cols // 32).copy()
    rng = np.random.default_rng(91)
    if sf:
        inf, ninf, nan = 0x7C00, 0xFC00, 0x7E00
        codes[3] = rng.integers(1, 0x400, cols // 32)            # subnormal f16 scales
        codes[4] = 0x0000
        codes[5, 2] = 0x8000
        codes[6] = codes[6] | 0x8000                              # negative scales
    else:
        f = lambda v: np.array(v, np.float32).view(np.uint32)
        inf, ninf, nan = f(np.inf), f(-np.inf), f(np.nan)
        codes[3] = f(rng.uniform(1e-30, 1e-28, cols // 32).astype(np.float32))  # small normal scales
        codes[4] = f(0.0)
        codes[5, 2] = f(-0.0)
        codes[6] = codes[6] | np.uint32(0x80000000)
    codes[0, 0] = inf
    codes[1, 3] = nan
    codes[2, 5] = ninf
    codes = codes.reshape(-1)
    W = inputs.assemble(wt, sf, rows, cols, m.q, codes)
    m2 = inputs.Matrix(wt, sf, rows, cols, W, m.q, codes)
    x = inputs.make_x(batch, cols, True, seed=92)
    y_ref, absref = oracle.matvec(W, wt, sf, rows, cols, x)
    y = run(qmv, m2, x).astype(np.float64)
    for r in range(3):
        nan_ref = np.isnan(y_ref[:, r])
        assert np.array_equal(np.isnan(y[:, r]), nan_ref), f"row {r}: NaN positions"
        assert np.array_equal(y[~nan_ref, r], y_ref[~nan_ref, r]), f"row {r}: infinities"
    check_product(y[:, 3:], y_ref[:, 3:], absref[:, 3:], TOL, f"special scales {wt},{sf}")
    check_product(y[:, 3:], y_ref[:, 3:], absref[:, 3:], HILO_TOL, f"special scales (hi + lo) {wt},{sf}")


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
