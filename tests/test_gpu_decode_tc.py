"""The decode kernels for 2..16 bf16 vectors vs the oracle: the tensor-memory kernel (passes of
8 vectors over 128 MB of weights, passes of 9..16 vectors over 8 MB) and the mma.sync kernel
(the other passes of 2..8).

The tensor-memory kernel splits the work into units of 128 rows x 256 columns shared out
evenly between two CTAs per SM, so a tile's columns may be summed by several CTAs; the parts
meet in a per-stream workspace and the last CTA to arrive adds them in CTA order.  The tests
at its sizes aim at that machinery: tiles split between many CTAs, tiles that end where a
problem of a grouped launch ends, repeated calls (the arrival counters must be back at zero
after every call), and the result's independence from timing (bit-identical across calls and
graph replays).  The small shapes check the mma.sync kernel the same way.
"""
import numpy as np
import pytest

import oracle
from block_quantized_weight_q4_gb300 import inputs
from helpers import assert_bits_equal, check_product, dev_u8, dev_x

pytestmark = pytest.mark.gpu

TOL = 1e-3
TYPES = [(1, 0), (1, 1), (2, 0), (2, 1)]
# launch sizes from which the tensor-memory kernel takes the bf16 passes
TC_MIN_BYTES = 128 << 20      # passes of 8 vectors
TC_WIDE_MIN_BYTES = 8 << 20   # passes of 9..16 vectors, one launch each


def weight_bytes(wt, sf, rows, cols):
    return rows * cols // 32 * ((16 if wt == 2 else 32) + (2 if sf else 4))


def sample_rows(rows, seed, n=160):
    rng = np.random.default_rng(seed)
    ids = np.unique(np.concatenate([rng.integers(0, rows, n), [0, 127, 128, rows - 1]]))
    return ids


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


def run(q, m, x, y=None):
    import torch
    y = q.matvec(m.wtype, m.scale_f16, m.rows, m.cols, dev_u8(m.W), dev_x(x), y)
    torch.cuda.synchronize()
    return y.cpu().numpy()


@pytest.mark.parametrize("wt,sf", TYPES)
@pytest.mark.parametrize("rows,cols", [(256, 256), (512, 4096), (300, 2048), (2000, 1024), (4096, 4096)])
@pytest.mark.parametrize("batch", [4, 5, 8, 9, 12, 15])
def test_tc_decode_matches_oracle(qmv, wt, sf, rows, cols, batch):
    # 512 x 4096: 64 units on 64 CTAs, each of the four tiles split 16 ways
    m = inputs.make_matrix(wt, sf, rows, cols, seed=rows * 7 + cols + batch)
    x = inputs.make_x(batch, cols, True, seed=batch + rows)
    y_ref, absref = oracle.matvec(m.W, wt, sf, rows, cols, x)
    check_product(run(qmv, m, x), y_ref, absref, TOL, f"tc {wt},{sf} {rows}x{cols} b{batch}")


@pytest.mark.parametrize("wt,sf", [(1, 0), (2, 1)])
@pytest.mark.parametrize("batch", [8, 13])
def test_tc_exact_pow2(qmv, wt, sf, batch):
    # power-of-two scales, integer activations: every partial sum is exact, in any split
    rows, cols = 600, 4096
    rng = np.random.default_rng(11 + wt)
    m = inputs.make_matrix(wt, sf, rows, cols, seed=12)
    codes = inputs.pow2_scales(rng, rows * cols // 32, sf)
    W = inputs.assemble(wt, sf, rows, cols, m.q, codes)
    x = inputs.make_int_x(batch, cols, True, seed=13)
    y_ref, _ = oracle.matvec(W, wt, sf, rows, cols, x)
    m2 = inputs.Matrix(wt, sf, rows, cols, W, m.q, codes)
    assert np.array_equal(run(qmv, m2, x).astype(np.float64), y_ref)


def test_tc_zero_rows_exact(qmv):
    rows, cols, batch = 700, 2048, 6
    m = inputs.make_matrix(2, 1, rows, cols, seed=14)
    q = m.q.copy().reshape(rows, -1)
    q[::7] = 0x88  # every level 0
    W = inputs.assemble(2, 1, rows, cols, q.reshape(-1), m.d_codes)
    m2 = inputs.Matrix(2, 1, rows, cols, W, q.reshape(-1), m.d_codes)
    x = inputs.make_x(batch, cols, True, seed=14)
    y_ref, absref = oracle.matvec(W, 2, 1, rows, cols, x)
    y = run(qmv, m2, x)
    assert np.all(y[:, ::7] == 0.0)
    check_product(y, y_ref, absref, TOL, "tc zero rows")


@pytest.mark.parametrize("wt,sf", [(2, 1), (1, 0)])
@pytest.mark.parametrize("batch", [8, 14])
def test_tc_repeated_calls_bit_identical(qmv, wt, sf, batch):
    # the split tiles' counters are reset by each call: later calls give the same bits
    rows, cols = 1536, 4096
    m = inputs.make_matrix(wt, sf, rows, cols, seed=15)
    x = inputs.make_x(batch, cols, True, seed=15)
    first = run(qmv, m, x)
    y_ref, absref = oracle.matvec(m.W, wt, sf, rows, cols, x)
    check_product(first, y_ref, absref, TOL, "tc first call")
    for _ in range(3):
        assert_bits_equal(run(qmv, m, x), first, "tc repeated call")


@pytest.mark.parametrize("batch", [7, 11])
def test_tc_grouped_problems(qmv, batch):
    # a grouped launch: units of all problems in one list, tiles ending at problem ends
    import torch
    shapes = [(300, 4096), (1024, 1024), (257, 2048), (4096, 256)]
    probs, refs = [], []
    for i, (rows, cols) in enumerate(shapes):
        m = inputs.make_matrix(2, 1, rows, cols, seed=70 + i)
        x = inputs.make_x(batch, cols, True, seed=80 + i)
        y = torch.full((batch, rows), 3.0, device="cuda")
        probs.append((rows, cols, dev_u8(m.W), dev_x(x), y))
        refs.append(oracle.matvec(m.W, 2, 1, rows, cols, x))
    for overlap in (False, True):
        qmv.matvec_grouped(2, 1, probs, overlap=overlap)
        torch.cuda.synchronize()
        for (rows, cols, _, _, y), (y_ref, absref) in zip(probs, refs):
            check_product(y.cpu().numpy(), y_ref, absref, TOL, f"tc grouped {rows}x{cols} overlap={overlap}")


def test_tc_graph_replay_bit_identical(qmv):
    # captured after an eager call on the same stream (which creates its workspace)
    import torch
    rows, cols, batch = 2048, 4096, 8
    m = inputs.make_matrix(2, 1, rows, cols, seed=16)
    W = dev_u8(m.W)
    x = dev_x(inputs.make_x(batch, cols, True, seed=16))
    s = torch.cuda.Stream()
    y = torch.empty((batch, rows), device="cuda")
    with torch.cuda.stream(s):
        qmv.matvec(2, 1, rows, cols, W, x, y)
    torch.cuda.synchronize()
    eager = y.cpu().numpy().copy()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            qmv.matvec(2, 1, rows, cols, W, x, y)
    y.fill_(0.0)
    for _ in range(4):
        g.replay()
    torch.cuda.synchronize()
    assert_bits_equal(y.cpu().numpy(), eager, "graph replay")


def test_tc_q8_large_launch_batch1(qmv):
    # a Q8_0 launch of 64M weights or more takes the kernel at batch 1 too; sampled rows
    import torch
    rows, cols = 65536, 1024
    m = inputs.make_matrix(1, 0, rows, cols, seed=17)
    x = inputs.make_x(1, cols, True, seed=17)
    y = run(qmv, m, x)
    ids = np.arange(0, rows, 97)
    y_ref, absref = oracle.matvec_rows(m.W, 1, 0, rows, cols, x, ids)
    check_product(y[:, ids], y_ref, absref, TOL, "q8 large b1")


@pytest.mark.parametrize("wt,sf,rows,cols", [(1, 0, 122880, 1024), (2, 1, 65536, 4096)])
@pytest.mark.parametrize("batch", [7, 8])
def test_tc_large_launch_sampled_rows(qmv, wt, sf, rows, cols, batch):
    # 142 / 151 MB: the tensor-memory kernel at 8 vectors (the mma.sync kernel at 7); rows
    # sampled over every part of the matrix (tiles split between CTAs at every CTA boundary)
    assert weight_bytes(wt, sf, rows, cols) >= TC_MIN_BYTES
    m = inputs.make_matrix(wt, sf, rows, cols, seed=30 + batch)
    x = inputs.make_x(batch, cols, True, seed=31 + batch)
    y = run(qmv, m, x)
    ids = sample_rows(rows, 32 + batch)
    y_ref, absref = oracle.matvec_rows(m.W, wt, sf, rows, cols, x, ids)
    check_product(y[:, ids], y_ref, absref, TOL, f"tc large {wt},{sf} b{batch}")


@pytest.mark.parametrize("wt,sf,rows,cols", [(2, 1, 8192, 4096), (1, 1, 4096, 4096)])
@pytest.mark.parametrize("batch", [9, 12, 16])
def test_tc_sixteen_vector_pass(qmv, wt, sf, rows, cols, batch):
    # 19 / 18 MB, 9..16 vectors: one pass of the tensor-memory kernel, all 16 MMA columns
    # vectors (zeros past the batch); batch 16 takes it too at these sizes
    assert weight_bytes(wt, sf, rows, cols) >= TC_WIDE_MIN_BYTES
    m = inputs.make_matrix(wt, sf, rows, cols, seed=40 + batch)
    x = inputs.make_x(batch, cols, True, seed=41 + batch)
    y = run(qmv, m, x)
    ids = sample_rows(rows, 42 + batch)
    y_ref, absref = oracle.matvec_rows(m.W, wt, sf, rows, cols, x, ids)
    check_product(y[:, ids], y_ref, absref, TOL, f"tc 16 {wt},{sf} b{batch}")
    check_product(y[:, ids], y_ref, absref, 1e-5, f"tc 16 tight {wt},{sf} b{batch}")


@pytest.mark.parametrize("batch", [10, 16])
def test_tc_sixteen_vector_pass_exact_and_repeatable(qmv, batch):
    # power-of-two scales and integer activations: every partial sum is exact in any split, so
    # the sampled rows equal the oracle bit for bit; repeated calls and graph replays give the
    # same bits (the arrival counters are back at zero after every launch)
    import torch
    wt, sf, rows, cols = 2, 1, 8192, 4096
    rng = np.random.default_rng(50 + batch)
    m = inputs.make_matrix(wt, sf, rows, cols, seed=51)
    codes = inputs.pow2_scales(rng, rows * cols // 32, sf)
    W = inputs.assemble(wt, sf, rows, cols, m.q, codes)
    x = inputs.make_int_x(batch, cols, True, seed=52 + batch)
    Wd, xd = dev_u8(W), dev_x(x)
    s = torch.cuda.Stream()
    y = torch.empty((batch, rows), device="cuda")
    with torch.cuda.stream(s):
        qmv.matvec(wt, sf, rows, cols, Wd, xd, y)
    torch.cuda.synchronize()
    first = y.cpu().numpy().copy()
    ids = sample_rows(rows, 53)
    y_ref, _ = oracle.matvec_rows(W, wt, sf, rows, cols, x, ids)
    assert np.array_equal(first[:, ids].astype(np.float64), y_ref)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            qmv.matvec(wt, sf, rows, cols, Wd, xd, y)
    for _ in range(3):
        y.fill_(0.0)
        g.replay()
        torch.cuda.synchronize()
        assert_bits_equal(y.cpu().numpy(), first, "tc 16 graph replay")


@pytest.mark.parametrize("batch", [6, 11])
def test_tc_grouped_large_launch(qmv, batch):
    # a grouped launch of 45 MB (11 vectors: one 16-vector pass of the tensor-memory kernel, tiles
    # of three problems in one unit list; 6 vectors: the mma.sync kernel), with overlap
    import torch
    shapes = [(14336, 4096), (4096, 4096), (1000, 4096)]
    assert sum(weight_bytes(2, 1, r, c) for r, c in shapes) >= TC_WIDE_MIN_BYTES
    probs, refs = [], []
    for i, (rows, cols) in enumerate(shapes):
        m = inputs.make_matrix(2, 1, rows, cols, seed=60 + i)
        x = inputs.make_x(batch, cols, True, seed=70 + i)
        y = torch.full((batch, rows), 3.0, device="cuda")
        ids = sample_rows(rows, 80 + i)
        probs.append((rows, cols, dev_u8(m.W), dev_x(x), y))
        refs.append((ids, oracle.matvec_rows(m.W, 2, 1, rows, cols, x, ids)))
    qmv.matvec_grouped(2, 1, probs, overlap=True)
    torch.cuda.synchronize()
    for (rows, cols, _, _, y), (ids, (y_ref, absref)) in zip(probs, refs):
        check_product(y.cpu().numpy()[:, ids], y_ref, absref, TOL, f"tc grouped {rows}x{cols} b{batch}")
