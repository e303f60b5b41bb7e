"""The single-vector decode kernel (batch 1, bfloat16 activations) vs the oracle.

That kernel spends the 8 columns of each MMA on the 8 weight blocks of a stage (the
activation fragment is block-diagonal), and takes IEEE-half operands for every stage whose
activations all convert exactly to half, bfloat16 operands otherwise.  These tests aim at
both: all four weight/scale types over shapes that span several tiles, a ragged row tail
and the column splits of launches with few tiles; stages that must take bfloat16 operands
(activations above the half range, inexact below it, NaN) next to stages that take half
ones in the same rows; exact results where every partial sum is representable (one-hot and
integer activations with power-of-two scales, activations that are half subnormals);
repeated calls and graph replays bit-identical.
"""
import numpy as np
import pytest

import oracle
from block_quantized_weight_q4_gb300 import inputs
from helpers import assert_bits_equal, check_product, dev_u8, dev_x

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


def with_pow2_scales(m, seed, lo_exp=-4, hi_exp=0):
    rng = np.random.default_rng(seed)
    codes = inputs.pow2_scales(rng, m.rows * m.cols // 32, m.scale_f16, lo_exp, hi_exp)
    W = inputs.assemble(m.wtype, m.scale_f16, m.rows, m.cols, m.q, codes)
    return inputs.Matrix(m.wtype, m.scale_f16, m.rows, m.cols, W, m.q, codes)


def bf16(v):
    return inputs.bf16_codes(np.asarray(v, np.float32).reshape(1, -1))


@pytest.mark.parametrize("wt,sf", TYPES)
@pytest.mark.parametrize("rows,cols", [(16, 256), (33, 256), (100, 4096), (300, 2048), (64, 11008),
                                       (1000, 1024), (4096, 4096), (129, 768)])
def test_b1_matches_oracle(qmv, wt, sf, rows, cols):
    # few tiles (16 x 256, 64 x 11008, 129 x 768) run with 8- or 16-warp CTAs whose warps
    # split the columns; 4096 x 4096 fills every SM with 4-warp CTAs
    m = inputs.make_matrix(wt, sf, rows, cols, seed=rows * 3 + cols + wt)
    x = inputs.make_x(1, cols, True, seed=rows + cols)
    y_ref, absref = oracle.matvec(m.W, wt, sf, rows, cols, x)
    check_product(run(qmv, m, x), y_ref, absref, TOL, f"b1 {wt},{sf} {rows}x{cols}")


@pytest.mark.parametrize("wt,sf", TYPES)
def test_b1_exact_integer_pow2(qmv, wt, sf):
    # integer x in [-4, 4], d = 2^e, e in [-4, 0]: every partial sum is exact in float32
    rows, cols = 200, 4096
    m = with_pow2_scales(inputs.make_matrix(wt, sf, rows, cols, seed=21), seed=22)
    x = inputs.make_int_x(1, cols, True, seed=23)
    y_ref, _ = oracle.matvec(m.W, wt, sf, rows, cols, x)
    assert np.array_equal(run(qmv, m, x).astype(np.float64), y_ref)


@pytest.mark.parametrize("wt,sf", TYPES)
def test_b1_one_hot_is_dequant(qmv, wt, sf):
    # x = e_c: y = level * d rounded once, the dequantized weight of column c
    rows, cols = 70, 1024
    m = inputs.make_matrix(wt, sf, rows, cols, seed=31)
    deq = oracle.dequant(m.W, wt, sf, rows, cols)
    for c in [0, 1, 15, 16, 31, 32, 255, 256, 517, cols - 1]:
        x = np.zeros((1, cols), np.float32)
        x[0, c] = 1.0
        assert_bits_equal(run(qmv, m, inputs.bf16_codes(x))[0], deq[:, c], f"one-hot {c}")


@pytest.mark.parametrize("wt", [1, 2])
def test_b1_half_subnormal_activations_exact(qmv, wt):
    # x = k * 2^-22 (|k| <= 4) are half subnormals, exact in half: those stages take half
    # operands; with power-of-two scales every partial sum is exact, so the result must be
    # bit-exact (a tensor core that flushed subnormal operands would give zeros)
    rows, cols = 96, 2048
    m = with_pow2_scales(inputs.make_matrix(wt, 1, rows, cols, seed=41), seed=42)
    rng = np.random.default_rng(43)
    x = np.ldexp(rng.integers(-4, 5, size=(1, cols)).astype(np.float32), -22)
    xc = inputs.bf16_codes(x)
    y_ref, _ = oracle.matvec(m.W, wt, 1, rows, cols, xc)
    assert np.any(y_ref != 0)
    assert np.array_equal(run(qmv, m, xc).astype(np.float64), y_ref)


@pytest.mark.parametrize("wt,sf", TYPES)
def test_b1_stages_outside_half_range(qmv, wt, sf):
    # N(0,1) activations with, in some 256-column stages, a value above the half range
    # (1e5, 3e30), one inexact below it (3e-9, 1e-30) or a half-range boundary value; those
    # stages take bfloat16 operands, the others half ones, in the same rows
    rows, cols = 160, 4096
    m = inputs.make_matrix(wt, sf, rows, cols, seed=51)
    x = np.random.default_rng(52).standard_normal((1, cols)).astype(np.float32)
    x[0, 3] = 1e5
    x[0, 256 + 40] = -3e-9
    x[0, 2 * 256 + 7] = 3e30
    x[0, 5 * 256 + 255] = 1e-30
    x[0, 9 * 256 + 100] = 65280.0    # largest bfloat16 below the half maximum: exact
    x[0, 11 * 256 + 1] = 2.0 ** -17  # exact half subnormal
    xc = inputs.bf16_codes(x)
    y_ref, absref = oracle.matvec(m.W, wt, sf, rows, cols, xc)
    check_product(run(qmv, m, xc), y_ref, absref, TOL, "mixed stages")


def test_b1_large_activations_exact(qmv):
    # Q4_0 (|level| <= 8), integer x with 2^16 (above the half maximum) in a few stages,
    # power-of-two scales 2^-4..2^-2: every partial sum is a multiple of 2^-4 below 2^19, exact
    # in float32, so the bfloat16-operand stages are bit-exact too
    wt, rows, cols = 2, 64, 2048
    m = with_pow2_scales(inputs.make_matrix(wt, 0, rows, cols, seed=61), seed=62, lo_exp=-4, hi_exp=-2)
    x = inputs.make_int_x(1, cols, False, seed=63).astype(np.float32)
    x[0, [10, 700, 1500]] = 65536.0
    xc = inputs.bf16_codes(x)
    y_ref, _ = oracle.matvec(m.W, wt, 0, rows, cols, xc)
    assert np.array_equal(run(qmv, m, xc).astype(np.float64), y_ref)


def test_b1_nan_activation_propagates(qmv):
    # NaN * level is NaN for every level, zero included: every row is NaN
    rows, cols = 48, 1024
    for wt in (1, 2):
        m = inputs.make_matrix(wt, 1, rows, cols, seed=71)
        x = np.random.default_rng(72).standard_normal((1, cols)).astype(np.float32)
        xc = inputs.bf16_codes(x)
        xc[0, 300] = 0x7FC0  # bfloat16 quiet NaN
        y_ref, _ = oracle.matvec(m.W, wt, 1, rows, cols, xc)
        y = run(qmv, m, xc)
        assert np.all(np.isnan(y_ref)) and np.all(np.isnan(y))


def test_b1_zero_activations_and_zero_rows(qmv):
    rows, cols = 80, 2048
    m = inputs.make_matrix(2, 1, rows, cols, seed=81)
    assert np.all(run(qmv, m, bf16(np.zeros(cols))) == 0.0)
    q = m.q.copy().reshape(rows, -1)
    q[::5] = 0x88  # every level 0
    W = inputs.assemble(2, 1, rows, cols, q.reshape(-1), m.d_codes)
    m2 = inputs.Matrix(2, 1, rows, cols, W, q.reshape(-1), m.d_codes)
    x = inputs.make_x(1, cols, True, seed=82)
    y_ref, absref = oracle.matvec(W, 2, 1, rows, cols, x)
    y = run(qmv, m2, x)
    assert np.all(y[:, ::5] == 0.0)
    check_product(y, y_ref, absref, TOL, "zero rows")


def test_b1_grouped_and_graph_replay_bit_identical(qmv):
    # a grouped launch of shapes with different column counts, eager and in a graph
    import torch
    shapes = [(512, 4096), (128, 4096), (300, 11008), (4096, 256)]
    probs, refs = [], []
    for i, (rows, cols) in enumerate(shapes):
        m = inputs.make_matrix(2, 1, rows, cols, seed=90 + i)
        x = inputs.make_x(1, cols, True, seed=95 + i)
        y = torch.full((1, rows), 7.0, device="cuda")
        probs.append((rows, cols, dev_u8(m.W), dev_x(x), y))
        refs.append(oracle.matvec(m.W, 2, 1, rows, cols, x))
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        qmv.matvec_grouped(2, 1, probs, overlap=True)
    torch.cuda.synchronize()
    eager = [p[4].cpu().numpy().copy() for p in probs]
    for (rows, cols, _, _, _), e, (y_ref, absref) in zip(probs, eager, refs):
        check_product(e, y_ref, absref, TOL, f"grouped {rows}x{cols}")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(2):
            qmv.matvec_grouped(2, 1, probs, overlap=True)
    for p in probs:
        p[4].fill_(0.0)
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for p, e in zip(probs, eager):
        assert_bits_equal(p[4].cpu().numpy(), e, "graph replay")


@pytest.mark.parametrize("sf", [1, 0])
def test_one_chunk_stages_large_q4(qmv, sf):
    # Q4_0 launches of 32 MB or more take one-chunk stages (five 4-warp CTAs per SM): 65536 x 4096
    # (151 / 168 MB) against the oracle on sampled rows, and exactly on an integer case
    import torch
    rows, cols = 65536, 4096
    m = inputs.make_matrix(2, sf, rows, cols, seed=500 + sf)
    x = inputs.make_x(1, cols, True, seed=501)
    y = run(qmv, m, x)
    rng = np.random.default_rng(502)
    ids = np.unique(np.concatenate([np.arange(40), rows - 1 - np.arange(40), rng.integers(0, rows, 200)]))
    y_ref, absref = oracle.matvec_rows(m.W, 2, sf, rows, cols, x, ids)
    check_product(y[:, ids], y_ref, absref, tol=TOL, what=f"one-chunk 65536x4096 sf{sf}")
    # integer activations with power-of-two scales: every partial sum exact, so bit-exact
    me = with_pow2_scales(m, 503)
    xe = inputs.make_int_x(1, cols, True, seed=504)
    ye = run(qmv, me, xe)
    ye_ref, _ = oracle.matvec_rows(me.W, 2, sf, rows, cols, xe, ids)
    assert_bits_equal(ye[:, ids], ye_ref.astype(np.float32), f"one-chunk exact sf{sf}")
    assert torch.cuda.is_available()


def test_one_chunk_stages_grouped_ffn(qmv):
    # the layer's {w1, w3} launch (2 x 11008 x 4096, 50.8 MB) in one grouped call, with overlap
    import torch
    dim, hidden = 4096, 11008
    ms = [inputs.make_matrix(2, 1, hidden, dim, seed=510 + i) for i in range(2)]
    x = inputs.make_x(1, dim, True, seed=512)
    xd = dev_x(x)
    ys = [torch.empty((1, hidden), device="cuda") for _ in ms]
    for _ in range(2):
        qmv.matvec_grouped(2, 1, [(hidden, dim, dev_u8(m.W), xd, y) for m, y in zip(ms, ys)], overlap=True)
    torch.cuda.synchronize()
    rng = np.random.default_rng(513)
    ids = np.unique(np.concatenate([np.arange(20), hidden - 1 - np.arange(20), rng.integers(0, hidden, 100)]))
    for m, y in zip(ms, ys):
        y_ref, absref = oracle.matvec_rows(m.W, 2, 1, hidden, dim, x, ids)
        check_product(y.cpu().numpy()[:, ids], y_ref, absref, tol=TOL, what="one-chunk grouped ffn")


@pytest.mark.parametrize("sf", [1, 0])
@pytest.mark.parametrize("rows,cols", [(4096, 4096), (4096, 11008), (2048, 4096)])
def test_few_tile_q4_launches(qmv, sf, rows, cols):
    # Q4_0 launches with fewer 32-row warp tiles than SMs (4096 rows: 128 tiles; the column split
    # and 8-warp CTAs fill the GPU): sampled rows against the oracle, an exact integer case bit for bit
    m = inputs.make_matrix(2, sf, rows, cols, seed=520 + rows + cols + sf)
    x = inputs.make_x(1, cols, True, seed=521)
    y = run(qmv, m, x)
    rng = np.random.default_rng(522)
    ids = np.unique(np.concatenate([np.arange(40), rows - 1 - np.arange(40), rng.integers(0, rows, 200)]))
    y_ref, absref = oracle.matvec_rows(m.W, 2, sf, rows, cols, x, ids)
    check_product(y[:, ids], y_ref, absref, tol=TOL, what=f"few tiles {rows}x{cols} sf{sf}")
    me = with_pow2_scales(m, 523)
    xe = inputs.make_int_x(1, cols, True, seed=524)
    ye = run(qmv, me, xe)
    ye_ref, _ = oracle.matvec_rows(me.W, 2, sf, rows, cols, xe, ids)
    assert_bits_equal(ye[:, ids], ye_ref.astype(np.float32), f"few tiles exact {rows}x{cols} sf{sf}")


@pytest.mark.parametrize("wt,sf", [(2, 1), (1, 0)])
def test_group_of_192_tiles_one_stage_per_warp(qmv, wt, sf):
    # the Llama-7B {wq, wk, wv} launch shape (6144 rows of 4096 columns in three problems): each
    # warp gets one 512-column stage, so 8-warp CTAs with a ring of one stage take it (every
    # stage requested before the dependency wait; the slot refilled only after it is read).
    # Sampled rows against the oracle; repeated calls and graph replays give the same bits.
    import torch
    from helpers import assert_bits_equal
    shapes = [(4096, 4096), (1024, 4096), (1024, 4096)]
    rng = np.random.default_rng(60 + wt)
    mats = [inputs.make_matrix(wt, sf, r, c, seed=600 + i) for i, (r, c) in enumerate(shapes)]
    x = inputs.make_x(1, 4096, True, seed=610)
    xd = dev_x(x)
    Ws = [dev_u8(m.W) for m in mats]
    ys = [torch.empty((1, r), device="cuda") for r, _ in shapes]
    probs = [(r, c, W, xd, y) for (r, c), W, y in zip(shapes, Ws, ys)]
    qmv.matvec_grouped(wt, sf, probs, overlap=True)
    torch.cuda.synchronize()
    first = [y.cpu().numpy().copy() for y in ys]
    for m, (r, c), y in zip(mats, shapes, first):
        ids = np.unique(np.concatenate([np.arange(0, r, 31), rng.integers(0, r, 64), [r - 1]]))
        y_ref, absref = oracle.matvec_rows(m.W, wt, sf, r, c, x, ids)
        check_product(y[:, ids], y_ref, absref, 1e-3, f"qkv group {r}x{c}")
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            qmv.matvec_grouped(wt, sf, probs, overlap=True)
    for _ in range(3):
        for y in ys:
            y.zero_()
        g.replay()
        torch.cuda.synchronize()
        for y, f in zip(ys, first):
            assert_bits_equal(y.cpu().numpy(), f, "qkv group graph replay")
    assert qmv.last_error() == 0
