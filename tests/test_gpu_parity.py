"""CUDA path vs the CPU oracle, through the C ABI (libqmv.so via the ctypes binding).

Bars: dequantization bit-exact; products within |y_gpu - y_ref| <= 1e-3 * sum_c |w x| per
element (exactly equal where that sum is 0); where every partial sum is exactly
representable (one-hot x, integer x with power-of-two scales) the product is bit-exact.
"""
import numpy as np
import pytest

import oracle
from block_quantized_weight_q4_gb300 import inputs
from helpers import HALF_TOL, assert_bits_equal, check_product, dev_u8, dev_x

pytestmark = pytest.mark.gpu

TOL = 1e-3


@pytest.fixture(scope="module", autouse=True)
def qmv():
    import torch
    from block_quantized_weight_q4_gb300.build import build
    import block_quantized_weight_q4_gb300 as q
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build()
    q.load_library()
    yield q
    assert q.last_error() == 0


def gpu_dequant(q, m):
    return q.dequant(m.wtype, m.scale_f16, m.rows, m.cols, dev_u8(m.W)).cpu().numpy()


def gpu_matvec(q, m, x):
    import torch
    y = q.matvec(m.wtype, m.scale_f16, m.rows, m.cols, dev_u8(m.W), dev_x(x))
    torch.cuda.synchronize()
    return y.cpu().numpy()


SHAPES = [(1, 32), (3, 96), (7, 64), (33, 256), (17, 160), (64, 1024), (100, 4096), (5, 11008)]
TYPES = [(1, 0), (1, 1), (2, 0), (2, 1)]


# ---------------------------------------------------------------- dequant
@pytest.mark.parametrize("wt,sf", TYPES)
@pytest.mark.parametrize("rows,cols", SHAPES)
def test_dequant_bit_exact(qmv, wt, sf, rows, cols):
    m = inputs.make_matrix(wt, sf, rows, cols, seed=rows + cols + 10 * wt + sf)
    assert_bits_equal(gpu_dequant(qmv, m), oracle.dequant(m.W, wt, sf, rows, cols), f"{wt},{sf},{rows}x{cols}")


@pytest.mark.parametrize("wt,sf", TYPES)
def test_dequant_special_scales(qmv, wt, sf):
    # every scale is valid input: negative, zero, subnormal, huge, inf, NaN scales
    rows, cols = 4, 256
    m = inputs.make_matrix(wt, sf, rows, cols, seed=5)
    if sf:
        specials = np.array([0x8000, 0x0000, 0x0001, 0x03FF, 0x7BFF, 0xFBFF, 0x7C00, 0xFC00, 0x7E00,
                             0x3C00, 0xBC00, 0x0400, 0x8001, 0x2E66, 0x1234, 0x7FFF], np.uint16)
    else:
        specials = np.array([-0.0, 0.0, 1e-45, 1.1754942e-38, 3.4028235e38, -3.4028235e38, np.inf, -np.inf,
                             np.nan, 1.0, -1.0, 1.1754944e-38, -1e-45, 0.1, 7e-39, 1e-40], np.float32).view(np.uint32)
    codes = m.d_codes.reshape(-1).copy()
    codes[:specials.size] = specials
    W = inputs.assemble(wt, sf, rows, cols, m.q, codes)
    m2 = inputs.Matrix(wt, sf, rows, cols, W, m.q, codes)
    assert_bits_equal(gpu_dequant(qmv, m2), oracle.dequant(W, wt, sf, rows, cols), "special scales")


# ---------------------------------------------------------------- products
@pytest.mark.parametrize("wt,sf", TYPES)
@pytest.mark.parametrize("rows,cols", SHAPES)
@pytest.mark.parametrize("xbf16", [True, False])
@pytest.mark.parametrize("batch", [1, 3, 8, 11])
def test_matvec_tolerance(qmv, wt, sf, rows, cols, xbf16, batch):
    m = inputs.make_matrix(wt, sf, rows, cols, seed=rows * 3 + cols + wt)
    x = inputs.make_x(batch, cols, xbf16, seed=rows + batch)
    y_ref, absref = oracle.matvec(m.W, wt, sf, rows, cols, x)
    check_product(gpu_matvec(qmv, m, x), y_ref, absref, TOL, f"{wt},{sf},{rows}x{cols},b{batch}")


@pytest.mark.parametrize("wt,sf", TYPES)
@pytest.mark.parametrize("rows,cols", [(16, 256), (21, 512), (3, 96), (40, 1024)])
@pytest.mark.parametrize("xbf16", [True, False])
def test_matvec_exact_integer_pow2(qmv, wt, sf, rows, cols, xbf16):
    # integer x in [-4, 4], d = 2^e with e in [-4, 0]: every partial sum is a multiple of
    # 2^-4 well below 2^20, exact in float32 in any order, so the result is bit-exact.
    rng = np.random.default_rng(rows + cols)
    m = inputs.make_matrix(wt, sf, rows, cols, seed=7)
    codes = inputs.pow2_scales(rng, rows * cols // 32, sf)
    W = inputs.assemble(wt, sf, rows, cols, m.q, codes)
    m2 = inputs.Matrix(wt, sf, rows, cols, W, m.q, codes)
    x = inputs.make_int_x(8, cols, xbf16, seed=3)
    y_ref, _ = oracle.matvec(W, wt, sf, rows, cols, x)
    y = gpu_matvec(qmv, m2, x)
    assert np.array_equal(y.astype(np.float64), y_ref)


@pytest.mark.parametrize("wt,sf", TYPES)
@pytest.mark.parametrize("cols", [96, 512])
def test_matvec_one_hot_is_dequant(qmv, wt, sf, cols):
    # x = e_c: one non-zero term, so y[b][r] is level * d rounded once: the dequantized weight.
    rows = 37
    m = inputs.make_matrix(wt, sf, rows, cols, seed=cols)
    picks = [0, 5, 31, 32, cols - 1, cols // 2, 17, cols - 33]
    x = np.zeros((8, cols), np.float32)
    for b, c in enumerate(picks):
        x[b, c] = 1.0
    deq = oracle.dequant(m.W, wt, sf, rows, cols)
    for xb in (x, inputs.bf16_codes(x)):
        y = gpu_matvec(qmv, m, xb)
        assert_bits_equal(y, deq[:, picks].T, "one-hot")


@pytest.mark.parametrize("wt", [1, 2])
def test_zero_level_rows_give_exact_zero(qmv, wt):
    # rows whose levels are all 0 have sum |w x| = 0: the product must be exactly 0
    rows, cols = 24, 512
    m = inputs.make_matrix(wt, 1, rows, cols, seed=2)
    q = m.q.copy().reshape(rows, -1)
    q[::3] = 0x88 if wt == 2 else 0x00
    W = inputs.assemble(wt, 1, rows, cols, q.reshape(-1), m.d_codes)
    m2 = inputs.Matrix(wt, 1, rows, cols, W, q.reshape(-1), m.d_codes)
    x = inputs.make_x(4, cols, True, seed=1)
    y_ref, absref = oracle.matvec(W, wt, 1, rows, cols, x)
    y = gpu_matvec(qmv, m2, x)
    assert np.all(y[:, ::3] == 0.0)
    check_product(y, y_ref, absref, TOL, "zero rows")


def test_q8_minus_128_decodes_faithfully(qmv):
    # -128 is not rejected by the product (only by validate); it decodes as -128 * d.
    rows, cols = 16, 256
    m = inputs.make_matrix(1, 0, rows, cols, seed=4)
    q = m.q.copy()
    q[::7] = 0x80
    W = inputs.assemble(1, 0, rows, cols, q, m.d_codes)
    m2 = inputs.Matrix(1, 0, rows, cols, W, q, m.d_codes)
    x = inputs.make_x(2, cols, True, seed=2)
    y_ref, absref = oracle.matvec(W, 1, 0, rows, cols, x)
    check_product(gpu_matvec(qmv, m2, x), y_ref, absref, TOL, "q8 -128")
    assert_bits_equal(gpu_dequant(qmv, m2), oracle.dequant(W, 1, 0, rows, cols), "q8 -128 dequant")


def test_output_guards_untouched(qmv):
    import torch
    for wt, rows, cols in [(2, 37, 512), (1, 5, 96), (2, 33, 4096)]:
        m = inputs.make_matrix(wt, 1, rows, cols, seed=9)
        x = dev_x(inputs.make_x(3, cols, True, seed=9))
        buf = torch.full((3 * rows + 64,), 12345.0, dtype=torch.float32, device="cuda")
        y = buf[32:32 + 3 * rows].view(3, rows)
        qmv.matvec(wt, 1, rows, cols, dev_u8(m.W), x, y)
        torch.cuda.synchronize()
        b = buf.cpu().numpy()
        assert np.all(b[:32] == 12345.0) and np.all(b[32 + 3 * rows:] == 12345.0)


def test_batch_zero_is_noop(qmv):
    import torch
    m = inputs.make_matrix(2, 1, 16, 256, seed=1)
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    y = torch.full((0, 16), 1.0, device="cuda")
    qmv.matvec(2, 1, 16, 256, dev_u8(m.W), x, y)
    torch.cuda.synchronize()


def test_nonfinite_scales_propagate_in_products(qmv):
    rows, cols = 16, 256
    m = inputs.make_matrix(2, 0, rows, cols, seed=3)
    codes = m.d_codes.reshape(-1).copy()
    codes[0] = np.array([np.inf], np.float32).view(np.uint32)[0]      # row 0 block 0
    codes[8 * 3 + 1] = np.array([np.nan], np.float32).view(np.uint32)[0]  # row 3 block 1
    W = inputs.assemble(2, 0, rows, cols, m.q, codes)
    m2 = inputs.Matrix(2, 0, rows, cols, W, m.q, codes)
    x = inputs.make_x(1, cols, True, seed=1)
    y_ref, absref = oracle.matvec(W, 2, 0, rows, cols, x)
    y = gpu_matvec(qmv, m2, x)
    assert np.isnan(y[0, 3]) and np.isnan(y_ref[0, 3])
    assert (np.isinf(y[0, 0]) or np.isnan(y[0, 0])) and (np.isinf(y_ref[0, 0]) or np.isnan(y_ref[0, 0]))
    ok = np.ones(rows, bool)
    ok[[0, 3]] = False
    check_product(y[:, ok], y_ref[:, ok], absref[:, ok], TOL, "finite rows")


# ---------------------------------------------------------------- validate
def test_validate_finds_first_minus_128(qmv):
    m = inputs.make_matrix(1, 0, 64, 1024, seed=1)
    assert qmv.validate(1, 0, 64, 1024, dev_u8(m.W)) == -1
    W = m.W.copy()
    W[[70000, 5000, 65535]] = 0x80
    assert qmv.validate(1, 0, 64, 1024, dev_u8(W)) == 5000
    assert oracle.validate(W, 1, 0, 64, 1024) == oracle.E_FORMAT
    m4 = inputs.make_matrix(2, 0, 64, 1024, seed=1)
    W4 = m4.W.copy()
    W4[:100] = 0x80
    assert qmv.validate(2, 0, 64, 1024, dev_u8(W4)) == -1


# ---------------------------------------------------------------- full-size workloads
def sample_rows(rows, rng, n=24):
    ids = set(range(min(8, rows))) | set(range(max(0, rows - 8), rows))
    ids |= set(rng.integers(0, rows, n).tolist())
    return np.array(sorted(ids), dtype=np.int64)


@pytest.mark.parametrize("name", ["q8_256", "q4_4096", "llama7b", "mixed_qwen", "prefill"])
def test_workload_full_size(qmv, name):
    """Every matrix of the workload at its full size, every batch size it names, through
    the same calls the benchmark times; checked on sampled rows (first, last, random)."""
    import torch
    wl = inputs.WORKLOADS[name]
    rng = np.random.default_rng(17)
    for i, spec in enumerate(wl.matrices):
        wt = spec.wtype
        if wl.q8_mask:
            wt = qmv.matrix_wtype(wl.file_wtype, wl.q8_mask, spec.cls)
            assert wt == spec.wtype
        m = inputs.make_matrix(wt, spec.scale_f16, spec.rows, spec.cols, seed=inputs.matrix_seed(name, i))
        Wd = dev_u8(m.W)
        ids = sample_rows(spec.rows, rng)
        xdt = [wl.x_bf16] + ([False] if wl.extra_x_f32 else [])
        for xb in xdt:
            for batch in wl.batches:
                x = inputs.make_x(batch, spec.cols, xb, seed=inputs.x_seed(name, i))
                y = qmv.matvec(wt, spec.scale_f16, spec.rows, spec.cols, Wd, dev_x(x))
                torch.cuda.synchronize()
                y_ref, absref = oracle.matvec_rows(m.W, wt, spec.scale_f16, spec.rows, spec.cols, x, ids)
                check_product(y.cpu().numpy()[:, ids], y_ref, absref, TOL, f"{name}/{spec.name}/b{batch}")
        # dequant of the sampled rows, bit-exact
        out = qmv.dequant(wt, spec.scale_f16, spec.rows, spec.cols, Wd)
        sub_q = m.q.reshape(spec.rows, -1)[ids].reshape(-1)
        sub_d = m.d_codes[ids].reshape(-1)
        sub = inputs.assemble(wt, spec.scale_f16, ids.size, spec.cols, sub_q, sub_d)
        assert_bits_equal(out[torch.from_numpy(ids).cuda()].cpu().numpy(), oracle.dequant(sub, wt, spec.scale_f16, ids.size, spec.cols),
                          f"{name}/{spec.name} dequant")
        del Wd, out


@pytest.mark.parametrize("wt,sf,rows,cols,batch", [
    (2, 1, 65536, 4096, 4),    # mma.sync kernel, four CTAs per SM without the reduction area (split tiles meet in q slots)
    (2, 1, 65536, 4096, 6),
    (2, 1, 14336, 4096, 2),    # fewer CTAs than the SMs hold: spread by their shared-memory request
    (1, 0, 151936, 1024, 4),
])
def test_small_batch_large_launches_sampled_and_repeatable(qmv, wt, sf, rows, cols, batch):
    import torch
    rng = np.random.default_rng(rows + batch)
    m = inputs.make_matrix(wt, sf, rows, cols, seed=rows + cols + wt + batch)
    x = inputs.make_x(batch, cols, True, seed=rows + batch)
    Wd, xd = dev_u8(m.W), dev_x(x)
    y1 = qmv.matvec(wt, sf, rows, cols, Wd, xd)
    y2 = qmv.matvec(wt, sf, rows, cols, Wd, xd)
    torch.cuda.synchronize()
    y1 = y1.cpu().numpy()
    assert_bits_equal(y1, y2.cpu().numpy(), f"repeat {rows}x{cols} b{batch}")
    ids = sample_rows(rows, rng)
    y_ref, absref = oracle.matvec_rows(m.W, wt, sf, rows, cols, x, ids)
    check_product(y1[:, ids], y_ref, absref, TOL, f"{rows}x{cols} b{batch}")


# ---------------------------------------------------------------- grouped launches
@pytest.mark.parametrize("wt,sf", TYPES)
@pytest.mark.parametrize("batch", [1, 5, 8])
@pytest.mark.parametrize("overlap", [False, True])
def test_grouped_matches_oracle(qmv, wt, sf, batch, overlap):
    # mixed shapes in one call, one of them on the general path (cols % 256 != 0)
    import torch
    shapes = [(40, 512), (7, 256), (100, 1024), (33, 96), (64, 2048)]
    probs, refs = [], []
    for i, (rows, cols) in enumerate(shapes):
        m = inputs.make_matrix(wt, sf, rows, cols, seed=50 + i)
        x = inputs.make_x(batch, cols, True, seed=60 + i)
        y = torch.full((batch, rows), 7.0, device="cuda")
        probs.append((rows, cols, dev_u8(m.W), dev_x(x), y))
        refs.append(oracle.matvec(m.W, wt, sf, rows, cols, x))
    qmv.matvec_grouped(wt, sf, probs, overlap=overlap)
    torch.cuda.synchronize()
    for (rows, cols, _, _, y), (y_ref, absref) in zip(probs, refs):
        check_product(y.cpu().numpy(), y_ref, absref, TOL, f"grouped {rows}x{cols}")


def test_grouped_in_graph_with_overlap(qmv):
    # a chain of grouped launches captured in a CUDA graph with programmatic overlap; each
    # stage's input is the previous stage's output (activations produced on the GPU)
    import torch
    rows, cols = 256, 256
    mats = [inputs.make_matrix(2, 1, rows, cols, seed=70 + i) for i in range(3)]
    Ws = [dev_u8(m.W) for m in mats]
    x0 = dev_x(inputs.make_x(1, cols, True, seed=5))
    ys = [torch.empty((1, rows), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    yf = [torch.empty((1, rows), device="cuda") for _ in range(3)]
    s = torch.cuda.Stream()
    def chain():
        x = x0
        for i in range(3):
            qmv.matvec_grouped(2, 1, [(rows, cols, Ws[i], x, yf[i])], overlap=True)
            ys[i].copy_(yf[i])  # a torch kernel between our launches
            x = ys[i]
    with torch.cuda.stream(s):
        chain()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        chain()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    x = inputs.make_x(1, cols, True, seed=5)
    for i in range(3):
        y_ref, absref = oracle.matvec(mats[i].W, 2, 1, rows, cols, x)
        got = yf[i].cpu().numpy()
        check_product(got, y_ref, absref, TOL, f"chain {i}")
        x = inputs.bf16_codes(got.astype(np.float32))


@pytest.mark.parametrize("wt,sf", TYPES)
@pytest.mark.parametrize("batch", [1, 2, 5, 8])
def test_f32_activations_needing_the_lo_part_exact(qmv, wt, sf, batch):
    # float32 x = k * 2^-6 with |k| < 2^10: up to 10 significant bits, more than bfloat16
    # holds, so a product that kept only the bfloat16 of x would be off; split as hi + lo
    # (both bfloat16) x is exact.  With |level| <= 8 (Q8_0 quants drawn in [-7, 7]) and
    # d = 2^e (e in [-2, 0]) every term is a multiple of 2^-8 below 2^7 and every partial sum
    # over 512 columns stays below 2^16: exact in float32 in any order, so the product must
    # equal the oracle bit for bit.
    rows, cols = 300, 512
    rng = np.random.default_rng(70 + wt + sf + batch)
    m = inputs.make_matrix(wt, sf, rows, cols, seed=71 + batch)
    q = m.q if wt == 2 else rng.integers(-7, 8, size=m.q.size).astype(np.int8).view(np.uint8)
    codes = inputs.pow2_scales(rng, rows * cols // 32, sf, -2, 0)
    W = inputs.assemble(wt, sf, rows, cols, q, codes)
    m2 = inputs.Matrix(wt, sf, rows, cols, W, q, codes)
    x = np.ldexp(rng.integers(-1023, 1024, size=(batch, cols)).astype(np.float32), -6)
    assert np.any(inputs.bf16_codes(x).astype(np.uint32) << 16 != x.view(np.uint32))
    y_ref, _ = oracle.matvec(W, wt, sf, rows, cols, x)
    y = gpu_matvec(qmv, m2, x)
    assert np.array_equal(y.astype(np.float64), y_ref)


@pytest.mark.parametrize("wt,sf", TYPES)
@pytest.mark.parametrize("rows,cols", [(600, 512), (300, 2048), (77, 4096)])
def test_f32_one_vector_split_in_the_product_exact(qmv, wt, sf, rows, cols):
    # one float32 vector over 256K weights or more: the block-diagonal kernel splits x into bf16
    # hi + lo in its activation stage (one launch); the exact case of the test above
    rng = np.random.default_rng(90 + wt + sf + rows)
    m = inputs.make_matrix(wt, sf, rows, cols, seed=91 + rows)
    q = m.q if wt == 2 else rng.integers(-7, 8, size=m.q.size).astype(np.int8).view(np.uint8)
    codes = inputs.pow2_scales(rng, rows * cols // 32, sf, -2, 0)
    W = inputs.assemble(wt, sf, rows, cols, q, codes)
    m2 = inputs.Matrix(wt, sf, rows, cols, W, q, codes)
    x = np.ldexp(rng.integers(-1023, 1024, size=(1, cols)).astype(np.float32), -6)
    y_ref, _ = oracle.matvec(W, wt, sf, rows, cols, x)
    assert np.array_equal(gpu_matvec(qmv, m2, x).astype(np.float64), y_ref)


@pytest.mark.parametrize("wt,sf", [(2, 1), (1, 0)])
def test_f32_one_vector_wide_magnitudes(qmv, wt, sf):
    # float32 activations over sixty decades (1e-30 .. 1e30, zeros, negative zeros), split in the
    # product: every stage spans far more than 2^28, so none is rounded to half and all keep
    # hi + lo: within the tolerance of the oracle, tight
    rows, cols = 512, 1024
    rng = np.random.default_rng(95 + wt)
    m = inputs.make_matrix(wt, sf, rows, cols, seed=96)
    x = (rng.standard_normal((1, cols)) * 10.0 ** rng.uniform(-30, 30, (1, cols))).astype(np.float32)
    x[0, ::37] = 0.0
    x[0, 5::41] = -0.0
    y_ref, absref = oracle.matvec(m.W, wt, sf, rows, cols, x)
    y = gpu_matvec(qmv, m, x)
    check_product(y, y_ref, absref, TOL, "wide f32 magnitudes")
    check_product(y, y_ref, absref, 1e-5, "wide f32 magnitudes, tight")


@pytest.mark.parametrize("rows,cols", [(1100, 2048), (12288, 8192)])
def test_f32_activations_batch8_graph_replay_bit_identical(qmv, rows, cols):
    # float32 activations, 8 vectors, eager on a stream (which creates its buffers) and then
    # replayed in a graph on it: 2.5 MB of weights take the mma.sync kernel (x split in its
    # stages), 113 MB the split kernel and the tensor-memory product
    import torch
    batch = 8
    m = inputs.make_matrix(1, 0, rows, cols, seed=81)
    x = inputs.make_x(batch, cols, False, seed=82)
    y_ref, absref = oracle.matvec(m.W, 1, 0, rows, cols, x)
    W, xd = dev_u8(m.W), dev_x(x)
    y = torch.empty((batch, rows), device="cuda")
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        qmv.matvec(1, 0, rows, cols, W, xd, y)
    torch.cuda.synchronize()
    first = y.cpu().numpy().copy()
    check_product(first, y_ref, absref, TOL, "f32 x batch 8")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            qmv.matvec(1, 0, rows, cols, W, xd, y)
    for _ in range(3):
        y.fill_(0.0)
        g.replay()
        torch.cuda.synchronize()
        assert_bits_equal(y.cpu().numpy(), first, "f32 x graph replay")


@pytest.mark.parametrize("route", ["f32", "pair", "f32_split"])
def test_one_vector_stages_rounded_to_half_and_exact(qmv, route):
    # one vector x = 1 + 2^-12 everywhere (Q8_0 levels 1..7 and scales 2^-2..1: positive weights,
    # so every error has one sign), except
    # that columns 1024..1535 also hold 2^-40 at four places.  Stages of 256 or 512 columns with
    # only 1 + 2^-12 are scaled into [2^14, 2^15) and rounded to half: 1 + 2^-12 becomes 1
    # exactly.  The stages over columns 1024..1535 span 2^40 > 2^28, so they keep hi + lo and
    # give x exactly.  The product must then equal the oracle's on x' (x with 1 outside columns
    # 1024..1535) up to float32 sums, and differ from the oracle's on x by about 2^-12 of y
    # (within HALF_TOL); the pair route (hi = 1, lo = 2^-12) and the float32 routes agree.  f32:
    # 1 MB of weights, rounded in the product's stages; f32_split: 18 MB, rounded per 256-column
    # chunk by the split kernel ahead of the product
    import torch
    rows, cols = (4096 if route == "f32_split" else 256), 4096
    rng = np.random.default_rng(97)
    q = rng.integers(1, 8, size=rows * cols).astype(np.int8).view(np.uint8)
    codes = inputs.pow2_scales(rng, rows * cols // 32, 1, -2, 0)
    W = inputs.assemble(1, 1, rows, cols, q, codes)
    x = np.full((1, cols), 1.0 + 2.0 ** -12, np.float32)
    x[0, [1024 + 17, 1024 + 300, 1024 + 301, 1024 + 511]] = 2.0 ** -40
    keep = np.zeros(cols, bool)
    keep[1024:1536] = True
    x_rounded = np.where(keep, x[0], np.float32(1.0))[None, :]
    y_ref, absref = oracle.matvec(W, 1, 1, rows, cols, x)
    y_exp, _ = oracle.matvec(W, 1, 1, rows, cols, x_rounded)
    Wd = dev_u8(W)
    y = torch.empty((1, rows), device="cuda")
    if route != "pair":
        qmv.matvec_grouped(1, 1, [(rows, cols, Wd, torch.from_numpy(x).cuda(), y)])
    else:
        hi = inputs.bf16_codes(x[0])
        lo = inputs.bf16_codes(x[0] - (hi.astype(np.uint32) << 16).view(np.float32))
        assert np.array_equal((hi.astype(np.uint32) << 16).view(np.float32)
                              + (lo.astype(np.uint32) << 16).view(np.float32), x[0])
        pair = torch.from_numpy(np.stack([hi, lo]).view(np.int16)).cuda().view(torch.bfloat16)
        qmv.matvec_grouped(1, 1, [(rows, cols, Wd, pair, y)], pair=True)
    torch.cuda.synchronize()
    yg = y.cpu().numpy()
    check_product(yg, y_ref, absref, HALF_TOL, f"{route}: against the oracle on x")
    check_product(yg, y_exp, absref, 1e-6, f"{route}: rounded stages 1, exact stages x")
    rel = (y_ref[0] - yg[0].astype(np.float64)) / absref[0]
    assert np.all(rel > 2.0 ** -12 * 0.7) and np.all(rel < 2.0 ** -12), f"{route}: {rel.min()} .. {rel.max()}"


def test_no_overlap_flag_reads_weights_written_just_before(qmv):
    # without the overlap flag a product may start during the preceding kernel's tail but must
    # read the weights that kernel writes: each replay writes one of two matrices into W with a
    # kernel right before the product (batch 1 and batch 4 routes), and y must be that matrix's
    import torch
    ma = inputs.make_matrix(2, 1, 2048, 4096, seed=70)
    mb = inputs.make_matrix(2, 1, 2048, 4096, seed=71)
    srcs = [dev_u8(ma.W), dev_u8(mb.W)]
    W = torch.zeros_like(srcs[0])
    for batch in (1, 4):
        x = inputs.make_x(batch, 4096, True, seed=72 + batch)
        xd = dev_x(x)
        want = []
        for s in srcs:
            yw = torch.empty((batch, 2048), device="cuda")
            qmv.matvec_grouped(2, 1, [(2048, 4096, s, xd, yw)])
            want.append(yw)
        torch.cuda.synchronize()
        ys = [torch.empty((batch, 2048), device="cuda") for _ in range(4)]
        g = torch.cuda.CUDAGraph()
        st = torch.cuda.Stream()
        with torch.cuda.stream(st):
            qmv.matvec_grouped(2, 1, [(2048, 4096, W, xd, ys[0])])
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=st):
            for i in range(4):
                torch.bitwise_or(srcs[i % 2], 0, out=W)      # a kernel writes the weights
                qmv.matvec_grouped(2, 1, [(2048, 4096, W, xd, ys[i])])
        for _ in range(3):
            W.zero_()
            g.replay()
            torch.cuda.synchronize()
            for i in range(4):
                assert_bits_equal(ys[i].cpu().numpy(), want[i % 2].cpu().numpy(), f"b{batch} product {i}")
    y_ref, absref = oracle.matvec(mb.W, 2, 1, 2048, 4096, x)
    check_product(ys[1].cpu().numpy(), y_ref, absref, TOL, "no overlap flag, batch 4")
