"""The activation-quantized product on the device vs the oracle.

qmv_quantize_x must give the oracle's activation image byte for byte (the Q8_0 rule decides
integers, and both sides take it in float32 round-to-nearest operations); qmv_matvec_qx must
agree with the oracle's exact evaluation to within the product's tolerance, and exactly
where every float32 step is exact.  Shapes cover one, two and four rows per warp, rows that
do not fill the last warp, block counts that do not fill the lanes, passes of 1, 2, 4 and 8
vectors and batches that take two passes; full-size matrices are checked on sampled rows.
"""
import numpy as np
import pytest

import oracle
from block_quantized_weight_q4_gb300 import inputs
from helpers import assert_bits_equal, check_product, dev_u8, dev_x

pytestmark = pytest.mark.gpu

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


def gpu_quantize_x(q, x):
    import torch
    xq = q.quantize_x(dev_x(x))
    torch.cuda.synchronize()
    return xq


def gpu_qx(q, m, xq_dev, batch):
    import torch
    y = q.matvec_qx(m.wtype, m.scale_f16, m.rows, m.cols, dev_u8(m.W), xq_dev, batch)
    torch.cuda.synchronize()
    return y.cpu().numpy()


def sub_matrix(m, ids):
    """The byte image of the listed rows of m (for checking full-size results row by row)."""
    ids = np.asarray(ids)
    qb = m.cols if m.wtype == 1 else m.cols // 2
    q = m.q.reshape(m.rows, qb)[ids]
    return inputs.assemble(m.wtype, m.scale_f16, ids.size, m.cols, q, m.d_codes[ids])


def activations(rng, batch, cols):
    # N(0, 1) with a per-block magnitude spread, plus blocks that probe the rule: all zero,
    # amax below the 1e-30 floor, and halves (rounded away from zero)
    x = (rng.standard_normal((batch, cols)) * np.exp(rng.uniform(-4, 4, (batch, cols // 32))).repeat(32, 1))
    x = x.astype(np.float32)
    nb = cols // 32
    if nb >= 4:
        x[0, 0:32] = 0.0
        x[-1, 32:64] = rng.standard_normal(32) * 1e-31
        x[0, 64:96] = np.arange(-16, 16) + 0.5
    return x


@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("batch,cols", [(1, 32), (3, 96), (8, 4096), (5, 11008), (2, 14336)])
def test_quantize_x_matches_oracle(qmv, bf16, batch, cols):
    rng = np.random.default_rng(batch * 31 + cols + bf16)
    x = activations(rng, batch, cols)
    xin = inputs.bf16_codes(x) if bf16 else x
    got = gpu_quantize_x(qmv, xin).cpu().numpy()
    want = oracle.quantize_x(xin)
    assert got.shape == want.shape
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[:8]}"


@pytest.mark.parametrize("wt,sf", TYPES)
@pytest.mark.parametrize("rows,cols,batch", [(1, 32, 1), (5, 96, 2), (37, 1024, 3), (100, 4128, 4),
                                             (300, 4096, 8), (70, 2048, 11)])
def test_matvec_qx_matches_oracle(qmv, wt, sf, rows, cols, batch):
    rng = np.random.default_rng(rows + cols + batch + 10 * wt + sf)
    m = inputs.make_matrix(wt, sf, rows, cols, seed=rows * 3 + cols)
    x = activations(rng, batch, cols)
    xq_host = oracle.quantize_x(x)
    y = gpu_qx(qmv, m, dev_u8(xq_host), batch)
    y_ref, absref = oracle.matvec_qx(m.W, wt, sf, rows, cols, xq_host, batch)
    check_product(y, y_ref, absref, what=f"qx {wt},{sf} {rows}x{cols} b{batch}")
    check_product(y, y_ref, absref, tol=1e-4, what=f"qx tight {wt},{sf} {rows}x{cols} b{batch}")


@pytest.mark.parametrize("wt", [1, 2])
@pytest.mark.parametrize("batch", [1, 2, 3, 8])
@pytest.mark.parametrize("cols", [128, 512])
def test_matvec_qx_exact_case(qmv, wt, batch, cols):
    # power-of-two weight scales and activations k * 2^e (one element per block at +-127):
    # every block term (d_w d_x) * isum is an integer times 2^-10 below 2^24 units, and so is
    # every partial sum, so the float32 result is exact in any order (cols 512 with 2..8 vectors:
    # the tensor-core route)
    rows = 9
    rng = np.random.default_rng(80 + wt + batch)
    if wt == 1:
        q = rng.integers(-127, 128, rows * cols).astype(np.int8).view(np.uint8)
    else:
        q = rng.integers(0, 256, rows * cols // 2).astype(np.uint8)
    d = np.full(rows * cols // 32, 2.0 ** -6, np.float32).view(np.uint32)
    W = inputs.assemble(wt, 0, rows, cols, q, d)
    m = inputs.Matrix(wt, 0, rows, cols, W, q, d.reshape(rows, cols // 32))
    k = rng.integers(-127, 128, (batch, cols // 32, 32))
    k[:, :, 3] = 127
    x = (k * 2.0 ** -4).reshape(batch, cols).astype(np.float32)
    xq_host = oracle.quantize_x(x)
    y = gpu_qx(qmv, m, dev_u8(xq_host), batch)
    y_ref, _ = oracle.matvec_qx(W, wt, 0, rows, cols, xq_host, batch)
    assert_bits_equal(y, y_ref.astype(np.float32), f"exact qx {wt} b{batch}")
    assert np.array_equal(y.astype(np.float64), y_ref)


@pytest.mark.parametrize("wt,sf,rows,cols,batch", [
    (2, 1, 65536, 4096, 1),    # four rows per warp
    (2, 1, 65536, 4096, 2),
    (2, 1, 14336, 4096, 3),    # two rows per warp, a pass of 4 with one repeated vector
    (1, 0, 11008, 4096, 8),    # Q8_0, two rows per warp
    (2, 0, 4096, 11008, 1),    # one row per warp, 344 blocks per row
    (1, 1, 151936, 1024, 1),   # the Q8_0 classifier shape
    (2, 1, 65536, 4096, 8),    # tensor-core mode, four CTAs per SM, split tiles meeting in the q slots
    (1, 0, 151936, 1024, 8),
])
def test_matvec_qx_full_size_sampled_rows(qmv, wt, sf, rows, cols, batch):
    import torch
    rng = np.random.default_rng(rows + batch)
    m = inputs.make_matrix(wt, sf, rows, cols, seed=rows + cols + wt)
    x = activations(rng, batch, cols)
    xq = qmv.quantize_x(dev_x(x))
    y = qmv.matvec_qx(wt, sf, rows, cols, dev_u8(m.W), xq, batch)
    torch.cuda.synchronize()
    y = y.cpu().numpy()
    xq_host = xq.cpu().numpy()
    assert np.array_equal(xq_host, oracle.quantize_x(x))
    ids = np.unique(np.concatenate([np.arange(8), rows - 1 - np.arange(8), rng.integers(0, rows, 48)]))
    y_ref, absref = oracle.matvec_qx(sub_matrix(m, ids), wt, sf, ids.size, cols, xq_host, batch)
    check_product(y[:, ids], y_ref, absref, what=f"full {wt},{sf} {rows}x{cols} b{batch}")
    check_product(y[:, ids], y_ref, absref, tol=1e-4, what=f"full tight {wt},{sf} {rows}x{cols} b{batch}")


def test_matvec_qx_repeat_and_graph_are_bit_identical(qmv):
    import torch
    rows, cols, batch = 14336, 4096, 2
    m = inputs.make_matrix(2, 1, rows, cols, seed=5)
    x = activations(np.random.default_rng(6), batch, cols)
    W = dev_u8(m.W)
    xd = dev_x(x)
    xq = qmv.quantize_x(xd)
    y1 = qmv.matvec_qx(2, 1, rows, cols, W, xq, batch).clone()
    y2 = torch.empty_like(y1)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        qmv.quantize_x(xd, xq=xq, stream=s)
        qmv.matvec_qx(2, 1, rows, cols, W, xq, batch, y=y2, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    y3 = torch.empty_like(y1)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        qmv.quantize_x(xd, xq=xq)
        qmv.matvec_qx(2, 1, rows, cols, W, xq, batch, y=y3)
    for _ in range(3):
        y3.zero_()
        g.replay()
    torch.cuda.synchronize()
    assert_bits_equal(y1.cpu().numpy(), y2.cpu().numpy(), "stream")
    assert_bits_equal(y1.cpu().numpy(), y3.cpu().numpy(), "graph replay")


def test_matvec_qx_empty_batch_and_y_untouched(qmv):
    import torch
    m = inputs.make_matrix(2, 1, 64, 64, seed=1)
    y = torch.full((0, 64), 7.0, device="cuda")
    out = qmv.matvec_qx(2, 1, 64, 64, dev_u8(m.W), torch.empty(0, dtype=torch.uint8, device="cuda"), 0, y=y)
    torch.cuda.synchronize()
    assert out.shape == (0, 64)


# --------------------------------------------- quantizer inside the product (qmv_matvec_qx_grouped)
def gpu_qx_grouped(q, wt, sf, mats, xs, bf16, overlap=False):
    import torch
    probs = []
    for m, x in zip(mats, xs):
        xin = inputs.bf16_codes(x) if bf16 else x
        probs.append((m.rows, m.cols, dev_u8(m.W), dev_x(xin), torch.full((x.shape[0], m.rows), 9.0, device="cuda")))
    q.matvec_qx_grouped(wt, sf, probs, overlap=overlap)
    torch.cuda.synchronize()
    return [p[4].cpu().numpy() for p in probs]


def oracle_qx(m, x, bf16):
    xin = inputs.bf16_codes(x) if bf16 else x
    xq = oracle.quantize_x(xin)
    return oracle.matvec_qx(m.W, m.wtype, m.scale_f16, m.rows, m.cols, xq, x.shape[0])


@pytest.mark.parametrize("wt,sf", TYPES)
@pytest.mark.parametrize("bf16", [False, True])
@pytest.mark.parametrize("shapes,batch", [([(37, 1024), (100, 1024)], 1), ([(300, 4096), (64, 4096), (64, 4096)], 3),
                                          ([(70, 2048), (40, 4128)], 8), ([(5, 96)], 11), ([(200, 512)], 2)])
def test_matvec_qx_grouped_matches_oracle(qmv, wt, sf, bf16, shapes, batch):
    rng = np.random.default_rng(sum(r for r, _ in shapes) + batch + 10 * wt + sf + bf16)
    mats = [inputs.make_matrix(wt, sf, r, c, seed=r * 3 + c + i) for i, (r, c) in enumerate(shapes)]
    xs = [activations(rng, batch, c) for _, c in shapes]
    ys = gpu_qx_grouped(qmv, wt, sf, mats, xs, bf16)
    for m, x, y in zip(mats, xs, ys):
        y_ref, absref = oracle_qx(m, x, bf16)
        what = f"qx grouped {wt},{sf} bf16={bf16} {m.rows}x{m.cols} b{batch}"
        check_product(y, y_ref, absref, what=what)
        check_product(y, y_ref, absref, tol=1e-4, what=what + " tight")


@pytest.mark.parametrize("wt", [1, 2])
@pytest.mark.parametrize("batch", [1, 3, 8])
def test_matvec_qx_grouped_exact_case(qmv, wt, batch):
    # the exact case of test_matvec_qx_exact_case for a group of two problems: bit-exact
    rng = np.random.default_rng(90 + wt + batch)
    mats, xs = [], []
    for rows, cols in [(9, 128), (17, 256)]:
        if wt == 1:
            q = rng.integers(-127, 128, rows * cols).astype(np.int8).view(np.uint8)
        else:
            q = rng.integers(0, 256, rows * cols // 2).astype(np.uint8)
        d = np.full(rows * cols // 32, 2.0 ** -6, np.float32).view(np.uint32)
        W = inputs.assemble(wt, 0, rows, cols, q, d)
        mats.append(inputs.Matrix(wt, 0, rows, cols, W, q, d.reshape(rows, cols // 32)))
        k = rng.integers(-127, 128, (batch, cols // 32, 32))
        k[:, :, 3] = 127
        xs.append((k * 2.0 ** -4).reshape(batch, cols).astype(np.float32))
    ys = gpu_qx_grouped(qmv, wt, 0, mats, xs, False)
    for m, x, y in zip(mats, xs, ys):
        y_ref, _ = oracle_qx(m, x, False)
        assert np.array_equal(y.astype(np.float64), y_ref), f"exact grouped qx {wt} b{batch} {m.rows}x{m.cols}"


@pytest.mark.parametrize("wt", [1, 2])
@pytest.mark.parametrize("bf16", [False, True])
def test_matvec_qx_grouped_one_vector_exact_case(qmv, wt, bf16):
    # one vector, cols multiples of 256 (the block-diagonal kernel, quants in its stages): the
    # exact case above (scales 2^-6 and 2^-4, integer block sums) must match bit for bit, with
    # zero blocks and blocks whose largest magnitude sits in any of the four lanes
    rng = np.random.default_rng(120 + wt + bf16)
    mats, xs = [], []
    for rows, cols in [(9, 256), (40, 512), (300, 512)]:  # block sums stay exact in float32
        if wt == 1:
            q = rng.integers(-127, 128, rows * cols).astype(np.int8).view(np.uint8)
        else:
            q = rng.integers(0, 256, rows * cols // 2).astype(np.uint8)
        d = np.full(rows * cols // 32, 2.0 ** -6, np.float32).view(np.uint32)
        W = inputs.assemble(wt, 0, rows, cols, q, d)
        mats.append(inputs.Matrix(wt, 0, rows, cols, W, q, d.reshape(rows, cols // 32)))
        k = rng.integers(-127, 128, (1, cols // 32, 32))
        k[0, np.arange(cols // 32), rng.integers(0, 32, cols // 32)] = 127 * rng.choice([-1, 1], cols // 32)
        k[0, ::7] = 0  # zero blocks
        xs.append((k * 2.0 ** -4).reshape(1, cols).astype(np.float32))
    ys = gpu_qx_grouped(qmv, wt, 0, mats, xs, bf16)
    for m, x, y in zip(mats, xs, ys):
        y_ref, _ = oracle_qx(m, x, bf16)
        assert np.array_equal(y.astype(np.float64), y_ref), f"exact one-vector qx {wt} {m.rows}x{m.cols}"


@pytest.mark.parametrize("batch", [1, 8])
def test_matvec_qx_grouped_llama7b_groups_sampled(qmv, batch):
    # the layer's groups as the layer step runs them ({wq,wk,wv} on one x, {w1,w3} on one x,
    # {w2} on 11008 columns): sampled rows of every matrix against the oracle
    rng = np.random.default_rng(95 + batch)
    spec = {s.name: s for s in inputs.WORKLOADS["llama7b"].matrices}
    for grp in (["wq", "wk", "wv"], ["w1", "w3"], ["w2"]):
        mats = [inputs.make_matrix(spec[n].wtype, spec[n].scale_f16, spec[n].rows, spec[n].cols, seed=300 + i)
                for i, n in enumerate(grp)]
        x = activations(rng, batch, mats[0].cols)
        ys = gpu_qx_grouped(qmv, 2, 1, mats, [x] * len(mats), True)
        xq = oracle.quantize_x(inputs.bf16_codes(x))
        for m, y in zip(mats, ys):
            ids = np.unique(np.concatenate([np.arange(8), m.rows - 1 - np.arange(8), rng.integers(0, m.rows, 32)]))
            y_ref, absref = oracle.matvec_qx(sub_matrix(m, ids), 2, 1, ids.size, m.cols, xq, batch)
            check_product(y[:, ids], y_ref, absref, tol=1e-4, what=f"layer group {grp} b{batch}")


def test_matvec_qx_grouped_repeat_overlap_and_graph_bit_identical(qmv):
    # the same launch eagerly, with the overlap flag after a kernel that writes x, and in graph
    # replays: the same bits; and the same sums as the two-step path within the tolerance
    import torch
    rows, cols, batch = 14336, 4096, 2
    m = inputs.make_matrix(2, 1, rows, cols, seed=7)
    x = activations(np.random.default_rng(8), batch, cols)
    W = dev_u8(m.W)
    xd = dev_x(inputs.bf16_codes(x))
    xsrc = xd.clone()
    y1 = torch.empty((batch, rows), device="cuda")
    qmv.matvec_qx_grouped(2, 1, [(rows, cols, W, xd, y1)])
    torch.cuda.synchronize()
    first = y1.cpu().numpy().copy()
    y2 = torch.empty_like(y1)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):  # the stream's first call creates its split buffer (not while captured)
        qmv.matvec_qx_grouped(2, 1, [(rows, cols, W, xd, y2)])
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        xd.copy_(xsrc)   # the activations come from the kernel just before the product
        qmv.matvec_qx_grouped(2, 1, [(rows, cols, W, xd, y2)], overlap=True)
    for _ in range(4):
        xd.zero_()
        y2.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert_bits_equal(y2.cpu().numpy(), first, "graph replay with overlap")
    xq = qmv.quantize_x(xd)
    y3 = qmv.matvec_qx(2, 1, rows, cols, W, xq, batch)
    torch.cuda.synchronize()
    ids = np.arange(0, rows, 97)
    y_ref, absref = oracle.matvec_qx(sub_matrix(m, ids), 2, 1, ids.size, cols, xq.cpu().numpy(), batch)
    check_product(first[:, ids], y_ref, absref, tol=1e-4, what="fused")
    check_product(y3.cpu().numpy()[:, ids], y_ref, absref, tol=1e-4, what="two-step")
    assert qmv.last_error() == 0


@pytest.mark.parametrize("wt", [1, 2])
@pytest.mark.parametrize("batch", [2, 8, 11])
def test_matvec_qx_grouped_two_step_exact_case(qmv, wt, batch):
    # two or more vectors, cols multiples of 256 (the quantizer launch, then the mma.sync
    # kernel's tensor-core mode on the images in the stream's split buffer): the exact case
    # (integer block sums, power-of-two scales) bit for bit, with two problems sharing one
    # activation array, one with its own, and 11 vectors taking two passes
    import torch
    rng = np.random.default_rng(140 + wt + batch)
    mats = []
    for rows, cols in [(33, 512), (100, 512), (17, 256)]:
        if wt == 1:
            q = rng.integers(-127, 128, rows * cols).astype(np.int8).view(np.uint8)
        else:
            q = rng.integers(0, 256, rows * cols // 2).astype(np.uint8)
        d = np.full(rows * cols // 32, 2.0 ** -6, np.float32).view(np.uint32)
        W = inputs.assemble(wt, 0, rows, cols, q, d)
        mats.append(inputs.Matrix(wt, 0, rows, cols, W, q, d.reshape(rows, cols // 32)))
    xs = []
    for cols in (512, 256):
        k = rng.integers(-127, 128, (batch, cols // 32, 32))
        k[:, :, 7] = 127
        k[:, ::5] = 0  # zero blocks
        xs.append((k * 2.0 ** -4).reshape(batch, cols).astype(np.float32))
    x512 = dev_x(xs[0])
    probs = [(m.rows, m.cols, dev_u8(m.W), x512 if m.cols == 512 else dev_x(xs[1]),
              torch.full((batch, m.rows), 9.0, device="cuda")) for m in mats]
    qmv.matvec_qx_grouped(wt, 0, probs)
    torch.cuda.synchronize()
    for m, p in zip(mats, probs):
        y_ref, _ = oracle_qx(m, xs[0] if m.cols == 512 else xs[1], False)
        assert np.array_equal(p[4].cpu().numpy().astype(np.float64), y_ref), \
            f"exact two-step qx {wt} b{batch} {m.rows}x{m.cols}"
    assert qmv.last_error() == 0


@pytest.mark.parametrize("bf16", [False, True])
def test_matvec_qx_grouped_two_step_equals_quantize_then_product(qmv, bf16):
    # one problem of 2..8 vectors: the grouped call's two launches are qmv_quantize_x and
    # qmv_matvec_qx's tensor-core mode, so the results are the same bits; a stream captured before
    # its first call (no split buffer yet) takes the dp4a kernel, within the tolerance
    import torch
    rows, cols, batch = 3000, 2048, 6
    m = inputs.make_matrix(2, 1, rows, cols, seed=71)
    x = activations(np.random.default_rng(72), batch, cols)
    xin = inputs.bf16_codes(x) if bf16 else x
    W, xd = dev_u8(m.W), dev_x(xin)
    y1 = torch.empty((batch, rows), device="cuda")
    qmv.matvec_qx_grouped(2, 1, [(rows, cols, W, xd, y1)])
    y2 = qmv.matvec_qx(2, 1, rows, cols, W, qmv.quantize_x(xd), batch)
    torch.cuda.synchronize()
    assert_bits_equal(y1.cpu().numpy(), y2.cpu().numpy(), "grouped two-step against the two calls")
    y3 = torch.empty_like(y1)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        qmv.matvec_qx_grouped(2, 1, [(rows, cols, W, xd, y3)])
    g.replay()
    torch.cuda.synchronize()
    y_ref, absref = oracle_qx(m, x, bf16)
    check_product(y3.cpu().numpy(), y_ref, absref, tol=1e-4, what="captured without a split buffer")
    check_product(y1.cpu().numpy(), y_ref, absref, tol=1e-4, what="two-step")
    assert qmv.last_error() == 0


def test_matvec_qx_grouped_two_step_edge_cases(qmv):
    # two problems reading one activation pointer with different cols (two images of the same
    # memory), and a group whose images exceed the stream's 2 MiB split buffer (the dp4a kernel
    # then quantizes them itself): both against the oracle
    import torch
    rng = np.random.default_rng(160)
    ma = inputs.make_matrix(2, 1, 40, 512, seed=161)
    mb = inputs.make_matrix(2, 1, 24, 256, seed=162)
    batch = 3
    x = activations(rng, batch, 512)
    xd = dev_x(x)
    ya = torch.full((batch, 40), 9.0, device="cuda")
    yb = torch.full((batch, 24), 9.0, device="cuda")
    xd256 = xd.view(-1)[:batch * 256].view(batch, 256)          # the same pointer, 256 columns
    assert xd256.data_ptr() == xd.data_ptr()
    qmv.matvec_qx_grouped(2, 1, [(40, 512, dev_u8(ma.W), xd, ya), (24, 256, dev_u8(mb.W), xd256, yb)])
    torch.cuda.synchronize()
    xb_view = x.reshape(-1)[:batch * 256].reshape(batch, 256)   # the same memory as [batch][256]
    for m, xv, y in ((ma, x, ya), (mb, xb_view, yb)):
        y_ref, absref = oracle_qx(m, xv, False)
        check_product(y.cpu().numpy(), y_ref, absref, tol=1e-4, what=f"shared pointer {m.rows}x{m.cols}")
    # 128 vectors of 16384 columns: 2.36 MB of images
    mc = inputs.make_matrix(1, 0, 16, 16384, seed=163)
    xc = activations(rng, 128, 16384)
    yc = torch.full((128, 16), 9.0, device="cuda")
    qmv.matvec_qx_grouped(1, 0, [(16, 16384, dev_u8(mc.W), dev_x(xc), yc)])
    torch.cuda.synchronize()
    y_ref, absref = oracle_qx(mc, xc, False)
    check_product(yc.cpu().numpy(), y_ref, absref, tol=1e-4, what="images beyond the split buffer")
    assert qmv.last_error() == 0
