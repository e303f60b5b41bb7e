"""Gated activations (the FFN down projection's input act(w1 x) * (w3 x)) on the device.

The product with x_dtype QMV_X_SILU_GLU_F32 / QMV_X_GELU_GLU_F32 must agree with the oracle's
product on act(gate) * up evaluated in double, within the product's tolerance taken against
the exact activations.  Cases: one vector (block-diagonal kernel), 3 and 8 vectors (tensor-memory
kernel), 11 vectors (two passes), a group of problems with different widths (each problem's up
array after its own gate), the Llama-7B FFN as a compiled step (w1 and w3 grouped, then w2 on
their outputs), and the refusals.
"""
import numpy as np
import pytest

import oracle
from block_quantized_weight_q4_gb300 import inputs
from helpers import HALF_TOL, check_product, dev_u8

pytestmark = pytest.mark.gpu

ACTS = [("silu", 0), ("gelu", 1)]


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


def gate_up(rng, batch, cols):
    g = (rng.standard_normal((batch, cols)) * 2).astype(np.float32)
    u = rng.standard_normal((batch, cols)).astype(np.float32)
    return g, u


@pytest.mark.parametrize("act,act_id", ACTS)
@pytest.mark.parametrize("wt,sf", [(1, 0), (1, 1), (2, 0), (2, 1)])
@pytest.mark.parametrize("batch", [1, 3, 8, 11])
def test_glu_product_matches_oracle(qmv, act, act_id, wt, sf, batch):
    import torch
    rows, cols = 300, 2048
    m = inputs.make_matrix(wt, sf, rows, cols, seed=400 + wt + sf)
    rng = np.random.default_rng(401 + batch + act_id)
    g, u = gate_up(rng, batch, cols)
    x = torch.from_numpy(np.stack([g, u])).cuda()             # (2, batch, cols): gate, up
    y = torch.empty((batch, rows), device="cuda")
    qmv.matvec_grouped(wt, sf, [(rows, cols, dev_u8(m.W), x, y)], act=act)
    torch.cuda.synchronize()
    y_ref, absref = oracle.matvec_glu(m.W, wt, sf, rows, cols, act_id, g, u)
    check_product(y.cpu().numpy(), y_ref, absref, what=f"glu {act} {wt},{sf} b{batch}")
    # one vector: the block-diagonal kernel rounds act(gate) * up once to half (2^-11 per term);
    # 2..8 vectors: the tensor-memory kernel keeps 16 bits of them
    tight = HALF_TOL if batch == 1 else 1e-4
    check_product(y.cpu().numpy(), y_ref, absref, tol=tight, what=f"glu tight {act} {wt},{sf} b{batch}")


def test_glu_one_vector_chunk_with_a_wide_range(qmv):
    # one vector: act(gate) * up is rounded to half per 256-column chunk ahead of the product;
    # the chunk holding a value 2^-60 below the rest cannot be rounded (that value would not be
    # a normal half) and keeps hi + lo, the others round: within HALF_TOL of the oracle
    import torch
    rows, cols = 512, 2048
    m = inputs.make_matrix(2, 1, rows, cols, seed=440)
    rng = np.random.default_rng(441)
    g, u = gate_up(rng, 1, cols)
    u[0, 700] = 2.0 ** -60
    x = torch.from_numpy(np.stack([g, u])).cuda()
    y = torch.empty((1, rows), device="cuda")
    qmv.matvec_grouped(2, 1, [(rows, cols, dev_u8(m.W), x, y)], act="silu")
    torch.cuda.synchronize()
    y_ref, absref = oracle.matvec_glu(m.W, 2, 1, rows, cols, 0, g, u)
    check_product(y.cpu().numpy(), y_ref, absref, tol=HALF_TOL, what="glu wide chunk")


@pytest.mark.parametrize("batch", [1, 4])
def test_glu_group_of_different_widths(qmv, batch):
    import torch
    shapes = [(256, 1024), (512, 2048), (128, 4096)]
    ms = [inputs.make_matrix(2, 1, r, c, seed=410 + i) for i, (r, c) in enumerate(shapes)]
    rng = np.random.default_rng(411)
    gus = [gate_up(rng, batch, c) for (_, c) in shapes]
    xs = [torch.from_numpy(np.stack(gu)).cuda() for gu in gus]
    ys = [torch.empty((batch, r), device="cuda") for (r, _) in shapes]
    qmv.matvec_grouped(2, 1, [(r, c, dev_u8(m.W), x, y) for (r, c), m, x, y in zip(shapes, ms, xs, ys)],
                       overlap=True, act="silu")
    torch.cuda.synchronize()
    for (r, c), m, (g, u), y in zip(shapes, ms, gus, ys):
        y_ref, absref = oracle.matvec_glu(m.W, 2, 1, r, c, 0, g, u)
        check_product(y.cpu().numpy(), y_ref, absref, tol=HALF_TOL if batch == 1 else 1e-4,
                      what=f"group {r}x{c} b{batch}")


def test_llama7b_ffn_as_compiled_step(qmv):
    # w1 and w3 (11008 x 4096) on bf16 x, grouped, write gate and up into one (2, 1, 11008)
    # buffer; w2 (4096 x 11008) takes SiLU(gate) * up from it; y comes back to pinned host
    import torch
    dim, hidden = 4096, 11008
    w1, w3 = (inputs.make_matrix(2, 1, hidden, dim, seed=s) for s in (420, 421))
    w2 = inputs.make_matrix(2, 1, dim, hidden, seed=422)
    W1, W3, W2 = dev_u8(w1.W), dev_u8(w3.W), dev_u8(w2.W)
    xh = torch.empty((1, dim), dtype=torch.bfloat16).pin_memory()
    xd = torch.empty_like(xh, device="cuda")
    gu = torch.empty((2, 1, hidden), device="cuda")
    y = torch.empty((1, dim), device="cuda")
    yh = torch.empty((1, dim)).pin_memory()
    groups = [(2, 1, [(hidden, dim, W1, xd, gu[0]), (hidden, dim, W3, xd, gu[1])], True),
              (2, 1, [(dim, hidden, W2, gu, y)], True, "silu")]
    rng = np.random.default_rng(423)
    xh.view(torch.int16).copy_(torch.from_numpy(inputs.bf16_codes(rng.standard_normal((1, dim))).view(np.int16)))
    step = qmv.Step(groups, before=[(xd, xh)], after=[(yh, y)])
    try:
        for _ in range(2):
            xh.view(torch.int16).copy_(
                torch.from_numpy(inputs.bf16_codes(rng.standard_normal((1, dim))).view(np.int16)))
            step.run()
            torch.cuda.current_stream().synchronize()
            g = gu[0].cpu().numpy()
            u = gu[1].cpu().numpy()
            y_ref, absref = oracle.matvec_glu(w2.W, 2, 1, dim, hidden, 0, g, u)
            check_product(yh.numpy(), y_ref, absref, tol=HALF_TOL, what="ffn step")
    finally:
        step.close()


def test_glu_refusals(qmv):
    import torch
    m = inputs.make_matrix(2, 1, 64, 96, seed=1)
    x = torch.zeros((2, 1, 96), device="cuda")
    y = torch.empty((1, 64), device="cuda")
    with pytest.raises(qmv.QmvError):        # cols % 256 != 0
        qmv.matvec_grouped(2, 1, [(64, 96, dev_u8(m.W), x, y)], act="silu")
    with pytest.raises(ValueError):          # x not (2, batch, cols)
        qmv.matvec_grouped(2, 1, [(64, 96, dev_u8(m.W), x[0], y)], act="gelu")


# ------------------------------------------------------- fused gate/up epilogue (qmv_matvec_glu)
# |act'| <= 1.1 for SiLU and <= 1.13 for GELU-tanh; 1.2 bounds both
ACT_LIPSCHITZ = 1.2


def _pair_values(h):
    """float64 hi + lo of a bfloat16 (2, rows) pair tensor."""
    import torch
    codes = h.view(torch.int16).cpu().numpy().view(np.uint16).astype(np.uint32)
    v = (codes << 16).view(np.float32).astype(np.float64)
    return v[0] + v[1], v


def _check_h(h_gpu, gate, G, up, U, act_id, what):
    # gate and up each meet the product bar (1e-3 of their sum |w x|); act changes by at most
    # ACT_LIPSCHITZ times a change of its argument; the float32 evaluation and the hi + lo pair
    # add a few parts in 2^17 of |h|
    h_ref = oracle.glu(act_id, gate, up)
    ag = np.abs(oracle.glu(act_id, gate, np.ones_like(gate)))
    dg, du = 1e-3 * G, 1e-3 * U
    bound = ACT_LIPSCHITZ * dg * (np.abs(up) + du) + ag * du + 2.0 ** -15 * np.abs(h_ref)
    err = np.abs(h_gpu - h_ref)
    assert np.all(err <= bound), f"{what}: {np.count_nonzero(err > bound)} values of h out of bound"
    return h_ref


@pytest.mark.parametrize("act,act_id", ACTS)
@pytest.mark.parametrize("sf", [0, 1])
@pytest.mark.parametrize("rows,cols", [(300, 2048), (64, 256), (1000, 4096)])
def test_fused_glu_matches_oracle(qmv, act, act_id, sf, rows, cols):
    import torch
    from helpers import dev_x
    m1 = inputs.make_matrix(2, sf, rows, cols, seed=500 + rows + sf)
    m3 = inputs.make_matrix(2, sf, rows, cols, seed=501 + rows + sf)
    x = inputs.make_x(1, cols, True, seed=502 + act_id)
    h = qmv.matvec_glu(2, sf, rows, cols, dev_u8(m1.W), dev_u8(m3.W), dev_x(x)[0], act=act)
    torch.cuda.synchronize()
    h_gpu, parts = _pair_values(h)
    gate, G = oracle.matvec(m1.W, 2, sf, rows, cols, x)
    up, U = oracle.matvec(m3.W, 2, sf, rows, cols, x)
    _check_h(h_gpu, gate[0], G[0], up[0], U[0], act_id, f"fused {act} {sf} {rows}x{cols}")
    # lo is the rounding of h - hi: at most half a bfloat16 ulp of hi
    hi, lo = parts
    assert np.all(np.abs(lo) <= np.abs(hi) * 2.0 ** -8)


@pytest.mark.parametrize("act,act_id", ACTS)
def test_fused_glu_then_down_projection(qmv, act, act_id):
    # the down projection reads the pair directly (x_dtype QMV_X_BF16_PAIR): against the oracle
    # on the pair's values hi + lo (exact in float32), within the product's tolerance and within
    # the one half rounding of each stage (HALF_TOL)
    import torch
    from helpers import dev_x
    dim, hidden = 1024, 2816
    m1 = inputs.make_matrix(2, 1, hidden, dim, seed=510)
    m3 = inputs.make_matrix(2, 1, hidden, dim, seed=511)
    m2 = inputs.make_matrix(2, 1, dim, hidden, seed=512)
    x = inputs.make_x(1, dim, True, seed=513)
    h = qmv.matvec_glu(2, 1, hidden, dim, dev_u8(m1.W), dev_u8(m3.W), dev_x(x)[0], act=act)
    y = torch.empty((1, dim), device="cuda")
    qmv.matvec_grouped(2, 1, [(dim, hidden, dev_u8(m2.W), h, y)], pair=True)
    torch.cuda.synchronize()
    h_gpu, _ = _pair_values(h)
    y_ref, absref = oracle.matvec(m2.W, 2, 1, dim, hidden, h_gpu.astype(np.float32)[None, :])
    check_product(y.cpu().numpy(), y_ref, absref, what=f"down projection on the pair ({act})")
    check_product(y.cpu().numpy(), y_ref, absref, tol=HALF_TOL, what=f"down projection tight ({act})")


def test_pair_route_equals_float32_route_bits(qmv):
    # a float32 vector x = hi + lo (hi, lo bfloat16, |lo| <= ulp(hi)/2) splits back into the same
    # hi and lo, so the float32 route (split kernel + the same product) and the pair route give
    # the same bits
    import torch
    from helpers import assert_bits_equal
    rows, cols = 512, 1024
    m = inputs.make_matrix(2, 1, rows, cols, seed=520)
    rng = np.random.default_rng(521)
    v = rng.standard_normal(cols).astype(np.float32)
    hi = inputs.bf16_codes(v)
    lo = inputs.bf16_codes(v - (hi.astype(np.uint32) << 16).view(np.float32))
    pair = torch.from_numpy(np.stack([hi, lo]).view(np.int16)).cuda().view(torch.bfloat16)
    xf = ((hi.astype(np.uint32) << 16).view(np.float32) + (lo.astype(np.uint32) << 16).view(np.float32))
    W = dev_u8(m.W)
    y1 = torch.empty((1, rows), device="cuda")
    y2 = torch.empty((1, rows), device="cuda")
    qmv.matvec_grouped(2, 1, [(rows, cols, W, pair, y1)], pair=True)
    qmv.matvec_grouped(2, 1, [(rows, cols, W, torch.from_numpy(xf[None, :]).cuda(), y2)])
    torch.cuda.synchronize()
    assert_bits_equal(y1.cpu().numpy(), y2.cpu().numpy(), "pair route vs float32 route")
    y_ref, absref = oracle.matvec(m.W, 2, 1, rows, cols, xf[None, :])
    check_product(y1.cpu().numpy(), y_ref, absref, what="pair route")


@pytest.mark.parametrize("act,act_id", ACTS)
def test_fused_glu_full_size_llama7b(qmv, act, act_id):
    # the Llama-7B FFN's w1 / w3 (11008 x 4096), every row against the oracle; the unfused path
    # (grouped {w1, w3} into float32 gate and up, h formed from them) is held to the same bound
    import torch
    from helpers import dev_x
    rows, cols = 11008, 4096
    m1 = inputs.make_matrix(2, 1, rows, cols, seed=530)
    m3 = inputs.make_matrix(2, 1, rows, cols, seed=531)
    x = inputs.make_x(1, cols, True, seed=532)
    W1, W3, xd = dev_u8(m1.W), dev_u8(m3.W), dev_x(x)
    h = qmv.matvec_glu(2, 1, rows, cols, W1, W3, xd[0], act=act)
    gu = torch.empty((2, 1, rows), device="cuda")
    qmv.matvec_grouped(2, 1, [(rows, cols, W1, xd, gu[0]), (rows, cols, W3, xd, gu[1])])
    torch.cuda.synchronize()
    h_gpu, _ = _pair_values(h)
    gate, G = oracle.matvec(m1.W, 2, 1, rows, cols, x)
    up, U = oracle.matvec(m3.W, 2, 1, rows, cols, x)
    _check_h(h_gpu, gate[0], G[0], up[0], U[0], act_id, f"full-size fused {act}")
    g, u = gu[0, 0].cpu().numpy().astype(np.float64), gu[1, 0].cpu().numpy().astype(np.float64)
    _check_h(oracle.glu(act_id, g, u), gate[0], G[0], up[0], U[0], act_id, f"full-size unfused {act}")
    assert qmv.last_error() == 0
