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
from helpers import check_product, dev_u8

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
    check_product(y.cpu().numpy(), y_ref, absref, tol=1e-4, what=f"glu tight {act} {wt},{sf} b{batch}")


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
        check_product(y.cpu().numpy(), y_ref, absref, tol=1e-4, what=f"group {r}x{c} b{batch}")


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
            check_product(yh.numpy(), y_ref, absref, tol=1e-4, what="ffn step")
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
