"""Compiled steps (qmv_step_create / run / destroy) on the device.

A step copies its inputs from pinned host memory, runs groups of products and copies the
results back; each run must give, bit for bit, what the same calls give eagerly (the step
records the kernels an eager call takes), and agree with the oracle.  Routes covered: one
bf16 vector (block-diagonal kernel), float32 activations of three vectors (split into bf16
pairs, tensor-memory kernel), a prefill batch of 32 (tcgen05 prefill kernel with split tiles).
"""
import numpy as np
import pytest

import oracle
from block_quantized_weight_q4_gb300 import inputs
from helpers import assert_bits_equal, check_product, dev_u8

pytestmark = pytest.mark.gpu


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


def to_dev_x(x):
    import torch
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(x).cuda()


@pytest.mark.parametrize("batch,bf16", [(1, True), (3, False), (32, True)])
def test_step_runs_match_eager_calls_and_oracle(qmv, batch, bf16):
    import torch
    shapes = [(2, 1, 1024, 4096), (2, 1, 3072, 4096), (1, 0, 2048, 4096)]   # (wtype, scale, rows, cols)
    ms = [inputs.make_matrix(wt, sf, r, c, seed=200 + i) for i, (wt, sf, r, c) in enumerate(shapes)]
    Ws = [dev_u8(m.W) for m in ms]
    cols = 4096
    xh = torch.empty((batch, cols), dtype=torch.bfloat16 if bf16 else torch.float32).pin_memory()
    xd = torch.empty_like(xh, device="cuda")
    ys = [torch.empty((batch, r), device="cuda") for (_, _, r, _) in shapes]
    yh = [torch.empty((batch, r)).pin_memory() for (_, _, r, _) in shapes]
    groups = [(2, 1, [(shapes[i][2], cols, Ws[i], xd, ys[i]) for i in (0, 1)], True),
              (1, 0, [(shapes[2][2], cols, Ws[2], xd, ys[2])], False)]
    rng = np.random.default_rng(300 + batch)

    def new_input():
        x = inputs.bf16_codes(rng.standard_normal((batch, cols))) if bf16 else \
            rng.standard_normal((batch, cols)).astype(np.float32)
        if bf16:
            xh.view(torch.int16).copy_(torch.from_numpy(x.view(np.int16)))
        else:
            xh.copy_(torch.from_numpy(x))
        return x

    new_input()
    step = qmv.Step(groups, before=[(xd, xh)], after=list(zip(yh, ys)))
    try:
        for it in range(3):
            x = new_input()
            step.run()
            torch.cuda.current_stream().synchronize()
            got = [y.clone() for y in yh]
            # the same calls, eagerly, on the same device input
            xe = to_dev_x(x)
            ye = [torch.empty_like(y) for y in ys]
            qmv.matvec_grouped(2, 1, [(shapes[i][2], cols, Ws[i], xe, ye[i]) for i in (0, 1)], overlap=True)
            qmv.matvec_grouped(1, 0, [(shapes[2][2], cols, Ws[2], xe, ye[2])])
            torch.cuda.synchronize()
            for i, (wt, sf, r, c) in enumerate(shapes):
                assert_bits_equal(got[i].numpy(), ye[i].cpu().numpy(), f"run {it} problem {i}")
                y_ref, absref = oracle.matvec(ms[i].W, wt, sf, r, c, x)
                check_product(got[i].numpy(), y_ref, absref, what=f"step {it} problem {i}")
        # another stream
        s = torch.cuda.Stream()
        step.run(stream=s)
        s.synchronize()
        for i in range(3):
            assert_bits_equal(yh[i].numpy(), got[i].numpy(), f"other stream problem {i}")
    finally:
        step.close()


def test_step_reports_a_bad_group(qmv):
    import torch
    m = inputs.make_matrix(2, 1, 64, 64, seed=1)
    x = torch.zeros((1, 48), dtype=torch.bfloat16, device="cuda")
    y = torch.empty((1, 64), device="cuda")
    with pytest.raises(qmv.QmvError):
        qmv.Step([(2, 1, [(64, 48, dev_u8(m.W), x, y)], False)])    # cols not a multiple of 32


def test_step_of_copies_only(qmv):
    import torch
    src = torch.arange(4096, dtype=torch.float32).pin_memory()
    mid = torch.empty(4096, device="cuda")
    dst = torch.zeros(4096).pin_memory()
    with qmv.Step([], before=[(mid, src)], after=[(dst, mid)]) as step:
        src.mul_(2.0)
        step.run()
        torch.cuda.current_stream().synchronize()
        assert torch.equal(dst, src)
    with pytest.raises(ValueError):
        step.run()                                   # closed on leaving the block
