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
from block_quantized_weight_q4_gb300 import binding, inputs
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
        # a run and its wait in one call
        for y in yh:
            y.zero_()
        step.run(stream=s, wait=True)
        for i in range(3):
            assert_bits_equal(yh[i].numpy(), got[i].numpy(), f"run and wait problem {i}")
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


def test_step_with_per_group_copies_and_a_chained_group(qmv):
    # per-group copies, as a decode step hands each group its input and takes each result back:
    # x0 and x2 come from the host, group 1 reads group 0's result y0 as float32 activations,
    # and y0, y2, y1 go back to the host; every run must give the bits of the same calls made
    # eagerly in order
    import torch
    cols = 4096
    m0 = inputs.make_matrix(2, 1, 4096, cols, seed=230)
    m1 = inputs.make_matrix(2, 1, 1024, 4096, seed=231)
    m2 = inputs.make_matrix(1, 1, 2048, cols, seed=232)
    W0, W1, W2 = dev_u8(m0.W), dev_u8(m1.W), dev_u8(m2.W)
    x0h = torch.empty((1, cols), dtype=torch.bfloat16).pin_memory()
    x2h = torch.empty((1, cols), dtype=torch.bfloat16).pin_memory()
    x0d, x2d = torch.empty_like(x0h, device="cuda"), torch.empty_like(x2h, device="cuda")
    y0 = torch.empty((1, 4096), device="cuda")
    y1 = torch.empty((1, 1024), device="cuda")
    y2 = torch.empty((1, 2048), device="cuda")
    y0h, y1h, y2h = (torch.empty(t.shape).pin_memory() for t in (y0, y1, y2))
    groups = [(2, 1, [(4096, cols, W0, x0d, y0)], True),
              (2, 1, [(1024, 4096, W1, y0, y1)], True),
              (1, 1, [(2048, cols, W2, x2d, y2)], True)]
    rng = np.random.default_rng(233)

    def new_inputs():
        xs = [inputs.bf16_codes(rng.standard_normal((1, cols))) for _ in range(2)]
        for h, x in zip((x0h, x2h), xs):
            h.view(torch.int16).copy_(torch.from_numpy(x.view(np.int16)))
        return xs

    new_inputs()
    step = qmv.Step(groups, before=[(x0d, x0h), (x2d, x2h)], after=[(y0h, y0), (y2h, y2), (y1h, y1)])
    try:
        for it in range(4):
            x0, x2 = new_inputs()
            step.run()
            torch.cuda.current_stream().synchronize()
            got = [t.clone().numpy() for t in (y0h, y1h, y2h)]
            e0 = torch.empty_like(y0)
            e1 = torch.empty_like(y1)
            e2 = torch.empty_like(y2)
            qmv.matvec_grouped(2, 1, [(4096, cols, W0, to_dev_x(x0), e0)], overlap=True)
            qmv.matvec_grouped(2, 1, [(1024, 4096, W1, e0, e1)], overlap=True)
            qmv.matvec_grouped(1, 1, [(2048, cols, W2, to_dev_x(x2), e2)], overlap=True)
            torch.cuda.synchronize()
            for g, e, what in zip(got, (e0, e1, e2), ("y0", "y1", "y2")):
                assert_bits_equal(g, e.cpu().numpy(), f"run {it} {what}")
            y_ref, absref = oracle.matvec(m0.W, 2, 1, 4096, cols, x0)
            check_product(got[0], y_ref, absref, what=f"run {it} y0")
            y_ref, absref = oracle.matvec(m1.W, 2, 1, 1024, 4096, got[0].astype(np.float32))
            check_product(got[1], y_ref, absref, what=f"run {it} y1")
    finally:
        step.close()


@pytest.mark.parametrize("nbytes,offset", [(1001, 3), (4096, 16), (65536 + 8, 8)])
def test_step_copies_of_any_size_and_offset(qmv, nbytes, offset):
    # host <-> device copies of a step (done by the GPU through the host memory's device address
    # when both ends allow it): any byte count and alignment, the exact bytes both ways
    import torch
    src = torch.randint(0, 256, (nbytes + 64,), dtype=torch.uint8).pin_memory()
    mid = torch.zeros(nbytes + 64, dtype=torch.uint8, device="cuda")
    dst = torch.zeros(nbytes + 64, dtype=torch.uint8).pin_memory()
    a, b = offset, offset + nbytes
    with qmv.Step([], before=[(mid[a:b], src[a:b])], after=[(dst[a:b], mid[a:b])]) as step:
        for _ in range(2):
            src.random_(0, 256)
            step.run(wait=True)
            assert torch.equal(dst[a:b], src[a:b])
            assert torch.equal(mid[a:b].cpu(), src[a:b])
            assert int(dst[:a].sum()) == 0 and int(dst[b:].sum()) == 0   # nothing outside the range


@pytest.mark.parametrize("batch,bf16", [(1, True), (3, False), (32, True)])
def test_products_store_y_into_pinned_host_memory(qmv, batch, bf16):
    # y in pinned host memory that the device addresses directly: the kernels' stores go there;
    # eager calls and a compiled step without a copy back give the bits of device-memory y
    import torch
    shapes = [(2, 1, 1024, 4096), (2, 1, 3072, 4096)]
    ms = [inputs.make_matrix(wt, sf, r, c, seed=240 + i) for i, (wt, sf, r, c) in enumerate(shapes)]
    Ws = [dev_u8(m.W) for m in ms]
    rng = np.random.default_rng(250 + batch)
    x = inputs.bf16_codes(rng.standard_normal((batch, 4096))) if bf16 else \
        rng.standard_normal((batch, 4096)).astype(np.float32)
    xd = to_dev_x(x)
    yd = [torch.empty((batch, r), device="cuda") for (_, _, r, _) in shapes]
    yh = [torch.full((batch, r), 7.0).pin_memory() for (_, _, r, _) in shapes]
    qmv.matvec_grouped(2, 1, [(r, 4096, Ws[i], xd, yd[i]) for i, (_, _, r, _) in enumerate(shapes)])
    qmv.matvec_grouped(2, 1, [(r, 4096, Ws[i], xd, yh[i]) for i, (_, _, r, _) in enumerate(shapes)], overlap=True)
    torch.cuda.synchronize()
    for i in range(2):
        assert_bits_equal(yh[i].numpy(), yd[i].cpu().numpy(), f"eager, problem {i}")
        y_ref, absref = oracle.matvec(ms[i].W, 2, 1, shapes[i][2], 4096, x)
        check_product(yh[i].numpy(), y_ref, absref, what=f"host y, problem {i}")
    xh = torch.from_numpy(x.view(np.int16) if bf16 else x).pin_memory()
    xs = torch.empty_like(xh, device="cuda")
    xsv = xs.view(torch.bfloat16) if bf16 else xs
    for y in yh:
        y.fill_(7.0)
    with qmv.Step([(2, 1, [(r, 4096, Ws[i], xsv, yh[i]) for i, (_, _, r, _) in enumerate(shapes)], True)],
                  before=[(xs, xh)]) as step:
        step.run(wait=True)
        for i in range(2):
            assert_bits_equal(yh[i].numpy(), yd[i].cpu().numpy(), f"step, problem {i}")


def test_gated_step_pipelined_runs_match_eager_calls(qmv):
    # a gated step as a decode loop drives it: the next run is enqueued while the current one
    # computes and opened only after the host has the current result and has written the next
    # input; every run's y (stored by the products into pinned host memory) must equal the
    # eager calls' bits for that input
    import torch
    shapes = [(2, 1, 4096, 4096), (2, 1, 1024, 4096)]
    ms = [inputs.make_matrix(wt, sf, r, c, seed=260 + i) for i, (wt, sf, r, c) in enumerate(shapes)]
    Ws = [dev_u8(m.W) for m in ms]
    xh = torch.empty((1, 4096), dtype=torch.bfloat16).pin_memory()
    xd = torch.empty_like(xh, device="cuda")
    yh = [torch.empty((1, r)).pin_memory() for (_, _, r, _) in shapes]
    groups = [(2, 1, [(shapes[0][2], 4096, Ws[0], xd, yh[0])], True),
              (2, 1, [(shapes[1][2], 4096, Ws[1], xd, yh[1])], True)]
    rng = np.random.default_rng(270)
    xs = [inputs.bf16_codes(rng.standard_normal((1, 4096))) for _ in range(5)]

    def put(x):
        xh.view(torch.int16).copy_(torch.from_numpy(x.view(np.int16)))

    put(xs[0])
    expect = []
    for x in xs:
        xe = to_dev_x(x)
        ye = [torch.empty((1, r), device="cuda") for (_, _, r, _) in shapes]
        for i, (_, _, r, _) in enumerate(shapes):
            qmv.matvec_grouped(2, 1, [(r, 4096, Ws[i], xe, ye[i])], overlap=True)
        torch.cuda.synchronize()
        expect.append([y.cpu().numpy() for y in ye])
    s = torch.cuda.Stream()
    with qmv.Step(groups, before=[(xd, xh)], gated=True) as step:
        step.run(stream=s)
        for it, x in enumerate(xs):
            put(x)
            step.open()
            if it + 1 < len(xs):
                step.run(stream=s)       # the next run waits at its gate
            step.wait()
            for i in range(2):
                assert_bits_equal(yh[i].numpy(), expect[it][i], f"gated run {it}, problem {i}")
        # the one-call forms: a run, its opening and the wait; the opening, the next run and the wait
        put(xs[2])
        step.run(stream=s, wait=True)
        for i in range(2):
            assert_bits_equal(yh[i].numpy(), expect[2][i], f"gated run_wait, problem {i}")
        step.run(stream=s)
        for it in (3, 4):
            put(xs[it])
            step.open_wait(step if it == 3 else None, stream=s)
            for i in range(2):
                assert_bits_equal(yh[i].numpy(), expect[it][i], f"gated open_wait {it}, problem {i}")
    y_ref, absref = oracle.matvec(ms[1].W, 2, 1, 1024, 4096, xs[4])   # the last run's input
    check_product(yh[1].numpy(), y_ref, absref, what="gated step against the oracle")


def test_gated_step_waits_and_reports(qmv):
    # the host's wait is bounded: an opened run still queued behind other work makes it run out
    # (QMV_E_TIMEOUT), and a later wait sees the run done; a run never opened holds its stream
    # until its gate's one-second bound, which the status word reports
    import torch
    m = inputs.make_matrix(2, 1, 256, 512, seed=280)
    W = dev_u8(m.W)
    xh = torch.zeros((1, 512), dtype=torch.bfloat16).pin_memory()
    xd = torch.empty_like(xh, device="cuda")
    yh = torch.full((1, 256), 5.0).pin_memory()
    s = torch.cuda.Stream()
    step = qmv.Step([(2, 1, [(256, 512, W, xd, yh)], False)], before=[(xd, xh)], gated=True)
    try:
        with pytest.raises(qmv.QmvError) as e:
            step.open()                      # no run enqueued
        assert e.value.status == binding.E_ARG
        with torch.cuda.stream(s):
            torch.cuda._sleep(50_000_000)    # tens of milliseconds of other work ahead of the run
        step.run(stream=s)
        step.open()
        with pytest.raises(qmv.QmvError) as e:
            step.wait(timeout_us=2000)
        assert e.value.status == binding.E_TIMEOUT
        step.wait()
        assert float(yh.abs().max()) == 0.0  # x = 0 gives y = 0
        assert qmv.last_error() == 0
        step.run(stream=s)
        assert not s.query()                 # held at the gate
        step.run(stream=s)                   # never opened
        s.synchronize()                      # returns after the gate's bound
        assert qmv.last_error() == binding.E_TIMEOUT
    finally:
        step.close()
    assert qmv.last_error() == 0


def test_gated_step_with_after_copies_and_without_before_copies(qmv):
    # a gated step whose results go back through `after` copies (the done kernel then follows the
    # copy), one with no `before` copies (the input already on the device: the gate only waits),
    # and the refusal of a `before` copy that is not pinned host -> device memory
    import torch
    m = inputs.make_matrix(2, 1, 512, 1024, seed=290)
    W = dev_u8(m.W)
    rng = np.random.default_rng(291)
    x = inputs.bf16_codes(rng.standard_normal((1, 1024)))
    xh = torch.from_numpy(x.view(np.int16)).pin_memory()
    xd = torch.empty_like(xh, device="cuda")
    yd = torch.empty((1, 512), device="cuda")
    yh = torch.zeros((1, 512)).pin_memory()
    xe = to_dev_x(x)
    ye = torch.empty((1, 512), device="cuda")
    qmv.matvec_grouped(2, 1, [(512, 1024, W, xe, ye)], overlap=True)
    torch.cuda.synchronize()
    want = ye.cpu().numpy()
    xdb = xd.view(torch.bfloat16)
    with qmv.Step([(2, 1, [(512, 1024, W, xdb, yd)], True)], before=[(xd, xh)], after=[(yh, yd)],
                  gated=True) as step:
        for _ in range(2):
            yh.zero_()
            step.run(wait=True)
            assert_bits_equal(yh.numpy(), want, "gated step with an after copy")
    xdb.copy_(xe)
    yd.zero_()
    with qmv.Step([(2, 1, [(512, 1024, W, xdb, yd)], True)], gated=True) as step:
        step.run(wait=True)
        assert_bits_equal(yd.cpu().numpy(), want, "gated step without before copies")
    with pytest.raises(qmv.QmvError) as e:
        qmv.Step([(2, 1, [(512, 1024, W, xdb, yd)], True)], before=[(xd, xe.view(torch.int16))], gated=True)
    assert e.value.status == binding.E_ARG
    assert qmv.last_error() == 0
