"""qmv_matvec_grouped_noalloc: the tensor-memory decode product with its scratch in a
fixed array inside the library, against the existing qmv_matvec_grouped and the oracle,
over two consecutive calls (the first call on a device does its one-time setup; the
second shows that the arrival counters were left, or set, back at zero).  Collected last so
that it also runs after every other GPU test in one process."""
import numpy as np
import pytest

import oracle
from block_quantized_weight_q4_gb300 import inputs
from helpers import assert_bits_equal, check_product, dev_u8, dev_x

pytestmark = pytest.mark.gpu

TOL = 1e-3


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


def _problems(wt, sf, shapes, batch, seed):
    import torch
    mats, probs = [], []
    for i, (rows, cols) in enumerate(shapes):
        m = inputs.make_matrix(wt, sf, rows, cols, seed=seed + i)
        x = inputs.make_x(batch, cols, True, seed=seed + 50 + i)
        mats.append((m, x))
        probs.append((rows, cols, dev_u8(m.W), dev_x(x), torch.full((batch, rows), 5.0, device="cuda")))
    return mats, probs


@pytest.mark.parametrize("wt,sf", [(2, 1), (1, 0)])
@pytest.mark.parametrize("batch", [1, 8])
def test_noalloc_matches_grouped_and_oracle(qmv, wt, sf, batch):
    import torch
    shapes = [(4096, 4096), (1000, 2048), (300, 256)]
    mats, probs = _problems(wt, sf, shapes, batch, seed=300 + 10 * wt + batch)
    refs = [oracle.matvec(m.W, wt, sf, p[0], p[1], x) for (m, x), p in zip(mats, probs)]
    # the existing entry point, twice
    qmv.matvec_grouped(wt, sf, probs)
    qmv.matvec_grouped(wt, sf, probs)
    torch.cuda.synchronize()
    base = [p[4].cpu().numpy().copy() for p in probs]
    # the allocation-free one, twice, on a stream no other entry point has used (so that no
    # per-stream workspace exists that it could have fallen back on)
    s = torch.cuda.Stream()
    outs = []
    for _ in range(2):
        for p in probs:
            p[4].fill_(5.0)
        torch.cuda.synchronize()
        qmv.matvec_grouped_noalloc(wt, sf, probs, stream=s)
        torch.cuda.synchronize()
        outs.append([p[4].cpu().numpy().copy() for p in probs])
    for k, (p, (y_ref, absref)) in enumerate(zip(probs, refs)):
        what = f"noalloc {wt},{sf} {p[0]}x{p[1]} b{batch}"
        check_product(outs[0][k], y_ref, absref, TOL, what)
        assert_bits_equal(outs[1][k], outs[0][k], what + " second call")
        # (the existing entry point takes the mma.sync kernel at this size: other sums)
        check_product(base[k], y_ref, absref, TOL, what + " (existing entry point)")


@pytest.mark.parametrize("batch", [8])
def test_noalloc_same_bits_as_grouped_at_tensor_memory_sizes(qmv, batch):
    # 142 MB of Q8_0 weights, 8 vectors: qmv_matvec_grouped takes the tensor-memory kernel too,
    # with the same grid and the same splits, so the two give the same bits (sampled rows
    # against the oracle)
    import torch
    wt, sf, rows, cols = 1, 0, 122880, 1024
    assert rows * cols // 32 * 36 >= 128 << 20
    mats, probs = _problems(wt, sf, [(rows, cols)], batch, seed=350 + batch)
    (m, x), = mats
    qmv.matvec_grouped(wt, sf, probs)
    torch.cuda.synchronize()
    base = probs[0][4].cpu().numpy().copy()
    probs[0][4].fill_(5.0)
    qmv.matvec_grouped_noalloc(wt, sf, probs, stream=torch.cuda.Stream())
    torch.cuda.synchronize()
    out = probs[0][4].cpu().numpy()
    ids = np.unique(np.random.default_rng(351).integers(0, rows, 128))
    y_ref, absref = oracle.matvec_rows(m.W, wt, sf, rows, cols, x, ids)
    check_product(out[:, ids], y_ref, absref, TOL, f"noalloc large b{batch}")
    assert_bits_equal(out, base, f"noalloc large b{batch} vs existing")


def test_noalloc_takes_no_device_memory_after_first_call(qmv):
    # after one call on the device (the library's device code and the scratch array are set up
    # lazily), further calls on a new stream leave the free device memory unchanged, with and
    # without the overlap flag, and match the oracle
    import torch
    wt, sf, batch = 2, 1, 8
    shapes = [(2048, 4096), (512, 1024)]
    mats, probs = _problems(wt, sf, shapes, batch, seed=400)
    refs = [oracle.matvec(m.W, wt, sf, p[0], p[1], x) for (m, x), p in zip(mats, probs)]
    s = torch.cuda.Stream()
    qmv.matvec_grouped_noalloc(wt, sf, probs, stream=s)  # warm-up
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for overlap in (False, True, False, True):
        qmv.matvec_grouped_noalloc(wt, sf, probs, overlap=overlap, stream=s)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0, "device memory taken by the allocation-free calls"
    for p, (y_ref, absref) in zip(probs, refs):
        check_product(p[4].cpu().numpy(), y_ref, absref, TOL, f"noalloc overlap {p[0]}x{p[1]}")
    assert qmv.last_error() == 0


def test_noalloc_rejects_what_it_cannot_run(qmv):
    import torch
    lib = qmv.load_library()
    m = inputs.make_matrix(2, 1, 256, 512, seed=1)
    W = dev_u8(m.W)
    xb = dev_x(inputs.make_x(9, 512, True, seed=1))
    y = torch.zeros((9, 256), device="cuda")
    # more vectors than the scratch holds
    with pytest.raises(RuntimeError, match="invalid argument"):
        qmv.matvec_grouped_noalloc(2, 1, [(256, 512, W, xb, y)])
    # float32 activations
    xf = dev_x(inputs.make_x(2, 512, False, seed=1))
    with pytest.raises(RuntimeError, match="format"):
        qmv.matvec_grouped_noalloc(2, 1, [(256, 512, W, xf, y[:2])])
    # columns the tensor-memory kernel does not take (a multiple of 32, not of 256)
    m2 = inputs.make_matrix(2, 1, 64, 288, seed=2)
    W2 = dev_u8(m2.W)
    x2 = dev_x(inputs.make_x(1, 288, True, seed=2))
    with pytest.raises(RuntimeError, match="shape"):
        qmv.matvec_grouped_noalloc(2, 1, [(64, 288, W2, x2, torch.zeros((1, 64), device="cuda"))])
    assert lib.qmv_check_device() == 0
