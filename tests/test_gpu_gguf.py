"""GGUF interleaved blocks on the device (qmv_gguf_to_mlb) vs the oracle, byte for byte.

Random records (any f16 code as d, any quant bytes) over shapes whose record counts fill
whole 32-record chunks, leave a partial last chunk, or hold a single record; the page's own
tensor shape (151,936 x 896, Q8_0 and Q4_0) at full size; and a product on the converted
image against the oracle's product on the oracle's conversion.
"""
import numpy as np
import pytest

import oracle
from helpers import check_product, dev_u8, dev_x

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


def random_gguf(rng, wt, rows, cols, finite_scales=True):
    n = oracle.gguf_bytes(wt, rows, cols)
    g = rng.integers(0, 256, n, dtype=np.int16).astype(np.uint8)
    if finite_scales:
        # d codes of moderate finite halves (products stay well inside float32)
        bs = 34 if wt == 1 else 18
        recs = g.reshape(-1, bs)
        d = rng.uniform(-0.05, 0.05, recs.shape[0]).astype(np.float16).view(np.uint16)
        recs[:, 0] = (d & 0xFF).astype(np.uint8)
        recs[:, 1] = (d >> 8).astype(np.uint8)
    return g


def gpu_convert(q, wt, rows, cols, g, fill=0xAB):
    import torch
    W = torch.full((q.weight_bytes(wt, 1, rows, cols),), fill, dtype=torch.uint8, device="cuda")
    q.gguf_to_mlb(wt, rows, cols, dev_u8(g), W=W)
    torch.cuda.synchronize()
    return W.cpu().numpy()


@pytest.mark.parametrize("wt", [1, 2])
@pytest.mark.parametrize("rows,cols", [(1, 32), (3, 96), (33, 1024), (7, 4128), (64, 4096), (5, 11008)])
def test_gguf_to_mlb_matches_oracle(qmv, wt, rows, cols):
    rng = np.random.default_rng(rows * 13 + cols + wt)
    g = random_gguf(rng, wt, rows, cols, finite_scales=False)   # every byte pattern, NaN codes included
    got = gpu_convert(qmv, wt, rows, cols, g)
    want = oracle.gguf_to_mlb(g, wt, rows, cols)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, f"{bad.size} bytes differ, first at {bad[:8]}"


@pytest.mark.parametrize("wt", [1, 2])
def test_gguf_to_mlb_page_tensor_full_size(qmv, wt):
    # output.weight (Q8_0) and token_embd.weight (Q4_0) of the page's model: 151,936 x 896
    rows, cols = 151936, 896
    rng = np.random.default_rng(90 + wt)
    g = random_gguf(rng, wt, rows, cols)
    assert g.size == (144643072 if wt == 1 else 76575744)
    got = gpu_convert(qmv, wt, rows, cols, g)
    want = oracle.gguf_to_mlb(g, wt, rows, cols)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("wt", [1, 2])
def test_product_on_converted_gguf(qmv, wt):
    # the converted image feeds the product kernels: y = W x against the oracle's product on
    # the oracle's conversion (bf16 activations, batch 1 and 3)
    import torch
    rows, cols = 2048, 4096
    rng = np.random.default_rng(95 + wt)
    g = random_gguf(rng, wt, rows, cols)
    W = qmv.gguf_to_mlb(wt, rows, cols, dev_u8(g))
    Wh = oracle.gguf_to_mlb(g, wt, rows, cols)
    for batch in (1, 3):
        x = rng.standard_normal((batch, cols)).astype(np.float32)
        y = qmv.matvec(wt, 1, rows, cols, W, dev_x(x))
        torch.cuda.synchronize()
        y_ref, absref = oracle.matvec(Wh, wt, 1, rows, cols, x)
        check_product(y.cpu().numpy(), y_ref, absref, what=f"gguf product {wt} b{batch}")
