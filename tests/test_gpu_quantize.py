"""The device writer rules (qmv_quantize) vs the oracle's writer, byte for byte.

The oracle's writer (oracle_quantize) evaluates the page's Q8_0 rule and the Q4_0 "round"
rule one float32 operation at a time; the device must produce the same bytes: the same
quants, the same scale bits, zeros in the padding.  Cases: workload-like data over shapes
whose block counts are not multiples of the four blocks a warp takes; blocks that probe
each step of the rules (all zero, below the 1e-30 amax floor, ties of magnitude for the
Q4_0 pivot, halves that round away from zero, scales that are f16 subnormals or round to
f16 zero, clamping); refused blocks (an f16 scale beyond the f16 range); a full-size
matrix of the prefill workload.
"""
import numpy as np
import pytest

import oracle
from helpers import dev_x

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


def gpu_quantize(q, wt, sf, src):
    import torch
    W, first = q.quantize(wt, sf, dev_x(np.ascontiguousarray(src, dtype=np.float32)))
    torch.cuda.synchronize()
    return W.cpu().numpy(), first


def assert_bytes_equal(got, want, what):
    assert got.shape == want.shape, what
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, f"{what}: {bad.size} bytes differ, first at {bad[:8]}"


def workload_like(rng, rows, cols):
    # N(0, 1) rows with a per-block magnitude spread over four decades, as trained weights
    x = rng.standard_normal((rows, cols)).astype(np.float32)
    s = np.exp(rng.uniform(-6, 3, size=(rows, cols // 32))).astype(np.float32)
    return (x.reshape(rows, -1, 32) * s[:, :, None]).reshape(rows, cols)


@pytest.mark.parametrize("wt,sf", TYPES)
@pytest.mark.parametrize("rows,cols", [(1, 32), (3, 96), (7, 64), (33, 256), (100, 4096), (5, 11008)])
def test_quantize_matches_oracle(qmv, wt, sf, rows, cols):
    rng = np.random.default_rng(rows * 7 + cols + wt + sf)
    src = workload_like(rng, rows, cols)
    W, first = gpu_quantize(qmv, wt, sf, src)
    assert first == -1
    assert_bytes_equal(W, oracle.quantize(src, wt, sf), f"{wt},{sf} {rows}x{cols}")


def special_blocks(rng):
    """Blocks that probe the rules' steps (each row of 32 is one block)."""
    blocks = []
    blocks.append(np.zeros(32))                                   # all zero (d = 0 / -0)
    blocks.append(np.full(32, -0.0))                              # negative zeros
    blocks.append(rng.standard_normal(32) * 1e-31)                # amax below the 1e-30 floor
    b = np.zeros(32); b[5] = 1e-30; blocks.append(b)              # amax exactly at the floor
    b = rng.integers(-4, 5, 32).astype(float); b[3] = 7; b[20] = -7; blocks.append(b)   # tie: first index
    b = rng.integers(-4, 5, 32).astype(float); b[9] = -6; b[2] = 6; blocks.append(b)    # tie, other sign
    b = np.arange(-16, 16, dtype=float) + 0.5; blocks.append(b)   # halves: round away from zero (Q8)
    b = np.linspace(-127, 127, 32); blocks.append(b)              # Q8 levels at the ends
    b = np.linspace(-8, 7, 32); blocks.append(b)                  # Q4 levels over the whole range
    b = rng.standard_normal(32) * 1e-6; blocks.append(b)          # f16 scale subnormal
    b = rng.standard_normal(32) * 1e-9; blocks.append(b)          # f16 scale rounds to zero (Q8, Q4)
    b = rng.standard_normal(32) * 3e-8; blocks.append(b)          # near the f16 subnormal floor
    b = rng.standard_normal(32) * 1e4; blocks.append(b)           # large, f16 scale still finite
    b = np.full(32, 3.0); b[31] = -3.0; blocks.append(b)          # all equal magnitudes
    b = rng.standard_normal(32); b[0] = 1e-3; b[1] = -50; blocks.append(b)   # one outlier
    return np.array(blocks, dtype=np.float32)


@pytest.mark.parametrize("wt,sf", TYPES)
def test_quantize_special_blocks(qmv, wt, sf):
    rng = np.random.default_rng(11 + wt + sf)
    blocks = special_blocks(rng)
    # the blocks as the rows of a 32-column matrix, and again side by side in one row
    for src in (blocks, blocks.reshape(1, -1), np.tile(blocks.reshape(3, -1), (2, 1))):
        W, first = gpu_quantize(qmv, wt, sf, src)
        assert first == -1
        assert_bytes_equal(W, oracle.quantize(src, wt, sf), f"special {wt},{sf} {src.shape}")


@pytest.mark.parametrize("wt", [1, 2])
def test_quantize_refuses_f16_overflow(qmv, wt):
    # an f16 scale beyond 65504 is refused: the block is written with d = 0 and *first_bad
    # names the first such block; every other block is the oracle's
    rows, cols = 6, 256
    rng = np.random.default_rng(21 + wt)
    src = workload_like(rng, rows, cols)
    big = 65504.0 * (127 if wt == 1 else 8) * 2
    src[2, 64:96] = rng.standard_normal(32) * big          # block 2 * 8 + 2 = 18
    src[4, 224:256] = rng.standard_normal(32) * big        # block 4 * 8 + 7 = 39
    W, first = gpu_quantize(qmv, wt, 1, src)
    assert first == 18
    ok = src.copy()
    ok[2, 64:96] = 0.0
    ok[4, 224:256] = 0.0
    want = oracle.quantize(ok, wt, 1)
    q_bytes = rows * cols if wt == 1 else rows * cols // 2
    d_off = oracle.scale_offset(wt, 1, rows, cols)
    qb = 32 if wt == 1 else 16
    refused = [18, 39]
    mask = np.ones(W.size, bool)
    for b in refused:
        mask[b * qb:(b + 1) * qb] = False
        mask[d_off + 2 * b:d_off + 2 * b + 2] = False
        # the refused block: d = +0 and zero quants (Q8_0) or nibbles 8 (Q4_0)
        assert np.all(W[b * qb:(b + 1) * qb] == (0 if wt == 1 else 0x88))
        assert W[d_off + 2 * b] == 0 and W[d_off + 2 * b + 1] == 0
    assert_bytes_equal(W[mask], want[mask], "blocks not refused")
    assert q_bytes <= d_off


def test_quantize_full_size_prefill_matrix(qmv):
    # the prefill workload's 14336 x 4096 matrix from float data, Q4_0 with f16 scales and
    # Q8_0 with f32 scales
    rows, cols = 14336, 4096
    rng = np.random.default_rng(31)
    src = workload_like(rng, rows, cols)
    for wt, sf in ((2, 1), (1, 0)):
        W, first = gpu_quantize(qmv, wt, sf, src)
        assert first == -1
        assert_bytes_equal(W, oracle.quantize(src, wt, sf), f"full size {wt},{sf}")


def test_quantize_then_dequant_is_the_rule(qmv):
    # round trip on the device: dequant(quantize(x)) equals the oracle's dequant of the
    # oracle's bytes, bit for bit
    import torch
    rows, cols = 64, 1024
    rng = np.random.default_rng(41)
    src = workload_like(rng, rows, cols)
    for wt, sf in TYPES:
        W, first = qmv.quantize(wt, sf, dev_x(src))
        out = qmv.dequant(wt, sf, rows, cols, W)
        torch.cuda.synchronize()
        want = oracle.dequant(oracle.quantize(src, wt, sf), wt, sf, rows, cols)
        got = out.cpu().numpy()
        assert np.array_equal(got.view(np.uint32), np.asarray(want, np.float32).view(np.uint32))


# ------------------------------------------------------------- Q4_0 best-fit writer
def gpu_quantize_fit(q, sf, src):
    import torch
    W, first = q.quantize_q4_fit(sf, dev_x(np.ascontiguousarray(src, dtype=np.float32)))
    torch.cuda.synchronize()
    return W.cpu().numpy(), first


@pytest.mark.parametrize("sf", [0, 1])
@pytest.mark.parametrize("rows,cols", [(1, 32), (3, 96), (33, 256), (256, 4096), (5, 11008)])
def test_quantize_q4_fit_matches_oracle(qmv, sf, rows, cols):
    rng = np.random.default_rng(rows * 5 + cols + sf)
    src = workload_like(rng, rows, cols)
    W, first = gpu_quantize_fit(qmv, sf, src)
    assert first == -1
    assert_bytes_equal(W, oracle.quantize_q4_fit(src, sf), f"fit {sf} {rows}x{cols}")


@pytest.mark.parametrize("sf", [0, 1])
def test_quantize_q4_fit_special_blocks(qmv, sf):
    rng = np.random.default_rng(31 + sf)
    blocks = list(special_blocks(rng))
    lv = rng.integers(-5, 6, 32).astype(np.float32)
    lv[4] = -6
    blocks.append(lv * np.float32(0.25))                 # exactly representable at level -6
    blocks.append(rng.standard_normal(32).astype(np.float32) * np.float32(3e-7))   # below 1e-6
    b = rng.standard_normal(32).astype(np.float32) * np.float32(1e-6)
    b[0] = np.float32(1e-6)
    blocks.append(b)                                     # the threshold itself (not scaled)
    src = np.array(blocks, dtype=np.float32)
    for s in (src, src.reshape(1, -1)):
        W, first = gpu_quantize_fit(qmv, sf, s)
        assert first == -1
        assert_bytes_equal(W, oracle.quantize_q4_fit(s, sf), f"fit special {sf} {s.shape}")


def test_quantize_q4_fit_refuses_f16_overflow(qmv):
    rows, cols = 4, 128
    rng = np.random.default_rng(41)
    src = workload_like(rng, rows, cols)
    src[1, 32:64] = rng.standard_normal(32) * 65504.0 * 40      # block 1 * 4 + 1 = 5
    W, first = gpu_quantize_fit(qmv, 1, src)
    assert first == 5
    ok = src.copy()
    ok[1, 32:64] = 0.0
    want = oracle.quantize_q4_fit(ok, 1)
    assert_bytes_equal(W, want, "fit with a refused block")       # refused: d = 0, nibbles 8


def test_quantize_q4_fit_full_size_sampled_rows(qmv):
    # the prefill workload's 14336 x 4096 matrix on the device; rows checked against the oracle
    # on a sample (the rule is per block, so the oracle runs on those rows alone)
    rows, cols = 14336, 4096
    rng = np.random.default_rng(51)
    src = workload_like(rng, rows, cols)
    W, first = gpu_quantize_fit(qmv, 1, src)
    assert first == -1
    ids = np.unique(np.concatenate([np.arange(4), rows - 1 - np.arange(4), rng.integers(0, rows, 40)]))
    want = oracle.quantize_q4_fit(src[ids], 1)
    qb, d_off = cols // 2, oracle.scale_offset(2, 1, rows, cols)
    wq = W[:rows * qb].reshape(rows, qb)[ids]
    wd = W[d_off:d_off + rows * cols // 16].reshape(rows, cols // 16)[ids]
    d_off_s = oracle.scale_offset(2, 1, ids.size, cols)
    assert np.array_equal(wq.reshape(-1), want[:ids.size * qb])
    assert np.array_equal(wd.reshape(-1), want[d_off_s:d_off_s + ids.size * cols // 16])
