"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Every test here runs on the CPU.  The facts are: byte counts printed on the pages,
hand-decoded blocks (tests/golden), IEEE half-precision conversion as numpy implements
it, closed forms of the product (one-hot, all-ones, exact integer arithmetic), and
invariants of the writer rules.  A plausible slip in the oracle (wrong nibble half,
wrong scale index, transposed product, dropped level offset, wrong padding) fails at
least one of them; tests/test_oracle_mutants.py checks that claim on planted mistakes.
"""
import math

import numpy as np
import pytest

import oracle
from block_quantized_weight_q4_gb300 import inputs
from conftest import read_cases, read_rows


# ----------------------------------------------------------------- sizes
def test_sizes_match_worked_examples():
    for wt, sf, rows, cols, expect, *src in read_rows("sizes_worked_examples.txt"):
        got = oracle.weight_bytes(int(wt), int(sf), int(rows), int(cols))
        assert got == int(expect), (wt, sf, rows, cols, " ".join(src))


def test_bits_per_weight():
    # Krafla "Body": Q4_0 4.5 bits/weight with f16 scales, 5 with f32; Q8_0 8.5 and 9.
    rows, cols = 4096, 4096
    for wt, sf, bits in [(2, 1, 4.5), (2, 0, 5.0), (1, 1, 8.5), (1, 0, 9.0)]:
        assert oracle.weight_bytes(wt, sf, rows, cols) * 8 / (rows * cols) == bits


def test_scale_offset_is_padded_q_size():
    assert oracle.scale_offset(2, 1, 1, 32) == 64
    assert oracle.scale_offset(1, 0, 1, 32) == 64
    assert oracle.scale_offset(1, 0, 2, 32) == 64
    assert oracle.scale_offset(1, 0, 3, 32) == 128
    assert oracle.scale_offset(2, 1, 151936, 896) == 151936 * 448


@pytest.mark.parametrize("args", [(2, 1, 1, 48), (2, 1, 0, 32), (2, 1, 1, 0), (1, 0, -1, 32),
                                  (3, 0, 1, 32), (2, 2, 1, 32), (2, 1, 2**40, 2**40)])
def test_sizes_reject_bad_shapes(args):
    assert oracle.weight_bytes(*args) == -1


# ----------------------------------------------------------------- number formats
def test_f16_all_codes_match_numpy():
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = codes.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_value(int(c)) for c in codes], dtype=np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f16_rne_matches_numpy():
    rng = np.random.default_rng(5)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(1e-3),
        rng.uniform(-7e4, 7e4, 20000).astype(np.float32),
        np.ldexp(rng.uniform(-1, 1, 20000), rng.integers(-30, 17, 20000)).astype(np.float32),
        # exact midpoints between neighbouring halves, and their neighbours
        (np.arange(0, 65504, 0.5, dtype=np.float64)[::97] + 0).astype(np.float32),
        np.array([65504, 65519.996, 65520, 65536, 6.1035156e-05, 5.9604645e-08,
                  2.9802322e-08, 2.9802326e-08, 8.940697e-08, 0.0, -0.0, 1.0009766, 1.0004883,
                  1.0014648, -2.0019531], dtype=np.float32),
    ])
    ref = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f16_bits_rne(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_bf16_value_is_upper_half():
    for v in [1.0, -2.5, 3.140625, 1e-40, -0.0, 65536.0]:
        u = np.array([v], dtype=np.float32).view(np.uint32)[0]
        code = int(u >> 16)
        assert oracle.bf16_value(code) == np.array([code << 16], dtype=np.uint32).view(np.float32)[0]
    assert oracle.bf16_value(0x3F80) == 1.0
    assert oracle.bf16_value(0xC020) == -2.5


# ----------------------------------------------------------------- hand-built blocks
def _block_image(case):
    wt = int(case["wtype"][0])
    sf = int(case["scale_f16"][0])
    qb = np.array([int(b, 16) for b in case["bytes"]], dtype=np.uint8)
    if sf:
        d = np.array([int(case["scale_code"][0], 16)], dtype=np.uint16)
    else:
        d = np.array([float(case["scale"][0])], dtype=np.float32).view(np.uint32)
    W = inputs.assemble(wt, sf, 1, 32, qb, d)
    return wt, sf, W


@pytest.mark.parametrize("case", read_cases("hand_blocks.txt"), ids=lambda c: c["name"])
def test_hand_blocks_dequant(case):
    wt, sf, W = _block_image(case)
    expect = np.array([float(v) for v in case["weights"]], dtype=np.float32)
    got = oracle.dequant(W, wt, sf, 1, 32)[0]
    assert np.array_equal(got, expect), (got, expect)
    # the product against one-hot x gives the same column values exactly
    for c in (0, 5, 16, 31):
        x = np.zeros((1, 32), dtype=np.float32)
        x[0, c] = 1.0
        y, a = oracle.matvec(W, wt, sf, 1, 32, x)
        assert y[0, 0] == expect[c] and a[0, 0] == abs(expect[c])


def test_scale_index_and_row_addressing():
    # 3 rows x 96 cols Q4_0: every nibble of row r block k is 9 (level 1), scale 2^(r*3+k);
    # so w[r][c] = 2^(3r + c//32) exactly.  A wrong scale index or row stride shows.
    rows, cols = 3, 96
    q = np.full(rows * cols // 2, 0x99, dtype=np.uint8)
    d = np.array([2.0 ** (3 * r + k) for r in range(rows) for k in range(3)], dtype=np.float32)
    for sf in (0, 1):
        codes = d.astype(np.float16).view(np.uint16) if sf else d.view(np.uint32)
        W = inputs.assemble(2, sf, rows, cols, q, codes)
        got = oracle.dequant(W, 2, sf, rows, cols)
        expect = np.array([[2.0 ** (3 * r + c // 32) for c in range(cols)] for r in range(rows)])
        assert np.array_equal(got, expect.astype(np.float32))


def test_q4_rows_hold_distinct_nibbles():
    # row r: low nibbles r+1, high nibbles 15-r, so elements 0..15 have level r-7 and
    # 16..31 level 7-r; d = 1.  A swapped nibble half or row stride shows.
    rows, cols = 4, 64
    q = np.zeros((rows, cols // 2), dtype=np.uint8)
    for r in range(rows):
        q[r, :] = (r + 1) | ((15 - r) << 4)
    d = np.ones(rows * cols // 32, dtype=np.float32).view(np.uint32)
    W = inputs.assemble(2, 0, rows, cols, q.reshape(-1), d)
    got = oracle.dequant(W, 2, 0, rows, cols)
    for r in range(rows):
        for c in range(cols):
            assert got[r, c] == ((r - 7) if (c % 32) < 16 else (7 - r))


def test_dequant_single_rounding_with_f32_scale():
    # level * d with one f32 rounding: d = 1 + 2^-23 (f32), level 3 -> 3 + 3*2^-23, which
    # rounds to 3 + 2^-22 (ties to even at 3 + 1.5*2^-22)...  computed here with numpy's
    # own float32 multiply, an independent IEEE implementation.
    d = np.array([1.0 + 2.0 ** -23], dtype=np.float32)
    q = np.full(16, 0xBB, dtype=np.uint8)  # level 3 everywhere
    W = inputs.assemble(2, 0, 1, 32, q, d.view(np.uint32))
    got = oracle.dequant(W, 2, 0, 1, 32)
    assert np.array_equal(got[0], np.full(32, np.float32(3.0) * d[0], dtype=np.float32))


def test_nonfinite_and_negative_scales_are_valid_input():
    # every scale is valid input: negative, zero, inf and NaN scales decode by IEEE.
    q = np.array([0x80 | 0x08] * 16, dtype=np.uint8)  # low nibble 8 (level 0), high 8 (level 0)
    q[0] = 0x9F  # element 0 level 7, element 16 level 1
    for dval in (-3.0, 0.0, np.inf, -np.inf, np.nan):
        d = np.array([dval], dtype=np.float32)
        W = inputs.assemble(2, 0, 1, 32, q, d.view(np.uint32))
        got = oracle.dequant(W, 2, 0, 1, 32)[0]
        with np.errstate(invalid="ignore"):
            expect = (np.array([7] + [0] * 15 + [1] + [0] * 15, dtype=np.float32) * d[0])
        assert np.array_equal(np.isnan(got), np.isnan(expect))
        ok = ~np.isnan(expect)
        assert np.array_equal(got[ok], expect[ok])


# ----------------------------------------------------------------- the product
def test_generator_layout_round_trip():
    # the byte image the generator assembles decodes back to the drawn q and d
    for wt, sf in [(1, 0), (1, 1), (2, 0), (2, 1)]:
        m = inputs.make_matrix(wt, sf, 5, 96, seed=3)
        for r in range(5):
            for k in range(3):
                code = int(m.d_codes[r, k])
                want = (np.array([code], np.uint16).view(np.float16).astype(np.float32)[0] if sf
                        else np.array([code], np.uint32).view(np.float32)[0])
                assert oracle.scale(m.W, wt, sf, 5, 96, r, k) == want
        if wt == 1:
            lv = m.q.view(np.int8).reshape(5, 96)
            for r, c in [(0, 0), (4, 95), (2, 33)]:
                assert oracle.level(m.W, wt, 96, r, c) == lv[r, c]


@pytest.mark.parametrize("wt,sf", [(1, 0), (1, 1), (2, 0), (2, 1)])
@pytest.mark.parametrize("rows,cols", [(1, 32), (3, 64), (5, 96)])
def test_product_one_hot_columns(wt, sf, rows, cols):
    # x = e_c picks column c of the dequantized matrix: one non-zero term, so exact.
    m = inputs.make_matrix(wt, sf, rows, cols, seed=rows * 7 + cols)
    deq = oracle.dequant(m.W, wt, sf, rows, cols)
    x = np.eye(cols, dtype=np.float32)  # batch = cols, batch row b is e_b
    y, a = oracle.matvec(m.W, wt, sf, rows, cols, x)
    # the double-precision term is the exact level * d; one IEEE float32 rounding of it is
    # the dequantized weight (and with f16 scales level * d is exact already)
    assert np.array_equal(y.astype(np.float32), deq.T)
    assert np.array_equal(a, np.abs(y))
    if sf:
        assert np.array_equal(y, deq.T.astype(np.float64))


def test_product_all_ones_closed_form():
    # x = 1: y[r] = sum_k d_rk * sum_j level_rkj; with Q4_0 bytes all equal to b the
    # levels of a block sum to 16*((b & 15) - 8) + 16*((b >> 4) - 8).
    rows, cols = 6, 128
    for b in (0x00, 0x88, 0xF0, 0x3C, 0xFF):
        q = np.full(rows * cols // 2, b, dtype=np.uint8)
        rng = np.random.default_rng(b)
        d = rng.uniform(-1, 1, rows * cols // 32).astype(np.float32)
        W = inputs.assemble(2, 0, rows, cols, q, d.view(np.uint32))
        y, _ = oracle.matvec(W, 2, 0, rows, cols, np.ones((1, cols), dtype=np.float32))
        per_block = 16 * ((b & 15) - 8) + 16 * ((b >> 4) - 8)
        expect = (d.astype(np.float64).reshape(rows, cols // 32) * per_block).sum(axis=1)
        assert np.allclose(y[0], expect, rtol=0, atol=1e-12)


def test_product_bf16_activations_match_their_f32_values():
    m = inputs.make_matrix(2, 1, 4, 64, seed=11)
    xb = inputs.make_x(3, 64, True, seed=12)
    xf = (xb.astype(np.uint32) << 16).view(np.float32)
    yb, ab = oracle.matvec(m.W, 2, 1, 4, 64, xb)
    yf, af = oracle.matvec(m.W, 2, 1, 4, 64, xf)
    assert np.array_equal(yb, yf) and np.array_equal(ab, af)


def test_product_linearity_and_batch_order():
    rows, cols = 7, 96
    m = inputs.make_matrix(1, 0, rows, cols, seed=21)
    x1 = inputs.make_int_x(1, cols, False, seed=1)
    x2 = inputs.make_int_x(1, cols, False, seed=2)
    y1, _ = oracle.matvec(m.W, 1, 0, rows, cols, x1)
    y2, _ = oracle.matvec(m.W, 1, 0, rows, cols, x2)
    yb, _ = oracle.matvec(m.W, 1, 0, rows, cols, np.concatenate([x2, x1]))
    y3, _ = oracle.matvec(m.W, 1, 0, rows, cols, 3 * x1 + x2)
    assert np.array_equal(yb[0], y2[0]) and np.array_equal(yb[1], y1[0])
    assert np.allclose(y3[0], 3 * y1[0] + y2[0], rtol=1e-13, atol=1e-13)


def test_product_exact_integer_case_equals_rational_sum():
    # integer x and power-of-two d: every term is an exact dyadic number, so the sum is
    # exact too; compare with a sum over Python fractions built from the hand rule.
    from fractions import Fraction
    rows, cols = 3, 64
    rng = np.random.default_rng(4)
    q = rng.integers(0, 256, rows * cols // 2).astype(np.uint8)
    d = inputs.pow2_scales(rng, rows * cols // 32, 0)
    W = inputs.assemble(2, 0, rows, cols, q, d)
    x = inputs.make_int_x(1, cols, False, seed=9)
    y, _ = oracle.matvec(W, 2, 0, rows, cols, x)
    dv = d.view(np.float32).reshape(rows, cols // 32)
    qb = q.reshape(rows, cols // 2)
    for r in range(rows):
        s = Fraction(0)
        for c in range(cols):
            k, j = divmod(c, 32)
            byte = int(qb[r, 16 * k + j % 16])
            nib = byte & 15 if j < 16 else byte >> 4
            s += Fraction(nib - 8) * Fraction(float(dv[r, k])) * Fraction(float(x[0, c]))
        assert Fraction(y[0, r]) == s


def test_matvec_rows_matches_full():
    m = inputs.make_matrix(2, 1, 9, 64, seed=5)
    x = inputs.make_x(2, 64, True, seed=6)
    y, a = oracle.matvec(m.W, 2, 1, 9, 64, x)
    ids = [8, 0, 3]
    ys, as_ = oracle.matvec_rows(m.W, 2, 1, 9, 64, x, ids)
    assert np.array_equal(ys, y[:, ids]) and np.array_equal(as_, a[:, ids])


# ----------------------------------------------------------------- validation
def test_validate_rejects_q8_minus_128_only():
    m = inputs.make_matrix(1, 0, 4, 64, seed=1)
    assert oracle.validate(m.W, 1, 0, 4, 64) == oracle.OK
    W = m.W.copy()
    W[77] = 0x80
    assert oracle.validate(W, 1, 0, 4, 64) == oracle.E_FORMAT
    # the same byte inside a Q4_0 matrix is just nibbles 0 and 8
    m4 = inputs.make_matrix(2, 0, 4, 64, seed=1)
    W4 = m4.W.copy()
    W4[7] = 0x80
    assert oracle.validate(W4, 2, 0, 4, 64) == oracle.OK
    assert oracle.validate(W4, 2, 0, 4, 48) == oracle.E_SHAPE


# ----------------------------------------------------------------- writer rules
def test_q8_rule_hand_example():
    (case,) = [c for c in read_cases("quant_rules.txt") if c["name"] == "q8_f32"]
    x = np.zeros(32, dtype=np.float32)
    vals = [float(v) for v in case["x"]]
    x[:len(vals)] = vals
    st, q, bits = oracle.quant_q8_block(x, 0)
    assert st == oracle.OK
    assert list(q[:len(vals)]) == [int(v) for v in case["q"]]
    assert np.array([bits], np.uint32).view(np.float32)[0] == np.float32(1.0) / np.float32(127.0)


def test_q4_round_rule_hand_example():
    (case,) = [c for c in read_cases("quant_rules.txt") if c["name"] == "q4_round"]
    x = np.zeros(32, dtype=np.float32)
    vals = [float(v) for v in case["x"]]
    x[:len(vals)] = vals
    st, qs, bits = oracle.quant_q4_round_block(x, 0)
    assert st == oracle.OK
    assert np.array([bits], np.uint32).view(np.float32)[0] == float(case["d"][0])
    nib = [int(qs[j] & 15) if j < 16 else int(qs[j - 16] >> 4) for j in range(32)]
    assert [n - 8 for n in nib[:len(vals)]] == [int(v) for v in case["level"]]


@pytest.mark.parametrize("sf", [0, 1])
def test_q8_rule_invariants(sf):
    rng = np.random.default_rng(31 + sf)
    for t in range(300):
        x = (rng.standard_normal(32) * 10.0 ** rng.uniform(-4, 3)).astype(np.float32)
        st, q, bits = oracle.quant_q8_block(x, sf)
        assert st == oracle.OK
        d = (np.array([bits], np.uint16).view(np.float16).astype(np.float32)[0] if sf
             else np.array([bits], np.uint32).view(np.float32)[0])
        amax = np.abs(x).max()
        if sf:
            # the stored scale is amax/127 rounded to the nearest half (numpy's rounding)
            assert bits == (np.float32(amax) / np.float32(127)).astype(np.float16).view(np.uint16)
        else:
            assert d == np.float32(amax) / np.float32(127)
        assert np.all(np.abs(q.astype(int)) <= 127)
        err = np.abs(x.astype(np.float64) - q.astype(np.float64) * float(d))
        # elements inside the +-127 range round to the nearest step; the rest clamp to
        # +-127 with their sign (an f16-rounded d can sit just below amax / 127)
        inside = np.abs(x.astype(np.float64)) / float(d) <= 127.0
        assert np.all(err[inside] <= float(d) * (0.5 + 1e-5) + 1e-30)
        assert np.all(q[~inside].astype(int) == np.sign(x[~inside]).astype(int) * 127)
        if not sf:
            assert abs(int(q[np.argmax(np.abs(x))])) == 127
    st, q, bits = oracle.quant_q8_block(np.zeros(32, np.float32), sf)
    assert st == oracle.OK and bits == 0 and not q.any()
    st, q, bits = oracle.quant_q8_block(np.full(32, 1e-31, np.float32), sf)
    assert st == oracle.OK and bits == 0 and not q.any()


def test_q8_f16_rule_refuses_scales_above_65504():
    x = np.zeros(32, np.float32)
    x[3] = 65504.0 * 127.0 * 1.01
    st, _, _ = oracle.quant_q8_block(x, 1)
    assert st == oracle.E_FORMAT
    st, _, _ = oracle.quant_q8_block(x, 0)
    assert st == oracle.OK


@pytest.mark.parametrize("sf", [0, 1])
def test_q4_round_rule_invariants(sf):
    rng = np.random.default_rng(41 + sf)
    for t in range(300):
        x = (rng.standard_normal(32) * 10.0 ** rng.uniform(-3, 2)).astype(np.float32)
        st, qs, bits = oracle.quant_q4_round_block(x, sf)
        assert st == oracle.OK
        d = (np.array([bits], np.uint16).view(np.float16).astype(np.float32)[0] if sf
             else np.array([bits], np.uint32).view(np.float32)[0])
        nib = np.array([qs[j] & 15 if j < 16 else qs[j - 16] >> 4 for j in range(32)], dtype=int)
        lv = nib - 8
        im = int(np.argmax(np.abs(x)))
        assert lv[im] == -8
        if not sf:
            assert np.float32(lv[im]) * d == x[im]  # the extreme element comes back exactly
        r = x.astype(np.float64) / float(d)
        ok = r <= 7.5 - 1e-4  # not clamped at level 7
        err = np.abs(x.astype(np.float64) - lv * float(d))
        tol = abs(float(d)) * (0.5 + 1e-3) if not sf else abs(float(d)) * 0.5 + abs(x[im] / 8 - d)
        assert np.all(err[ok] <= tol + 1e-30)


def test_quantize_matrix_round_trip_q8():
    rng = np.random.default_rng(8)
    src = rng.standard_normal((4, 64)).astype(np.float32)
    W = oracle.quantize(src, 1, 0)
    deq = oracle.dequant(W, 1, 0, 4, 64)
    # each weight within half a step of the block's scale
    d = src.reshape(4, 2, 32)
    step = (np.abs(d).max(axis=2) / 127.0).repeat(32, axis=1).reshape(4, 64)
    assert np.all(np.abs(deq - src) <= step * 0.5 * (1 + 1e-5))
    # quantizing the dequantized matrix again gives the same bytes when the block max is hit
    W2 = oracle.quantize(deq, 1, 0)
    q_bytes = 4 * 64
    assert np.array_equal(W2[:q_bytes], W[:q_bytes])


# ----------------------------------------------------- activation-quantized product
def _exact_activations(rng, batch, cols, e_lo=-6, e_hi=3):
    """x = k * 2^e per block: integers |k| <= 127 with one element of each block at +-127,
    and a power-of-two step 2^e per block.  The Q8_0 rule must give back k and d = 2^e
    exactly: amax = 127 * 2^e, 127 / amax = 2^-e, x * 2^-e = k, k +- 0.5 truncates to k."""
    nb = cols // 32
    k = rng.integers(-127, 128, size=(batch, nb, 32))
    pos = rng.integers(0, 32, size=(batch, nb))
    sign = np.where(rng.random((batch, nb)) < 0.5, -1, 1)
    for b in range(batch):
        for blk in range(nb):
            k[b, blk, pos[b, blk]] = 127 * sign[b, blk]
    e = rng.integers(e_lo, e_hi + 1, size=(batch, nb))
    x = (k * np.exp2(e)[:, :, None]).reshape(batch, cols).astype(np.float32)
    return x, k.reshape(batch, cols).astype(np.int8), np.exp2(e).astype(np.float32).reshape(-1)


@pytest.mark.parametrize("bf16", [False, True])
def test_quantize_x_gives_back_exact_activations(bf16):
    rng = np.random.default_rng(51)
    batch, cols = 3, 128
    x, k, step = _exact_activations(rng, batch, cols)
    xin = inputs.bf16_codes(x) if bf16 else x   # k * 2^e has at most 8 significant bits
    if bf16:
        assert np.array_equal((xin.astype(np.uint32) << 16).view(np.float32), x)
    xq = oracle.quantize_x(xin)
    off = oracle.scale_offset(1, 0, batch, cols)
    assert np.array_equal(xq[:batch * cols].view(np.int8), k.reshape(-1))
    assert np.array_equal(xq[off:off + 4 * step.size].view(np.float32), step)
    assert not xq[batch * cols:off].any()


def test_quantize_x_is_the_q8_writer_rule():
    # the runtime's activation quantizer and the writer share the rule ("Quantization rule")
    rng = np.random.default_rng(52)
    x = (rng.standard_normal((4, 96)) * np.exp(rng.uniform(-5, 5, (4, 1)))).astype(np.float32)
    assert np.array_equal(oracle.quantize_x(x), oracle.quantize(x, 1, 0))
    xb = inputs.bf16_codes(x)
    assert np.array_equal(oracle.quantize_x(xb), oracle.quantize((xb.astype(np.uint32) << 16).view(np.float32), 1, 0))


@pytest.mark.parametrize("wt", [1, 2])
def test_matvec_qx_equals_plain_product_on_exact_activations(wt):
    # activations that the rule represents exactly leave the product unchanged: with f16
    # weight scales every term level * d_w * k * 2^e has <= 26 significant bits and the
    # whole sum stays within double's 53, so both evaluations are exact
    rng = np.random.default_rng(53 + wt)
    rows, cols, batch = 6, 256, 3
    m = inputs.make_matrix(wt, 1, rows, cols, seed=54 + wt)
    x, _, _ = _exact_activations(rng, batch, cols, e_lo=-3, e_hi=0)
    yq, aq = oracle.matvec_qx(m.W, wt, 1, rows, cols, oracle.quantize_x(x), batch)
    y, a = oracle.matvec(m.W, wt, 1, rows, cols, x)
    assert np.array_equal(yq, y)
    assert np.array_equal(aq, a)


@pytest.mark.parametrize("wt,sf", [(1, 0), (1, 1), (2, 0), (2, 1)])
def test_matvec_qx_equals_product_with_dequantized_activations(wt, sf):
    # sum_k d_w d_x sum_j level q_x = sum_c w_c * (q_x d_x)_c: the product against the
    # dequantized activations; the f32 dequant rounds each q_x * d_x once (<= 2^-24 relative)
    rows, cols, batch = 5, 320, 2
    m = inputs.make_matrix(wt, sf, rows, cols, seed=60 + 2 * wt + sf)
    x = inputs.make_x(batch, cols, False, seed=61)
    xq = oracle.quantize_x(x)
    xhat = oracle.dequant(xq, 1, 0, batch, cols)
    yq, aq = oracle.matvec_qx(m.W, wt, sf, rows, cols, xq, batch)
    y, a = oracle.matvec(m.W, wt, sf, rows, cols, xhat)
    assert np.all(np.abs(yq - y) <= 2.0 ** -22 * a)
    assert np.allclose(aq, a, rtol=2.0 ** -22, atol=0)
    # and it differs from the product with the unquantized activations by about one step
    y0, a0 = oracle.matvec(m.W, wt, sf, rows, cols, x)
    assert np.all(np.abs(yq - y0) <= 0.01 * a0)


def test_matvec_qx_hand_block():
    # Q4_0, one block, every byte 0x99 (levels +1), d_w = 0.5.  x = [127, -63.5, 0, ...]:
    # amax = 127, d_x = 1, 127 / amax = 1; q_0 = trunc(127 + 0.5) = 127, q_1 = trunc(-63.5 - 0.5)
    # = -64 (rounded away from zero); isum = 127 - 64 = 63, y = 0.5 * 1 * 63 = 31.5 (the float
    # product would be 0.5 * 63.5 = 31.75); absref = 0.5 * (127 + 64) = 95.5.
    W = inputs.assemble(2, 0, 1, 32, np.full(16, 0x99, np.uint8), np.array([0.5], np.float32).view(np.uint32))
    x = np.zeros((1, 32), np.float32)
    x[0, 0], x[0, 1] = 127.0, -63.5
    y, a = oracle.matvec_qx(W, 2, 0, 1, 32, oracle.quantize_x(x), 1)
    assert y[0, 0] == 31.5 and a[0, 0] == 95.5
    # Q8_0: quants [2, -3, 0, ...], d_w = 0.25; x = [127, 1.5, 0, ...] gives q_x = [127, 2]
    # (1.5 + 0.5 = 2): isum = 254 - 6 = 248, y = 62
    q = np.zeros(32, np.int8)
    q[0], q[1] = 2, -3
    W = inputs.assemble(1, 0, 1, 32, q.view(np.uint8), np.array([0.25], np.float32).view(np.uint32))
    x = np.zeros((1, 32), np.float32)
    x[0, 0], x[0, 1] = 127.0, 1.5
    y, a = oracle.matvec_qx(W, 1, 0, 1, 32, oracle.quantize_x(x), 1)
    assert y[0, 0] == 62.0 and a[0, 0] == 0.25 * 260


def test_matvec_qx_batch_rows_are_independent():
    rows, cols = 4, 128
    m = inputs.make_matrix(2, 1, rows, cols, seed=70)
    x = inputs.make_x(3, cols, False, seed=71)
    y, _ = oracle.matvec_qx(m.W, 2, 1, rows, cols, oracle.quantize_x(x), 3)
    for b in range(3):
        yb, _ = oracle.matvec_qx(m.W, 2, 1, rows, cols, oracle.quantize_x(x[b:b + 1]), 1)
        assert np.array_equal(y[b], yb[0])


# ----------------------------------------------------------- GGUF interleaved blocks
def test_gguf_sizes_match_the_page():
    for wt, rows, cols, expect, *src in read_rows("gguf_sizes.txt"):
        assert oracle.gguf_bytes(int(wt), int(rows), int(cols)) == int(expect), " ".join(src)


@pytest.mark.parametrize("case", [c for c in read_cases("hand_blocks.txt") if c["scale_f16"][0] == "1"],
                         ids=lambda c: c["name"])
def test_gguf_hand_blocks(case):
    # the hand blocks with f16 scales, written as one GGUF record each: d (little-endian f16
    # code) then the quant bytes; converted, they must hold the weights worked out by hand
    wt = int(case["wtype"][0])
    code = int(case["scale_code"][0], 16)
    qb = [int(b, 16) for b in case["bytes"]]
    rec = np.array([code & 0xFF, code >> 8] + qb, np.uint8)
    assert rec.size == oracle.gguf_bytes(wt, 1, 32)
    W = oracle.gguf_to_mlb(rec, wt, 1, 32)
    expect = np.array([float(v) for v in case["weights"]], np.float32)
    assert np.array_equal(oracle.dequant(W, wt, 1, 1, 32)[0], expect)


@pytest.mark.parametrize("wt", [1, 2])
def test_gguf_record_addressing(wt):
    # record (r, k) of a 3 x 96 tensor: d = 2^(3r + k), every weight level +1 (Q4_0 byte 0x99,
    # Q8_0 byte 1), so w[r][c] = 2^(3r + c // 32): checks the record stride, row stride and
    # the place of d in the record
    rows, cols = 3, 96
    qb = 32 if wt == 1 else 16
    recs = []
    for r in range(rows):
        for k in range(cols // 32):
            code = int(np.array([2.0 ** (3 * r + k)], np.float16).view(np.uint16)[0])
            recs += [code & 0xFF, code >> 8] + [1 if wt == 1 else 0x99] * qb
    g = np.array(recs, np.uint8)
    assert g.size == oracle.gguf_bytes(wt, rows, cols)
    W = oracle.gguf_to_mlb(g, wt, rows, cols)
    expect = np.array([[2.0 ** (3 * r + c // 32) for c in range(cols)] for r in range(rows)], np.float32)
    assert np.array_equal(oracle.dequant(W, wt, 1, rows, cols), expect)


# ------------------------------------------------- gated activation (FFN down projection)
@pytest.mark.parametrize("act", [0, 1])
@pytest.mark.parametrize("wt,sf", [(1, 0), (2, 1)])
def test_glu_odd_part_gives_the_plain_product(act, wt, sf):
    # both activations satisfy act(g) - act(-g) = g (SiLU: g s(g) + g s(-g) = g since
    # s(g) + s(-g) = 1; GELU-tanh: tanh is odd), so y(g, u) - y(-g, u) = W (g * u): the plain
    # product, pinned separately, with x = g * u (exact in float32 for these small integers)
    rows, cols, batch = 5, 96, 2
    m = inputs.make_matrix(wt, sf, rows, cols, seed=110 + act)
    rng = np.random.default_rng(111)
    g = rng.integers(-6, 7, (batch, cols)).astype(np.float32) / 4
    u = rng.integers(-8, 9, (batch, cols)).astype(np.float32) / 8
    yp, _ = oracle.matvec_glu(m.W, wt, sf, rows, cols, act, g, u)
    yn, _ = oracle.matvec_glu(m.W, wt, sf, rows, cols, act, -g, u)
    y, a = oracle.matvec(m.W, wt, sf, rows, cols, (g * u).astype(np.float32))
    assert np.all(np.abs((yp - yn) - y) <= 1e-12 * a)


def test_glu_silu_and_gelu_values():
    # one-hot weights pick h itself: W = one block, level +1 at column 0 only, d = 1
    q = np.full(16, 0x88, np.uint8)
    q[0] = 0x89                                         # element 0: nibble 9 (level +1)
    W = inputs.assemble(2, 0, 1, 32, q, np.array([1.0], np.float32).view(np.uint32))
    up = np.zeros((1, 32), np.float32)
    up[0, 0] = 1.0
    # SiLU at ln 3: the sigmoid is exactly 3/4, so SiLU(g) = 3g/4 (g rounded to float32)
    g = np.zeros((1, 32), np.float32)
    g[0, 0] = np.float32(np.log(3.0))
    y, _ = oracle.matvec_glu(W, 2, 0, 1, 32, 0, g, up)
    assert abs(y[0, 0] - 0.75 * float(g[0, 0])) < 1e-7
    # GELU-tanh where its tanh is exactly 1/2: sqrt(2/pi)(g + 0.044715 g^3) = atanh(1/2), found
    # by bisection here; then GELU(g) = g/2 * 3/2 = 3g/4
    k, target = np.sqrt(2 / np.pi), np.arctanh(0.5)
    lo, hi = 0.0, 2.0
    for _ in range(200):
        mid = (lo + hi) / 2
        lo, hi = (mid, hi) if k * (mid + 0.044715 * mid ** 3) < target else (lo, mid)
    g[0, 0] = np.float32(lo)
    y, _ = oracle.matvec_glu(W, 2, 0, 1, 32, 1, g, up)
    assert abs(y[0, 0] - 0.75 * float(g[0, 0])) < 1e-6
    # zero up or zero gate give zero; a large gate passes through SiLU unchanged
    y, a = oracle.matvec_glu(W, 2, 0, 1, 32, 0, g, np.zeros_like(up))
    assert y[0, 0] == 0 and a[0, 0] == 0
    y, _ = oracle.matvec_glu(W, 2, 0, 1, 32, 0, np.zeros_like(g), up)
    assert y[0, 0] == 0
    g[0, 0] = 40.0
    y, _ = oracle.matvec_glu(W, 2, 0, 1, 32, 0, g, up)
    assert abs(y[0, 0] - 40.0) < 1e-12


@pytest.mark.parametrize("act", [0, 1])
def test_glu_values_odd_part_and_limits(act):
    # h = act(g) * u value by value: the odd part act(g) - act(-g) = g (both activations), act(0)
    # = 0, and for large |g| the activation tends to max(g, 0)
    rng = np.random.default_rng(120 + act)
    g = rng.standard_normal(200) * 3
    u = rng.standard_normal(200)
    hp, hn = oracle.glu(act, g, u), oracle.glu(act, -g, u)
    assert np.all(np.abs((hp - hn) - g * u) <= 1e-14 * (np.abs(g * u) + 1))
    assert np.all(oracle.glu(act, np.zeros(3), np.ones(3)) == 0)
    big = np.array([40.0, -40.0])
    h = oracle.glu(act, big, np.ones(2))
    assert abs(h[0] - 40.0) < 1e-12 and abs(h[1]) < 1e-12


def test_glu_silu_and_gelu_three_quarters():
    # SiLU at ln 3 (sigmoid exactly 3/4) and GELU-tanh where its tanh is exactly 1/2 both give
    # 3g/4, times u
    g = np.array([np.log(3.0)])
    assert abs(oracle.glu(0, g, np.array([2.0]))[0] - 1.5 * g[0]) < 1e-15
    k, target = np.sqrt(2 / np.pi), np.arctanh(0.5)
    lo, hi = 0.0, 2.0
    for _ in range(200):
        mid = (lo + hi) / 2
        lo, hi = (mid, hi) if k * (mid + 0.044715 * mid ** 3) < target else (lo, mid)
    assert abs(oracle.glu(1, np.array([lo]), np.array([-1.0]))[0] + 0.75 * lo) < 1e-14


# ------------------------------------------------------------- Q4_0 best-fit writer
def _weighted_err(x, w):
    x = x.astype(np.float64)
    return float(np.sum(x * x * (x - w.astype(np.float64)) ** 2))


@pytest.mark.parametrize("sf", [0, 1])
def test_q4_fit_exact_blocks_come_back_exactly(sf):
    # x = c * l with integer levels l in [-7, 7], one element at -8 (the unique largest
    # magnitude) and c a power of two: the candidate that maps the largest element to -8 reproduces
    # l, the weighted least-squares d is c itself, and the error is zero; so dequant gives x back
    rng = np.random.default_rng(120 + sf)
    rows, cols = 6, 128
    lv = rng.integers(-7, 8, (rows, cols // 32, 32))
    lv[:, :, 5] = -8
    c = np.exp2(rng.integers(-10, 3, (rows, cols // 32))).astype(np.float32)
    x = (lv * c[:, :, None]).reshape(rows, cols).astype(np.float32)
    W = oracle.quantize_q4_fit(x, sf)
    assert np.array_equal(oracle.dequant(W, 2, sf, rows, cols), x)


def test_q4_fit_never_worse_than_the_round_rule():
    # the candidate at -8 starts from the round rule's own scale, and a weighted least-squares d
    # over the same levels cannot raise the weighted error; the winner is no worse than that
    rng = np.random.default_rng(130)
    rows, cols = 64, 256
    x = (rng.standard_normal((rows, cols)) * np.exp(rng.uniform(-3, 3, (rows, 1)))).astype(np.float32)
    fit = oracle.dequant(oracle.quantize_q4_fit(x, 0), 2, 0, rows, cols)
    rnd = oracle.dequant(oracle.quantize(x, 2, 0), 2, 0, rows, cols)
    better = 0
    for r in range(rows):
        for k in range(cols // 32):
            sl = slice(32 * k, 32 * k + 32)
            ef, er = _weighted_err(x[r, sl], fit[r, sl]), _weighted_err(x[r, sl], rnd[r, sl])
            assert ef <= er * (1 + 1e-5) + 1e-30, (r, k, ef, er)
            better += ef < er * (1 - 1e-3)
    assert better > rows * cols // 32 // 2   # the search usually finds a strictly better fit


def test_q4_fit_scales_with_the_block():
    # every step scales exactly under a power-of-two factor (away from the 1e-6 threshold and
    # float32's range ends): the nibbles stay, d scales by the factor
    rng = np.random.default_rng(140)
    for _ in range(20):
        x = rng.standard_normal(32).astype(np.float32)
        st, q1, d1 = oracle.quant_q4_fit_block(x, 0)
        st2, q2, d2 = oracle.quant_q4_fit_block(x * np.float32(2.0 ** 7), 0)
        assert st == st2 == 0 and np.array_equal(q1, q2)
        assert np.array([d2], np.uint32).view(np.float32)[0] == np.array([d1], np.uint32).view(np.float32)[0] * 2.0 ** 7


def test_q4_fit_small_and_zero_blocks():
    # a block below 1e-6 is fitted at unit scale: the same nibbles as the block scaled up to a
    # largest magnitude of 1, and d scaled back; the all-zero block is d = 0 with level 0
    rng = np.random.default_rng(150)
    y = rng.standard_normal(32).astype(np.float32)
    y[7] = 1.0
    y = np.clip(y, -0.99, 1.0).astype(np.float32)     # element 7 is the unique largest, exactly 1
    a = np.float32(2.0 ** -30)
    st, qs, ds = oracle.quant_q4_fit_block(y * a, 0)
    st1, q1, d1 = oracle.quant_q4_fit_block(y, 0)
    assert st == st1 == 0 and np.array_equal(qs, q1)
    assert np.array([ds], np.uint32).view(np.float32)[0] == np.array([d1], np.uint32).view(np.float32)[0] * a
    st, q0, d0 = oracle.quant_q4_fit_block(np.zeros(32, np.float32), 1)
    assert st == 0 and d0 == 0 and np.all(q0 == 0x88)


@pytest.mark.parametrize("top", [-6, -7, 6])
def test_q4_fit_exact_blocks_at_other_levels(top):
    # the candidates run from -6 to -8.4: a block that is exactly c * l with its largest element
    # at level -6 or -7 (others strictly smaller) is reproduced only by the candidate that maps
    # it there; a positive largest element maps to the same levels with d negative
    rng = np.random.default_rng(160 + top)
    rows, cols = 4, 96
    lim = abs(top) - 1
    lv = rng.integers(-lim, lim + 1, (rows, cols // 32, 32))
    lv[:, :, 11] = top
    c = np.exp2(rng.integers(-8, 2, (rows, cols // 32))).astype(np.float32)
    x = (lv * c[:, :, None]).reshape(rows, cols).astype(np.float32)
    W = oracle.quantize_q4_fit(x, 0)
    assert np.array_equal(oracle.dequant(W, 2, 0, rows, cols), x)
