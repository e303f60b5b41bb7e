"""The pins catch plausible mistakes in the oracle.

Each case copies oracle/qmv_oracle.c, plants one mistake by text substitution (a swapped
nibble half, a dropped level offset, a transposed index, wrong padding, a lost sign...),
each of which keeps every write inside its buffer (the copies run in this process),
builds the copy with gcc into a temporary directory and runs the page-derived pin checks
against it.  At least one check must fail for every mutant, and all checks must pass for
the unmodified copy.  Everything happens on the CPU; the real oracle is not touched.
"""
import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest

from block_quantized_weight_q4_gb300 import inputs
from conftest import read_cases, read_rows

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "qmv_oracle.c")

MUTANTS = {
    "nibble_halves_swapped": ("(j < 16) ? (byte & 0x0f) : (byte >> 4)", "(j < 16) ? (byte >> 4) : (byte & 0x0f)"),
    "level_offset_dropped": ("return nibble - 8;", "return nibble;"),
    "level_offset_off_by_one": ("return nibble - 8;", "return nibble - 7;"),
    "scale_index_transposed": ("int64_t idx = r * (cols / 32) + k;", "int64_t idx = k * rows + r;"),
    "pad_to_32": ("return ((n + 63) / 64) * 64;", "return ((n + 31) / 32) * 32;"),
    "q4_row_stride": ("W[r * (cols / 2) + 16 * k + (j % 16)]", "W[r * cols + 16 * k + (j % 16)]"),
    "q4_byte_in_block": ("W[r * (cols / 2) + 16 * k + (j % 16)]", "W[r * (cols / 2) + 16 * k + j / 2]"),
    "q8_unsigned": ("return (int)(int8_t)W[r * cols + c];", "return (int)W[r * cols + c];"),
    "f16_bias": ("mag = ldexp((double)(1024 + m), e - 25);", "mag = ldexp((double)(1024 + m), e - 24);"),
    "f16_subnormal": ("mag = ldexp((double)m, -24);", "mag = ldexp((double)m, -23);"),
    "f16_implicit_bit": ("mag = ldexp((double)(1024 + m), e - 25);", "mag = ldexp((double)m, e - 25);"),
    "x_transposed": ("((const float *)x)[b * cols + c]", "((const float *)x)[c * cols + b]"),
    "absref_not_abs": ("acc_abs += fabs(t);", "acc_abs += t;"),
    "validate_wrong_byte": ("if (W[i] == 0x80)", "if (W[i] == 0x7f)"),
    "q8_size_halved": ("int64_t q = (wtype == ORACLE_Q8_0) ? n : n / 2;", "int64_t q = n / 2;"),
    "f16_scale_size": ("int64_t dsz = nscales * (scale_f16 ? 2 : 4);", "int64_t dsz = nscales * 4;"),
    "f16_scale_read_as_f32": ("if (scale_f16) {\n        const uint8_t *p = W + off + 2 * idx;",
                              "if (0) {\n        const uint8_t *p = W + off + 2 * idx;"),
    "qx_x_scale_of_vector_0": ("oracle_scale(xq, ORACLE_Q8_0, 0, batch, cols, b, k)",
                               "oracle_scale(xq, ORACLE_Q8_0, 0, batch, cols, 0, k)"),
    "qx_x_quants_of_vector_0": ("oracle_level(xq, ORACLE_Q8_0, cols, b, 32 * k + j)",
                                "oracle_level(xq, ORACLE_Q8_0, cols, 0, 32 * k + j)"),
    "qx_block_scale_dropped": ("acc += s * (double)isum;", "acc += (double)isum;"),
    "qx_x_scale_byte_order": ("xq[off + 4 * idx + i] = (uint8_t)((bits >> (8 * i)) & 0xff);",
                              "xq[off + 4 * idx + i] = (uint8_t)((bits >> (8 * (3 - i))) & 0xff);"),
    "q8_rule_without_half": ("float u = t + copysignf(0.5f, x[j]);", "float u = t;"),
    "fit_den_unweighted_level": ("den += (t * (float)l[j]) * (float)l[j];", "den += t * (float)l[j];"),
    "fit_clamp_high_8": ("if (r > 7.0f) r = 7.0f;", "if (r > 8.0f) r = 8.0f;"),
    "fit_candidates_from_minus_7": ("const float L = (float)(-(60 + 2 * k)) / 10.0f;",
                                    "const float L = (float)(-(70 + 2 * k)) / 10.0f;"),
    "glu_silu_sign": ("if (act == 0) return g / (1.0 + exp(-g));", "if (act == 0) return g / (1.0 + exp(g));"),
    "glu_gelu_cubic": ("(g + 0.044715 * g * g * g)", "(g + 0.044715 * g * g)"),
    "glu_up_dropped": ("glu_act(act, (double)gate[(int64_t)b * cols + c]) * (double)up[(int64_t)b * cols + c]",
                       "glu_act(act, (double)gate[(int64_t)b * cols + c])"),
    "gguf_record_without_d": ("int64_t block_bytes = 2 + qb;", "int64_t block_bytes = qb;"),
    "gguf_d_bytes_swapped": ("W[off + 2 * idx] = rec[0];\n            W[off + 2 * idx + 1] = rec[1];",
                             "W[off + 2 * idx] = rec[1];\n            W[off + 2 * idx + 1] = rec[0];"),
    "gguf_quants_at_record_start": ("W[idx * qb + j] = rec[2 + j];", "W[idx * qb + j] = rec[j];"),
    "glu_values_up_dropped": ("for (int64_t i = 0; i < n; i++) h[i] = glu_act(act, gate[i]) * up[i];",
                              "for (int64_t i = 0; i < n; i++) h[i] = glu_act(act, gate[i]);"),
    "glu_values_gate_for_up": ("for (int64_t i = 0; i < n; i++) h[i] = glu_act(act, gate[i]) * up[i];",
                               "for (int64_t i = 0; i < n; i++) h[i] = glu_act(act, gate[i]) * gate[i];"),
    "gguf_q8_block_32": ("int64_t block_bytes = (wtype == ORACLE_Q8_0) ? 34 : 18;",
                         "int64_t block_bytes = (wtype == ORACLE_Q8_0) ? 32 : 18;"),
}


class Orc:
    """Minimal ctypes view of one build of the oracle source."""

    def __init__(self, so):
        lib = ctypes.CDLL(so)
        i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
        lib.oracle_weight_bytes.restype = i64
        lib.oracle_weight_bytes.argtypes = [i32, i32, i64, i64]
        lib.oracle_f16_value.restype = ctypes.c_float
        lib.oracle_f16_value.argtypes = [ctypes.c_uint16]
        lib.oracle_dequant.restype = i32
        lib.oracle_dequant.argtypes = [i32, i32, i64, i64, vp, vp]
        lib.oracle_matvec.restype = i32
        lib.oracle_matvec.argtypes = [i32, i32, i64, i64, vp, vp, i32, i32, vp, vp]
        lib.oracle_validate.restype = i32
        lib.oracle_validate.argtypes = [i32, i32, i64, i64, vp]
        lib.oracle_quantize_x.restype = i32
        lib.oracle_quantize_x.argtypes = [i32, i64, i64, vp, vp]
        lib.oracle_matvec_qx.restype = i32
        lib.oracle_matvec_qx.argtypes = [i32, i32, i64, i64, vp, vp, i32, vp, vp]
        lib.oracle_gguf_bytes.restype = i64
        lib.oracle_gguf_bytes.argtypes = [i32, i64, i64]
        lib.oracle_quantize_q4_fit.restype = i32
        lib.oracle_quantize_q4_fit.argtypes = [i32, i64, i64, vp, vp]
        lib.oracle_quantize.restype = i32
        lib.oracle_quantize.argtypes = [i32, i32, i64, i64, vp, vp]
        lib.oracle_matvec_glu.restype = i32
        lib.oracle_matvec_glu.argtypes = [i32, i32, i64, i64, vp, i32, vp, vp, i32, vp, vp]
        lib.oracle_glu.restype = i32
        lib.oracle_glu.argtypes = [i32, i64, vp, vp, vp]
        lib.oracle_gguf_to_mlb.restype = i32
        lib.oracle_gguf_to_mlb.argtypes = [i32, i64, i64, vp, vp]
        self.lib = lib

    def dequant(self, W, wt, sf, rows, cols):
        out = np.empty((rows, cols), np.float32)
        assert self.lib.oracle_dequant(wt, sf, rows, cols, W.ctypes.data, out.ctypes.data) == 0
        return out

    def matvec(self, W, wt, sf, rows, cols, x):
        x = np.ascontiguousarray(x)
        y = np.empty((x.shape[0], rows))
        a = np.empty_like(y)
        assert self.lib.oracle_matvec(wt, sf, rows, cols, W.ctypes.data, x.ctypes.data,
                                      int(x.dtype == np.uint16), x.shape[0], y.ctypes.data, a.ctypes.data) == 0
        return y, a

    def quantize_x(self, x):
        batch, cols = x.shape
        # room for whatever layout a mutant computes (a mutated size may undercount)
        xq = np.zeros(4 * batch * cols + 1024, np.uint8)
        assert self.lib.oracle_quantize_x(0, batch, cols, x.ctypes.data, xq.ctypes.data) == 0
        return xq

    def matvec_qx(self, W, wt, sf, rows, cols, xq, batch):
        y = np.empty((batch, rows))
        a = np.empty_like(y)
        assert self.lib.oracle_matvec_qx(wt, sf, rows, cols, W.ctypes.data, xq.ctypes.data, batch,
                                         y.ctypes.data, a.ctypes.data) == 0
        return y, a


def pin_checks(o):
    """Yields (name, passed) for the page-derived checks."""
    for wt, sf, rows, cols, expect, *_ in read_rows("sizes_worked_examples.txt"):
        yield "size", o.lib.oracle_weight_bytes(int(wt), int(sf), int(rows), int(cols)) == int(expect)
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = codes.view(np.float16).astype(np.float32)
    got = np.array([o.lib.oracle_f16_value(int(c)) for c in codes], np.float32)
    fin = ~np.isnan(ref)
    yield "f16", bool(np.array_equal(got[fin], ref[fin]))
    for case in read_cases("hand_blocks.txt"):
        wt, sf = int(case["wtype"][0]), int(case["scale_f16"][0])
        qb = np.array([int(b, 16) for b in case["bytes"]], np.uint8)
        d = (np.array([int(case["scale_code"][0], 16)], np.uint16) if sf
             else np.array([float(case["scale"][0])], np.float32).view(np.uint32))
        W = inputs.assemble(wt, sf, 1, 32, qb, d)
        expect = np.array([float(v) for v in case["weights"]], np.float32)
        yield "hand", bool(np.array_equal(o.dequant(W, wt, sf, 1, 32)[0], expect))
    # scale index / row addressing: w[r][c] = 2^(3r + c//32)
    rows, cols = 3, 96
    q = np.full(rows * cols // 2, 0x99, np.uint8)
    dv = np.array([2.0 ** (3 * r + k) for r in range(rows) for k in range(3)], np.float32)
    for sf in (0, 1):
        codes2 = dv.astype(np.float16).view(np.uint16) if sf else dv.view(np.uint32)
        W = inputs.assemble(2, sf, rows, cols, q, codes2)
        exp = np.array([[2.0 ** (3 * r + c // 32) for c in range(cols)] for r in range(rows)], np.float32)
        yield "scale_index", bool(np.array_equal(o.dequant(W, 2, sf, rows, cols), exp))
    # one-hot product on random Q4_0 / Q8_0 matrices vs the dequantized columns
    for wt in (1, 2):
        m = inputs.make_matrix(wt, 0, 5, 96, seed=3)
        deq = o.dequant(m.W, wt, 0, 5, 96)
        y, a = o.matvec(m.W, wt, 0, 5, 96, np.eye(96, dtype=np.float32))
        yield "one_hot", bool(np.array_equal(y.astype(np.float32), deq.T) and np.array_equal(a, np.abs(y)))
    # the Q8 -128 check
    m = inputs.make_matrix(1, 0, 4, 64, seed=1)
    W = m.W.copy()
    W[77] = 0x80
    yield "validate", o.lib.oracle_validate(1, 0, 4, 64, W.ctypes.data) == 2 and \
        o.lib.oracle_validate(1, 0, 4, 64, m.W.ctypes.data) == 0
    # activation-quantized product: activations k * 2^e (one element of each block at +-127)
    # quantize to k and 2^e exactly, so the product equals the plain one (exact sums)
    rng = np.random.default_rng(5)
    batch, cols = 2, 96
    k = rng.integers(-127, 128, size=(batch, 3, 32))
    k[:, :, 7] = 127
    x = (k * np.exp2(rng.integers(-3, 1, size=(batch, 3)))[:, :, None]).reshape(batch, cols).astype(np.float32)
    xq = o.quantize_x(x)
    yield "qx_quants", bool(np.array_equal(xq[:batch * cols].view(np.int8), k.reshape(-1).astype(np.int8)))
    for wt in (1, 2):
        m = inputs.make_matrix(wt, 1, 4, cols, seed=8 + wt)
        yq, _ = o.matvec_qx(m.W, wt, 1, 4, cols, xq, batch)
        y, _ = o.matvec(m.W, wt, 1, 4, cols, x)
        yield "qx_exact", bool(np.array_equal(yq, y))
    # a hand block: levels +1, d_w = 0.5, x = [127, -63.5, 0...] -> q_x = [127, -64], y = 31.5
    W = inputs.assemble(2, 0, 1, 32, np.full(16, 0x99, np.uint8), np.array([0.5], np.float32).view(np.uint32))
    xh = np.zeros((1, 32), np.float32)
    xh[0, 0], xh[0, 1] = 127.0, -63.5
    yield "qx_hand", o.matvec_qx(W, 2, 0, 1, 32, o.quantize_x(xh), 1)[0][0, 0] == 31.5
    # GGUF: the page's tensor sizes, and records with d = 2^(3r + k), levels +1
    for wt, rows, cols, expect, *_ in read_rows("gguf_sizes.txt"):
        yield "gguf_size", o.lib.oracle_gguf_bytes(int(wt), int(rows), int(cols)) == int(expect)
    for wt in (1, 2):
        qb = 32 if wt == 1 else 16
        recs = []
        for r in range(3):
            for k in range(3):
                code = int(np.array([2.0 ** (3 * r + k)], np.float16).view(np.uint16)[0])
                recs += [code & 0xFF, code >> 8] + [1 if wt == 1 else 0x99] * qb
        g = np.array(recs + [0] * 256, np.uint8)       # slack: a mutated record size stays in bounds
        Wg = np.zeros(4096, np.uint8)
        assert o.lib.oracle_gguf_to_mlb(wt, 3, 96, g.ctypes.data, Wg.ctypes.data) == 0
        exp = np.array([[2.0 ** (3 * r + c // 32) for c in range(96)] for r in range(3)], np.float32)
        yield "gguf_records", bool(np.array_equal(o.dequant(Wg, wt, 1, 3, 96), exp))
    # Q4_0 best fit: exact blocks come back exactly; never worse than the round rule (weighted)
    rng = np.random.default_rng(14)
    lv = rng.integers(-7, 8, (4, 3, 32))
    lv[:, :, 5] = -8
    cc = np.exp2(rng.integers(-6, 2, (4, 3))).astype(np.float32)
    xe = np.ascontiguousarray((lv * cc[:, :, None]).reshape(4, 96).astype(np.float32))
    Wf = np.zeros(4096, np.uint8)
    o.lib.oracle_quantize_q4_fit(0, 4, 96, xe.ctypes.data, Wf.ctypes.data)
    yield "fit_exact", bool(np.array_equal(o.dequant(Wf, 2, 0, 4, 96), xe))
    lv6 = rng.integers(-5, 6, (4, 3, 32))
    lv6[:, :, 9] = -6
    x6 = np.ascontiguousarray((lv6 * cc[:, :, None]).reshape(4, 96).astype(np.float32))
    o.lib.oracle_quantize_q4_fit(0, 4, 96, x6.ctypes.data, Wf.ctypes.data)
    yield "fit_exact_at_minus_6", bool(np.array_equal(o.dequant(Wf, 2, 0, 4, 96), x6))
    xr = np.ascontiguousarray((rng.standard_normal((8, 96)) * 3).astype(np.float32))
    Wr = np.zeros(4096, np.uint8)
    o.lib.oracle_quantize_q4_fit(0, 8, 96, xr.ctypes.data, Wf.ctypes.data)
    o.lib.oracle_quantize(2, 0, 8, 96, xr.ctypes.data, Wr.ctypes.data)
    df, dr = o.dequant(Wf, 2, 0, 8, 96).astype(np.float64), o.dequant(Wr, 2, 0, 8, 96).astype(np.float64)
    xd = xr.astype(np.float64)
    ef = (xd ** 2 * (xd - df) ** 2).reshape(8, 3, 32).sum(axis=2)
    er = (xd ** 2 * (xd - dr) ** 2).reshape(8, 3, 32).sum(axis=2)
    yield "fit_vs_round", bool(np.all(ef <= er * (1 + 1e-5) + 1e-30) and np.sum(ef < er * (1 - 1e-3)) > 12)
    # gated activation: act(g) - act(-g) = g turns two gated products into the plain one, and a
    # one-hot weight reads SiLU(ln 3) = 3/4 ln 3, GELU-tanh at a known point = 3g/4
    m = inputs.make_matrix(2, 1, 4, 64, seed=12)
    rng = np.random.default_rng(13)
    g = np.ascontiguousarray((rng.integers(-6, 7, (1, 64)) / 4).astype(np.float32))
    u = np.ascontiguousarray((rng.integers(-8, 9, (1, 64)) / 8).astype(np.float32))
    ng = np.ascontiguousarray(-g)
    for act in (0, 1):
        yp, yn, a = (np.empty((1, 4)) for _ in range(3))
        o.lib.oracle_matvec_glu(2, 1, 4, 64, m.W.ctypes.data, act, g.ctypes.data, u.ctypes.data, 1,
                                yp.ctypes.data, a.ctypes.data)
        o.lib.oracle_matvec_glu(2, 1, 4, 64, m.W.ctypes.data, act, ng.ctypes.data, u.ctypes.data, 1,
                                yn.ctypes.data, a.ctypes.data)
        y, a = o.matvec(m.W, 2, 1, 4, 64, np.ascontiguousarray((g * u).astype(np.float32)))
        yield "glu_odd", bool(np.all(np.abs((yp - yn) - y) <= 1e-12 * a + 1e-300))
    qh = np.full(16, 0x88, np.uint8)
    qh[0] = 0x89
    Wh = inputs.assemble(2, 0, 1, 32, qh, np.array([1.0], np.float32).view(np.uint32))
    uh = np.zeros((1, 32), np.float32)
    uh[0, 0] = 1.0
    gh = np.zeros((1, 32), np.float32)
    gh[0, 0] = np.float32(np.log(3.0))
    yv, av = np.empty((1, 1)), np.empty((1, 1))
    o.lib.oracle_matvec_glu(2, 0, 1, 32, Wh.ctypes.data, 0, gh.ctypes.data, uh.ctypes.data, 1, yv.ctypes.data,
                            av.ctypes.data)
    yield "glu_silu_ln3", abs(yv[0, 0] - 0.75 * float(gh[0, 0])) < 1e-7
    # GELU-tanh where its tanh is 1/2 (the point found by bisection): GELU(g) = 3g/4
    kk, target = np.sqrt(2 / np.pi), np.arctanh(0.5)
    lo, hi = 0.0, 2.0
    for _ in range(200):
        mid = (lo + hi) / 2
        lo, hi = (mid, hi) if kk * (mid + 0.044715 * mid ** 3) < target else (lo, mid)
    gh[0, 0] = np.float32(lo)
    o.lib.oracle_matvec_glu(2, 0, 1, 32, Wh.ctypes.data, 1, gh.ctypes.data, uh.ctypes.data, 1, yv.ctypes.data,
                            av.ctypes.data)
    yield "glu_gelu_value", abs(yv[0, 0] - 0.75 * float(gh[0, 0])) < 1e-6
    # h = act(g) * u value by value: the odd part gives g * u
    gv = np.ascontiguousarray(rng.standard_normal(50) * 3)
    uv = np.ascontiguousarray(rng.standard_normal(50))
    for act in (0, 1):
        hp, hn = np.empty(50), np.empty(50)
        o.lib.oracle_glu(act, 50, gv.ctypes.data, uv.ctypes.data, hp.ctypes.data)
        ngv = np.ascontiguousarray(-gv)
        o.lib.oracle_glu(act, 50, ngv.ctypes.data, uv.ctypes.data, hn.ctypes.data)
        yield "glu_values_odd", bool(np.all(np.abs((hp - hn) - gv * uv) <= 1e-14 * (np.abs(gv * uv) + 1)))


def build_variant(tmp, name, text):
    c = os.path.join(tmp, f"{name}.c")
    so = os.path.join(tmp, f"{name}.so")
    with open(c, "w") as f:
        f.write(text)
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", "-o", so, c, "-lm"],
                   check=True)
    return Orc(so)


@pytest.fixture(scope="module")
def tmpdir():
    with tempfile.TemporaryDirectory() as d:
        yield d


def test_unmodified_copy_passes_all_pins(tmpdir):
    o = build_variant(tmpdir, "orig", open(SRC).read())
    failed = [n for n, ok in pin_checks(o) if not ok]
    assert not failed, failed


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmpdir, name):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) >= 1, f"mutation site not found: {old}"
    o = build_variant(tmpdir, name, text.replace(old, new))
    results = list(pin_checks(o))
    assert any(not ok for _, ok in results), f"mutant {name} passed every pin"
