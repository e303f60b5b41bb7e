"""Plain CPU oracle for block-quantized (Q8_0 / Q4_0) weight matrices.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may use this package; the CUDA library and its Python binding never
import it.  The arithmetic lives in ``qmv_oracle.c`` (plain C, one weight at a time,
products in double precision), written from the Krafla ".mlb model format v1" page:
sections "Body" (two arrays q then d, each padded to 64 bytes), "Q8_0", "Q4_0",
"Quantization rule" and "Validation done by the loader".  This module only compiles
that file with gcc and marshals numpy arrays to it.

Parity unpinned: the writer-only corner readings (an f16 Q8_0 scale that rounds to
zero, the all-zero Q4_0 block, ties of the largest magnitude); everything else is
pinned by ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmv_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle.so")

Q8_0 = 1
Q4_0 = 2
OK = 0
E_FORMAT = 2
E_SHAPE = 3

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    lib.oracle_weight_bytes.restype = i64
    lib.oracle_weight_bytes.argtypes = [i32, i32, i64, i64]
    lib.oracle_scale_offset.restype = i64
    lib.oracle_scale_offset.argtypes = [i32, i32, i64, i64]
    lib.oracle_f16_value.restype = ctypes.c_float
    lib.oracle_f16_value.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_bits_rne.restype = ctypes.c_uint16
    lib.oracle_f16_bits_rne.argtypes = [ctypes.c_float]
    lib.oracle_bf16_value.restype = ctypes.c_float
    lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
    lib.oracle_level.restype = i32
    lib.oracle_level.argtypes = [vp, i32, i64, i64, i64]
    lib.oracle_scale.restype = ctypes.c_float
    lib.oracle_scale.argtypes = [vp, i32, i32, i64, i64, i64, i64]
    lib.oracle_dequant.restype = i32
    lib.oracle_dequant.argtypes = [i32, i32, i64, i64, vp, vp]
    lib.oracle_matvec.restype = i32
    lib.oracle_matvec.argtypes = [i32, i32, i64, i64, vp, vp, i32, i32, vp, vp]
    lib.oracle_matvec_rows.restype = i32
    lib.oracle_matvec_rows.argtypes = [i32, i32, i64, i64, vp, vp, i32, i32, vp, i64, vp, vp]
    lib.oracle_validate.restype = i32
    lib.oracle_validate.argtypes = [i32, i32, i64, i64, vp]
    lib.oracle_quant_q8_block.restype = i32
    lib.oracle_quant_q8_block.argtypes = [vp, i32, vp, vp]
    lib.oracle_quant_q4_round_block.restype = i32
    lib.oracle_quant_q4_round_block.argtypes = [vp, i32, vp, vp]
    lib.oracle_quantize.restype = i32
    lib.oracle_quantize.argtypes = [i32, i32, i64, i64, vp, vp]
    lib.oracle_quantize_x.restype = i32
    lib.oracle_quantize_x.argtypes = [i32, i64, i64, vp, vp]
    lib.oracle_matvec_qx.restype = i32
    lib.oracle_matvec_qx.argtypes = [i32, i32, i64, i64, vp, vp, i32, vp, vp]
    lib.oracle_glu.restype = i32
    lib.oracle_glu.argtypes = [i32, i64, vp, vp, vp]
    lib.oracle_matvec_glu.restype = i32
    lib.oracle_matvec_glu.argtypes = [i32, i32, i64, i64, vp, i32, vp, vp, i32, vp, vp]
    lib.oracle_quant_q4_fit_block.restype = i32
    lib.oracle_quant_q4_fit_block.argtypes = [vp, i32, vp, vp]
    lib.oracle_quantize_q4_fit.restype = i32
    lib.oracle_quantize_q4_fit.argtypes = [i32, i64, i64, vp, vp]
    lib.oracle_gguf_bytes.restype = i64
    lib.oracle_gguf_bytes.argtypes = [i32, i64, i64]
    lib.oracle_gguf_to_mlb.restype = i32
    lib.oracle_gguf_to_mlb.argtypes = [i32, i64, i64, vp, vp]
    _lib = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def weight_bytes(wtype: int, scale_f16: int, rows: int, cols: int) -> int:
    return int(_load().oracle_weight_bytes(wtype, scale_f16, rows, cols))


def scale_offset(wtype: int, scale_f16: int, rows: int, cols: int) -> int:
    return int(_load().oracle_scale_offset(wtype, scale_f16, rows, cols))


def f16_value(code: int) -> float:
    return float(_load().oracle_f16_value(code))


def f16_bits_rne(v: float) -> int:
    return int(_load().oracle_f16_bits_rne(v))


def bf16_value(code: int) -> float:
    return float(_load().oracle_bf16_value(code))


def level(W: np.ndarray, wtype: int, cols: int, r: int, c: int) -> int:
    return int(_load().oracle_level(_ptr(W), wtype, cols, r, c))


def scale(W: np.ndarray, wtype: int, scale_f16: int, rows: int, cols: int, r: int, k: int) -> float:
    return float(_load().oracle_scale(_ptr(W), wtype, scale_f16, rows, cols, r, k))


def dequant(W: np.ndarray, wtype: int, scale_f16: int, rows: int, cols: int) -> np.ndarray:
    """float32 rows x cols, w = level * d (one float32 multiply)."""
    out = np.empty((rows, cols), dtype=np.float32)
    st = _load().oracle_dequant(wtype, scale_f16, rows, cols, _ptr(W), _ptr(out))
    if st != OK:
        raise ValueError(f"oracle_dequant status {st}")
    return out


def _x_args(x: np.ndarray):
    if x.dtype == np.float32:
        return 0
    if x.dtype == np.uint16:  # bfloat16 codes
        return 1
    raise TypeError("x must be float32 or uint16 bfloat16 codes")


def matvec(W: np.ndarray, wtype: int, scale_f16: int, rows: int, cols: int, x: np.ndarray):
    """y (batch x rows, float64) and absref = sum |w x| (same shape) for x (batch x cols)."""
    x = np.ascontiguousarray(x)
    batch = x.shape[0]
    assert x.shape == (batch, cols)
    y = np.empty((batch, rows), dtype=np.float64)
    a = np.empty((batch, rows), dtype=np.float64)
    st = _load().oracle_matvec(wtype, scale_f16, rows, cols, _ptr(W), _ptr(x), _x_args(x),
                               batch, _ptr(y), _ptr(a))
    if st != OK:
        raise ValueError(f"oracle_matvec status {st}")
    return y, a


def matvec_rows(W: np.ndarray, wtype: int, scale_f16: int, rows: int, cols: int,
                x: np.ndarray, row_ids):
    """Like matvec but only for the listed rows: returns (batch x len(row_ids)) arrays."""
    x = np.ascontiguousarray(x)
    batch = x.shape[0]
    ids = np.ascontiguousarray(np.asarray(row_ids, dtype=np.int64))
    y = np.empty((batch, ids.size), dtype=np.float64)
    a = np.empty((batch, ids.size), dtype=np.float64)
    st = _load().oracle_matvec_rows(wtype, scale_f16, rows, cols, _ptr(W), _ptr(x), _x_args(x),
                                    batch, _ptr(ids), ids.size, _ptr(y), _ptr(a))
    if st != OK:
        raise ValueError(f"oracle_matvec_rows status {st}")
    return y, a


def validate(W: np.ndarray, wtype: int, scale_f16: int, rows: int, cols: int) -> int:
    return int(_load().oracle_validate(wtype, scale_f16, rows, cols, _ptr(W)))


def quant_q8_block(x: np.ndarray, scale_f16: int):
    """(status, q int8[32], stored scale bits) for one block by the Q8_0 rule."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.size == 32
    q = np.zeros(32, dtype=np.int8)
    bits = np.zeros(1, dtype=np.uint32)
    st = _load().oracle_quant_q8_block(_ptr(x), scale_f16, _ptr(q), _ptr(bits))
    return int(st), q, int(bits[0])


def quant_q4_round_block(x: np.ndarray, scale_f16: int):
    """(status, 16 packed bytes, stored scale bits) for one block by the Q4_0 round rule."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.size == 32
    qs = np.zeros(16, dtype=np.uint8)
    bits = np.zeros(1, dtype=np.uint32)
    st = _load().oracle_quant_q4_round_block(_ptr(x), scale_f16, _ptr(qs), _ptr(bits))
    return int(st), qs, int(bits[0])


def quantize(src: np.ndarray, wtype: int, scale_f16: int) -> np.ndarray:
    """Matrix bytes (two-array layout) from float32 rows x cols by the writer rules."""
    src = np.ascontiguousarray(src, dtype=np.float32)
    rows, cols = src.shape
    n = weight_bytes(wtype, scale_f16, rows, cols)
    if n < 0:
        raise ValueError("bad shape")
    W = np.zeros(n, dtype=np.uint8)
    st = _load().oracle_quantize(wtype, scale_f16, rows, cols, _ptr(src), _ptr(W))
    if st != OK:
        raise ValueError(f"oracle_quantize status {st}")
    return W


def quantize_x(x: np.ndarray) -> np.ndarray:
    """Activations (batch x cols, float32 or uint16 bfloat16 codes) by the Q8_0 rule into the
    Q8_0 / f32-scale two-array image of a batch x cols matrix (uint8)."""
    x = np.ascontiguousarray(x)
    batch, cols = x.shape
    n = weight_bytes(Q8_0, 0, batch, cols)
    if n < 0:
        raise ValueError("bad shape")
    xq = np.zeros(n, dtype=np.uint8)
    st = _load().oracle_quantize_x(_x_args(x), batch, cols, _ptr(x), _ptr(xq))
    if st != OK:
        raise ValueError(f"oracle_quantize_x status {st}")
    return xq


def matvec_qx(W: np.ndarray, wtype: int, scale_f16: int, rows: int, cols: int, xq: np.ndarray, batch: int):
    """Activation-quantized product: y (batch x rows, float64) = per block d_w d_x times the exact
    integer dot of weight levels and activation quants, and absref (same shape)."""
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    assert xq.size >= weight_bytes(Q8_0, 0, batch, cols)
    y = np.empty((batch, rows), dtype=np.float64)
    a = np.empty((batch, rows), dtype=np.float64)
    st = _load().oracle_matvec_qx(wtype, scale_f16, rows, cols, _ptr(W), _ptr(xq), batch, _ptr(y), _ptr(a))
    if st != OK:
        raise ValueError(f"oracle_matvec_qx status {st}")
    return y, a


def gguf_bytes(wtype: int, rows: int, cols: int) -> int:
    """Bytes of a rows x cols tensor in GGUF interleaved blocks (18 / 34 bytes per block)."""
    return int(_load().oracle_gguf_bytes(wtype, rows, cols))


def gguf_to_mlb(gguf: np.ndarray, wtype: int, rows: int, cols: int) -> np.ndarray:
    """The two-array image (f16 scales) of a tensor given in GGUF interleaved blocks."""
    gguf = np.ascontiguousarray(gguf, dtype=np.uint8)
    assert gguf.size >= gguf_bytes(wtype, rows, cols)
    W = np.zeros(weight_bytes(wtype, 1, rows, cols), dtype=np.uint8)
    st = _load().oracle_gguf_to_mlb(wtype, rows, cols, _ptr(gguf), _ptr(W))
    if st != OK:
        raise ValueError(f"oracle_gguf_to_mlb status {st}")
    return W


def matvec_glu(W: np.ndarray, wtype: int, scale_f16: int, rows: int, cols: int, act: int,
               gate: np.ndarray, up: np.ndarray):
    """y = W (act(gate) * up) for batch x cols float32 gate and up (act 0 SiLU, 1 GELU-tanh),
    float64 y and absref (batch x rows)."""
    gate = np.ascontiguousarray(gate, dtype=np.float32)
    up = np.ascontiguousarray(up, dtype=np.float32)
    batch = gate.shape[0]
    assert gate.shape == up.shape == (batch, cols)
    y = np.empty((batch, rows), dtype=np.float64)
    a = np.empty((batch, rows), dtype=np.float64)
    st = _load().oracle_matvec_glu(wtype, scale_f16, rows, cols, _ptr(W), act, _ptr(gate), _ptr(up), batch,
                                   _ptr(y), _ptr(a))
    if st != OK:
        raise ValueError(f"oracle_matvec_glu status {st}")
    return y, a


def glu(act: int, gate: np.ndarray, up: np.ndarray) -> np.ndarray:
    """h = act(gate) * up (act 0 SiLU, 1 GELU-tanh) for float64 arrays of one shape, in float64."""
    gate = np.ascontiguousarray(gate, dtype=np.float64)
    up = np.ascontiguousarray(up, dtype=np.float64)
    assert gate.shape == up.shape
    h = np.empty_like(gate)
    st = _load().oracle_glu(act, gate.size, _ptr(gate), _ptr(up), _ptr(h))
    if st != OK:
        raise ValueError(f"oracle_glu status {st}")
    return h


def quant_q4_fit_block(x: np.ndarray, scale_f16: int):
    """(status, 16 packed bytes, stored scale bits) for one block by the best-fit rule."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    assert x.size == 32
    qs = np.zeros(16, dtype=np.uint8)
    bits = ctypes.c_uint32(0)
    st = _load().oracle_quant_q4_fit_block(_ptr(x), scale_f16, _ptr(qs), ctypes.addressof(bits))
    return st, qs, int(bits.value)


def quantize_q4_fit(src: np.ndarray, scale_f16: int) -> np.ndarray:
    """Q4_0 matrix bytes (two-array layout) from float32 rows x cols by the best-fit rule."""
    src = np.ascontiguousarray(src, dtype=np.float32)
    rows, cols = src.shape
    W = np.zeros(weight_bytes(Q4_0, scale_f16, rows, cols), dtype=np.uint8)
    st = _load().oracle_quantize_q4_fit(scale_f16, rows, cols, _ptr(src), _ptr(W))
    if st != OK:
        raise ValueError(f"oracle_quantize_q4_fit status {st}")
    return W
