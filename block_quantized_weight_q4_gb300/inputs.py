"""Seeded synthetic inputs for the quantized matrix-vector product.

This module only draws random numbers and lays bytes out; it holds none of the
method's arithmetic (no decoding, no products).  Both the CUDA path's tests and the
CPU oracle consume what it makes, so neither side's arithmetic leaks into the other.

Byte layout of a matrix image (Krafla ".mlb model format v1", section "Body"): the q
array, zero padding up to the next multiple of 64 bytes, then the d array.  The
optional padding after d is left out unless asked for, so that a reader that strays
past the end of d is caught by the bounds of the buffer.

Workloads (the shapes the benchmark and the full-size tests use):
  q8_256       Q8_0 256 x 256, f32 scales, x f32, batch 1, seed 0
  q4_4096      Q4_0 4096 x 4096, f16 scales, x bf16, batch 1
  llama7b      Llama-7B-shaped decode layer (wq, wk, wv, wo, w1, w3, w2), Q4_0 f16, batch 1
  mixed_qwen   q8_mask = 2: Q4_0 body of one dim-1024 layer + Q8_0 classifier
               151936 x 1024, f32 scales, batch 1 and 8
  prefill      Q4_0 f16, W 14336 x 4096 and 4096 x 14336, X bf16 of 16, 64, 128 tokens
Matrix i of a workload (in listed order) is drawn with seed i and its activations
with seed 1000 + i, except q8_256 whose matrix and activations use seed 0.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

Q8_0 = 1
Q4_0 = 2

# q8_mask class bits (the header's mask has a bit for each class of matrix)
CLASS_TOK_EMB = 1
CLASS_WCLS = 2
CLASS_WQ_WK = 4
CLASS_WV = 8
CLASS_WO = 16
CLASS_W1_W3 = 32
CLASS_W2 = 64


@dataclass
class MatrixSpec:
    name: str
    rows: int
    cols: int
    wtype: int
    scale_f16: int
    cls: int = 0  # q8_mask class bit, 0 when not part of a model


@dataclass
class Workload:
    name: str
    matrices: list
    batches: tuple
    x_bf16: bool
    q8_mask: int = 0
    file_wtype: int = Q4_0
    extra_x_f32: bool = False  # also exercised with f32 activations
    notes: str = ""
    seeds: list = field(default_factory=list)


def _llama7b():
    s = [("wq", 4096, 4096, CLASS_WQ_WK), ("wk", 1024, 4096, CLASS_WQ_WK),
         ("wv", 1024, 4096, CLASS_WV), ("wo", 4096, 4096, CLASS_WO),
         ("w1", 11008, 4096, CLASS_W1_W3), ("w3", 11008, 4096, CLASS_W1_W3),
         ("w2", 4096, 11008, CLASS_W2)]
    return [MatrixSpec(n, r, c, Q4_0, 1, cl) for n, r, c, cl in s]


def _mixed_body():
    s = [("wq", 2048, 1024, CLASS_WQ_WK), ("wk", 1024, 1024, CLASS_WQ_WK),
         ("wv", 1024, 1024, CLASS_WV), ("wo", 1024, 2048, CLASS_WO),
         ("w1", 3072, 1024, CLASS_W1_W3), ("w3", 3072, 1024, CLASS_W1_W3),
         ("w2", 1024, 3072, CLASS_W2)]
    return [MatrixSpec(n, r, c, Q4_0, 0, cl) for n, r, c, cl in s]


WORKLOADS = {
    "q8_256": Workload("q8_256", [MatrixSpec("w", 256, 256, Q8_0, 0)], (1,), x_bf16=False),
    "q4_4096": Workload("q4_4096", [MatrixSpec("w", 4096, 4096, Q4_0, 1)], (1,), x_bf16=True),
    "llama7b": Workload("llama7b", _llama7b(), (1,), x_bf16=True),
    "mixed_qwen": Workload("mixed_qwen",
                           _mixed_body() + [MatrixSpec("wcls", 151936, 1024, Q8_0, 0, CLASS_WCLS)],
                           (1, 8), x_bf16=True, q8_mask=CLASS_WCLS, file_wtype=Q4_0,
                           extra_x_f32=True),
    "prefill": Workload("prefill", [MatrixSpec("w_up", 14336, 4096, Q4_0, 1),
                                    MatrixSpec("w_down", 4096, 14336, Q4_0, 1)],
                        (16, 64, 128), x_bf16=True),
}


def matrix_seed(workload: str, i: int) -> int:
    return 0 if workload == "q8_256" else i


def x_seed(workload: str, i: int) -> int:
    return 0 if workload == "q8_256" else 1000 + i


def array_offsets(wtype: int, scale_f16: int, rows: int, cols: int):
    """(q bytes, offset of d, d bytes) of the byte image: q, zeros to 64, d."""
    n = rows * cols
    q_bytes = n if wtype == Q8_0 else n // 2
    d_off = -(-q_bytes // 64) * 64
    d_bytes = (n // 32) * (2 if scale_f16 else 4)
    return q_bytes, d_off, d_bytes


@dataclass
class Matrix:
    wtype: int
    scale_f16: int
    rows: int
    cols: int
    W: np.ndarray       # uint8 byte image
    q: np.ndarray       # uint8 view of the q array as drawn
    d_codes: np.ndarray  # uint16 (f16 codes) or uint32 (f32 bits), rows x cols/32


def assemble(wtype: int, scale_f16: int, rows: int, cols: int, q: np.ndarray,
             d_codes: np.ndarray, trailing_pad: bool = False) -> np.ndarray:
    q_bytes, d_off, d_bytes = array_offsets(wtype, scale_f16, rows, cols)
    total = d_off + d_bytes
    if trailing_pad:
        total = -(-total // 64) * 64
    W = np.zeros(total, dtype=np.uint8)
    W[:q_bytes] = np.ascontiguousarray(q).reshape(-1).view(np.uint8)
    W[d_off:d_off + d_bytes] = np.ascontiguousarray(d_codes).astype(
        np.uint16 if scale_f16 else np.uint32).reshape(-1).view(np.uint8)
    return W


def random_scales(rng: np.random.Generator, n: int, scale_f16: int,
                  low: float = 1e-3, high: float = 2e-2) -> np.ndarray:
    d = rng.uniform(low, high, size=n).astype(np.float32)
    if scale_f16:
        return d.astype(np.float16).view(np.uint16)
    return d.view(np.uint32)


def make_matrix(wtype: int, scale_f16: int, rows: int, cols: int, seed: int,
                trailing_pad: bool = False, d_low: float = 1e-3, d_high: float = 2e-2) -> Matrix:
    """Uniform quants (Q8_0 integers in [-127, 127], Q4_0 bytes 0..255) and d ~ U[low, high]."""
    rng = np.random.default_rng(seed)
    if wtype == Q8_0:
        q = rng.integers(-127, 128, size=rows * cols, dtype=np.int16).astype(np.int8).view(np.uint8)
    else:
        q = rng.integers(0, 256, size=rows * cols // 2, dtype=np.int16).astype(np.uint8)
    d_codes = random_scales(rng, rows * cols // 32, scale_f16, d_low, d_high)
    W = assemble(wtype, scale_f16, rows, cols, q, d_codes, trailing_pad)
    return Matrix(wtype, scale_f16, rows, cols, W, q, d_codes.reshape(rows, cols // 32))


def bf16_codes(x: np.ndarray) -> np.ndarray:
    """bfloat16 codes nearest to finite float32 values (ties to even)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def make_x(batch: int, cols: int, bf16: bool, seed: int) -> np.ndarray:
    """Activations ~ N(0, 1): float32, or bfloat16 codes (uint16) when bf16."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(size=(batch, cols)).astype(np.float32)
    return bf16_codes(x) if bf16 else x


def make_int_x(batch: int, cols: int, bf16: bool, seed: int, lo: int = -4, hi: int = 4) -> np.ndarray:
    """Small integer activations (exact in every format): for exact-arithmetic cases."""
    rng = np.random.default_rng(seed)
    x = rng.integers(lo, hi + 1, size=(batch, cols)).astype(np.float32)
    return bf16_codes(x) if bf16 else x


def pow2_scales(rng: np.random.Generator, n: int, scale_f16: int, lo_exp: int = -4,
                hi_exp: int = 0) -> np.ndarray:
    """Power-of-two scales 2^e, e uniform in [lo_exp, hi_exp] (exact-arithmetic cases)."""
    d = np.ldexp(np.ones(n, dtype=np.float32), rng.integers(lo_exp, hi_exp + 1, size=n)).astype(np.float32)
    if scale_f16:
        return d.astype(np.float16).view(np.uint16)
    return d.view(np.uint32)
