"""Block-quantized (Q8_0 / Q4_0) weight matrix-vector product for GB300 (sm_103a).

The compute path is the C-ABI library ``libqmv.so`` built from ``csrc/``; this package
is a thin ctypes binding over it (argument marshalling only).  The library is loaded on
first use, and every entry point raises if it is missing: there is no CPU fallback.
"""
from .binding import (  # noqa: F401
    Q8_0, Q4_0, SCALE_F32, SCALE_F16, X_F32, X_BF16,
    QmvError, library_path, load_library, weight_bytes, scale_offset,
    matvec, matvec_grouped, matvec_grouped_noalloc, matvec_glu, FLAG_OVERLAP, FLAG_BF16_WEIGHTS, MAX_GROUP, NOALLOC_MAX_BATCH, dequant,
    validate, quantize, quantize_q4_fit, quantize_x, matvec_qx, matvec_qx_grouped, gguf_bytes, gguf_to_mlb, Step, matrix_wtype, strerror, last_error,
)
