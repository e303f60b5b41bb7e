"""ctypes binding over libqmv.so (C ABI declared in include/qmv.h).

Argument marshalling only: tensors are passed as raw device pointers with the current
torch CUDA stream; every step of the computation runs in the library's kernels.  If the
library has not been built, every call raises: there is no CPU fallback.

Format (Krafla ".mlb model format v1", "Body"): a matrix image is the q array, zero
padding to 64 bytes, then the d array; W below is a uint8 CUDA tensor holding it.
"""
from __future__ import annotations

import ctypes
import os

Q8_0 = 1
Q4_0 = 2
SCALE_F32 = 0
SCALE_F16 = 1
X_F32 = 0
X_BF16 = 1

OK = 0
E_FORMAT = 2
E_SHAPE = 3
E_ARG = 4
E_ALIGN = 5
E_CUDA = 6
E_TIMEOUT = 7

_HERE = os.path.dirname(os.path.abspath(__file__))
_lib = None


class QmvError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: status {status} ({strerror(status)})")


def library_path() -> str:
    return os.path.join(_HERE, "libqmv.so")


def load_library():
    """Load libqmv.so (raises OSError if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise OSError(f"libqmv.so not built ({path}); run block_quantized_weight_q4_gb300.build")
    lib = ctypes.CDLL(path)
    i64, i32, vp, sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
    lib.qmv_weight_bytes.restype = sz
    lib.qmv_weight_bytes.argtypes = [i32, i32, i64, i64]
    lib.qmv_scale_offset.restype = i64
    lib.qmv_scale_offset.argtypes = [i32, i32, i64, i64]
    lib.qmv_matrix_wtype.restype = i32
    lib.qmv_matrix_wtype.argtypes = [i32, ctypes.c_uint32, i32, i32]
    lib.qmv_matvec.restype = i32
    lib.qmv_matvec.argtypes = [i32, i32, i64, i64, vp, vp, i32, vp, i32, vp]
    lib.qmv_matvec_grouped.restype = i32
    lib.qmv_matvec_grouped.argtypes = [i32, i32, i32, i32, vp, i32, ctypes.c_uint, vp]
    lib.qmv_matvec_grouped_noalloc.argtypes = [i32, i32, i32, i32, vp, i32, ctypes.c_uint, vp]
    lib.qmv_matvec_glu.restype = i32
    lib.qmv_matvec_glu.argtypes = [i32, i32, i64, i64, vp, vp, vp, i32, i32, vp, ctypes.c_uint, vp]
    lib.qmv_dequant.restype = i32
    lib.qmv_dequant.argtypes = [i32, i32, i64, i64, vp, vp, vp]
    lib.qmv_validate.restype = i32
    lib.qmv_validate.argtypes = [i32, i32, i64, i64, vp, vp, vp]
    lib.qmv_quantize.restype = i32
    lib.qmv_quantize.argtypes = [i32, i32, i64, i64, vp, vp, vp, vp]
    lib.qmv_step_create.restype = i32
    lib.qmv_step_create.argtypes = [vp, i32, vp, i32, vp, i32, ctypes.POINTER(vp)]
    lib.qmv_step_run.restype = i32
    lib.qmv_step_run.argtypes = [vp, vp]
    lib.qmv_step_run_wait.restype = i32
    lib.qmv_step_run_wait.argtypes = [vp, vp]
    lib.qmv_step_destroy.restype = i32
    lib.qmv_step_destroy.argtypes = [vp]
    lib.qmv_step_create_gated.restype = i32
    lib.qmv_step_create_gated.argtypes = [vp, i32, vp, i32, vp, i32, ctypes.POINTER(vp)]
    lib.qmv_step_open.restype = i32
    lib.qmv_step_open.argtypes = [vp]
    lib.qmv_step_wait.restype = i32
    lib.qmv_step_wait.argtypes = [vp, ctypes.c_longlong]
    lib.qmv_step_open_wait.restype = i32
    lib.qmv_step_open_wait.argtypes = [vp, vp, vp, ctypes.c_longlong]
    lib.qmv_gguf_bytes.restype = ctypes.c_size_t
    lib.qmv_gguf_bytes.argtypes = [i32, i64, i64]
    lib.qmv_gguf_to_mlb.restype = i32
    lib.qmv_gguf_to_mlb.argtypes = [i32, i64, i64, vp, vp, vp]
    lib.qmv_quantize_q4_fit.restype = i32
    lib.qmv_quantize_q4_fit.argtypes = [i32, i64, i64, vp, vp, vp, vp]
    lib.qmv_quantize_x.restype = i32
    lib.qmv_quantize_x.argtypes = [i32, i64, i64, vp, vp, vp]
    lib.qmv_matvec_qx_grouped.restype = i32
    lib.qmv_matvec_qx_grouped.argtypes = [i32, i32, i32, i32, vp, i32, ctypes.c_uint, vp]
    lib.qmv_matvec_qx.restype = i32
    lib.qmv_matvec_qx.argtypes = [i32, i32, i64, i64, vp, vp, vp, i32, vp]
    lib.qmv_check_device.restype = i32
    lib.qmv_check_device.argtypes = []
    lib.qmv_strerror.restype = ctypes.c_char_p
    lib.qmv_strerror.argtypes = [i32]
    _lib = lib
    return lib


def strerror(status: int) -> str:
    try:
        return load_library().qmv_strerror(status).decode()
    except OSError:
        return "libqmv not loaded"


def _check(status: int, where: str):
    if status != OK:
        raise QmvError(status, where)


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _x_dtype(x) -> int:
    import torch
    if x.dtype == torch.float32:
        return X_F32
    if x.dtype == torch.bfloat16:
        return X_BF16
    raise TypeError("x must be float32 or bfloat16")


def weight_bytes(wtype: int, scale_dtype: int, rows: int, cols: int) -> int:
    return int(load_library().qmv_weight_bytes(wtype, scale_dtype, rows, cols))


def scale_offset(wtype: int, scale_dtype: int, rows: int, cols: int) -> int:
    return int(load_library().qmv_scale_offset(wtype, scale_dtype, rows, cols))


def matrix_wtype(file_wtype: int, q8_mask: int, class_bit: int, shared_classifier: bool = False) -> int:
    return int(load_library().qmv_matrix_wtype(file_wtype, q8_mask, class_bit, int(bool(shared_classifier))))


def matvec(wtype: int, scale_dtype: int, rows: int, cols: int, W, x, y=None, stream=None):
    """y = W x.  W: uint8 CUDA tensor (matrix image); x: (batch, cols) float32/bfloat16
    CUDA tensor; y: optional (batch, rows) float32 CUDA tensor.  Returns y."""
    import torch
    if x.dim() == 1:
        x = x.unsqueeze(0)
    batch = x.shape[0]
    if x.shape[1] != cols or not x.is_contiguous():
        raise ValueError("x must be a contiguous (batch, cols) tensor")
    if y is None:
        y = torch.empty((batch, rows), dtype=torch.float32, device=x.device)
    if y.dtype != torch.float32 or tuple(y.shape) != (batch, rows) or not y.is_contiguous():
        raise ValueError("y must be a contiguous float32 (batch, rows) tensor")
    st = load_library().qmv_matvec(wtype, scale_dtype, rows, cols, W.data_ptr(), x.data_ptr(), _x_dtype(x),
                                   y.data_ptr(), batch, _stream(stream))
    _check(st, "qmv_matvec")
    return y


class Problem(ctypes.Structure):
    """qmv_problem of include/qmv.h."""
    _fields_ = [("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("W", ctypes.c_void_p),
                ("x", ctypes.c_void_p), ("y", ctypes.c_void_p)]


FLAG_OVERLAP = 1
FLAG_BF16_WEIGHTS = 2
MAX_GROUP = 8
X_SILU_GLU_F32 = 2
X_GELU_GLU_F32 = 3
X_BF16_PAIR = 4
ACTS = {"silu": X_SILU_GLU_F32, "gelu": X_GELU_GLU_F32}
ACT_SILU = 0
ACT_GELU_TANH = 1
ACT_CODES = {"silu": ACT_SILU, "gelu": ACT_GELU_TANH}
NOALLOC_MAX_BATCH = 8


def _problem_array(problems, act=None, pair=False):
    """act: None, or "silu" / "gelu" for gated activations (x of each problem: float32
    (2, batch, cols), gate then up).  pair: one vector given as bfloat16 (2, cols), hi parts
    then lo parts (the layout matvec_glu writes)."""
    n = len(problems)
    if not 1 <= n <= MAX_GROUP:
        raise ValueError("1..8 problems per group")
    arr = (Problem * n)()
    if pair:
        import torch
        for i, (rows, cols, W, x, y) in enumerate(problems):
            if x.dtype != torch.bfloat16 or tuple(x.shape) != (2, cols) or not x.is_contiguous():
                raise ValueError("a pair x is a contiguous bfloat16 (2, cols) tensor: hi, lo")
            if tuple(y.shape) != (1, rows) or not y.is_contiguous():
                raise ValueError("y must be a contiguous (1, rows) tensor")
            arr[i] = Problem(rows, cols, W.data_ptr(), x.data_ptr(), y.data_ptr())
        return arr, n, 1, X_BF16_PAIR
    if act is not None:
        import torch
        if act not in ACTS:
            raise ValueError("act must be 'silu' or 'gelu'")
        batch = problems[0][3].shape[1]
        for (rows, cols, W, x, y) in problems:
            if x.dtype != torch.float32 or tuple(x.shape) != (2, batch, cols):
                raise ValueError("gated activations need float32 x of shape (2, batch, cols)")
        xdt = ACTS[act]
    else:
        batch = problems[0][3].shape[0]
        xdt = _x_dtype(problems[0][3])
    for i, (rows, cols, W, x, y) in enumerate(problems):
        xshape = (2, batch, cols) if act is not None else (batch, cols)
        xdt_i = xdt if act is not None else _x_dtype(x)
        if tuple(x.shape) != xshape or tuple(y.shape) != (batch, rows) or xdt_i != xdt:
            raise ValueError("every problem needs x (batch, cols) of one dtype and y (batch, rows)")
        if not (x.is_contiguous() and y.is_contiguous()):
            raise ValueError("x and y must be contiguous")
        arr[i] = Problem(rows, cols, W.data_ptr(), x.data_ptr(), y.data_ptr())
    return arr, n, batch, xdt


def _flags(overlap: bool, bf16_weights: bool = False) -> int:
    return (FLAG_OVERLAP if overlap else 0) | (FLAG_BF16_WEIGHTS if bf16_weights else 0)


def matvec_grouped(wtype: int, scale_dtype: int, problems, overlap: bool = False, stream=None, act=None,
                   bf16_weights: bool = False, pair: bool = False):
    """Several products in one launch.  problems: list of (rows, cols, W, x, y) with W a
    uint8 CUDA tensor, x (batch, cols) and y (batch, rows) CUDA tensors; all share wtype,
    scale_dtype, the x dtype and batch.  overlap: QMV_FLAG_OVERLAP (the weights must not be
    written by the preceding kernel on the stream).  act: "silu" / "gelu" for gated
    activations, x then float32 (2, batch, cols): gate, up; the product takes act(gate) * up.
    bf16_weights: QMV_FLAG_BF16_WEIGHTS (prefill passes round each weight once to bfloat16).
    pair: each x is one vector as a bfloat16 (2, cols) pair (QMV_X_BF16_PAIR), y (1, rows)."""
    arr, n, batch, xdt = _problem_array(problems, act, pair)
    st = load_library().qmv_matvec_grouped(wtype, scale_dtype, xdt, batch, ctypes.addressof(arr), n,
                                           _flags(overlap, bf16_weights), _stream(stream))
    _check(st, "qmv_matvec_grouped")


def matvec_glu(wtype: int, scale_dtype: int, rows: int, cols: int, W1, W3, x, act: str = "silu", h=None,
               overlap: bool = False, stream=None):
    """The FFN's gate and up projections with the gated activation as their epilogue
    (qmv_matvec_glu): x a bfloat16 (cols,) or (1, cols) CUDA tensor; returns h, a bfloat16 (2, rows)
    CUDA tensor holding act(W1 x) * (W3 x) as hi and lo parts (the pair layout matvec_grouped
    takes with pair=True)."""
    import torch
    if act not in ACT_CODES:
        raise ValueError("act must be 'silu' or 'gelu'")
    if x.dtype != torch.bfloat16 or x.numel() != cols or not x.is_contiguous():
        raise ValueError("x must be one contiguous bfloat16 vector of cols values")
    if h is None:
        h = torch.empty((2, rows), dtype=torch.bfloat16, device=x.device)
    if h.dtype != torch.bfloat16 or tuple(h.shape) != (2, rows) or not h.is_contiguous():
        raise ValueError("h must be a contiguous bfloat16 (2, rows) tensor")
    st = load_library().qmv_matvec_glu(wtype, scale_dtype, rows, cols, W1.data_ptr(), W3.data_ptr(), x.data_ptr(),
                                       X_BF16, ACT_CODES[act], h.data_ptr(), FLAG_OVERLAP if overlap else 0,
                                       _stream(stream))
    _check(st, "qmv_matvec_glu")
    return h


def matvec_grouped_noalloc(wtype: int, scale_dtype: int, problems, overlap: bool = False, stream=None):
    """matvec_grouped that allocates no device memory (qmv_matvec_grouped_noalloc): bfloat16
    x, at most NOALLOC_MAX_BATCH vectors, cols % 256 == 0; its scratch is one fixed array
    in the library, so calls that may overlap in time must be ordered on one stream."""
    arr, n, batch, xdt = _problem_array(problems)
    st = load_library().qmv_matvec_grouped_noalloc(wtype, scale_dtype, xdt, batch, ctypes.addressof(arr), n,
                                                   FLAG_OVERLAP if overlap else 0, _stream(stream))
    _check(st, "qmv_matvec_grouped_noalloc")


class Copy(ctypes.Structure):
    """qmv_copy of include/qmv.h."""
    _fields_ = [("dst", ctypes.c_void_p), ("src", ctypes.c_void_p), ("bytes", ctypes.c_size_t)]


class Group(ctypes.Structure):
    """qmv_group of include/qmv.h."""
    _fields_ = [("wtype", ctypes.c_int), ("scale_dtype", ctypes.c_int), ("x_dtype", ctypes.c_int),
                ("batch", ctypes.c_int), ("problems", ctypes.c_void_p), ("n", ctypes.c_int),
                ("flags", ctypes.c_uint)]


def _copies(pairs):
    arr = (Copy * max(len(pairs), 1))()
    for i, (dst, src) in enumerate(pairs):
        nbytes = src.numel() * src.element_size()
        if dst.numel() * dst.element_size() != nbytes or not (dst.is_contiguous() and src.is_contiguous()):
            raise ValueError("a copy needs contiguous tensors of equal size")
        arr[i] = Copy(dst.data_ptr(), src.data_ptr(), nbytes)
    return arr


class Step:
    """A compiled step (qmv_step_create): `before` copies, product groups, `after` copies,
    recorded once as a CUDA graph; run() enqueues it with one library call.

    before / after: lists of (dst, src) tensors (device or pinned host); groups: list of
    (wtype, scale_dtype, problems, overlap[, act[, bf16_weights]]) with problems as for
    matvec_grouped.  Creating the
    step runs it once.  The tensors are kept alive with the step; a run reads and writes the
    same buffers.  Runs of one step must not overlap in time.  close() (or leaving a `with`
    block) waits for the device and frees the step.

    gated=True (qmv_step_create_gated): each run waits on the device until open() (its `before`
    copies: pinned host to device memory), and wait() spins on the host until the opened runs
    are done; a decode loop enqueues the next run before it needs it and only opens it then."""

    def __init__(self, groups, before=(), after=(), gated=False):
        keep = [list(before), list(after)]
        garr = (Group * max(len(groups), 1))()
        for i, grp in enumerate(groups):
            wtype, scale_dtype, problems, overlap = grp[:4]
            parr, n, batch, xdt = _problem_array(problems, grp[4] if len(grp) > 4 else None)
            keep.append((parr, problems))
            garr[i] = Group(wtype, scale_dtype, xdt, batch, ctypes.addressof(parr), n,
                            _flags(overlap, len(grp) > 5 and bool(grp[5])))
        b, a = _copies(list(before)), _copies(list(after))
        handle = ctypes.c_void_p()
        create = load_library().qmv_step_create_gated if gated else load_library().qmv_step_create
        st = create(ctypes.addressof(b), len(before), ctypes.addressof(garr), len(groups),
                    ctypes.addressof(a), len(after), ctypes.byref(handle))
        _check(st, "qmv_step_create_gated" if gated else "qmv_step_create")
        self._handle = handle
        self._keep = keep

    def run(self, stream=None, wait=False):
        """Enqueue one run on `stream` (the current stream by default); wait=True also waits for
        the stream in the same library call (qmv_step_run_wait)."""
        if self._handle is None:
            raise ValueError("step destroyed")
        if wait:
            _check(load_library().qmv_step_run_wait(self._handle, _stream(stream)), "qmv_step_run_wait")
        else:
            _check(load_library().qmv_step_run(self._handle, _stream(stream)), "qmv_step_run")

    def open(self):
        """Open the oldest enqueued run of a gated step (qmv_step_open)."""
        if self._handle is None:
            raise ValueError("step destroyed")
        _check(load_library().qmv_step_open(self._handle), "qmv_step_open")

    def wait(self, timeout_us=0):
        """Wait on the host until the opened runs of a gated step are done (qmv_step_wait)."""
        if self._handle is None:
            raise ValueError("step destroyed")
        _check(load_library().qmv_step_wait(self._handle, int(timeout_us)), "qmv_step_wait")

    def open_wait(self, next_step=None, stream=None, timeout_us=0):
        """open(), then next_step.run(stream) when given, then wait(): one library call
        (qmv_step_open_wait), a decode loop's step with the next run enqueued behind it."""
        if self._handle is None or (next_step is not None and next_step._handle is None):
            raise ValueError("step destroyed")
        _check(load_library().qmv_step_open_wait(self._handle, None if next_step is None else next_step._handle,
                                                 _stream(stream), int(timeout_us)), "qmv_step_open_wait")

    def close(self):
        if self._handle is not None:
            st = load_library().qmv_step_destroy(self._handle)
            self._handle = None
            self._keep = None
            _check(st, "qmv_step_destroy")

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
        return False


def dequant(wtype: int, scale_dtype: int, rows: int, cols: int, W, out=None, stream=None):
    """float32 (rows, cols) = level * d.  Returns out."""
    import torch
    if out is None:
        out = torch.empty((rows, cols), dtype=torch.float32, device=W.device)
    st = load_library().qmv_dequant(wtype, scale_dtype, rows, cols, W.data_ptr(), out.data_ptr(), _stream(stream))
    _check(st, "qmv_dequant")
    return out


def validate(wtype: int, scale_dtype: int, rows: int, cols: int, W, stream=None) -> int:
    """Index of the first Q8_0 quant byte equal to -128, or -1 (waits for the stream)."""
    import torch
    first = torch.empty(1, dtype=torch.int64, device=W.device)
    st = load_library().qmv_validate(wtype, scale_dtype, rows, cols, W.data_ptr(), first.data_ptr(),
                                     _stream(stream))
    _check(st, "qmv_validate")
    return int(first.item())


def quantize(wtype: int, scale_dtype: int, src, W=None, stream=None):
    """Matrix bytes (uint8 CUDA tensor of weight_bytes()) from float32 (rows, cols) by the
    writer rules.  Returns (W, first refused block index or -1); waits for the stream."""
    import torch
    rows, cols = src.shape
    if src.dtype != torch.float32 or not src.is_contiguous():
        raise ValueError("src must be a contiguous float32 (rows, cols) tensor")
    if W is None:
        W = torch.empty(weight_bytes(wtype, scale_dtype, rows, cols), dtype=torch.uint8, device=src.device)
    first = torch.empty(1, dtype=torch.int64, device=src.device)
    st = load_library().qmv_quantize(wtype, scale_dtype, rows, cols, src.data_ptr(), W.data_ptr(), first.data_ptr(),
                                     _stream(stream))
    _check(st, "qmv_quantize")
    return W, int(first.item())


def gguf_bytes(wtype: int, rows: int, cols: int) -> int:
    """Bytes of a rows x cols tensor in GGUF interleaved blocks (0 when invalid)."""
    return int(load_library().qmv_gguf_bytes(wtype, rows, cols))


def gguf_to_mlb(wtype: int, rows: int, cols: int, src, W=None, stream=None):
    """A tensor in GGUF interleaved blocks (uint8 CUDA tensor) into the two-array layout with
    f16 scales (uint8 CUDA tensor of weight_bytes(wtype, SCALE_F16, rows, cols)).  Returns W."""
    import torch
    if W is None:
        W = torch.empty(max(weight_bytes(wtype, SCALE_F16, rows, cols), 0), dtype=torch.uint8, device=src.device)
    st = load_library().qmv_gguf_to_mlb(wtype, rows, cols, src.data_ptr(), W.data_ptr(), _stream(stream))
    _check(st, "qmv_gguf_to_mlb")
    return W


def quantize_x(x, xq=None, stream=None):
    """The runtime's activation quantizer: x (batch, cols) float32/bfloat16 CUDA tensor into
    xq, the Q8_0 / f32-scale image of the batch x cols matrix (uint8 CUDA tensor of
    weight_bytes(Q8_0, SCALE_F32, batch, cols)).  Returns xq."""
    import torch
    if x.dim() == 1:
        x = x.unsqueeze(0)
    batch, cols = x.shape
    if not x.is_contiguous():
        raise ValueError("x must be a contiguous (batch, cols) tensor")
    if xq is None:
        xq = torch.empty(max(weight_bytes(Q8_0, SCALE_F32, batch, cols), 0), dtype=torch.uint8, device=x.device)
    st = load_library().qmv_quantize_x(_x_dtype(x), batch, cols, x.data_ptr(), xq.data_ptr(), _stream(stream))
    _check(st, "qmv_quantize_x")
    return xq


def matvec_qx(wtype: int, scale_dtype: int, rows: int, cols: int, W, xq, batch: int, y=None, stream=None):
    """Activation-quantized product: y[v][r] = sum_b d_w d_x (exact integer block dot) for the
    quantized activations xq (as quantize_x returns them, batch vectors).  Returns y."""
    import torch
    if y is None:
        y = torch.empty((batch, rows), dtype=torch.float32, device=xq.device)
    if y.dtype != torch.float32 or tuple(y.shape) != (batch, rows) or not y.is_contiguous():
        raise ValueError("y must be a contiguous float32 (batch, rows) tensor")
    st = load_library().qmv_matvec_qx(wtype, scale_dtype, rows, cols, W.data_ptr(), xq.data_ptr(), y.data_ptr(),
                                      batch, _stream(stream))
    _check(st, "qmv_matvec_qx")
    return y


def matvec_qx_grouped(wtype: int, scale_dtype: int, problems, overlap: bool = False, stream=None):
    """The activation-quantized product with the activation quantizer inside the launch
    (qmv_matvec_qx_grouped): problems as for matvec_grouped, x float32 or bfloat16 (batch, cols);
    each y receives matvec_qx(W, quantize_x(x))."""
    arr, n, batch, xdt = _problem_array(problems)
    st = load_library().qmv_matvec_qx_grouped(wtype, scale_dtype, xdt, batch, ctypes.addressof(arr), n,
                                              FLAG_OVERLAP if overlap else 0, _stream(stream))
    _check(st, "qmv_matvec_qx_grouped")


def quantize_q4_fit(scale_dtype: int, src, W=None, stream=None):
    """Q4_0 matrix bytes from float32 (rows, cols) by the best-fit rule (qmv_quantize_q4_fit).
    Returns (W, first refused block index or -1); waits for the stream."""
    import torch
    rows, cols = src.shape
    if src.dtype != torch.float32 or not src.is_contiguous():
        raise ValueError("src must be a contiguous float32 (rows, cols) tensor")
    if W is None:
        W = torch.empty(weight_bytes(Q4_0, scale_dtype, rows, cols), dtype=torch.uint8, device=src.device)
    first = torch.empty(1, dtype=torch.int64, device=src.device)
    st = load_library().qmv_quantize_q4_fit(scale_dtype, rows, cols, src.data_ptr(), W.data_ptr(), first.data_ptr(),
                                            _stream(stream))
    _check(st, "qmv_quantize_q4_fit")
    return W, int(first.item())


def last_error() -> int:
    """Synchronize the device; return and clear the kernels' status word."""
    return int(load_library().qmv_check_device())
