"""The C-ABI library on the CPU: it builds, loads, exports every declared symbol, and its
host-only logic (sizes, class dispatch, argument checks) behaves as include/qmv.h states.
No test here launches a kernel: every call with device pointers fails its checks first."""
import ctypes
import os
import re

import pytest

import oracle
from block_quantized_weight_q4_gb300 import binding
from block_quantized_weight_q4_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build()
    return binding.load_library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "qmv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(qmv_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "qmv_matvec" in names and "qmv_dequant" in names
    for n in names:
        assert hasattr(lib, n), n


def test_weight_bytes_agree_with_oracle(lib):
    for wt in (1, 2):
        for sf in (0, 1):
            for rows, cols in [(1, 32), (3, 96), (7, 64), (256, 256), (151936, 896), (4096, 11008)]:
                assert binding.weight_bytes(wt, sf, rows, cols) == oracle.weight_bytes(wt, sf, rows, cols)
                assert binding.scale_offset(wt, sf, rows, cols) == oracle.scale_offset(wt, sf, rows, cols)


@pytest.mark.parametrize("args", [(2, 1, 1, 48), (2, 1, 0, 32), (2, 1, 1, 0), (1, 0, -1, 32),
                                  (3, 0, 1, 32), (2, 2, 1, 32), (2, 1, 2**40, 2**40)])
def test_weight_bytes_invalid(lib, args):
    assert binding.weight_bytes(*args) == 0
    assert binding.scale_offset(*args) == -1


def test_q8_mask_dispatch(lib):
    # Krafla header offset 72: classes with their bit set are Q8_0 in a Q4_0 file.
    m = binding.matrix_wtype
    assert m(2, 2, 2) == 1 and m(2, 2, 4) == 2 and m(2, 0, 2) == 2
    assert m(2, 4 | 64, 4) == 1 and m(2, 4 | 64, 64) == 1 and m(2, 4 | 64, 32) == 2
    # a Q8_0 file stores everything as Q8_0
    assert all(m(1, 0, c) == 1 for c in (1, 2, 4, 8, 16, 32, 64))
    # with a shared classifier, tok_emb takes Q8_0 when the mask has bit 1 or bit 2
    assert m(2, 2, 1, True) == 1 and m(2, 2, 1, False) == 2 and m(2, 1, 1, True) == 1
    assert m(2, 0, 3) == -1 and m(5, 0, 2) == -1


FAKE = 0x10000  # never dereferenced: every call below fails its host checks first


def call_matvec(lib, wt=2, sf=1, rows=64, cols=64, W=FAKE, x=FAKE, xd=1, y=FAKE, batch=1):
    return lib.qmv_matvec(wt, sf, rows, cols, W, x, xd, y, batch, None)


def test_matvec_argument_errors(lib):
    assert call_matvec(lib, wt=3) == binding.E_FORMAT
    assert call_matvec(lib, sf=2) == binding.E_FORMAT
    assert call_matvec(lib, xd=5) == binding.E_FORMAT
    assert call_matvec(lib, xd=-1) == binding.E_FORMAT
    # a bfloat16 pair (4) is one vector with cols % 256 == 0
    assert call_matvec(lib, xd=4, cols=64) == binding.E_SHAPE
    assert call_matvec(lib, xd=4, cols=256, batch=2) == binding.E_ARG
    # gated activations (2: SiLU, 3: GELU-tanh) need cols % 256 == 0: checked before any launch
    assert call_matvec(lib, xd=2, cols=64) == binding.E_SHAPE
    assert call_matvec(lib, xd=3, cols=96) == binding.E_SHAPE
    assert call_matvec(lib, cols=48) == binding.E_SHAPE
    assert call_matvec(lib, rows=0) == binding.E_SHAPE
    assert call_matvec(lib, rows=2**40, cols=2**40) == binding.E_SHAPE
    assert call_matvec(lib, W=0) == binding.E_ARG
    assert call_matvec(lib, x=0) == binding.E_ARG
    assert call_matvec(lib, y=0) == binding.E_ARG
    assert call_matvec(lib, batch=-1) == binding.E_ARG
    assert call_matvec(lib, W=FAKE + 8) == binding.E_ALIGN
    assert call_matvec(lib, x=FAKE + 4) == binding.E_ALIGN
    assert call_matvec(lib, y=FAKE + 2) == binding.E_ALIGN
    # an empty batch is a no-op, checked before any device work
    assert call_matvec(lib, batch=0, x=0, y=0) == binding.OK


def test_dequant_and_validate_argument_errors(lib):
    assert lib.qmv_dequant(2, 1, 64, 48, FAKE, FAKE, None) == binding.E_SHAPE
    assert lib.qmv_dequant(2, 1, 64, 64, FAKE, 0, None) == binding.E_ARG
    assert lib.qmv_dequant(2, 1, 64, 64, FAKE, FAKE + 4, None) == binding.E_ALIGN
    assert lib.qmv_dequant(0, 1, 64, 64, FAKE, FAKE, None) == binding.E_FORMAT
    assert lib.qmv_validate(1, 0, 64, 64, FAKE, 0, None) == binding.E_ARG
    assert lib.qmv_validate(1, 0, 64, 64, FAKE, FAKE + 4, None) == binding.E_ALIGN
    assert lib.qmv_validate(1, 0, 0, 64, FAKE, FAKE, None) == binding.E_SHAPE
    # qmv_quantize: shape, format, null and alignment checks before any launch
    assert lib.qmv_quantize(2, 1, 64, 48, FAKE, FAKE, FAKE, None) == binding.E_SHAPE
    assert lib.qmv_quantize(3, 1, 64, 64, FAKE, FAKE, FAKE, None) == binding.E_FORMAT
    assert lib.qmv_quantize(2, 1, 64, 64, 0, FAKE, FAKE, None) == binding.E_ARG
    assert lib.qmv_quantize(2, 1, 64, 64, FAKE, FAKE, 0, None) == binding.E_ARG
    assert lib.qmv_quantize(2, 1, 64, 64, FAKE + 4, FAKE, FAKE, None) == binding.E_ALIGN
    assert lib.qmv_quantize(2, 1, 64, 64, FAKE, FAKE + 8, FAKE, None) == binding.E_ALIGN
    assert lib.qmv_quantize(2, 1, 64, 64, FAKE, FAKE, FAKE + 4, None) == binding.E_ALIGN
    # qmv_step_create / run / destroy: argument checks before any CUDA call
    out = ctypes.c_void_p(123)
    assert lib.qmv_step_create(None, 0, None, 0, None, 0, None) == binding.E_ARG
    assert lib.qmv_step_create(None, 1, None, 0, None, 0, ctypes.byref(out)) == binding.E_ARG
    assert out.value is None                                  # *step is cleared on failure
    assert lib.qmv_step_create(None, 0, None, -1, None, 0, ctypes.byref(out)) == binding.E_ARG
    assert lib.qmv_step_create(None, 0, None, 2, None, 0, ctypes.byref(out)) == binding.E_ARG
    assert lib.qmv_step_create(None, 0, None, 0, None, -1, ctypes.byref(out)) == binding.E_ARG
    bad = (binding.Copy * 1)(binding.Copy(0, FAKE, 64))
    assert lib.qmv_step_create(ctypes.addressof(bad), 1, None, 0, None, 0, ctypes.byref(out)) == binding.E_ARG
    assert lib.qmv_step_run(None, None) == binding.E_ARG
    assert lib.qmv_step_run_wait(None, None) == binding.E_ARG
    assert lib.qmv_step_destroy(None) == binding.OK
    # the gated step: the same argument checks, and open / wait need a step
    assert lib.qmv_step_create_gated(None, 0, None, 0, None, 0, None) == binding.E_ARG
    assert lib.qmv_step_create_gated(ctypes.addressof(bad), 1, None, 0, None, 0, ctypes.byref(out)) == binding.E_ARG
    assert out.value is None
    assert lib.qmv_step_open(None) == binding.E_ARG
    assert lib.qmv_step_wait(None, 0) == binding.E_ARG
    assert lib.qmv_step_open_wait(None, None, None, 0) == binding.E_ARG
    # qmv_gguf_bytes / qmv_gguf_to_mlb: sizes, then shape, format, null and alignment checks
    assert lib.qmv_gguf_bytes(1, 151936, 896) == 144643072
    assert lib.qmv_gguf_bytes(2, 151936, 896) == 76575744
    assert lib.qmv_gguf_bytes(2, 1, 896) == 504
    assert lib.qmv_gguf_bytes(2, 1, 48) == 0 and lib.qmv_gguf_bytes(3, 1, 32) == 0
    assert lib.qmv_gguf_to_mlb(3, 4, 64, FAKE, FAKE, None) == binding.E_FORMAT
    assert lib.qmv_gguf_to_mlb(2, 4, 48, FAKE, FAKE, None) == binding.E_SHAPE
    assert lib.qmv_gguf_to_mlb(2, 0, 64, FAKE, FAKE, None) == binding.E_SHAPE
    assert lib.qmv_gguf_to_mlb(2, 4, 64, 0, FAKE, None) == binding.E_ARG
    assert lib.qmv_gguf_to_mlb(1, 4, 64, FAKE, 0, None) == binding.E_ARG
    assert lib.qmv_gguf_to_mlb(2, 4, 64, FAKE + 2, FAKE, None) == binding.E_ALIGN
    assert lib.qmv_gguf_to_mlb(2, 4, 64, FAKE, FAKE + 8, None) == binding.E_ALIGN
    # qmv_quantize_q4_fit: the checks of qmv_quantize
    assert lib.qmv_quantize_q4_fit(2, 64, 64, FAKE, FAKE, FAKE, None) == binding.E_FORMAT
    assert lib.qmv_quantize_q4_fit(1, 64, 48, FAKE, FAKE, FAKE, None) == binding.E_SHAPE
    assert lib.qmv_quantize_q4_fit(1, 64, 64, 0, FAKE, FAKE, None) == binding.E_ARG
    assert lib.qmv_quantize_q4_fit(0, 64, 64, FAKE, FAKE, 0, None) == binding.E_ARG
    assert lib.qmv_quantize_q4_fit(1, 64, 64, FAKE + 4, FAKE, FAKE, None) == binding.E_ALIGN
    assert lib.qmv_quantize_q4_fit(1, 64, 64, FAKE, FAKE, FAKE + 4, None) == binding.E_ALIGN
    # qmv_quantize_x: dtype, shape, batch, null and alignment checks before any launch
    assert lib.qmv_quantize_x(2, 1, 64, FAKE, FAKE, None) == binding.E_FORMAT
    assert lib.qmv_quantize_x(0, 1, 48, FAKE, FAKE, None) == binding.E_SHAPE
    assert lib.qmv_quantize_x(0, 1, 0, FAKE, FAKE, None) == binding.E_SHAPE
    assert lib.qmv_quantize_x(0, -1, 64, FAKE, FAKE, None) == binding.E_ARG
    assert lib.qmv_quantize_x(1, 0, 64, 0, 0, None) == binding.OK          # batch 0: nothing to do
    assert lib.qmv_quantize_x(0, 2, 64, 0, FAKE, None) == binding.E_ARG
    assert lib.qmv_quantize_x(1, 2, 64, FAKE, 0, None) == binding.E_ARG
    assert lib.qmv_quantize_x(0, 2, 64, FAKE + 8, FAKE, None) == binding.E_ALIGN
    assert lib.qmv_quantize_x(0, 2, 64, FAKE, FAKE + 4, None) == binding.E_ALIGN
    # qmv_matvec_qx: the matrix checks of qmv_matvec, then the activation image and y
    assert lib.qmv_matvec_qx(3, 0, 64, 64, FAKE, FAKE, FAKE, 1, None) == binding.E_FORMAT
    assert lib.qmv_matvec_qx(2, 1, 64, 48, FAKE, FAKE, FAKE, 1, None) == binding.E_SHAPE
    assert lib.qmv_matvec_qx(2, 1, 64, 64, 0, FAKE, FAKE, 1, None) == binding.E_ARG
    assert lib.qmv_matvec_qx(2, 1, 64, 64, FAKE + 8, FAKE, FAKE, 1, None) == binding.E_ALIGN
    assert lib.qmv_matvec_qx(2, 1, 64, 64, FAKE, FAKE, FAKE, -1, None) == binding.E_ARG
    assert lib.qmv_matvec_qx(2, 1, 64, 64, FAKE, 0, 0, 0, None) == binding.OK   # batch 0
    assert lib.qmv_matvec_qx(2, 1, 64, 64, FAKE, 0, FAKE, 1, None) == binding.E_ARG
    assert lib.qmv_matvec_qx(1, 0, 64, 64, FAKE, FAKE, 0, 1, None) == binding.E_ARG
    assert lib.qmv_matvec_qx(2, 1, 64, 64, FAKE, FAKE + 8, FAKE, 1, None) == binding.E_ALIGN
    assert lib.qmv_matvec_qx(2, 1, 64, 64, FAKE, FAKE, FAKE + 2, 1, None) == binding.E_ALIGN


def test_matvec_glu_argument_errors(lib):
    def glu(wt=2, sf=1, rows=64, cols=256, W1=FAKE, W3=FAKE, x=FAKE, xd=1, act=0, h=FAKE, flags=0):
        return lib.qmv_matvec_glu(wt, sf, rows, cols, W1, W3, x, xd, act, h, flags, None)
    assert glu(wt=1) == binding.E_FORMAT          # the fused epilogue takes Q4_0
    assert glu(wt=3) == binding.E_FORMAT
    assert glu(xd=0) == binding.E_FORMAT          # one bfloat16 vector
    assert glu(act=2) == binding.E_FORMAT
    assert glu(flags=2) == binding.E_ARG
    assert glu(cols=64) == binding.E_SHAPE        # cols % 256
    assert glu(cols=48) == binding.E_SHAPE
    assert glu(rows=0) == binding.E_SHAPE
    assert glu(W1=0) == binding.E_ARG and glu(W3=0) == binding.E_ARG
    assert glu(x=0) == binding.E_ARG and glu(h=0) == binding.E_ARG
    assert glu(W3=FAKE + 8) == binding.E_ALIGN
    assert glu(x=FAKE + 2) == binding.E_ALIGN and glu(h=FAKE + 4) == binding.E_ALIGN


def test_matvec_qx_grouped_argument_errors(lib):
    def call(wt=2, sf=1, xd=1, batch=1, rows=64, cols=64, W=FAKE, x=FAKE, y=FAKE, n=1, flags=0, null=False):
        arr = (binding.Problem * 1)(binding.Problem(rows, cols, W, x, y))
        return lib.qmv_matvec_qx_grouped(wt, sf, xd, batch, None if null else ctypes.addressof(arr), n, flags, None)
    assert call(null=True) == binding.E_ARG
    assert call(n=0) == binding.E_ARG and call(n=9) == binding.E_ARG
    assert call(xd=2) == binding.E_FORMAT and call(xd=4) == binding.E_FORMAT
    assert call(batch=-1) == binding.E_ARG
    assert call(flags=2) == binding.E_ARG
    assert call(wt=3) == binding.E_FORMAT and call(sf=2) == binding.E_FORMAT
    assert call(cols=48) == binding.E_SHAPE and call(rows=0) == binding.E_SHAPE
    # one pass of 8 vectors keeps 8 * cols quants in shared memory
    assert call(batch=8, cols=25120 * 2) == binding.E_SHAPE
    assert call(batch=1, cols=200704 + 32) == binding.E_SHAPE
    assert call(W=0) == binding.E_ARG and call(x=0) == binding.E_ARG and call(y=0) == binding.E_ARG
    assert call(W=FAKE + 8) == binding.E_ALIGN and call(x=FAKE + 8) == binding.E_ALIGN
    assert call(y=FAKE + 2) == binding.E_ALIGN
    assert call(batch=0, x=0, y=0) == binding.OK


def test_strerror_never_null(lib):
    for s in (0, 2, 3, 4, 5, 6, 7, 99, -1):
        assert isinstance(lib.qmv_strerror(s), bytes) and lib.qmv_strerror(s)


def test_binding_prototypes_match_the_header(lib):
    # every function the header declares has a ctypes prototype in the binding with the same
    # number of parameters (a mismatch would pass garbage through the C ABI)
    text = open(os.path.join(ROOT, "include", "qmv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    decls = re.findall(r"\b(qmv_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text)
    assert len(decls) >= 19
    for name, params in decls:
        params = params.strip()
        n = 0 if params in ("", "void") else params.count(",") + 1
        fn = getattr(lib, name)
        assert fn.argtypes is not None, f"{name}: no prototype in the binding"
        assert len(fn.argtypes) == n, f"{name}: header has {n} parameters, binding {len(fn.argtypes)}"
