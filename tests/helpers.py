"""Shared test helpers: device transfer, the tolerance check, bit-exact comparison."""
import numpy as np


# Batch-1 products on float32, bfloat16-pair or gated activations round each activation once to
# IEEE half after a power-of-two scale of its stage: at most 2^-11 relative error per term, plus
# the float32 sums (a few parts in 2^20 of sum |w x| at the sizes of the tests)
HALF_TOL = 2.0 ** -11 + 2.0 ** -16


def dev_u8(W):
    import torch
    return torch.from_numpy(np.ascontiguousarray(W)).cuda()


def dev_x(x):
    """float32 array -> float32 CUDA tensor; uint16 bfloat16 codes -> bfloat16 CUDA tensor."""
    import torch
    x = np.ascontiguousarray(x)
    if x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(x.astype(np.float32)).cuda()


def check_product(y_gpu, y_ref, absref, tol=1e-3, what=""):
    """|y_gpu - y_ref| <= tol * sum|w x| for every element (exact zero when the sum is 0)."""
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(y_gpu - y_ref)
    bound = tol * absref
    bad = ~(err <= bound)
    if bad.any():
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {bad.sum()} elements out of tolerance; first at {tuple(i)}: "
                             f"gpu={y_gpu[tuple(i)]!r} ref={y_ref[tuple(i)]!r} bound={bound[tuple(i)]!r}")
    return float(np.max(err / np.where(absref > 0, absref, 1.0))) if err.size else 0.0


def assert_bits_equal(a, b, what=""):
    """Bit-exact float32 comparison; NaNs compare equal to NaNs (payloads may differ)."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    b = np.ascontiguousarray(b, dtype=np.float32)
    na, nb = np.isnan(a), np.isnan(b)
    assert np.array_equal(na, nb), f"{what}: NaN positions differ"
    ua, ub = a[~na].view(np.uint32), b[~nb].view(np.uint32)
    if not np.array_equal(ua, ub):
        i = int(np.argmax(ua != ub))
        raise AssertionError(f"{what}: {int((ua != ub).sum())} values differ; first {a[~na][i]!r} vs {b[~nb][i]!r}")
