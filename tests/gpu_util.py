"""Shared helpers for the GPU parity tests (the CUDA path through the C ABI
against the CPU oracle)."""

import numpy as np
import pytest


def require_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import __graft_entry__

    __graft_entry__.build()
    import gradient_synchronisation_gb300 as zr

    return torch, zr


def bits_equal(a, b):
    """Bitwise equality of float arrays; NaNs compared by class only."""
    a = np.ascontiguousarray(a)
    b = np.ascontiguousarray(b)
    if a.dtype == np.uint16:
        fa = (a.astype(np.uint32) << 16).view(np.float32)
        fb = (b.astype(np.uint32) << 16).view(np.float32)
        ua, ub = a, b
    else:
        fa, fb = a, b
        ua, ub = a.view(np.uint32), b.view(np.uint32)
    na, nb = np.isnan(fa), np.isnan(fb)
    if not np.array_equal(na, nb):
        return False
    return np.array_equal(ua[~na], ub[~nb])


def ulp_report(a, b):
    """(count of differing elements, max ULP distance) for float32 arrays."""
    ia = a.view(np.int32).astype(np.int64)
    ib = b.view(np.int32).astype(np.int64)
    ia = np.where(ia < 0, -(ia & 0x7FFFFFFF), ia)
    ib = np.where(ib < 0, -(ib & 0x7FFFFFFF), ib)
    d = np.abs(ia - ib)
    return int((d != 0).sum()), int(d.max()) if d.size else 0
