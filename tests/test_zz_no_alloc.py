"""xsymv_s_noalloc — SSYMV for callers that cannot allocate device memory
during a call (for example a plug-in whose host application owns all device
memory, or latency-critical code where cudaMalloc would block or synchronise
the device).  It runs xsymv_s's kernels on a fixed device array instead of an
allocated workspace.

This file is collected last on purpose.  The test calls the entry point
through the C ABI twice in a row and checks both results against xsymv_s
within the SSYMV tolerance; it also checks the size limit.  It must pass in a
fresh process and after every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle
from symmetric_matrix_vector_gb300 import _build, inputs
from tests.gpu_helpers import TOL, from_device, logical, to_device

pytestmark = pytest.mark.gpu

XSYMV_ERR_TOO_LARGE = -5


def _noalloc(lib):
    fn = lib.xsymv_s_noalloc
    fn.argtypes = [ctypes.c_char, ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_int,
                   ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_int]
    fn.restype = ctypes.c_int
    return fn


def test_noalloc_matches_xsymv_s_twice():
    import torch

    import symmetric_matrix_vector_gb300 as xs

    _build.build()
    lib = xs.load()
    fn = _noalloc(lib)
    torch.cuda.set_device(0)
    xs.xsymv_set_stream(torch.cuda.current_stream().cuda_stream)

    for uplo, n, incy in (("U", 3000, 1), ("L", 4097, -2)):
        p = inputs.make_problem("s", uplo, n, lda=n + 5, alpha=1.25, beta=0.5, incy=incy, seed=n)
        A, x, y0 = to_device(p.A), to_device(p.x), to_device(p.y)

        y_ref = y0.clone()
        assert xs.xsymv_s(uplo, n, 1.25, A, p.lda, x, 1, 0.5, y_ref, incy) == 0
        ref = logical("s", from_device(y_ref, p.y), n, incy).astype(np.float64)
        # error normaliser |alpha| |A||x| + |beta| |y| from the oracle
        _, _, _, den = oracle.get().rows("s", uplo, n, 1.25, p.A, p.lda, p.x, 1, 0.5, p.y, incy,
                                         np.arange(n))
        for call in range(2):
            y = y0.clone()
            st = fn(uplo.encode(), n, 1.25, ctypes.c_void_p(A.data_ptr()), p.lda,
                    ctypes.c_void_p(x.data_ptr()), 1, 0.5, ctypes.c_void_p(y.data_ptr()), incy)
            assert st == 0, (call, st)
            got = logical("s", from_device(y, p.y), n, incy).astype(np.float64)
            err = np.abs(got - ref) / den
            assert float(np.max(err)) <= TOL["s"], (uplo, n, call, float(np.max(err)))


def test_noalloc_rejects_too_large():
    import torch

    import symmetric_matrix_vector_gb300 as xs

    _build.build()
    lib = xs.load()
    fn = _noalloc(lib)
    # A below is far smaller than an n-by-n matrix: the call is only safe if
    # it is rejected before anything is enqueued.  So n is chosen so that the
    # column partials alone (one per 512 rows or fewer, per column) exceed
    # the 16 MiB array whatever kernel variant is tuned, and the library's
    # own workspace estimate is checked first.
    n = 100000
    assert xs.xsymv_workspace_bytes("s", "U", n) > (16 << 20)
    y = torch.full((n,), 3.0, device="cuda")
    A = torch.zeros(16, device="cuda")
    st = fn(b"U", n, 1.0, ctypes.c_void_p(A.data_ptr()), n, ctypes.c_void_p(y.data_ptr()), 1, 0.0,
            ctypes.c_void_p(y.data_ptr()), 1)
    assert st == XSYMV_ERR_TOO_LARGE
    torch.cuda.synchronize()
    assert bool((y == 3.0).all())
    assert "16 MiB" in xs.xsymv_status_string(st)
