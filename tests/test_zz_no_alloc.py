"""xsymv_s_noalloc — SSYMV for callers that cannot allocate device memory
during a call (for example a plug-in whose host application owns all device
memory, or latency-critical code where cudaMalloc would block or synchronise
the device).  It runs xsymv_s's kernels on a fixed device array instead of an
allocated workspace.

This file is collected last on purpose.  The tests call the entry point
through the C ABI twice in a row and check both results against the oracle
within the SSYMV tolerance and, bit for bit, against xsymv_s (the same kernels
on the same plan); they cover a size just below the array's limit, alpha = 0,
the refusal of a problem that does not fit (with every buffer as large as its
arguments say), and the timeout status of the kernels' bounded waits.  They
must pass in a fresh process and after every other test.
"""
import ctypes

import numpy as np
import pytest

import oracle
from symmetric_matrix_vector_gb300 import _build, inputs
from tests.gpu_helpers import TOL, errors, from_device, sample_rows, to_device

pytestmark = pytest.mark.gpu

XSYMV_ERR_TOO_LARGE = -5
XSYMV_ERR_TIMEOUT = -6
SCRATCH_BYTES = 16 << 20
# the plan's warp and row tables share the array with the workspace: a
# generous bound on their size (an int4 per warp, an int2 per block row)
TABLES_MARGIN = 256 << 10


@pytest.fixture(scope="module")
def lib():
    import torch

    import symmetric_matrix_vector_gb300 as xs

    _build.build()
    xs.load()
    torch.cuda.set_device(0)
    xs.xsymv_set_variant("s", -1)
    xs.xsymv_set_stream(torch.cuda.current_stream().cuda_stream)
    yield xs
    xs.xsymv_set_variant("s", -1)


def _noalloc(xs):
    fn = xs.load().xsymv_s_noalloc
    fn.argtypes = [ctypes.c_char, ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_int,
                   ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_int]
    fn.restype = ctypes.c_int
    return fn


def _call(fn, uplo, n, alpha, A, lda, x, incx, beta, y, incy):
    return fn(uplo.encode(), n, alpha, ctypes.c_void_p(A.data_ptr()), lda,
              ctypes.c_void_p(x.data_ptr()), incx, beta, ctypes.c_void_p(y.data_ptr()), incy)


def largest_accepted_n(xs, uplo="U"):
    """the largest n (a multiple of 64, below 32768) whose workspace and plan
    tables fit the 16 MiB array, by the library's own workspace estimate"""
    for n in range(32768, 1024, -64):
        ws = xs.xsymv_workspace_bytes("s", uplo, n)
        if 0 < ws and (ws + 255) // 256 * 256 + TABLES_MARGIN <= SCRATCH_BYTES:
            return n
    raise AssertionError("no size fits the array")


def _check_case(xs, fn, uplo, n, lda, alpha, beta, incy, rows=None):
    p = inputs.make_problem("s", uplo, n, lda=lda, alpha=alpha, beta=beta, incy=incy, seed=n)
    A, x, y0 = to_device(p.A), to_device(p.x), to_device(p.y)
    y_ref = y0.clone()
    assert xs.xsymv_s(uplo, n, alpha, A, p.lda, x, 1, beta, y_ref, incy) == 0
    for call in range(2):
        y = y0.clone()
        st = _call(fn, uplo, n, alpha, A, p.lda, x, 1, beta, y, incy)
        assert st == 0, (call, st)
        assert xs.xsymv_sync_status() == 0
        got = from_device(y, p.y)
        # against the oracle (componentwise, normalised by |alpha||A||x| + |beta||y|)
        err, _ = errors(oracle.get(), p, got, rows=rows)
        assert float(np.max(err)) <= TOL["s"], (uplo, n, call, float(np.max(err)))
        # the same kernels on the same plan as xsymv_s: the same bytes
        assert bool((y == y_ref).all()), ("differs from xsymv_s", uplo, n, call)
        # the gap elements of a strided y are never written
        if abs(incy) > 1:
            idx = set((np.arange(n) * abs(incy)).tolist())
            assert all(np.isnan(got[k]) for k in range(len(got)) if k not in idx)


def test_noalloc_matches_oracle_and_xsymv_s_twice(lib):
    fn = _noalloc(lib)
    for uplo, n, incy in (("U", 3000, 1), ("L", 4097, -2), ("U", 1, 1), ("L", 257, 3)):
        _check_case(lib, fn, uplo, n, n + 5, 1.25, 0.5, incy)


def test_noalloc_largest_accepted_size(lib):
    """just below the array's limit (n about 31000): sampled rows against the
    oracle, bitwise equal to xsymv_s, two calls in a row"""
    fn = _noalloc(lib)
    n = largest_accepted_n(lib)
    assert n > 24576, n
    _check_case(lib, fn, "U", n, n, 1.0, 0.0, 1, rows=sample_rows(n, count=128, seed=n))


def test_noalloc_one_launch_variant(lib):
    """the allocation-free entry with a one-launch variant forced (its grid
    barrier's word lives in the array's header): against the oracle and, bit
    for bit, against xsymv_s with the same variant, two calls in a row"""
    fn = _noalloc(lib)
    fused = [v for v in range(lib.xsymv_variant_count("s"))
             if lib.xsymv_variant_name("s", v).endswith("_f")]
    assert fused
    try:
        for v in fused[:2]:
            assert lib.xsymv_set_variant("s", v) == 0
            _check_case(lib, fn, "U", 8192, 8192 + 4, 1.25, 0.5, 1,
                        rows=sample_rows(8192, count=128, seed=v))
            _check_case(lib, fn, "L", 3001, 3001, 1.0, 0.0, -1)
    finally:
        lib.xsymv_set_variant("s", -1)


def test_noalloc_alpha_zero(lib):
    """alpha = 0: y := beta*y, neither A nor x read (NaN bytes there are
    harmless), equal to xsymv_s's result"""
    import torch

    fn = _noalloc(lib)
    n = 513
    p = inputs.make_problem("s", "L", n, lda=n, alpha=0.0, beta=0.5, seed=3)
    nanA = torch.full((n * n,), float("nan"), device="cuda")
    x = to_device(p.x).view(torch.float32)
    y0 = to_device(p.y).view(torch.float32)
    y_ref = y0.clone()
    assert lib.xsymv_s("L", n, 0.0, nanA, n, x, 1, 0.5, y_ref, 1) == 0
    for _ in range(2):
        y = y0.clone()
        assert _call(fn, "L", n, 0.0, nanA, n, x, 1, 0.5, y, 1) == 0
        got = y.cpu().numpy()
        err, _ = errors(oracle.get(), p, got)
        assert float(np.max(err)) <= TOL["s"]
        assert bool((y == y_ref).all())


def test_noalloc_rejects_too_large(lib):
    """A problem whose workspace exceeds the 16 MiB array is refused before
    anything is enqueued.  Every buffer handed over is as large as the
    arguments say (a full n-by-n matrix, x and y of n elements), so even a
    call that were wrongly accepted would only read and write valid memory."""
    import torch

    fn = _noalloc(lib)
    n = 36864
    assert lib.xsymv_workspace_bytes("s", "U", n) > SCRATCH_BYTES
    A = torch.zeros(n * n, dtype=torch.float32, device="cuda")    # 5.4 GB
    x = torch.ones(n, dtype=torch.float32, device="cuda")
    y = torch.full((n,), 3.0, dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    launches = lib.xsymv_launch_count()
    st = _call(fn, "U", n, 1.0, A, n, x, 1, 0.0, y, 1)
    assert st == XSYMV_ERR_TOO_LARGE
    assert lib.xsymv_launch_count() == launches
    torch.cuda.synchronize()
    assert bool((y == 3.0).all())
    assert "16 MiB" in lib.xsymv_status_string(st)
    del A
    torch.cuda.empty_cache()


def _tma_variant(xs):
    tma = [v for v in range(xs.xsymv_variant_count("s")) if "_t" in xs.xsymv_variant_name("s", v)
           and not xs.xsymv_variant_name("s", v).endswith("_tk")]
    assert tma
    return tma[0]


def test_noalloc_timeout_status_and_call_number_wrap(lib):
    """The bounded waits of the bulk-copy variant run out under the test hook
    (bytes announced on every ring barrier that never arrive; nothing
    faults): xsymv_sync_status reports the allocation-free call's timeout
    from the array's status word, y is NaN, and the next normal call is
    correct.  Call numbers that start again at 1 clear the status word
    first, so a failure under a large old number hides no later failure."""
    import torch

    fn = _noalloc(lib)
    n = 700
    p = inputs.make_problem("s", "U", n, lda=n, alpha=1.0, beta=0.0, seed=4)
    A = to_device(p.A).view(torch.float32)
    x = to_device(p.x).view(torch.float32)
    y0 = to_device(p.y).view(torch.float32)

    def run():
        y = y0.clone()
        st = _call(fn, "U", n, 1.0, A, n, x, 1, 0.0, y, 1)
        assert st == 0
        return y, lib.xsymv_sync_status()

    assert lib.xsymv_set_variant("s", _tma_variant(lib)) == 0
    try:
        good, st = run()
        assert st == 0
        err, _ = errors(oracle.get(), p, good.cpu().numpy())
        assert float(np.max(err)) <= TOL["s"]
        lib.xsymv_set_wait_limit(2_000_000)          # 2 ms
        lib.xsymv_test_stall(True)
        bad, st = run()
        assert st == XSYMV_ERR_TIMEOUT
        assert bool(torch.isnan(bad).all())
        lib.xsymv_test_stall(False)
        again, st = run()
        assert st == 0 and bool((again == good).all())
        # across the wrap of the call numbers
        assert lib.xsymv_test_set_call_number(0x7ffffffd) == 0
        lib.xsymv_test_stall(True)
        _, st = run()                                # call 0x7ffffffe fails
        assert st == XSYMV_ERR_TIMEOUT
        lib.xsymv_test_stall(False)
        again, st = run()                            # call 1: the word is cleared
        assert st == 0 and bool((again == good).all())
        lib.xsymv_test_stall(True)
        bad, st = run()                              # call 2 fails: reported
        assert st == XSYMV_ERR_TIMEOUT and bool(torch.isnan(bad).all())
    finally:
        lib.xsymv_test_stall(False)
        lib.xsymv_set_wait_limit(0)
        lib.xsymv_set_variant("s", -1)
    good2, st = run()
    assert st == 0
    err, _ = errors(oracle.get(), p, good2.cpu().numpy())
    assert float(np.max(err)) <= TOL["s"]
