"""The worked examples of tests/golden/ (equation (1) of "CUDA-xSYMV の実装と
評価", IPSJ 2014-HPC-146, written out by hand) through the C ABI on the GPU,
with every compiled variant: all values and intermediate results there are
exact, so every variant must return them bit for bit."""
import numpy as np
import pytest

from tests import golden_cases as G
from tests.gpu_helpers import from_device, to_device

pytestmark = pytest.mark.gpu

CASES = G.cases()


@pytest.fixture(scope="module")
def lib():
    import torch

    import symmetric_matrix_vector_gb300 as xs

    assert torch.cuda.is_available()
    xs.load()
    assert xs.xsymv_set_stream(torch.cuda.current_stream().cuda_stream) == 0
    yield xs
    for k in "sdczw":
        xs.xsymv_set_variant(k, -1)


@pytest.mark.parametrize("case", CASES, ids=[c["name"] for c in CASES])
def test_worked_examples_every_variant(lib, case):
    kind, uplo, n = case["kind"], case["uplo"], case["n"]
    A, lda = G.stored_matrix(case)
    x = G.stored_vector(case, "x", case["incx"])
    y0 = G.stored_vector(case, "y0", case["incy"])
    al, be = G.scalars(case)
    want = G.expected(case)
    dA, dx = to_device(A), to_device(x)
    try:
        for v in [-1] + list(range(lib.xsymv_variant_count(kind))):
            assert lib.xsymv_set_variant(kind, v) == 0
            dy = to_device(y0)
            st = lib.symv(kind, uplo, n, al, dA, lda, dx, case["incx"], be, dy, case["incy"])
            assert st == 0
            got = G.logical(case, from_device(dy, y0), case["incy"])
            name = "tuned" if v < 0 else lib.xsymv_variant_name(kind, v)
            assert np.array_equal(got, want), (case["name"], name, got, want)
            assert lib.xsymv_sync_status() == 0
    finally:
        lib.xsymv_set_variant(kind, -1)
