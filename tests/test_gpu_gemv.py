"""GPU parity of the general product xgemv_s / xgemv_d (the comparison the
CUDA-xSYMV report makes in §1) against the oracle's definition, through the
C ABI: sizes spanning several tiles with ragged tails, strides, every
compiled variant, special scalars, run-to-run bit identity and the full
comparison size on sampled rows."""
import numpy as np
import pytest

import oracle
import symmetric_matrix_vector_gb300 as xs
from symmetric_matrix_vector_gb300 import inputs
from tests.gpu_helpers import TOL, from_device, logical, sample_rows, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def o():
    return oracle.get()


def run_gemv(p, alpha=None, beta=None, y=None, A=None):
    A_d = to_device(p.A) if A is None else A
    x_d = to_device(p.x)
    y_d = to_device(p.y) if y is None else y
    st = xs.gemv(p.kind, p.n, p.alpha if alpha is None else alpha, A_d, p.lda, x_d, p.incx,
                 p.beta if beta is None else beta, y_d, p.incy)
    return st, y_d


def gemv_errors(o, p, y_gpu, rows=None, alpha=None, beta=None):
    rows = np.arange(p.n) if rows is None else np.asarray(rows, dtype=np.int64)
    info, hi, lo, den = o.gemv_rows(p.kind, p.n, p.alpha if alpha is None else alpha, p.A, p.lda,
                                    p.x, p.incx, p.beta if beta is None else beta, p.y, p.incy,
                                    rows)
    assert info == 0
    yl = logical(p.kind, y_gpu, p.n, p.incy)[rows].astype(np.float64)
    with np.errstate(invalid="ignore", divide="ignore"):
        err = np.abs((yl - hi) - lo)
        rel = np.where(den > 0, err / np.where(den > 0, den, 1.0), err)
    rel[~np.isfinite(rel)] = np.inf
    return rel


@pytest.mark.parametrize("kind", ["s", "d"])
@pytest.mark.parametrize("n", [1, 3, 31, 128, 129, 257, 1000, 2111])
def test_sizes(o, kind, n):
    p = inputs.make_general(kind, n, lda=n + 5, alpha=1.25, beta=-0.5, seed=n)
    st, y = run_gemv(p)
    assert st == 0
    yh = from_device(y, p.y)
    assert gemv_errors(o, p, yh).max() <= TOL[kind]


@pytest.mark.parametrize("kind", ["s", "d"])
@pytest.mark.parametrize("incx,incy", [(2, 1), (-1, 3), (1, -2), (-3, -1)])
def test_strides(o, kind, incx, incy):
    n = 700
    p = inputs.make_general(kind, n, lda=n, alpha=-0.75, beta=2.0, incx=incx, incy=incy, seed=3)
    st, y = run_gemv(p)
    assert st == 0
    yh = from_device(y, p.y)
    assert gemv_errors(o, p, yh).max() <= TOL[kind]
    # gap elements of y stay untouched (NaN)
    idx = set((np.arange(n) * abs(incy)).tolist())
    gaps = [k for k in range(len(p.y)) if k not in idx]
    assert np.all(np.isnan(yh[gaps]))


@pytest.mark.parametrize("kind", ["s", "d"])
def test_every_variant(o, kind):
    n = 1543
    p = inputs.make_general(kind, n, lda=n + 3, alpha=0.5, beta=1.5, seed=4)
    A_d = to_device(p.A)
    try:
        for v in range(xs.xgemv_variant_count(kind)):
            assert xs.xgemv_set_variant(kind, v) == 0
            st, y = run_gemv(p, A=A_d)
            assert st == 0
            err = gemv_errors(o, p, from_device(y, p.y)).max()
            assert err <= TOL[kind], (xs.xgemv_variant_name(kind, v), err)
    finally:
        xs.xgemv_set_variant(kind, -1)


@pytest.mark.parametrize("kind", ["s", "d"])
def test_unaligned_matrix(o, kind):
    # lda*sizeof not a multiple of 16: the element-load path
    n = 601
    p = inputs.make_general(kind, n, lda=n, alpha=1.0, beta=0.0, seed=5)
    st, y = run_gemv(p)
    assert st == 0
    assert gemv_errors(o, p, from_device(y, p.y)).max() <= TOL[kind]


@pytest.mark.parametrize("kind", ["s", "d"])
def test_special_scalars(o, kind):
    import torch

    n = 300
    p = inputs.make_general(kind, n, lda=n, alpha=1.0, beta=0.5, seed=6)
    # alpha = 0: y := beta*y without reading A or x (NaN there)
    nanA = torch.full_like(to_device(p.A), 255)
    st, y = run_gemv(p, alpha=0.0, A=nanA)
    assert st == 0
    assert np.array_equal(from_device(y, p.y), (p.y * p.y.dtype.type(0.5)))
    # beta = 0: y is overwritten without being read
    ynan = torch.full_like(to_device(p.y), 255)
    st, y = run_gemv(p, beta=0.0, y=ynan)
    assert st == 0
    assert gemv_errors(o, p, from_device(y, p.y), beta=0.0).max() <= TOL[kind]
    # alpha = 0, beta = 1: nothing is written
    ynan = torch.full_like(to_device(p.y), 255)
    st, y = run_gemv(p, alpha=0.0, beta=1.0, y=ynan)
    assert st == 0 and torch.all(y == 255)


@pytest.mark.parametrize("kind", ["s", "d"])
def test_bitwise_repeatable(kind):
    import torch

    n = 4099
    d = inputs.device_general(kind, n, lda=n + 1, alpha=1.0, beta=0.25, seed=8)
    outs = []
    for _ in range(3):
        y = d["y"].clone()
        assert xs.gemv(kind, n, 1.0, d["A"], n + 1, d["x"], 1, 0.25, y, 1) == 0
        outs.append(y)
    torch.cuda.synchronize()
    assert all(torch.equal(outs[0], t) for t in outs[1:])


@pytest.mark.parametrize("kind,n", [("s", 32768), ("d", 24576)])
def test_full_size_sampled(o, kind, n):
    """the size the benchmark compares SYMV and GEMV at, sampled rows"""
    import torch

    d = inputs.device_general(kind, n, lda=n + 32, alpha=1.0, beta=0.0, seed=n)
    y = torch.empty_like(d["y"])
    assert xs.gemv(kind, n, 1.0, d["A"], n + 32, d["x"], 1, 0.0, y, 1) == 0
    torch.cuda.synchronize()
    A = d["A"].cpu().numpy()
    x = d["x"].cpu().numpy()
    yh = y.cpu().numpy()
    del d
    p = inputs.Problem(kind=kind, uplo="G", n=n, lda=n + 32, alpha=1.0, beta=0.0, A=A, x=x,
                       y=np.zeros_like(yh))
    rows = sample_rows(n, count=48, seed=n)
    assert gemv_errors(o, p, yh, rows=rows).max() <= TOL[kind]
