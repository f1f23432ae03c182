"""GPU parity of the block-column split (one xSYMV / xHEMV call cut into
panels of stored columns, one per GPU, each streamed by the ``*_shard``
entry point into a full-length partial vector, then added in rank order and
merged with alpha and beta by ``*_reduce``).  The report cites multi-GPU
Level-2 BLAS (its reference [7], KBLAS, §1 of "CUDA-xSYMV の実装と評価", IPSJ
2014-HPC-146) without a split of its own; this is the plainest reading.

Here every shard runs on the one GPU, one after another, each panel in its
own allocation (as it would sit in its own GPU's memory); nothing waits on
anything but the stream.  Results are compared with the CPU oracle on every
row and must repeat bit for bit."""
import numpy as np
import pytest

import oracle
from symmetric_matrix_vector_gb300 import inputs
from tests.gpu_helpers import TOL, errors, from_device, to_device

pytestmark = pytest.mark.gpu

KINDS = ("s", "d", "c", "z", "w")
SCAL = {
    "s": (1.25, 0.5), "d": (-0.75, 2.0), "c": (complex(1.0, 0.5), complex(0.5, -0.25)),
    "z": (complex(1.0, 0.5), complex(0.5, -0.25)), "w": ((1.0, 2.0 ** -60), (0.5, 0.0)),
}
SIZE = {"s": 1300, "d": 1100, "c": 900, "z": 700, "w": 520}


@pytest.fixture(scope="module")
def o():
    return oracle.get()


@pytest.fixture(scope="module", autouse=True)
def lib():
    import torch

    import symmetric_matrix_vector_gb300 as xs

    assert torch.cuda.is_available()
    xs.load()
    for k in KINDS:
        xs.xsymv_set_variant(k, -1)
    yield xs


def run_shards(xs, p, bounds, alpha=None, beta=None, y=None, pad=0):
    """every panel in its own device array, its shard into row r of one
    partials buffer, then the reduction; returns the device y"""
    import torch

    from symmetric_matrix_vector_gb300 import sharded

    A = to_device(p.A)
    x = to_device(p.x)
    yd = to_device(p.y) if y is None else y
    es = inputs.ELEM_BYTES[p.kind]
    N = len(bounds) - 1
    parts = torch.full((N, p.n * es), 0xFF, dtype=torch.uint8, device="cuda")   # NaN bytes
    panels = []
    for r in range(N):
        c0, c1 = bounds[r], bounds[r + 1]
        panel, ldp = sharded.extract_panel(torch, A, p.kind, p.uplo, p.n, p.lda, c0, c1, pad=pad)
        panels.append(panel)
        st = xs.symv_shard(p.kind, p.uplo, p.n, c0, c1, panel, ldp, x, p.incx, parts[r])
        assert st == 0, (r, st)
    st = xs.symv_reduce(p.kind, p.n, N, p.alpha if alpha is None else alpha, parts, p.n,
                        p.beta if beta is None else beta, yd, p.incy)
    assert st == 0, st
    return yd, parts


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("uplo", ["U", "L"])
def test_shards_match_oracle(o, lib, kind, uplo):
    """N = 1, 2, 3 and 8 even panels: all rows against the oracle, and the
    same bytes on a second run"""
    al, be = SCAL[kind]
    n = SIZE[kind]
    p = inputs.make_problem(kind, uplo, n, lda=n + 3, alpha=al, beta=be, seed=50 + n)
    for N in (1, 2, 3, 8):
        bounds = lib.xsymv_shard_bounds(uplo, n, N)
        y1, _ = run_shards(lib, p, bounds)
        err, _ = errors(o, p, from_device(y1, p.y))
        assert np.max(err) <= TOL[kind], (kind, uplo, N, float(np.max(err)))
        y2, _ = run_shards(lib, p, bounds)
        assert bool((y1 == y2).all()), ("not bitwise repeatable", kind, uplo, N)


@pytest.mark.parametrize("kind", KINDS)
def test_single_shard_equals_plain_call(lib, kind):
    """one panel holding the whole triangle, reduced with N = 1, gives the
    plain call's bytes (same kernels, plan and final rounding)"""
    from tests.gpu_helpers import DeviceProblem

    al, be = SCAL[kind]
    n = SIZE[kind]
    for uplo in ("U", "L"):
        p = inputs.make_problem(kind, uplo, n, lda=n, alpha=al, beta=be, seed=60 + n)
        ys, _ = run_shards(lib, p, [0, n])
        st, yp = DeviceProblem(p).run()
        assert st == 0
        assert bool((ys == yp).all()), (kind, uplo)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("uplo", ["U", "L"])
def test_shards_odd_boundaries_and_strides(o, lib, kind, uplo):
    """panels whose edges are off the 16-byte grid (element loads), padded
    panels on the grid (vector loads), empty panels, negative and strided
    vectors, NaN in y with beta = 0"""
    import torch

    al, be = SCAL[kind]
    n = 611
    p = inputs.make_problem(kind, uplo, n, lda=n + 1, alpha=al, beta=be, incx=-2, incy=3,
                            seed=70)
    for bounds, pad in (([0, 37, 301, 302, 555, n], 0), ([0, 0, 160, 160, 448, n], 5),
                        ([0, n, n], 3)):
        y, _ = run_shards(lib, p, bounds, pad=pad)
        yl = from_device(y, p.y)
        err, _ = errors(o, p, yl)
        assert np.max(err) <= TOL[kind], (kind, uplo, bounds, float(np.max(err)))
        # the gaps of a strided y are never written
        idx = set((np.arange(n) * 3).tolist())
        assert all(np.all(np.isnan(yl[k])) for k in range(len(yl)) if k not in idx)
    zero = (0.0, 0.0) if kind == "w" else 0.0
    ynan = torch.full_like(to_device(p.y), 0xFF)
    y, _ = run_shards(lib, p, lib.xsymv_shard_bounds(uplo, n, 4), beta=zero, y=ynan)
    err, _ = errors(o, p, from_device(y, p.y), beta=zero)
    assert np.max(err) <= TOL[kind]


@pytest.mark.parametrize("kind", KINDS)
def test_reduce_special_scalars(o, lib, kind):
    """alpha = 0 reads no partial vector (NaN there is harmless); alpha = 0
    and beta = 1 touches nothing"""
    import torch

    n = 300
    al, be = SCAL[kind]
    zero = (0.0, 0.0) if kind == "w" else 0.0
    one = (1.0, 0.0) if kind == "w" else 1.0
    p = inputs.make_problem(kind, "U", n, lda=n, alpha=al, beta=be, seed=80)
    es = inputs.ELEM_BYTES[kind]
    nan_parts = torch.full((3, n * es), 0xFF, dtype=torch.uint8, device="cuda")
    y = to_device(p.y)
    assert lib.symv_reduce(kind, n, 3, zero, nan_parts, n, be, y, 1) == 0
    err, _ = errors(o, p, from_device(y, p.y), alpha=zero)
    assert np.max(err) <= TOL[kind]
    y0 = y.clone()
    assert lib.symv_reduce(kind, n, 3, zero, nan_parts, n, one, y, 1) == 0
    torch.cuda.synchronize()
    assert bool((y == y0).all())


def test_reduce_adds_in_rank_order(lib):
    """fp32 partials 1e8, -1e8, 1 (in rank order) sum to 1 only when added
    left to right; the reverse order gives 0"""
    import torch

    n = 1000
    P = torch.empty((3, n), dtype=torch.float32, device="cuda")
    P[0], P[1], P[2] = 1e8, -1e8, 1.0
    y = torch.full((n,), 5.0, device="cuda")
    assert lib.xsymv_s_reduce(n, 3, 1.0, P, n, 0.0, y, 1) == 0
    assert bool((y == 1.0).all())
    Pr = P.flip(0).contiguous()
    assert lib.xsymv_s_reduce(n, 3, 1.0, Pr, n, 0.0, y, 1) == 0
    assert bool((y == 0.0).all())


@pytest.mark.parametrize("kind,uplo,n,N", [("s", "U", 16384, 8), ("s", "L", 12288, 3),
                                           ("c", "U", 8192, 4), ("d", "L", 8192, 2)])
def test_shards_large(o, lib, kind, uplo, n, N):
    """larger problems: every row against the oracle, bitwise repeats"""
    al, be = SCAL[kind]
    p = inputs.make_problem(kind, uplo, n, lda=n, alpha=al, beta=be, seed=n + N)
    bounds = lib.xsymv_shard_bounds(uplo, n, N)
    y1, _ = run_shards(lib, p, bounds)
    err, _ = errors(o, p, from_device(y1, p.y))
    assert np.max(err) <= TOL[kind], (kind, uplo, n, N, float(np.max(err)))
    y2, _ = run_shards(lib, p, bounds)
    assert bool((y1 == y2).all())
