"""GPU parity of the ordered-ticket variants ("_tk"): the report's own
accumulation ("CUDA-xSYMV の実装と評価", IPSJ 2014-HPC-146, §2.1, figures
"kernel" and "Atomic": dynamic block IDs, per-chunk tickets passed on in a
fixed order), in one launch.  Checked through the C ABI against the CPU
oracle element by element, for bit-identical repeats, for its bounded waits
(a withheld ticket makes them run out: the host reads XSYMV_ERR_TIMEOUT, the
outputs whose sums could not complete are NaN, and the next call is correct),
and against the workspace variants' results."""
import numpy as np
import pytest

from symmetric_matrix_vector_gb300 import inputs
from tests.gpu_helpers import TOL, DeviceProblem, errors, from_device, logical, sample_rows

pytestmark = pytest.mark.gpu

KINDS = ("s", "d", "c", "z", "w")
SCAL = {
    "s": (1.25, 0.5), "d": (-0.75, 2.0), "c": (complex(1.0, 0.5), complex(0.5, -0.25)),
    "z": (complex(1.0, 0.5), complex(0.5, -0.25)), "w": ((1.0, 2.0 ** -60), (0.5, 0.0)),
}
ERR_TIMEOUT = -6
ERR_VALUE = -4


@pytest.fixture(scope="module")
def o():
    import oracle

    return oracle.get()


@pytest.fixture(scope="module")
def lib():
    import torch

    import symmetric_matrix_vector_gb300 as xs

    assert torch.cuda.is_available()
    xs.load()
    assert xs.xsymv_set_stream(torch.cuda.current_stream().cuda_stream) == 0
    yield xs
    for k in KINDS:
        xs.xsymv_set_variant(k, -1)


def ticket_variants(lib, kind):
    v = [i for i in range(lib.xsymv_variant_count(kind))
         if lib.xsymv_variant_name(kind, i).endswith("_tk")]
    assert v, kind
    return v


class forced:
    """force one variant of a kind for the duration of a with-block"""

    def __init__(self, lib, kind, index):
        self.lib, self.kind, self.index = lib, kind, index

    def __enter__(self):
        assert self.lib.xsymv_set_variant(self.kind, self.index) == 0

    def __exit__(self, *a):
        self.lib.xsymv_set_variant(self.kind, -1)


def check(o, p, y, rows=None):
    err, _ = errors(o, p, y, rows=rows)
    assert np.max(err) <= TOL[p.kind], (p.kind, p.uplo, p.n, float(np.max(err)))


SIZES = [1, 2, 3, 31, 32, 33, 127, 128, 129, 255, 256, 257, 300, 513, 1000]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("uplo", ["U", "L"])
def test_ticket_sizes(o, lib, kind, uplo):
    """every ticket variant, ragged tails and tile boundaries, both triangles"""
    al, be = SCAL[kind]
    for v in ticket_variants(lib, kind):
        with forced(lib, kind, v):
            for n in SIZES:
                p = inputs.make_problem(kind, uplo, n, lda=n + (n % 3), alpha=al, beta=be,
                                        seed=n + 17 * v)
                st, yd = DeviceProblem(p).run()
                assert st == 0
                check(o, p, from_device(yd, p.y))


@pytest.mark.parametrize("kind", KINDS)
def test_ticket_strides_and_beta_zero(o, lib, kind):
    """negative and non-unit strides; beta = 0 with NaN in y (not read)"""
    import torch

    al, _ = SCAL[kind]
    zero = (0.0, 0.0) if kind == "w" else 0.0
    with forced(lib, kind, ticket_variants(lib, kind)[0]):
        for uplo, incx, incy in (("U", -2, 3), ("L", 3, -1)):
            p = inputs.make_problem(kind, uplo, 600, lda=601, alpha=al, beta=zero, incx=incx,
                                    incy=incy, seed=5)
            dp = DeviceProblem(p)
            st, yd = dp.run(y=torch.full_like(dp.y0, 0xFF))
            assert st == 0
            y = from_device(yd, p.y)
            check(o, p, y)
            # the gaps between y's elements are not written (still all-ones bytes)
            idx = set((np.arange(p.n) * abs(incy)).tolist())
            raw = yd.cpu().numpy().reshape(len(y), -1)
            assert all(np.all(raw[k] == 0xFF) for k in range(len(y)) if k not in idx)


@pytest.mark.parametrize("kind", KINDS)
def test_ticket_bitwise_repeatable(lib, kind):
    """ten repeats give identical bytes, also with other work running on a
    second stream (which changes which blocks start first, hence which warp
    gets which dynamic ID)"""
    import torch

    al, be = SCAL[kind]
    n = {"s": 6000, "d": 4000, "c": 3000, "z": 2500, "w": 1500}[kind]
    p = inputs.make_problem(kind, "U", n, lda=n + 8, alpha=al, beta=be, seed=21)
    dp = DeviceProblem(p)
    noise_stream = torch.cuda.Stream()
    big = torch.randn(1 << 24, device="cuda")
    for v in ticket_variants(lib, kind):
        with forced(lib, kind, v):
            st, first = dp.run()
            assert st == 0
            for r in range(10):
                if r % 2:
                    with torch.cuda.stream(noise_stream):
                        for _ in range(4):
                            big.mul_(1.0001)
                st, again = dp.run()
                assert st == 0
                assert bool((first == again).all()), (kind, v, "repeat", r)
    torch.cuda.synchronize()


FULL = [("ssymv_sweep", 32768), ("ssymv_sweep", 8192), ("dsymv", None), ("chemv", None),
        ("zhemv", None), ("wsymv", None)]


@pytest.mark.parametrize("name,n", FULL, ids=["%s_%s" % (a, b or "full") for a, b in FULL])
def test_ticket_full_size_sampled(o, lib, name, n):
    """the workloads at full size, sampled rows against the oracle, bitwise
    repeats, and agreement with the workspace variant within tolerance"""
    p = inputs.workload(name, n=n)
    dp = DeviceProblem(p)
    rows = sample_rows(p.n, count=128, seed=p.n + 1)
    st, yw = dp.run()                      # the tuned (workspace) variant
    assert st == 0
    for v in ticket_variants(lib, p.kind):
        with forced(lib, p.kind, v):
            st, y1 = dp.run()
            assert st == 0
            y = from_device(y1, p.y)
            assert np.all(np.isfinite(logical(p.kind, y, p.n, p.incy)))
            check(o, p, y, rows=rows)
            st, y2 = dp.run()
            assert st == 0 and bool((y1 == y2).all())
    check(o, p, from_device(yw, p.y), rows=rows)


def test_ticket_single_launch(lib):
    """an ordered-ticket call is one kernel launch (no finaliser)"""
    p = inputs.make_problem("s", "U", 1000, alpha=1.0, beta=0.5, seed=1)
    dp = DeviceProblem(p)
    with forced(lib, "s", ticket_variants(lib, "s")[0]):
        st, _ = dp.run()    # a new plan: its tables are built once (one more launch)
        assert st == 0
        c0 = lib.xsymv_launch_count()
        for _ in range(5):
            st, _ = dp.run()
            assert st == 0
        assert lib.xsymv_launch_count() - c0 == 5


@pytest.mark.parametrize("kind", ["s", "z"])
def test_ticket_withheld_reports_timeout(o, lib, kind):
    """The test hook makes every chain's first contributor keep its ticket:
    every other contributor's bounded wait runs out (nothing faults), the
    host reads XSYMV_ERR_TIMEOUT, every output whose sum could not complete
    is NaN, and the next normal call on the same context is correct."""
    al, be = SCAL[kind]
    n = 1500
    p = inputs.make_problem(kind, "L", n, lda=n, alpha=al, beta=be, seed=2)
    dp = DeviceProblem(p)
    with forced(lib, kind, ticket_variants(lib, kind)[0]):
        st, good = dp.run()
        assert st == 0 and lib.xsymv_sync_status() == 0
        try:
            lib.xsymv_set_wait_limit(2_000_000)          # 2 ms
            lib.xsymv_test_stall(True)
            st, bad = dp.run()
            assert st == 0
            assert lib.xsymv_sync_status() == ERR_TIMEOUT
            yb = logical(kind, from_device(bad, p.y), n, 1)
            # at this size every chunk has several contributors: no chain completes
            assert np.all(np.isnan(yb.astype(np.complex128) if kind == "z" else yb))
        finally:
            lib.xsymv_test_stall(False)
            lib.xsymv_set_wait_limit(0)
        st, again = dp.run()
        assert st == 0 and lib.xsymv_sync_status() == 0
        assert bool((again == good).all())
        check(o, p, from_device(again, p.y))


def test_noalloc_refuses_ticket_variant(lib):
    """the allocation-free entry point has no ticket buffer: a forced ticket
    variant is refused with nothing enqueued"""
    import torch

    import ctypes

    fn = lib.load().xsymv_s_noalloc
    fn.argtypes = [ctypes.c_char, ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_int,
                   ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_int]
    fn.restype = ctypes.c_int
    p = inputs.make_problem("s", "U", 500, alpha=1.0, beta=0.0, seed=3)
    dp = DeviceProblem(p)
    y = dp.y0.clone()
    with forced(lib, "s", ticket_variants(lib, "s")[0]):
        st = fn(b"U", p.n, 1.0, dp.A.data_ptr(), p.lda, dp.x.data_ptr(), 1, 0.0, y.data_ptr(), 1)
    assert st == ERR_VALUE
    torch.cuda.synchronize()
    assert bool((y == dp.y0).all())
