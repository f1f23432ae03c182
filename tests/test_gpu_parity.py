"""GPU parity: the CUDA library through its C ABI against the CPU oracle,
element by element on seeded inputs (componentwise error normalised by
|alpha||A||x| + |beta||y|), plus bitwise run-to-run identity and the BLAS
edge cases.  The operation is equation (1) of "CUDA-xSYMV の実装と評価"
(IPSJ 2014-HPC-146): y := alpha*A*x + beta*y, one triangle of A stored."""
import numpy as np
import pytest

import oracle
from symmetric_matrix_vector_gb300 import inputs
from tests.gpu_helpers import TOL, DeviceProblem, errors, from_device, logical, sample_rows

pytestmark = pytest.mark.gpu

KINDS = ("s", "d", "c", "z", "w")
SCAL = {
    "s": (1.25, 0.5), "d": (-0.75, 2.0), "c": (complex(1.0, 0.5), complex(0.5, -0.25)),
    "z": (complex(1.0, 0.5), complex(0.5, -0.25)), "w": ((1.0, 2.0 ** -60), (0.5, 0.0)),
}


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
    for k in KINDS:
        xs.xsymv_set_variant(k, -1)


def run_and_check(o, p, rows=None, **kw):
    dp = DeviceProblem(p)
    st, yd = dp.run(**kw)
    assert st == 0, st
    y = from_device(yd, p.y)
    err, _ = errors(o, p, y, rows=rows, alpha=kw.get("alpha"), beta=kw.get("beta"))
    assert np.max(err) <= TOL[p.kind], (p.kind, p.uplo, p.n, float(np.max(err)))
    return y


# ---------------------------------------------------------------- sizes ----
SIZES = [1, 2, 3, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257, 300, 513]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("uplo", ["U", "L"])
def test_sizes_and_ragged_tails(o, kind, uplo):
    al, be = SCAL[kind]
    for n in SIZES:
        p = inputs.make_problem(kind, uplo, n, lda=n + (n % 3), alpha=al, beta=be, seed=n)
        run_and_check(o, p)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("uplo", ["U", "L"])
@pytest.mark.parametrize("incx,incy", [(2, -1), (-3, 2), (-1, -1)])
def test_strides(o, kind, uplo, incx, incy):
    al, be = SCAL[kind]
    for n in (45, 200):
        p = inputs.make_problem(kind, uplo, n, lda=n + 1, alpha=al, beta=be, incx=incx,
                                incy=incy, seed=7 + n)
        y = run_and_check(o, p)
        # gap elements of y are never written (they stay NaN)
        idx = set((np.arange(n) * abs(incy)).tolist())
        gaps = [k for k in range(len(y)) if k not in idx]
        assert all(np.all(np.isnan(y[k])) for k in gaps)


@pytest.mark.parametrize("kind", KINDS)
def test_every_variant(o, lib, kind):
    """each compiled kernel variant (the tuner's space) is correct"""
    al, be = SCAL[kind]
    try:
        for v in range(lib.xsymv_variant_count(kind)):
            assert lib.xsymv_set_variant(kind, v) == 0
            for uplo in ("U", "L"):
                # 16-byte aligned columns (vector loads, also in the diagonal
                # tiles) and unaligned ones (element loads), ragged tails;
                # 1300: three block rows of 512
                for n, lda in ((97, 99), (700, 704), (1300, 1302), (1301, 1304)):
                    p = inputs.make_problem(kind, uplo, n, lda=lda, alpha=al, beta=be,
                                            seed=100 + v)
                    run_and_check(o, p)
    finally:
        lib.xsymv_set_variant(kind, -1)


@pytest.mark.parametrize("kind", KINDS)
def test_unaligned_matrix(o, kind):
    """lda and base address off the 16-byte grid take the element-load path"""
    import torch

    al, be = SCAL[kind]
    n = 301
    p = inputs.make_problem(kind, "U", n, lda=n, alpha=al, beta=be, seed=3)
    dp = DeviceProblem(p)
    esz = p.A.itemsize * (2 if kind == "w" else 1)
    # shift A off the 16-byte grid (by one element, or half of a 16-byte one)
    off = esz if esz < 16 else 8
    buf = torch.zeros(dp.A.numel() + 64, dtype=torch.uint8, device="cuda")
    buf[off:off + dp.A.numel()] = dp.A
    st, yd = dp.run(A=buf[off:])
    assert st == 0
    err, _ = errors(o, p, from_device(yd, p.y))
    assert np.max(err) <= TOL[kind]


# ------------------------------------------------------------ workloads ----
@pytest.mark.parametrize("name", ["ssymv_small", "dsymv", "chemv", "zhemv", "wsymv"])
def test_workloads_small_n(o, name):
    """the five named workloads' recipes (uplo, lda, scalars, NaN sentinels)
    at sizes the oracle checks row by row in seconds"""
    n = {"ssymv_small": 1024, "dsymv": 1100, "chemv": 900, "zhemv": 700, "wsymv": 520}[name]
    p = inputs.workload(name, n=n)
    run_and_check(o, p)


@pytest.mark.parametrize("n", [4096, 8192])
def test_sweep_points_all_rows(o, n):
    """two points of the size sweep, every row against the oracle's row-by-row
    coding of the definition"""
    p = inputs.workload("ssymv_sweep", n=n)
    run_and_check(o, p)


def all_rows_error(o, p, y_gpu):
    """Componentwise error of every row against the oracle's three-part
    algorithm (its binary64 / binary128 accumulator, for all n rows in one
    streaming pass), normalised by |alpha|(|A||x|)_i + |beta||y_i|: the
    normaliser is the same algorithm run on the moduli (real symmetric; a
    Hermitian diagonal counts with its real part only)."""
    n, k = p.n, p.kind
    assert p.incx == 1 and p.incy == 1
    info, _, hi, lo = o.symv(k, p.uplo, n, p.alpha, p.A, p.lda, p.x, 1, p.beta, p.y, 1)
    assert info == 0
    idx = np.arange(n)
    if k == "w":      # moduli of the high words (the low words change them by 2^-53 at most)
        M = np.abs(p.A[:, :p.lda, 0]).astype(np.float32)
        ax, ay = np.abs(p.x[:, 0]), np.abs(p.y[:, 0])
        al, be = abs(p.alpha[0]), abs(p.beta[0])
    else:
        M = np.abs(p.A[:, :p.lda]).astype(np.float32)
        if k in ("c", "z"):
            M[idx, idx] = np.abs(p.A[idx, idx].real)
        ax, ay = np.abs(p.x), np.abs(p.y)
        al, be = abs(complex(p.alpha)), abs(complex(p.beta))
    info, _, den, _ = o.symv("s", p.uplo, n, al, M, p.lda, ax.astype(np.float32), 1, be,
                             ay.astype(np.float32), 1)
    assert info == 0
    yl = logical(k, y_gpu, n, 1)
    if k == "w":
        err = np.abs((yl[:, 0] - hi) + (yl[:, 1] - lo))
    elif k in ("c", "z"):
        err = np.hypot((yl.real.astype(np.float64) - hi[:, 0]) - lo[:, 0],
                       (yl.imag.astype(np.float64) - hi[:, 1]) - lo[:, 1])
    else:
        err = np.abs((yl.astype(np.float64) - hi) - lo)
    return err / den


@pytest.mark.parametrize("name,n", [("ssymv_sweep", 32768), ("chemv", 16384), ("wsymv", 8192)])
def test_workloads_full_size_all_rows(o, name, n):
    """the largest single-precision workloads and the double-double one, in
    the benchmark's launch configuration, checked on every row"""
    p = inputs.workload(name, n=n)
    dp = DeviceProblem(p)
    st, yd = dp.run()
    assert st == 0
    err = all_rows_error(o, p, from_device(yd, p.y))
    assert np.all(np.isfinite(err))
    assert float(np.max(err)) <= TOL[p.kind], (name, float(np.max(err)))


FULL = [("ssymv_sweep", 16384), ("ssymv_sweep", 32768), ("dsymv", None), ("chemv", None),
        ("zhemv", None), ("wsymv", None)]


@pytest.mark.parametrize("name,n", FULL, ids=["%s_%s" % (a, b or "full") for a, b in FULL])
def test_workloads_full_size_sampled(o, name, n):
    """full sizes, in the benchmark's launch configuration, checked on
    sampled rows (each recomputed by the oracle from the definition), and
    bitwise identical across repeated calls"""
    p = inputs.workload(name, n=n)
    dp = DeviceProblem(p)
    st, y1 = dp.run()
    assert st == 0
    y = from_device(y1, p.y)
    assert np.all(np.isfinite(logical(p.kind, y, p.n, p.incy)))
    rows = sample_rows(p.n, count=160, seed=p.n)
    err, _ = errors(o, p, y, rows=rows)
    assert np.max(err) <= TOL[p.kind], (name, float(np.max(err)))
    for _ in range(3):
        st, y2 = dp.run()
        assert st == 0
        assert bool((y1 == y2).all()), "results differ between runs"


# --------------------------------------------------------- determinism -----
@pytest.mark.parametrize("kind", KINDS)
def test_bitwise_repeatable(kind):
    """ten repeats give identical bytes, also with other work running
    concurrently on a second stream"""
    import torch

    al, be = SCAL[kind]
    n = {"s": 6000, "d": 4000, "c": 3000, "z": 2500, "w": 1500}[kind]
    p = inputs.make_problem(kind, "U", n, lda=n + 8, alpha=al, beta=be, seed=21)
    dp = DeviceProblem(p)
    st, first = dp.run()
    assert st == 0
    noise_stream = torch.cuda.Stream()
    big = torch.randn(1 << 24, device="cuda")
    for r in range(10):
        if r % 2:
            with torch.cuda.stream(noise_stream):
                for _ in range(4):
                    big.mul_(1.0001)
        st, again = dp.run()
        assert st == 0
        assert bool((first == again).all()), ("repeat", r)
    torch.cuda.synchronize()


# ---------------------------------------------------------- edge cases -----
@pytest.mark.parametrize("kind", KINDS)
def test_special_scalars(o, kind):
    import torch

    n = 150
    p = inputs.make_problem(kind, "L", n, lda=n, alpha=SCAL[kind][0], beta=SCAL[kind][1],
                            seed=5)
    dp = DeviceProblem(p)
    zero = (0.0, 0.0) if kind == "w" else 0.0
    one = (1.0, 0.0) if kind == "w" else 1.0
    nanA = torch.full_like(dp.A, 0xFF)          # all-ones bytes: NaN in every type
    # alpha = 0: y := beta*y, A and x not read
    st, yd = dp.run(alpha=zero, A=nanA)
    assert st == 0
    err, _ = errors(o, p, from_device(yd, p.y), alpha=zero)
    assert np.max(err) <= TOL[kind]
    # alpha = 0, beta = 1: nothing is touched
    st, yd = dp.run(alpha=zero, beta=one, A=nanA)
    assert st == 0 and bool((yd == dp.y0).all())
    # beta = 0: y is not read (NaN input does not propagate)
    ynan = torch.full_like(dp.y0, 0xFF)
    st, yd = dp.run(beta=zero, y=ynan)
    assert st == 0
    err, _ = errors(o, p, from_device(yd, p.y), beta=zero)
    assert np.max(err) <= TOL[kind]


def test_n_zero_and_errors(lib):
    import torch

    y = torch.full((16,), 7.0, device="cuda")
    assert lib.xsymv_s("U", 0, 1.0, 0, 1, 0, 1, 0.0, y, 1) == 0
    assert lib.xsymv_s("Q", 4, 1.0, y, 4, y, 1, 0.0, y, 1) == 1
    assert lib.xsymv_s("U", -2, 1.0, y, 4, y, 1, 0.0, y, 1) == 2
    assert lib.xsymv_s("U", 4, 1.0, y, 3, y, 1, 0.0, y, 1) == 5
    assert lib.xsymv_s("U", 4, 1.0, y, 4, y, 0, 0.0, y, 1) == 7
    assert lib.xsymv_s("U", 4, 1.0, y, 4, y, 1, 0.0, y, 0) == 10
    torch.cuda.synchronize()
    assert bool((y == 7.0).all())


@pytest.mark.parametrize("kind", KINDS)
def test_y_guard_words(o, kind):
    """elements just before and after y are never written"""
    import torch

    n = 333
    p = inputs.make_problem(kind, "U", n, lda=n, alpha=SCAL[kind][0], beta=SCAL[kind][1],
                            seed=9)
    dp = DeviceProblem(p)
    guard = 64
    buf = torch.full((dp.y0.numel() + 2 * guard,), 0x5A, dtype=torch.uint8, device="cuda")
    buf[guard:guard + dp.y0.numel()] = dp.y0
    st, _ = dp.run(y=buf[guard:guard + dp.y0.numel()])
    assert st == 0
    torch.cuda.synchronize()
    assert bool((buf[:guard] == 0x5A).all()) and bool((buf[-guard:] == 0x5A).all())
    err, _ = errors(o, p, from_device(buf[guard:guard + dp.y0.numel()], p.y))
    assert np.max(err) <= TOL[kind]


def test_non_default_stream(o):
    import torch

    p = inputs.make_problem("s", "U", 2000, lda=2000, alpha=1.0, beta=0.0, seed=11)
    dp = DeviceProblem(p)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        st, yd = dp.run()
    assert st == 0
    s.synchronize()
    err, _ = errors(o, p, from_device(yd, p.y))
    assert np.max(err) <= TOL["s"]


@pytest.mark.parametrize("variant,per_call", [("vr2_u2_r0_w8_b4_g13", 2),
                                               ("vr2_u2_r0_w8_b4_g13_c2_f", 1)])
def test_launch_count_and_timing(lib, variant, per_call):
    """every call of a two-kernel variant launches exactly the main kernel and
    the finaliser, a one-launch variant one kernel (plus, on the first call of
    a plan, the kernel that builds its tables); a forced variant is used as
    is, even back to back"""
    names = [lib.xsymv_variant_name("s", i) for i in range(lib.xsymv_variant_count("s"))]
    assert lib.xsymv_set_variant("s", names.index(variant)) == 0
    try:
        p = inputs.make_problem("s", "U", 1000, alpha=1.0, beta=0.5, seed=1)
        dp = DeviceProblem(p)
        st, _ = dp.run()    # a new plan: its warp and row tables are built once (one more launch)
        assert st == 0
        c0 = lib.xsymv_launch_count()
        lib.xsymv_timing_enable(True)
        for _ in range(5):
            st, _ = dp.run()
            assert st == 0
        calls, main_ms, call_ms = lib.xsymv_timing_read()
        lib.xsymv_timing_enable(False)
        assert lib.xsymv_launch_count() - c0 == 5 * per_call
        assert calls == 5 and 0 < main_ms <= call_ms
    finally:
        lib.xsymv_set_variant("s", -1)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("uplo", ["U", "L"])
def test_host_buffer_entry(o, lib, kind, uplo):
    """the *_host entry points take host arrays, copy the triangle in panels
    and return with y written"""
    al, be = SCAL[kind]
    for n, incx, incy in ((1, 1, 1), (129, 1, 1), (300, -2, 3), (5000, 1, -1)):
        if kind in ("z", "w") and n == 5000:
            n = 2100
        p = inputs.make_problem(kind, uplo, n, lda=n + 3, alpha=al, beta=be, incx=incx, incy=incy,
                                seed=31 + n)
        y = p.y.copy()
        st = lib.symv_host(kind, uplo, n, al, p.A, p.lda, p.x, incx, be, y, incy)
        assert st == 0
        err, _ = errors(o, p, y)
        assert np.max(err) <= TOL[kind], (kind, uplo, n, float(np.max(err)))
        h2d, d2h = lib.xsymv_host_traffic()
        es = p.A.itemsize * (2 if kind == "w" else 1)
        assert d2h == n * es
        # only the triangle (plus a few percent in panel corners) travels
        assert h2d <= (n * (n + 1) / 2 * 1.05 + 2 * n + 64 * n) * es


@pytest.mark.parametrize("kind", KINDS)
def test_host_buffer_entry_pinned_zero_copy(o, lib, kind):
    """with page-locked host buffers the kernels read A, x and write y in
    place; the result is bitwise the device-buffer result"""
    import torch

    al, be = SCAL[kind]
    n = 777
    p = inputs.make_problem(kind, "L", n, lda=n + 4, alpha=al, beta=be, incx=2, incy=-1, seed=41)

    def pinned(a):
        return torch.from_numpy(np.ascontiguousarray(a).reshape(-1).view(np.uint8)).pin_memory()

    hA, hx, hy = pinned(p.A), pinned(p.x), pinned(p.y)
    st = lib.symv_host(kind, "L", n, al, hA.data_ptr(), p.lda, hx.data_ptr(), 2, be,
                       hy.data_ptr(), -1)
    assert st == 0
    y = hy.numpy().view(p.y.dtype).reshape(p.y.shape)
    err, _ = errors(o, p, y)
    assert np.max(err) <= TOL[kind]
    dp = DeviceProblem(p)
    st, yd = dp.run()
    assert st == 0
    assert np.array_equal(from_device(yd, p.y).view(np.uint8), y.view(np.uint8))
    h2d, d2h = lib.xsymv_host_traffic()
    es = p.A.itemsize * (2 if kind == "w" else 1)
    assert d2h == n * es and h2d == (n * (n + 1) // 2 + 2 * n) * es


def test_bounded_wait_reports_timeout(lib):
    """A bulk-copy barrier that never completes (test hook: 16 bytes are
    announced that never arrive) makes the kernel's bounded waits run out:
    the call's y becomes NaN, the host reads XSYMV_ERR_TIMEOUT, and the next
    normal call on the same context is correct again."""
    import torch

    p = inputs.make_problem("s", "U", 1500, lda=1500, alpha=1.0, beta=0.0, seed=2)
    dp = DeviceProblem(p)
    assert lib.xsymv_set_stream(torch.cuda.current_stream().cuda_stream) == 0
    # the waits live in the bulk-copy (TMA) ring variants
    tma = [v for v in range(lib.xsymv_variant_count("s")) if "_t" in lib.xsymv_variant_name("s", v)]
    assert tma and lib.xsymv_set_variant("s", tma[0]) == 0
    st, good = dp.run()
    assert st == 0 and lib.xsymv_sync_status() == 0
    try:
        lib.xsymv_set_wait_limit(2_000_000)          # 2 ms
        lib.xsymv_test_stall(True)
        st, bad = dp.run()
        assert st == 0
        assert lib.xsymv_sync_status() == -6
        yb = from_device(bad, p.y)
        assert np.all(np.isnan(yb))
    finally:
        lib.xsymv_test_stall(False)
        lib.xsymv_set_wait_limit(0)
    st, again = dp.run()
    lib.xsymv_set_variant("s", -1)
    assert st == 0 and lib.xsymv_sync_status() == 0
    assert bool((again == good).all())


def test_call_numbers_wrap(lib):
    """Calls tag failures in the status word with their call number; when the
    numbers start again at 1 the word is cleared first, so a failure recorded
    under a large old number does not hide the failures that follow."""
    import torch

    p = inputs.make_problem("s", "U", 700, lda=700, alpha=1.0, beta=0.0, seed=4)
    dp = DeviceProblem(p)
    assert lib.xsymv_set_stream(torch.cuda.current_stream().cuda_stream) == 0
    tma = [v for v in range(lib.xsymv_variant_count("s")) if "_t" in lib.xsymv_variant_name("s", v)]
    assert tma and lib.xsymv_set_variant("s", tma[0]) == 0
    try:
        st, good = dp.run()
        assert st == 0 and lib.xsymv_sync_status() == 0
        assert lib.xsymv_test_set_call_number(0x7ffffffd) == 0
        lib.xsymv_set_wait_limit(2_000_000)          # 2 ms
        lib.xsymv_test_stall(True)
        st, _ = dp.run()                             # call 0x7ffffffe fails
        assert st == 0 and lib.xsymv_sync_status() == -6
        lib.xsymv_test_stall(False)
        st, again = dp.run()                         # call 1: the word is cleared
        assert st == 0 and lib.xsymv_sync_status() == 0
        assert bool((again == good).all())
        lib.xsymv_test_stall(True)
        st, bad = dp.run()                           # call 2 fails: reported
        assert st == 0 and lib.xsymv_sync_status() == -6
        assert np.all(np.isnan(from_device(bad, p.y)))
    finally:
        lib.xsymv_test_stall(False)
        lib.xsymv_set_wait_limit(0)
        lib.xsymv_set_variant("s", -1)
    assert lib.xsymv_test_set_call_number(-1) == -4
    assert lib.xsymv_test_set_call_number(0x7fffffff) == -4


@pytest.mark.parametrize("kind", ["s", "d", "z"])
def test_chained_calls_read_previous_result(lib, kind):
    """Each call's main kernel may be scheduled while the previous call's
    finaliser still runs (programmatic launch); it must not read x before
    that finaliser has written it.  Five calls y_{k+1} := A y_k, each
    reading the previous call's y as its x, enqueued back to back on one
    stream, give the same bytes as the same calls with the host waiting for
    the GPU after each one."""
    import torch

    n = {"s": 3000, "d": 2000, "z": 1500}[kind]
    al, _ = SCAL[kind]
    zero = 0.0
    p = inputs.make_problem(kind, "U", n, lda=n + 4, alpha=al, beta=zero, seed=77)
    dp = DeviceProblem(p)
    assert lib.xsymv_set_stream(torch.cuda.current_stream().cuda_stream) == 0

    def iterate(sync):
        a, b = dp.x.clone(), dp.x.clone()
        for _ in range(5):
            st = lib.symv(kind, "U", n, al, dp.A, p.lda, a, 1, zero, b, 1)
            assert st == 0
            if sync:
                torch.cuda.synchronize()
            a, b = b, a
        torch.cuda.synchronize()
        return a

    chained = iterate(False)
    waited = iterate(True)
    assert bool((chained == waited).all())


@pytest.mark.parametrize("kind,n", [("s", 8192), ("d", 4096), ("z", 2048), ("w", 1024)])
def test_one_launch_gives_way_to_its_twin_back_to_back(lib, kind, n):
    """At sizes where the tuned variant is a one-launch kernel, isolated
    calls run in one launch each; calls that run back to back (the GPU never
    idle between them) switch to the variant's two-kernel twin, whose calls
    fill each other's tails, and isolated calls switch back.  Both compute the
    same plan's sums in the same order: every call gives the same bytes."""
    import torch

    name = lib.xsymv_variant_name(kind, lib.xsymv_selected_variant(kind, "U", n))
    if not name.endswith("_f"):
        pytest.skip("the tuned variant at this size is not a one-launch one: " + name)
    al, _ = SCAL[kind]
    p = inputs.make_problem(kind, "U", n, lda=n, alpha=al, beta=0.0, seed=n)
    dp = DeviceProblem(p)
    es = inputs.ELEM_BYTES[kind]
    assert lib.xsymv_set_stream(torch.cuda.current_stream().cuda_stream) == 0
    ref = torch.zeros(n * es, dtype=torch.uint8, device="cuda")
    assert lib.symv(kind, "U", n, al, dp.A, n, dp.x, 1, 0.0, ref, 1) == 0
    torch.cuda.synchronize()

    def isolated(k):
        c0 = lib.xsymv_launch_count()
        for _ in range(k):
            y = torch.zeros_like(ref)
            assert lib.symv(kind, "U", n, al, dp.A, n, dp.x, 1, 0.0, y, 1) == 0
            torch.cuda.synchronize()
            assert bool((y == ref).all())
        return lib.xsymv_launch_count() - c0

    isolated(2)
    assert isolated(4) == 4                       # one launch per isolated call
    calls = 40
    ys = torch.zeros((calls, n * es), dtype=torch.uint8, device="cuda")
    ev = [torch.cuda.Event() for _ in range(calls)]
    c0 = lib.xsymv_launch_count()
    for i in range(calls):
        if i >= 4:
            ev[i - 4].synchronize()               # four calls queued: the GPU is never idle
        assert lib.symv(kind, "U", n, al, dp.A, n, dp.x, 1, 0.0, ys[i], 1) == 0
        ev[i].record()
    torch.cuda.synchronize()
    launched = lib.xsymv_launch_count() - c0
    assert launched >= calls + calls // 2, launched   # most calls ran as two kernels
    assert bool((ys == ref.unsqueeze(0)).all())
    isolated(2)                                   # (the first may still be a twin)
    assert isolated(4) == 4


@pytest.mark.parametrize("kind", ["s", "d", "c", "w"])
def test_caller_kernels_between_calls_are_ordered(lib, kind):
    """An iterative method: each step's x is rebuilt from the previous
    product by the caller's own kernels on the same stream (a slow one on a
    large buffer, then the write of x), and the next call reads it.  A main
    kernel that starts streaming early must still see every byte those
    kernels wrote: the loop enqueued without host waits gives the bytes of
    the same loop with the host waiting after every step."""
    import torch

    n = 3000 if kind != "w" else 900
    al, _ = SCAL[kind]
    p = inputs.make_problem(kind, "U", n, lda=n + 4, alpha=al, beta=0.0, seed=99)
    dp = DeviceProblem(p)
    assert lib.xsymv_set_stream(torch.cuda.current_stream().cuda_stream) == 0
    big = torch.ones(64 << 20, dtype=torch.float32, device="cuda")   # 256 MB
    es = inputs.ELEM_BYTES[kind]
    dt = torch.float32 if kind in "sc" else torch.float64

    def iterate(sync):
        x = dp.x.clone()
        y = torch.zeros_like(x)
        for k in range(6):
            st = lib.symv(kind, "U", n, al, dp.A, p.lda, x, 1, 0.0, y, 1)
            assert st == 0
            # the caller's kernels: a slow pass over 256 MB, then x := y / 4 + 1 + k,
            # written element by element as the real components of the kind
            s = (big * 1.0000001).sum() * 0.0
            xv, yv = x.view(dt), y.view(dt)
            xv.copy_(yv * 0.25 + s.to(dt) + (1.0 + k))
            if sync:
                torch.cuda.synchronize()
        torch.cuda.synchronize()
        return x.clone(), y.clone()

    waited = iterate(True)
    chained = iterate(False)
    assert bool((waited[0] == chained[0]).all()) and bool((waited[1] == chained[1]).all())


@pytest.mark.parametrize("kind", KINDS)
def test_one_launch_variants_barrier_timeout(lib, kind):
    """The one-launch ("_f") variants meet at a grid barrier with a bounded
    wait.  The test hook makes every block wait for one block more than the
    grid has (nothing faults): the wait runs out, the host reads
    XSYMV_ERR_TIMEOUT, the call's y is NaN, and the next normal call on the
    same context is correct and bit-identical to the one before."""
    import torch

    fused = [v for v in range(lib.xsymv_variant_count(kind))
             if lib.xsymv_variant_name(kind, v).endswith("_f")]
    assert fused
    al, be = SCAL[kind]
    p = inputs.make_problem(kind, "U", 900, lda=900, alpha=al, beta=be, seed=12)
    dp = DeviceProblem(p)
    assert lib.xsymv_set_stream(torch.cuda.current_stream().cuda_stream) == 0
    assert lib.xsymv_set_variant(kind, fused[0]) == 0
    try:
        st, good = dp.run()
        assert st == 0 and lib.xsymv_sync_status() == 0
        assert lib.xsymv_launch_count() > 0
        lib.xsymv_set_wait_limit(2_000_000)          # 2 ms
        lib.xsymv_test_stall(True)
        st, bad = dp.run()
        assert st == 0
        assert lib.xsymv_sync_status() == -6
        assert np.all(np.isnan(from_device(bad, p.y)))
        lib.xsymv_test_stall(False)
        lib.xsymv_set_wait_limit(0)
        st, again = dp.run()
        assert st == 0 and lib.xsymv_sync_status() == 0
        assert bool((again == good).all())
    finally:
        lib.xsymv_test_stall(False)
        lib.xsymv_set_wait_limit(0)
        lib.xsymv_set_variant(kind, -1)


@pytest.mark.parametrize("kind", ["s", "c"])
def test_one_launch_equals_two_kernels_same_plan(o, lib, kind):
    """A one-launch variant and the two-kernel variant of the same tile shape,
    register cap and costs (so the same resident warps and the same plan)
    compute the same partial sums and add them in the same order: the same
    bytes."""
    names = [lib.xsymv_variant_name(kind, v) for v in range(lib.xsymv_variant_count(kind))]
    al, be = SCAL[kind]
    pairs = [(v, names.index(nm[:-len("_c2_f")])) for v, nm in enumerate(names)
             if nm.endswith("_c2_f") and nm[:-len("_c2_f")] in names]
    assert pairs
    for vf, vt in pairs:
        for uplo in ("U", "L"):
            for n in (700, 3001):
                p = inputs.make_problem(kind, uplo, n, lda=n + 4, alpha=al, beta=be, seed=n + vf)
                dp = DeviceProblem(p)
                try:
                    assert lib.xsymv_set_variant(kind, vf) == 0
                    st, yf = dp.run()
                    assert st == 0
                    assert lib.xsymv_set_variant(kind, vt) == 0
                    st, yt = dp.run()
                    assert st == 0
                finally:
                    lib.xsymv_set_variant(kind, -1)
                err, _ = errors(o, p, from_device(yf, p.y))
                assert np.max(err) <= TOL[kind]
                assert bool((yf == yt).all()), (names[vf], names[vt], uplo, n)


@pytest.mark.parametrize("kind", ["s", "d"])
def test_one_launch_calls_on_two_streams(o, lib, kind):
    """One-launch calls issued on two streams at once, each with its own
    problem and workspace: their grids are cooperative (the driver starts a
    grid only when all of its blocks fit), so neither waits at its barrier for
    blocks the other holds; both results stay correct and bit-identical to the
    same calls made one at a time."""
    import torch

    fused = [v for v in range(lib.xsymv_variant_count(kind))
             if lib.xsymv_variant_name(kind, v).endswith("_f")]
    al, be = SCAL[kind]
    probs = [inputs.make_problem(kind, u, 2500 + 300 * i, lda=2600 + 300 * i, alpha=al, beta=be,
                                 seed=90 + i) for i, u in enumerate("UL")]
    dps = [DeviceProblem(p) for p in probs]
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    assert lib.xsymv_set_variant(kind, fused[0]) == 0
    try:
        torch.cuda.synchronize()
        ref = []
        for dp, s in zip(dps, streams):
            with torch.cuda.stream(s):          # y's copy and the call on the same stream
                st, y = dp.run(stream=s)
            assert st == 0
            s.synchronize()
            ref.append(y)
        outs = [[], []]
        for _ in range(10):
            for i, (dp, s) in enumerate(zip(dps, streams)):
                with torch.cuda.stream(s):
                    st, y = dp.run(stream=s)
                assert st == 0
                outs[i].append(y)
        torch.cuda.synchronize()
        for i, s in enumerate(streams):
            assert lib.xsymv_set_stream(s.cuda_stream) == 0
            assert lib.xsymv_sync_status() == 0
            for y in outs[i]:
                assert bool((y == ref[i]).all())
        for p, y in zip(probs, ref):
            err, _ = errors(o, p, from_device(y, p.y))
            assert np.max(err) <= TOL[kind]
    finally:
        lib.xsymv_set_variant(kind, -1)
        lib.xsymv_set_stream(torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("kind", ["s", "c", "d"])
def test_back_to_back_calls_overlap_safely(lib, kind):
    """A call's main kernel may start streaming while the previous call's
    finaliser still runs, when the host sees that the finaliser's y misses
    the new call's A and x (the two calls' partial sums sit in different
    halves of the workspace).  Calls of two different sizes alternating on one
    stream with no host wait, and calls whose x or A overlaps the previous
    call's y (which must wait), give the bytes of the same calls made one at a
    time."""
    import torch

    al, be = SCAL[kind]
    sizes = (1500, 4100) if kind != "d" else (1200, 2900)
    probs = [inputs.make_problem(kind, u, n, lda=n + 2, alpha=al, beta=be, seed=n)
             for u, n in zip("UL", sizes)]
    dps = [DeviceProblem(p) for p in probs]
    order = [0, 1, 1, 0, 1, 0, 0, 1]

    def run_all(sync):
        outs = []
        for i in order:
            st, y = dps[i].run()
            assert st == 0
            if sync:
                torch.cuda.synchronize()
            outs.append(y)
        torch.cuda.synchronize()
        return outs

    waited = run_all(True)
    chained = run_all(False)
    for a, b in zip(waited, chained):
        assert bool((a == b).all())
    # the next call reads as its A a buffer the previous call's finaliser is
    # writing (y): the host must not let it start early
    n = 512
    p = inputs.make_problem(kind, "U", n, lda=n, alpha=al, beta=0.0, seed=5)
    dp = DeviceProblem(p)
    big = torch.zeros(dp.A.numel(), dtype=torch.uint8, device="cuda")
    big.copy_(dp.A)
    es = inputs.ELEM_BYTES[kind]

    def pair(sync):
        y1 = big[: n * es]                          # call 1 writes the first column of A2
        st, _ = dp.run(y=y1)
        assert st == 0
        if sync:
            torch.cuda.synchronize()
        y2 = dp.y0.clone()
        st, _ = dp.run(A=big, y=y2)                 # call 2 reads it as A
        assert st == 0
        torch.cuda.synchronize()
        return y2.clone(), big.clone()

    big.copy_(dp.A)
    ref = pair(True)
    big.copy_(dp.A)
    got = pair(False)
    assert bool((ref[0] == got[0]).all()) and bool((ref[1] == got[1]).all())
