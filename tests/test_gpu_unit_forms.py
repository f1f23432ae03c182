"""The double-double kernels issue every rounded sum, difference and product
of two doubles as a fused multiply-add with a unit operand (a + b =
fma(a, 1, b), a - b = fma(b, -1, a), a * b = fma(a, b, -0)).  IEEE 754
makes each the same single rounding of the same exact value; this checks
it on the GPU, bit for bit, against the plain instructions and against the
host's IEEE arithmetic, on random operands of every exponent gap, on
near-cancellation, on double-double-like pairs, in the subnormal range and
on the special values."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu


def _operands():
    rng = np.random.default_rng(20141)
    n = 1 << 16
    a1 = rng.uniform(-1, 1, n) * 2.0 ** rng.integers(-60, 60, n)
    b1 = a1 * rng.uniform(-1, 1, n) * 2.0 ** (-rng.integers(0, 120, n).astype(float))
    a2 = rng.uniform(-1, 1, n)
    b2 = -a2 * (1 + rng.uniform(-1e-15, 1e-15, n))                 # near cancellation
    a3 = rng.uniform(-4, 4, n)
    b3 = rng.uniform(-1, 1, n) * np.abs(a3) * 2.0 ** -53           # hi + lo of a DD
    a4 = rng.uniform(-1, 1, n) * 2.0 ** -1000                       # subnormal results
    b4 = rng.uniform(-1, 1, n) * 2.0 ** rng.integers(-1074, -1000, n).astype(float)
    a5 = rng.uniform(-1, 1, n) * 2.0 ** 1000                        # overflow of products
    b5 = rng.uniform(-1, 1, n) * 2.0 ** rng.integers(0, 40, n).astype(float)
    sp = np.array([0.0, -0.0, 1.0, -1.0, np.inf, -np.inf, np.nan, 5e-324, -5e-324,
                   np.finfo(np.float64).max, -np.finfo(np.float64).max, 2.0 ** -1022])
    a6, b6 = (x.ravel() for x in np.meshgrid(sp, sp))
    a = np.concatenate([a1, a2, a3, a4, a5, a6])
    b = np.concatenate([b1, b2, b3, b4, b5, b6])
    return a, b


def _same_bits(x, y):
    both_nan = np.isnan(x) & np.isnan(y)
    return (x.view(np.int64) == y.view(np.int64)) | both_nan


def test_fused_unit_forms_equal_plain_operations():
    import symmetric_matrix_vector_gb300 as xs

    a, b = _operands()
    n = a.size
    da = torch.from_numpy(a).cuda()
    db = torch.from_numpy(b).cuda()
    out = torch.full((6 * n,), 7.0, dtype=torch.float64, device="cuda")
    xs.check(xs.xsymv_probe_unit_forms(da, db, out, n))
    torch.cuda.synchronize()
    o = out.cpu().numpy().reshape(n, 6)
    with np.errstate(all="ignore"):
        host = [a + b, a - b, a * b]
    for j, name in enumerate(("add", "sub", "mul")):
        plain, fused = o[:, j], o[:, 3 + j]
        assert _same_bits(plain, host[j]).all(), name + ": plain instruction vs host IEEE"
        bad = ~_same_bits(fused, plain)
        assert not bad.any(), "%s: fused form differs at a=%r b=%r" % (
            name, a[bad][:3].tolist(), b[bad][:3].tolist())

