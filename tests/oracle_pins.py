"""Pins for the CPU oracle, each a plain function ``check_*(o)`` that raises
AssertionError when the oracle handle ``o`` disagrees with something fixed
outside it: exact brute force on tiny inputs (Python rationals), closed forms,
invariants of the mathematics, and a library BLAS.

The same checks run against the real oracle (test_oracle_pins.py) and against
deliberately broken copies of it (test_oracle_mutants.py), which shows that a
plausible mistake anywhere in the oracle fails at least one of them.

The operation is equation (1) of "CUDA-xSYMV の実装と評価" (IPSJ
2014-HPC-146, §1): y := alpha*A*x + beta*y, A symmetric (Hermitian for the
complex kinds), one triangle stored.
"""
from __future__ import annotations

from fractions import Fraction as Fr

import numpy as np

from symmetric_matrix_vector_gb300.inputs import DTYPES, make_general, make_problem

KINDS = ("s", "d", "c", "z", "w")
# unit roundoff of the oracle's accumulator per kind
ACC_U = {"s": 2.0 ** -53, "c": 2.0 ** -53, "d": 2.0 ** -113, "z": 2.0 ** -113, "w": 2.0 ** -113}
OUT_U = {"s": 2.0 ** -24, "c": 2.0 ** -24, "d": 2.0 ** -53, "z": 2.0 ** -53, "w": 2.0 ** -105}
# the oracle reports a binary128 value as a pair of doubles: ~106 bits
REP_U = {"s": 0.0, "c": 0.0, "d": 2.0 ** -105, "z": 2.0 ** -105, "w": 2.0 ** -105}


def acc_bound(kind, n, den, mag=None):
    """rounding bound of an n-term accumulation plus the pair representation;
    ``mag`` defaults to ``den`` (an upper bound on |y_i|)"""
    return 4 * (n + 2) * ACC_U[kind] * den + 2 * REP_U[kind] * (den if mag is None else mag)


# ----------------------------------------------------------------------------
# exact arithmetic helpers (brute force, independent of the oracle)
# ----------------------------------------------------------------------------

def _flat(kind, arr):
    return arr.reshape(-1, 2) if kind == "w" else arr.reshape(-1)


def exact_elem(kind, arr, k):
    """element k of a storage array as an exact (re, im) pair of Fractions"""
    v = _flat(kind, arr)[k]
    if kind in ("s", "d"):
        return Fr(float(v)), Fr(0)
    if kind in ("c", "z"):
        return Fr(float(v.real)), Fr(float(v.imag))
    return Fr(float(v[0])) + Fr(float(v[1])), Fr(0)


def exact_scalar(kind, s):
    if kind == "s":
        return Fr(float(np.float32(s))), Fr(0)
    if kind == "d":
        return Fr(float(s)), Fr(0)
    if kind == "c":
        s = complex(s)
        return Fr(float(np.float32(s.real))), Fr(float(np.float32(s.imag)))
    if kind == "z":
        s = complex(s)
        return Fr(s.real), Fr(s.imag)
    if isinstance(s, (tuple, list)):
        return Fr(float(s[0])) + Fr(float(s[1])), Fr(0)
    return Fr(float(s)), Fr(0)


def cmul(a, b):
    return a[0] * b[0] - a[1] * b[1], a[0] * b[1] + a[1] * b[0]


def cadd(a, b):
    return a[0] + b[0], a[1] + b[1]


def vidx(n, inc, i):
    return (i if inc > 0 else i - (n - 1)) * inc


def full_exact(kind, uplo, A, lda, i, j):
    """A(i, j) of the full matrix, mirrored from the stored triangle"""
    herm = kind in ("c", "z")
    inside = i <= j if uplo == "U" else i >= j
    if herm and i == j:                  # real diagonal: imaginary part not read
        v = _flat(kind, A)[i + j * lda]
        return Fr(float(v.real)), Fr(0)
    if inside:
        re, im = exact_elem(kind, A, i + j * lda)
    else:
        re, im = exact_elem(kind, A, j + i * lda)
        if herm:
            im = -im
    return re, im


def exact_symv(p, alpha=None, beta=None):
    """y := alpha*A*x + beta*y by the definition, in exact rationals"""
    kind, n = p.kind, p.n
    al = exact_scalar(kind, p.alpha if alpha is None else alpha)
    be = exact_scalar(kind, p.beta if beta is None else beta)
    out = []
    for i in range(n):
        s = (Fr(0), Fr(0))
        if al != (0, 0):
            for j in range(n):
                s = cadd(s, cmul(full_exact(kind, p.uplo, p.A, p.lda, i, j),
                                 exact_elem(kind, p.x, vidx(n, p.incx, j))))
        r = cmul(al, s)
        if be != (0, 0):
            r = cadd(r, cmul(be, exact_elem(kind, p.y, vidx(n, p.incy, i))))
        out.append(r)
    return out


def exact_denom(p):
    """|alpha| * sum_j |A(i,j)| |x_j| + |beta| |y_i| in float64"""
    kind, n = p.kind, p.n
    al = [float(v) for v in exact_scalar(kind, p.alpha)]
    be = [float(v) for v in exact_scalar(kind, p.beta)]
    out = []
    for i in range(n):
        d = 0.0
        for j in range(n):
            a = [float(v) for v in full_exact(kind, p.uplo, p.A, p.lda, i, j)]
            xv = [float(v) for v in exact_elem(kind, p.x, vidx(n, p.incx, j))]
            d += np.hypot(*a) * np.hypot(*xv)
        yv = [0.0, 0.0]
        if be != [0.0, 0.0]:
            yv = [float(v) for v in exact_elem(kind, p.y, vidx(n, p.incy, i))]
        out.append(np.hypot(*al) * d + np.hypot(*be) * np.hypot(*yv))
    return out


def ref_pairs(kind, hi, lo):
    """oracle's unrounded output (hi + lo) as exact (re, im) Fractions"""
    res = []
    for i in range(hi.shape[0]):
        if kind in ("c", "z"):
            res.append((Fr(float(hi[i, 0])) + Fr(float(lo[i, 0])),
                        Fr(float(hi[i, 1])) + Fr(float(lo[i, 1]))))
        else:
            res.append((Fr(float(hi[i])) + Fr(float(lo[i])), Fr(0)))
    return res


def y_pairs(kind, y, n, inc):
    return [exact_elem(kind, y, vidx(n, inc, i)) for i in range(n)]


def run(o, p, alpha=None, beta=None):
    return o.symv(p.kind, p.uplo, p.n, p.alpha if alpha is None else alpha, p.A, p.lda, p.x,
                  p.incx, p.beta if beta is None else beta, p.y, p.incy)


def _absdiff(a, b):
    return float(max(abs(a[0] - b[0]), abs(a[1] - b[1])))


# ----------------------------------------------------------------------------
# input builders
# ----------------------------------------------------------------------------

def int_problem(kind, uplo, n, *, lda=None, incx=1, incy=1, alpha=1.25, beta=0.5, seed=0,
                lo_scale=2.0 ** -20):
    """Small-integer data (DD: integer hi plus a dyadic lo): every oracle
    operation on it is exact, so results must equal exact arithmetic."""
    p = make_problem(kind, uplo, n, lda=lda, incx=incx, incy=incy, alpha=alpha, beta=beta,
                     seed=seed)
    rng = np.random.default_rng(1000 + seed)

    def ints(shape):
        return rng.integers(-4, 5, size=shape).astype(np.float64)

    A = p.A
    for j in range(n):
        rows = range(0, j + 1) if uplo == "U" else range(j, n)
        for i in rows:
            if kind in ("s", "d"):
                A[j, i] = ints(())
            elif kind in ("c", "z"):
                re, im = ints(()), ints(())
                A[j, i] = complex(re, np.nan if i == j else im)
            else:
                A[j, i, 0] = ints(())
                A[j, i, 1] = ints(()) * lo_scale
    for v, inc in ((p.x, incx), (p.y, incy)):
        for i in range(n):
            k = vidx(n, inc, i)
            if kind in ("s", "d"):
                v[k] = ints(())
            elif kind in ("c", "z"):
                v[k] = complex(ints(()), ints(()))
            else:
                v[k, 0] = ints(())
                v[k, 1] = ints(()) * lo_scale
    return p


def _alpha_beta(kind, i):
    if kind in ("c", "z"):
        return [(complex(1.25, -0.5), complex(0.5, 0.25)), (complex(-2.0, 0.75), complex(0.0, 0.0))][i]
    if kind == "w":
        return [((1.25, 2.0 ** -20), (0.5, 0.0)), ((-2.0, 0.0), (0.0, 0.0))][i]
    return [(1.25, 0.5), (-2.0, 0.0)][i]


# ----------------------------------------------------------------------------
# the checks
# ----------------------------------------------------------------------------

def check_quad_type(o):
    assert o.quad_mant_dig() == 113


def check_integer_bruteforce(o):
    """exact data: the oracle's output must equal brute-force rationals"""
    for kind in KINDS:
        for uplo in ("U", "L"):
            for n, incx, incy, ab in ((1, 1, 1, 0), (2, 2, -1, 0), (3, -3, 2, 1), (5, 1, 1, 0),
                                      (8, -1, -2, 1), (13, 1, 3, 0)):
                alpha, beta = _alpha_beta(kind, ab)
                p = int_problem(kind, uplo, n, lda=n + 2, incx=incx, incy=incy, alpha=alpha,
                                beta=beta, seed=n)
                info, y, hi, lo = run(o, p)
                assert info == 0
                want = exact_symv(p)
                got = ref_pairs(kind, hi, lo)
                for i in range(n):
                    assert got[i] == want[i], (kind, uplo, n, i, got[i], want[i])
                if kind != "w":
                    yo = y_pairs(kind, y, n, incy)
                    for i in range(n):
                        assert yo[i] == want[i], (kind, uplo, n, i)


def check_random_vs_exact(o):
    """random data: error within the accumulator's rounding bound"""
    for kind in KINDS:
        for uplo in ("U", "L"):
            for n, seed in ((7, 1), (19, 2)):
                alpha, beta = _alpha_beta(kind, seed % 2)
                p = make_problem(kind, uplo, n, lda=n + 1, alpha=alpha, beta=beta, seed=seed)
                info, y, hi, lo = run(o, p)
                assert info == 0
                want = exact_symv(p)
                den = exact_denom(p)
                got = ref_pairs(kind, hi, lo)
                yo = y_pairs(kind, y, n, p.incy) if kind != "w" else None
                for i in range(n):
                    err = _absdiff(got[i], want[i])
                    assert err <= acc_bound(kind, n, den[i]), (kind, uplo, n, i, err, den[i])
                    if yo is not None:
                        e2 = _absdiff(yo[i], want[i])
                        mag = float(max(abs(want[i][0]), abs(want[i][1])))
                        assert e2 <= 2 * OUT_U[kind] * mag + acc_bound(kind, n, den[i])


def check_closed_forms(o):
    """identity, all-ones, diagonal and rank-one matrices"""
    for kind in KINDS:
        for uplo in ("U", "L"):
            n = 9
            alpha, beta = _alpha_beta(kind, 0)
            base = int_problem(kind, uplo, n, lda=n, alpha=alpha, beta=beta, seed=5)
            al, be = exact_scalar(kind, alpha), exact_scalar(kind, beta)
            xs = [exact_elem(kind, base.x, i) for i in range(n)]
            ys = [exact_elem(kind, base.y, i) for i in range(n)]
            rng = np.random.default_rng(9)
            u = rng.integers(-3, 4, size=n).astype(np.float64)
            d = rng.integers(-3, 4, size=n).astype(np.float64)
            for form in ("identity", "ones", "diag", "rank1"):
                A = base.A.copy()
                for j in range(n):
                    rows = range(0, j + 1) if uplo == "U" else range(j, n)
                    for i in rows:
                        if form == "identity":
                            v = 1.0 if i == j else 0.0
                        elif form == "ones":
                            v = 1.0
                        elif form == "diag":
                            v = d[i] if i == j else 0.0
                        else:
                            v = u[i] * u[j]
                        if kind == "w":
                            A[j, i] = (v, 0.0)
                        elif kind in ("c", "z"):
                            A[j, i] = complex(v, np.nan if i == j else 0.0)
                        else:
                            A[j, i] = v
                p = base
                p2 = type(p)(**{**p.__dict__, "A": A})
                info, y, hi, lo = run(o, p2)
                got = ref_pairs(kind, hi, lo)
                sx = (sum(v[0] for v in xs), sum(v[1] for v in xs))
                ux = (sum(Fr(u[k]) * xs[k][0] for k in range(n)),
                      sum(Fr(u[k]) * xs[k][1] for k in range(n)))
                for i in range(n):
                    if form == "identity":
                        core = xs[i]
                    elif form == "ones":
                        core = sx
                    elif form == "diag":
                        core = (Fr(d[i]) * xs[i][0], Fr(d[i]) * xs[i][1])
                    else:
                        core = (Fr(u[i]) * ux[0], Fr(u[i]) * ux[1])
                    want = cadd(cmul(al, core), cmul(be, ys[i]))
                    assert got[i] == want, (kind, uplo, form, i)


def _transpose_storage(p):
    """the same matrix stored in the other triangle"""
    n, lda = p.n, p.lda
    A = p.A.copy()
    herm = p.kind in ("c", "z")
    for j in range(n):
        for i in range(n):
            inside_new = i >= j if p.uplo == "U" else i <= j
            if inside_new and i != j:
                v = p.A[i, j].copy() if p.kind == "w" else p.A[i, j]
                if herm:
                    v = np.conj(v)
                A[j, i] = v
            elif not inside_new:
                A[j, i] = np.nan if p.kind != "w" else (np.nan, np.nan)
    return type(p)(**{**p.__dict__, "A": A, "uplo": "L" if p.uplo == "U" else "U"})


def check_mirror(o):
    """upper storage of A equals lower storage of the same A"""
    for kind in KINDS:
        for uplo in ("U", "L"):
            p = int_problem(kind, uplo, 11, lda=12, seed=3)
            q = _transpose_storage(p)
            _, _, h1, l1 = run(o, p)
            _, _, h2, l2 = run(o, q)
            assert ref_pairs(kind, h1, l1) == ref_pairs(kind, h2, l2), (kind, uplo)
            pr = make_problem(kind, uplo, 16, lda=16, alpha=_alpha_beta(kind, 0)[0],
                              beta=_alpha_beta(kind, 0)[1], seed=4)
            qr = _transpose_storage(pr)
            _, _, h1, l1 = run(o, pr)
            _, _, h2, l2 = run(o, qr)
            den = exact_denom(pr)
            g1, g2 = ref_pairs(kind, h1, l1), ref_pairs(kind, h2, l2)
            for i in range(pr.n):
                assert _absdiff(g1[i], g2[i]) <= 2 * acc_bound(kind, 16, den[i]), (kind, uplo, i)


def check_linearity(o):
    """y(a1 + a2, b) = y(a1, b) + y(a2, 0) within rounding"""
    for kind in KINDS:
        for uplo in ("U", "L"):
            p = make_problem(kind, uplo, 14, lda=15, seed=6)
            if kind in ("c", "z"):
                a1, a2, b = complex(0.75, 0.25), complex(-1.5, 0.5), complex(0.25, -1.0)
                a12 = a1 + a2
            elif kind == "w":
                a1, a2, b, a12 = (0.75, 0.0), (-1.5, 0.0), (0.25, 0.0), (-0.75, 0.0)
            else:
                a1, a2, b = 0.75, -1.5, 0.25
                a12 = a1 + a2
            _, _, h12, l12 = run(o, p, alpha=a12, beta=b)
            _, _, h1, l1 = run(o, p, alpha=a1, beta=b)
            _, _, h2, l2 = run(o, p, alpha=a2, beta=0.0 if kind != "w" else (0.0, 0.0))
            g12, g1, g2 = (ref_pairs(kind, h, l) for h, l in ((h12, l12), (h1, l1), (h2, l2)))
            den = exact_denom(type(p)(**{**p.__dict__, "alpha": 2.0 if kind != "w" else (2.0, 0.0),
                                          "beta": 1.0 if kind != "w" else (1.0, 0.0)}))
            for i in range(p.n):
                assert _absdiff(g12[i], cadd(g1[i], g2[i])) <= 3 * acc_bound(kind, 14, den[i]), (kind, i)


def check_hermitian_real(o):
    """HEMV of a real matrix is SYMV; DD with lo = 0 is DSYMV in binary128"""
    for uplo in ("U", "L"):
        for ck, rk in (("c", "s"), ("z", "d")):
            pr = make_problem(rk, uplo, 17, lda=18, alpha=1.5, beta=-0.5, seed=8)
            A = pr.A.astype(DTYPES[ck])
            for j in range(pr.n):
                A[j, j] = complex(A[j, j].real, np.nan)
            pc = type(pr)(**{**pr.__dict__, "kind": ck, "A": A, "x": pr.x.astype(DTYPES[ck]),
                             "y": pr.y.astype(DTYPES[ck]), "alpha": complex(1.5, 0.0),
                             "beta": complex(-0.5, 0.0)})
            _, _, hr, lr = run(o, pr)
            _, _, hc, lc = run(o, pc)
            assert np.array_equal(hc[:, 0], hr) and np.array_equal(lc[:, 0], lr), (ck, uplo)
            assert not np.any(hc[:, 1]), (ck, uplo)
        pd = make_problem("d", uplo, 17, lda=17, alpha=-0.75, beta=2.0, seed=9)
        Aw = np.stack([pd.A, np.where(np.isnan(pd.A), np.nan, 0.0)], axis=-1)
        pw = type(pd)(**{**pd.__dict__, "kind": "w", "A": Aw,
                         "x": np.stack([pd.x, np.zeros_like(pd.x)], -1),
                         "y": np.stack([pd.y, np.zeros_like(pd.y)], -1),
                         "alpha": (-0.75, 0.0), "beta": (2.0, 0.0)})
        _, _, hd, ld = run(o, pd)
        _, _, hw, lw = run(o, pw)
        assert np.array_equal(hd, hw) and np.array_equal(ld, lw), uplo


def check_library_blas(o):
    """working-precision agreement with scipy's BLAS ?symv / ?hemv"""
    from scipy.linalg import blas

    for kind, fn in (("s", blas.ssymv), ("d", blas.dsymv), ("c", blas.chemv), ("z", blas.zhemv)):
        for uplo in ("U", "L"):
            n = 96
            alpha, beta = _alpha_beta(kind, 0)
            p = make_problem(kind, uplo, n, lda=n, alpha=alpha, beta=beta, seed=10)
            full = p.A[:, :n].T.copy()          # (i, j) = A(i, j)
            a = np.where(np.isnan(full.real) if kind in "cz" else np.isnan(full), 0, full)
            if kind in "cz":
                a = np.where(np.isnan(a.imag), a.real.astype(a.dtype), a)
            ys = fn(alpha, a, p.x, beta=beta, y=p.y.copy(), lower=int(uplo == "L"))
            _, y, hi, lo = run(o, p)
            rows = np.arange(n)
            _, _, _, den = o.rows(kind, uplo, n, alpha, p.A, p.lda, p.x, 1, beta, p.y, 1, rows)
            tol = {"s": 5e-5, "c": 5e-5, "d": 1e-12, "z": 1e-12}[kind]
            ref = hi[:, 0] + 1j * hi[:, 1] if kind in "cz" else hi
            err = np.abs(ys - ref) / den
            assert np.max(err) <= tol, (kind, uplo, np.max(err))


def check_rows_vs_symv(o):
    """the definition (rows) and the three-part algorithm (symv) agree"""
    for kind in KINDS:
        for uplo in ("U", "L"):
            n = 40
            alpha, beta = _alpha_beta(kind, 0)
            p = make_problem(kind, uplo, n, lda=n + 3, alpha=alpha, beta=beta, incx=-2, incy=3,
                             seed=12)
            _, _, hi, lo = run(o, p)
            rows = np.arange(n)
            info, rh, rl, den = o.rows(kind, uplo, n, alpha, p.A, p.lda, p.x, p.incx, beta, p.y,
                                       p.incy, rows)
            assert info == 0
            g1, g2 = ref_pairs(kind, hi, lo), ref_pairs(kind, rh, rl)
            for i in range(n):
                assert _absdiff(g1[i], g2[i]) <= 2 * acc_bound(kind, n, den[i]), (kind, uplo, i)


def check_denominator(o):
    """the error normaliser matches |alpha| |A||x| + |beta| |y|"""
    for kind in KINDS:
        for uplo in ("U", "L"):
            alpha, beta = _alpha_beta(kind, 0)
            p = make_problem(kind, uplo, 12, lda=12, alpha=alpha, beta=beta, incy=-1, seed=14)
            _, _, _, den = o.rows(kind, uplo, p.n, alpha, p.A, p.lda, p.x, p.incx, beta, p.y,
                                  p.incy, np.arange(p.n))
            want = exact_denom(p)
            assert np.allclose(den, want, rtol=1e-12, atol=0), kind


def check_unused_never_read(o):
    """NaN outside the stored triangle (and in Hermitian diagonal imaginary
    parts and vector gaps) never reaches the result"""
    for kind in KINDS:
        for uplo in ("U", "L"):
            alpha, beta = _alpha_beta(kind, 0)
            p = make_problem(kind, uplo, 33, lda=35, alpha=alpha, beta=beta, incx=2, incy=-2,
                             seed=15)
            info, y, hi, lo = run(o, p)
            assert info == 0 and np.all(np.isfinite(hi)) and np.all(np.isfinite(lo)), (kind, uplo)
            # y's gap elements are left untouched
            idx = set(vidx(p.n, p.incy, i) for i in range(p.n))
            gaps = [k for k in range(len(y)) if k not in idx]
            for k in gaps:
                assert np.all(np.isnan(y[k] if kind != "w" else y[k]))


def check_special_scalars(o):
    """alpha = 0 reads neither A nor x; beta = 0 does not read y;
    alpha = 0, beta = 1 leaves y unchanged; n = 0 does nothing"""
    for kind in KINDS:
        for uplo in ("U", "L"):
            p = make_problem(kind, uplo, 10, lda=10, seed=16)
            zero = (0.0, 0.0) if kind == "w" else 0.0
            one = (1.0, 0.0) if kind == "w" else 1.0
            half = (0.5, 0.0) if kind == "w" else 0.5
            Anan = np.full_like(p.A, np.nan)
            xnan = np.full_like(p.x, np.nan)
            info, y, hi, lo = o.symv(kind, uplo, p.n, zero, Anan, p.lda, xnan, 1, half, p.y, 1)
            want = y_pairs(kind, p.y, p.n, 1)
            got = ref_pairs(kind, hi, lo)
            for i in range(p.n):
                assert got[i] == (want[i][0] / 2, want[i][1] / 2), (kind, i)
            info, y, hi, lo = o.symv(kind, uplo, p.n, zero, Anan, p.lda, xnan, 1, one, p.y, 1)
            assert np.array_equal(y, p.y)
            ynan = np.full_like(p.y, np.nan)
            info, y, hi, lo = o.symv(kind, uplo, p.n, one, p.A, p.lda, p.x, 1, zero, ynan, 1)
            assert np.all(np.isfinite(hi))
            info, y, hi, lo = o.symv(kind, uplo, 0, one, p.A, 1, p.x, 1, zero, p.y, 1)
            assert info == 0 and np.array_equal(y, p.y)


def check_arg_errors(o):
    """BLAS argument-error positions"""
    p = make_problem("d", "U", 4, seed=17)
    cases = [(("X", 4, 4, 1, 1), 1), (("U", -1, 4, 1, 1), 2), (("L", 4, 3, 1, 1), 5),
             (("U", 4, 4, 0, 1), 7), (("U", 4, 4, 1, 0), 10), (("l", 4, 4, -1, -1), 0)]
    for (uplo, n, lda, incx, incy), want in cases:
        info, y, _, _ = o.symv("d", uplo, n, 1.0, p.A, lda, p.x, incx, 0.0, p.y, incy)
        assert info == want, (uplo, n, lda, incx, incy, info)
        if want:
            assert np.array_equal(y, p.y, equal_nan=True)


# ----------------------------------------------------------------------------
# the general product the report compares SYMV with (§1): oracle_gemv_rows
# ----------------------------------------------------------------------------

def int_general(kind, n, *, lda=None, incx=1, incy=1, alpha=1.25, beta=0.5, seed=0):
    """Unsymmetric small-integer problem: every oracle operation is exact."""
    p = make_general(kind, n, lda=lda, incx=incx, incy=incy, alpha=alpha, beta=beta, seed=seed)
    rng = np.random.default_rng(2000 + seed)
    p.A[:, :n] = rng.integers(-4, 5, size=(n, n)).astype(p.A.dtype)
    for v, inc in ((p.x, incx), (p.y, incy)):
        for i in range(n):
            v[vidx(n, inc, i)] = rng.integers(-4, 5)
    return p


def exact_gemv(p, rows=None):
    """rows of alpha*A*x + beta*y by the definition, in exact rationals"""
    n = p.n
    al, be = Fr(float(np.float32(p.alpha) if p.kind == "s" else p.alpha)), \
        Fr(float(np.float32(p.beta) if p.kind == "s" else p.beta))
    out = []
    for i in (range(n) if rows is None else rows):
        s = Fr(0)
        if al != 0:
            for j in range(n):
                s += Fr(float(p.A[j, i])) * Fr(float(p.x[vidx(n, p.incx, j)]))
        r = al * s
        if be != 0:
            r += be * Fr(float(p.y[vidx(n, p.incy, i)]))
        out.append(r)
    return out


def gemv(o, p, rows=None, alpha=None, beta=None, A=None, x=None, y=None):
    rows = np.arange(p.n) if rows is None else np.asarray(rows)
    return o.gemv_rows(p.kind, p.n, p.alpha if alpha is None else alpha, p.A if A is None else A,
                       p.lda, p.x if x is None else x, p.incx, p.beta if beta is None else beta,
                       p.y if y is None else y, p.incy, rows)


def check_gemv_integer_bruteforce(o):
    """exact unsymmetric data: the oracle equals brute-force rationals (a
    transposed operand, a wrong stride or a dropped term changes the value)"""
    for kind in ("s", "d"):
        for n, incx, incy, (alpha, beta) in ((1, 1, 1, (1.25, 0.5)), (2, -1, 2, (1.25, 0.5)),
                                             (3, 2, -3, (-2.0, 0.0)), (7, 1, 1, (0.75, -1.5)),
                                             (12, -2, -1, (1.25, 0.5))):
            p = int_general(kind, n, lda=n + 3, incx=incx, incy=incy, alpha=alpha, beta=beta,
                            seed=n)
            info, hi, lo, den = gemv(o, p)
            assert info == 0
            want = exact_gemv(p)
            for i in range(n):
                assert Fr(float(hi[i])) + Fr(float(lo[i])) == want[i], (kind, n, i)


def check_gemv_closed_forms(o):
    """A = I gives alpha*x + beta*y; A = u v^T gives alpha*(v.x)*u + beta*y"""
    n = 9
    for kind in ("s", "d"):
        p = int_general(kind, n, lda=n + 1, seed=3)
        A = p.A.copy()
        A[:, :n] = 0
        for j in range(n):
            A[j, j] = 1
        _, hi, lo, _ = gemv(o, p, A=A)
        for i in range(n):
            want = Fr(1.25) * Fr(float(p.x[i])) + Fr(0.5) * Fr(float(p.y[i]))
            assert Fr(float(hi[i])) + Fr(float(lo[i])) == want, (kind, i)
        u = np.arange(1, n + 1, dtype=np.float64)
        v = np.arange(n, 0, -1, dtype=np.float64) - 4
        A[:, :n] = np.outer(v, u)            # A[j, i] = A(i, j) = u_i v_j
        vx = sum(Fr(float(v[j])) * Fr(float(p.x[j])) for j in range(n))
        _, hi, lo, _ = gemv(o, p, A=A)
        for i in range(n):
            want = Fr(1.25) * vx * Fr(float(u[i])) + Fr(0.5) * Fr(float(p.y[i]))
            assert Fr(float(hi[i])) + Fr(float(lo[i])) == want, (kind, i)


def check_gemv_random_and_library(o):
    """random data: within the binary128 accumulation bound of exact
    arithmetic, and within working-precision tolerance of scipy's ?gemv"""
    from scipy.linalg import blas

    for kind, fn, tol in (("s", blas.sgemv, 5e-5), ("d", blas.dgemv, 1e-12)):
        n = 23
        p = make_general(kind, n, lda=n + 2, alpha=-0.75, beta=1.5, incx=-2, incy=3, seed=4)
        info, hi, lo, den = gemv(o, p)
        assert info == 0
        want = exact_gemv(p)
        for i in range(n):
            err = abs(float(Fr(float(hi[i])) + Fr(float(lo[i])) - want[i]))
            assert err <= 4 * (n + 2) * 2.0 ** -113 * den[i] + 2.0 ** -104 * den[i], (kind, i)
        a = p.A[:, :n].T.copy()
        xs = np.array([p.x[vidx(n, p.incx, j)] for j in range(n)])
        ys = np.array([p.y[vidx(n, p.incy, i)] for i in range(n)])
        ref = fn(p.alpha, a, xs, beta=p.beta, y=ys.copy())
        assert np.max(np.abs(ref - hi) / den) <= tol, kind


def check_gemv_symmetric_matches_symv(o):
    """on the explicitly mirrored matrix the general product is SYMV"""
    n = 17
    p = make_problem("d", "L", n, lda=n, alpha=1.25, beta=0.5, seed=5)
    full = np.where(np.isnan(p.A), p.A.T, p.A)        # A[j, i] for i < j from A[i, j]
    g = make_general("d", n, lda=n, alpha=1.25, beta=0.5, seed=5)
    _, gh, gl, gden = gemv(o, g, A=full, x=p.x, y=p.y)
    _, sy, sh, sl = run(o, p)
    for i in range(n):
        d = abs((gh[i] - sh[i]) + (gl[i] - sl[i]))
        assert d <= 8 * (n + 2) * 2.0 ** -105 * gden[i], i


def check_gemv_special_and_errors(o):
    """alpha = 0 reads neither A nor x; beta = 0 does not read y; padding rows
    are never read; BLAS argument positions 1 n, 4 lda, 6 incx, 9 incy"""
    for kind in ("s", "d"):
        p = make_general(kind, 6, lda=8, alpha=1.25, beta=0.5, seed=6)
        _, hi, lo, den = gemv(o, p)
        assert np.all(np.isfinite(hi)) and np.all(np.isfinite(den))
        nanA = np.full_like(p.A, np.nan)
        _, hi, lo, _ = gemv(o, p, alpha=0.0, A=nanA, x=np.full_like(p.x, np.nan))
        assert np.array_equal(hi, 0.5 * p.y.astype(np.float64)) and not np.any(lo)
        _, hi, lo, _ = gemv(o, p, beta=0.0, y=np.full_like(p.y, np.nan))
        assert np.all(np.isfinite(hi))
    p = make_general("d", 4, seed=7)
    for (n, lda, incx, incy), want in (((-1, 4, 1, 1), 1), ((4, 3, 1, 1), 4), ((4, 4, 0, 1), 6),
                                       ((4, 4, 1, 0), 9), ((4, 4, -1, -1), 0)):
        info, _, _, _ = o.gemv_rows("d", n, 1.0, p.A, lda, p.x, incx, 0.0, p.y, incy,
                                    np.arange(max(n, 0)))
        assert info == want, (n, lda, incx, incy, info)


ALL_CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]
