"""Loader of the worked examples in tests/golden/symv_worked_examples.json:
turns a case into the stored arrays the oracle and the library take (only
the uplo triangle of A in column-major order, NaN elsewhere; strided x and
y with NaN gaps).  exact_result() evaluates the definition on a case's
logical data in rational arithmetic; it serves only to check the fixture
file itself (its hand-written results), never as a reference for the oracle
or the library."""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np

PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                    "symv_worked_examples.json")
DTYPES = {"s": np.float32, "d": np.float64, "c": np.complex64, "z": np.complex128,
          "w": np.float64}


def cases():
    with open(PATH) as f:
        return json.load(f)["cases"]


def _num(kind, v):
    """a scalar of the case as a Python number (complex for c/z, (hi, lo) for w)"""
    if kind in "cz":
        return complex(v[0], v[1])
    if kind == "w":
        return (float(v[0]), float(v[1]))
    return float(v)


def _put(arr, idx, kind, v):
    """arr[idx] = v; idx an int or a tuple of ints (w: v is (hi, lo))"""
    idx = idx if isinstance(idx, tuple) else (idx,)
    if kind == "w":
        arr[idx + (0,)], arr[idx + (1,)] = v
    else:
        arr[idx] = v


def stored_matrix(case, lda_pad=1):
    """(A, lda): numpy array of shape (n, lda) (w: (n, lda, 2)); row j of the
    array is column j of the matrix; only the uplo triangle holds values"""
    kind, n, upper = case["kind"], case["n"], case["uplo"] in "Uu"
    lda = n + lda_pad
    shape = (n, lda, 2) if kind == "w" else (n, lda)
    A = np.full(shape, np.nan, dtype=DTYPES[kind])
    if kind in "cz":
        A[...] = complex(np.nan, np.nan)
    if case["A"] is None:
        return A, lda
    for j in range(n):
        for i in range(n):
            if (i <= j) if upper else (i >= j):
                v = _num(kind, case["A"][i][j])
                if kind in "cz" and i == j:
                    v = complex(v.real, np.nan)   # the diagonal's imaginary part is never used
                _put(A, (j, i), kind, v)
    return A, lda


def stored_vector(case, key, inc):
    """strided storage of the logical vector case[key] (None: all NaN)"""
    kind, n = case["kind"], case["n"]
    m = 1 + (n - 1) * abs(inc)
    v = np.full((m, 2) if kind == "w" else (m,), np.nan, dtype=DTYPES[kind])
    if kind in "cz":
        v[...] = complex(np.nan, np.nan)
    if case[key] is None:
        return v
    for i in range(n):
        k = i * abs(inc) if inc > 0 else (n - 1 - i) * abs(inc)
        _put(v, k, kind, _num(kind, case[key][i]))
    return v


def logical(case, stored, inc):
    """the n logical elements of a strided result (w: (n, 2))"""
    n = case["n"]
    idx = [(i * abs(inc) if inc > 0 else (n - 1 - i) * abs(inc)) for i in range(n)]
    return stored[idx]


def expected(case):
    kind = case["kind"]
    y = case["y"]
    if kind == "w":
        return np.array(y, dtype=np.float64).reshape(case["n"], 2)
    if kind in "cz":
        return np.array([complex(a, b) for a, b in y], dtype=DTYPES[kind])
    return np.array(y, dtype=DTYPES[kind])


def scalars(case):
    kind = case["kind"]
    return _num(kind, case["alpha"]), _num(kind, case["beta"])


# ---- exact rational evaluation of the definition, to check the fixture ----

def _frac(kind, v):
    """exact value: Fraction, or (re, im) Fractions for c/z; w: hi + lo"""
    if kind in "cz":
        return (Fraction(v[0]), Fraction(v[1]))
    if kind == "w":
        return Fraction(v[0]) + Fraction(v[1])
    return Fraction(v)


def _mul(kind, a, b):
    if kind in "cz":
        return (a[0] * b[0] - a[1] * b[1], a[0] * b[1] + a[1] * b[0])
    return a * b


def _add(kind, a, b):
    if kind in "cz":
        return (a[0] + b[0], a[1] + b[1])
    return a + b


def exact_result(case):
    """alpha * A * x + beta * y0 on the fixture's logical data, in exact
    rational arithmetic (beta = 0: y0 not used; alpha = 0: A, x not used)"""
    kind, n = case["kind"], case["n"]
    zero = (Fraction(0), Fraction(0)) if kind in "cz" else Fraction(0)
    al, be = _frac(kind, case["alpha"]), _frac(kind, case["beta"])
    out = []
    for i in range(n):
        s = zero
        if al != zero:
            for j in range(n):
                s = _add(kind, s, _mul(kind, _frac(kind, case["A"][i][j]), _frac(kind, case["x"][j])))
        r = _mul(kind, al, s)
        if be != zero:
            r = _add(kind, r, _mul(kind, be, _frac(kind, case["y0"][i])))
        out.append(r)
    return out
