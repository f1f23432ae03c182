"""The worked examples of tests/golden/ (y := alpha*A*x + beta*y, equation (1)
of "CUDA-xSYMV の実装と評価", IPSJ 2014-HPC-146, written out by hand): the
fixture is consistent with itself, and the CPU oracle reproduces every case
bit for bit (all values and intermediate results there are exact)."""
from fractions import Fraction

import numpy as np
import pytest

from tests import golden_cases as G

CASES = G.cases()
IDS = [c["name"] for c in CASES]


@pytest.fixture(scope="module")
def o():
    import oracle

    return oracle.get()


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_fixture_is_consistent(case):
    """the stated results equal the definition evaluated exactly, the matrix
    is symmetric (Hermitian for c, z), and double-double results are
    normalised"""
    kind, n = case["kind"], case["n"]
    if case["A"] is not None:
        for i in range(n):
            for j in range(n):
                a, b = case["A"][i][j], case["A"][j][i]
                if kind in "cz":
                    assert a[0] == b[0] and a[1] == -b[1], (i, j)
                else:
                    assert a == b, (i, j)
    want = G.exact_result(case)
    for i, y in enumerate(case["y"]):
        if kind in "cz":
            assert (Fraction(y[0]), Fraction(y[1])) == want[i], (case["name"], i)
        elif kind == "w":
            assert Fraction(y[0]) + Fraction(y[1]) == want[i], (case["name"], i)
            assert abs(y[1]) <= np.spacing(abs(y[0])) / 2
        else:
            assert Fraction(y) == want[i], (case["name"], i)


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_oracle_reproduces_worked_examples(o, case):
    kind, uplo, n = case["kind"], case["uplo"], case["n"]
    A, lda = G.stored_matrix(case)
    x = G.stored_vector(case, "x", case["incx"])
    y0 = G.stored_vector(case, "y0", case["incy"])
    al, be = G.scalars(case)
    info, y, _, _ = o.symv(kind, uplo, n, al, A, lda, x, case["incx"], be, y0, case["incy"])
    assert info == 0
    got = G.logical(case, y, case["incy"])
    want = G.expected(case)
    assert np.array_equal(got, want), (case["name"], got, want)
