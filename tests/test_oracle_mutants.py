"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that
the pins in oracle_pins.py catch every one of them.

Each mutant is a textual edit of oracle.c inside one function (or at file
scope), compiled to a temporary library.  A mutant that passes every pin
would mean the pins cannot tell that mistake from the correct algorithm.
"""
import re

import pytest

import oracle
from tests import oracle_pins as pins

# (id, function name or None for file scope, old text, new text)
MUTANTS = [
    ("s_part_two_dropped", "oracle_ssymv",
     "acc[i] += al * ((double)A[i + (long)i * lda] * X(i));", ";"),
    ("s_part_three_dropped", "oracle_ssymv", "for (int i = 0; i < n; i++) acc[i] += al * v[i];", ";"),
    ("s_row_term_wrong_x", "oracle_ssymv", "v[i] += a * X(j);", "v[i] += a * X(i);"),
    ("s_col_term_wrong_x", "oracle_ssymv", "t += a * X(i);", "t += a * X(j);"),
    ("s_alpha_missing_part_one", "oracle_ssymv", "acc[j] += al * t;", "acc[j] += t;"),
    ("s_beta_ignored", "oracle_ssymv", "be * (double)Y(i)", "(double)Y(i)"),
    ("s_beta_zero_reads_y", "oracle_ssymv",
     "acc[i] = (beta == 0.0f) ? 0.0 : be * (double)Y(i);", "acc[i] = be * (double)Y(i);"),
    ("d_accumulator_double", "oracle_dsymv", "quad_t t = 0;", "double t = 0;"),
    ("d_part_two_dropped", "oracle_dsymv",
     "acc[i] += al * ((quad_t)A[i + (long)i * lda] * X(i));", ";"),
    ("upper_strict_includes_diagonal", None,
     "if (upper) { *i0 = 0;     *i1 = j; }", "if (upper) { *i0 = 0;     *i1 = j + 1; }"),
    ("lower_reads_upper_positions", None,
     "else       { *i0 = j + 1; *i1 = n; }", "else       { *i0 = 0; *i1 = j; }"),
    ("c_conj_missing", "oracle_chemv",
     "t = cd_add(t, cd_mul(cd_conj(a), XE(i)));", "t = cd_add(t, cd_mul(a, XE(i)));"),
    ("c_conj_on_row_term", "oracle_chemv",
     "v[i] = cd_add(v[i], cd_mul(a, XE(j)));", "v[i] = cd_add(v[i], cd_mul(cd_conj(a), XE(j)));"),
    ("z_diag_imag_read", "oracle_zhemv", "cquad d = {AE(i, i).re, 0};", "cquad d = AE(i, i);"),
    ("z_complex_mul_sign", None,
     "return (cquad){a.re * b.re - a.im * b.im, a.re * b.im + a.im * b.re};",
     "return (cquad){a.re * b.re + a.im * b.im, a.re * b.im + a.im * b.re};"),
    ("z_alpha_conj", "oracle_zhemv", "acc[j] = cq_add(acc[j], cq_mul(al, t));",
     "acc[j] = cq_add(acc[j], cq_mul(cq_conj(al), t));"),
    ("w_lo_dropped", "oracle_wsymv",
     "#define DD(p, k) ((quad_t)(p)[2 * (k)] + (quad_t)(p)[2 * (k) + 1])",
     "#define DD(p, k) ((quad_t)(p)[2 * (k)])"),
    ("w_part_three_dropped", "oracle_wsymv", "for (int i = 0; i < n; i++) acc[i] += al * v[i];", ";"),
    ("split_lo_dropped", None, "*lo = (double)(q - (quad_t)h);", "*lo = 0.0;"),
    ("rows_mirror_conj_missing", None, "if (herm) a.im = -a.im;", ";"),
    ("rows_beta_term_missing_in_denominator", "oracle_rows",
     "dy = modulus(be) * modulus(yi);", "dy = 0.0;"),
    ("negative_inc_not_reversed", None,
     "static long first_index(int n, int inc) { return inc > 0 ? 0 : (long)(1 - n) * inc; }",
     "static long first_index(int n, int inc) { return inc > 0 ? 0 : 0 * n; }\n"
     "#define ORACLE_ABS_INC 1"),
    ("bad_lda_check", None, "if (lda < (n > 1 ? n : 1)) return 5;", "if (lda < 1) return 5;"),
    ("gemv_transposed", "oracle_gemv_rows",
     "load_val(kind, A, i + j * (long)lda)", "load_val(kind, A, j + i * (long)lda)"),
    ("gemv_beta_dropped", "oracle_gemv_rows", "out += be * yi;", "out += yi;"),
    ("gemv_alpha_dropped", "oracle_gemv_rows", "quad_t out = al * s;", "quad_t out = s;"),
    ("gemv_last_column_dropped", "oracle_gemv_rows",
     "for (long j = 0; j < n; j++) {", "for (long j = 0; j + 1 < n; j++) {"),
    ("gemv_accumulator_double", "oracle_gemv_rows", "quad_t s = 0;", "double s = 0;"),
]


def _function_span(src, name):
    """[start, end) of the definition of C function ``name``"""
    m = re.search(r"^int %s\(" % re.escape(name), src, flags=re.M)
    assert m, name
    end = src.index("\n}\n", m.start()) + 3
    return m.start(), end


def mutate(src, func, old, new):
    if func is None:
        lo, hi = 0, len(src)
    else:
        lo, hi = _function_span(src, func)
    body = src[lo:hi]
    assert body.count(old) == 1, "mutation anchor must occur once: %r" % old
    return src[:lo] + body.replace(old, new) + src[hi:]


def _fix_negative_inc(src):
    # a mutant that forgets to reverse negative strides must still index inside
    # the arrays: take |inc| as the step wherever the stride is applied
    for a, b in (("(long)(i) * incx", "(long)(i) * (incx < 0 ? -incx : incx)"),
                 ("(long)(i) * incy", "(long)(i) * (incy < 0 ? -incy : incy)"),
                 ("kx + j * incx", "kx + j * (incx < 0 ? -incx : incx)"),
                 ("ky + i * incy", "ky + i * (incy < 0 ? -incy : incy)")):
        assert a in src, a
        src = src.replace(a, b)
    return src


@pytest.fixture(scope="module")
def source():
    with open(oracle.SOURCE) as f:
        return f.read()


@pytest.mark.parametrize("mid,func,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_mutant(tmp_path, source, mid, func, old, new):
    src = mutate(source, func, old, new)
    if "ORACLE_ABS_INC" in src:
        src = _fix_negative_inc(src)
    path = tmp_path / "oracle_mutant.c"
    path.write_text(src)
    lib = oracle.build(str(path), str(tmp_path / "liboracle_mutant.so"), force=True)
    o = oracle.Oracle(lib)
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(o)
        except (AssertionError, ValueError, ArithmeticError):
            # a wrong value, or a NaN/Inf that cannot be compared exactly
            failed.append(check.__name__)
    assert failed, "no pin detects mutant %s" % mid


def test_unmutated_copy_passes(tmp_path, source):
    path = tmp_path / "oracle_copy.c"
    path.write_text(source)
    o = oracle.Oracle(oracle.build(str(path), str(tmp_path / "liboracle_copy.so"), force=True))
    for check in pins.ALL_CHECKS:
        check(o)
