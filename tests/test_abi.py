"""The C-ABI library without a GPU: it loads, exports every entry point that
include/xsymv.h declares, and rejects bad BLAS arguments (checked on the host
before any CUDA call) with the xerbla positions."""
import ctypes
import os
import re

import numpy as np
import pytest

import symmetric_matrix_vector_gb300 as xs
from symmetric_matrix_vector_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "xsymv.h")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return xs.load()


def declared_symbols():
    src = open(HEADER).read()
    return re.findall(r"XSYMV_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)


def test_header_declares_the_five_entry_points():
    names = declared_symbols()
    for n in ("xsymv_s", "xsymv_d", "xhemv_c", "xhemv_z", "xsymv_w"):
        assert n in names
    assert len(names) == len(set(names))


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(xs.library_path())
    for name in declared_symbols():
        assert hasattr(raw, name), name


def test_only_declared_symbols_are_exported(lib):
    import subprocess

    out = subprocess.run(["nm", "-D", "--defined-only", xs.library_path()], check=True,
                         capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if l.split() and l.split()[-2] in "TDBR"}
    exported = {e for e in exported if not e.startswith("_")}
    assert exported == set(declared_symbols()), exported ^ set(declared_symbols())


@pytest.mark.parametrize("kind", ["s", "d", "c", "z", "w"])
def test_argument_errors_on_host(lib, kind):
    one = (1.0, 0.0) if kind == "w" else 1.0
    zero = (0.0, 0.0) if kind == "w" else 0.0
    f = getattr(xs, xs.ENTRY_POINTS[kind])
    # pointers are never dereferenced: the checks come first
    bogus = 0x1000
    assert f("X", 4, one, bogus, 4, bogus, 1, zero, bogus, 1, stream=0) == 1
    assert f("U", -1, one, bogus, 4, bogus, 1, zero, bogus, 1, stream=0) == 2
    assert f("L", 4, one, bogus, 3, bogus, 1, zero, bogus, 1, stream=0) == 5
    assert f("U", 4, one, bogus, 4, bogus, 0, zero, bogus, 1, stream=0) == 7
    assert f("u", 4, one, bogus, 4, bogus, 1, zero, bogus, 0, stream=0) == 10
    # first bad argument wins, as in xerbla
    assert f("X", -1, one, bogus, 0, bogus, 0, zero, bogus, 0, stream=0) == 1
    assert f("U", 5, one, bogus, 1, bogus, 0, zero, bogus, 1, stream=0) == 5
    # quick returns touch nothing
    assert f("U", 0, one, bogus, 1, bogus, 1, zero, bogus, 1, stream=0) == 0
    assert f("l", 7, zero, bogus, 7, bogus, 1, one, bogus, 1, stream=0) == 0


def test_status_strings(lib):
    for st in (0, 1, 2, 5, 7, 10, -1, -2, -3, -4, -5, -6):
        assert xs.xsymv_status_string(st) != "unknown status"
    assert xs.xsymv_status_string(12345) == "unknown status"


def test_variants_introspection(lib):
    for kind in "sdczw":
        cnt = xs.xsymv_variant_count(kind)
        assert cnt >= 1
        for i in range(cnt):
            assert re.fullmatch(r"vr\d+_u\d+_[rt]\d+_w\d+(_b\d+)?(_x\d+)?(_g\d+)?(_c\d+)?(_tk|_f)?", xs.xsymv_variant_name(kind, i))
        assert xs.xsymv_variant_name(kind, cnt) is None
        assert xs.xsymv_set_variant(kind, cnt) == -4
        assert xs.xsymv_set_variant(kind, -1) == 0
    assert xs.xsymv_variant_count("q") == 0


def test_stream_round_trip(lib):
    assert xs.xsymv_set_stream(0x1234) == 0
    assert xs.xsymv_get_stream() == 0x1234
    assert xs.xsymv_set_stream(0) == 0


def test_cpu_tensor_is_refused(lib):
    import torch

    a = torch.zeros(4)
    with pytest.raises(ValueError):
        xs.xsymv_s("U", 2, 1.0, a, 2, a, 1, 0.0, a, 1, stream=0)


@pytest.mark.parametrize("kind", ["s", "d"])
def test_gemv_argument_errors_on_host(lib, kind):
    bogus = 0x1000
    f = getattr(xs, "xgemv_" + kind)
    assert f(-1, 1.0, bogus, 4, bogus, 1, 0.0, bogus, 1, stream=0) == 1
    assert f(4, 1.0, bogus, 3, bogus, 1, 0.0, bogus, 1, stream=0) == 4
    assert f(4, 1.0, bogus, 4, bogus, 0, 0.0, bogus, 1, stream=0) == 6
    assert f(4, 1.0, bogus, 4, bogus, 1, 0.0, bogus, 0, stream=0) == 9
    assert f(-1, 1.0, bogus, 0, bogus, 0, 0.0, bogus, 0, stream=0) == 1
    # quick returns touch nothing
    assert f(0, 1.0, bogus, 1, bogus, 1, 0.0, bogus, 1, stream=0) == 0
    assert f(5, 0.0, bogus, 5, bogus, 1, 1.0, bogus, 1, stream=0) == 0
    with pytest.raises(ValueError):
        xs.gemv("c", 1, 1.0, bogus, 1, bogus, 1, 0.0, bogus, 1)


def test_gemv_variants_introspection(lib):
    for kind in "sd":
        cnt = xs.xgemv_variant_count(kind)
        assert cnt >= 1
        for i in range(cnt):
            assert re.fullmatch(r"vr\d+_u\d+_r0_w\d+(_b\d+)?", xs.xgemv_variant_name(kind, i))
        assert xs.xgemv_variant_name(kind, cnt) is None
        assert xs.xgemv_set_variant(kind, cnt) == -4
        assert xs.xgemv_set_variant(kind, 1) == 0 and xs.xgemv_selected_variant(kind) == 1
        assert xs.xgemv_set_variant(kind, -1) == 0 and xs.xgemv_selected_variant(kind) == 0
    assert xs.xgemv_variant_count("c") == -4
    assert xs.xgemv_variant_name("c", 0) is None


def tuned_entries():
    """(kind, upper, n_max, variant name) of every row of the tuned table"""
    src = open(os.path.join(ROOT, "symmetric_matrix_vector_gb300", "csrc", "xsymv_tuned.h")).read()
    body = src.split("// BEGIN TUNED TABLE", 1)[1].split("// END TUNED TABLE", 1)[0]
    return [(k, int(u), int(nmax), name) for k, u, nmax, name in
            re.findall(r"\{'(\w)', (-?\d+), (\d+), \"([^\"]*)\"\}", body)]


def test_tuned_table_names_compiled_variants(lib):
    """Every row of the tuned table names a variant compiled for its kind,
    and the library resolves a call of that row's largest size to exactly
    that variant (rows are looked up by name, not by position)."""
    rows = tuned_entries()
    assert len(rows) >= 5
    for kind, upper, n_max, name in rows:
        compiled = [xs.xsymv_variant_name(kind, i) for i in range(xs.xsymv_variant_count(kind))]
        if not name:          # an untuned kind: variant 0
            continue
        assert name in compiled, (kind, name)
        for uplo in (("U", "L") if upper < 0 else (("U",) if upper else ("L",))):
            n = min(n_max, 1 << 20)
            got = xs.xsymv_variant_name(kind, xs.xsymv_selected_variant(kind, uplo, n))
            assert got == name, (kind, uplo, n, name, got)


@pytest.mark.parametrize("kind", ["s", "d", "c", "z", "w"])
def test_shard_and_reduce_argument_errors_on_host(lib, kind):
    """the shard and reduce entry points check their arguments before any
    CUDA call (positions in their own signatures)"""
    one = (1.0, 0.0) if kind == "w" else 1.0
    zero = (0.0, 0.0) if kind == "w" else 0.0
    bogus = 0x1000
    sh = lambda *a: xs.symv_shard(kind, *a, stream=0)          # noqa: E731
    assert sh("X", 10, 0, 5, bogus, 10, bogus, 1, bogus) == 1
    assert sh("U", -1, 0, 0, bogus, 10, bogus, 1, bogus) == 2
    assert sh("U", 10, -1, 5, bogus, 10, bogus, 1, bogus) == 3
    assert sh("U", 10, 11, 11, bogus, 10, bogus, 1, bogus) == 3
    assert sh("U", 10, 6, 5, bogus, 10, bogus, 1, bogus) == 4
    assert sh("U", 10, 0, 11, bogus, 10, bogus, 1, bogus) == 4
    assert sh("U", 10, 2, 8, bogus, 7, bogus, 1, bogus) == 6     # upper panel: 8 rows
    assert sh("L", 10, 2, 8, bogus, 7, bogus, 1, bogus) == 6     # lower panel: 8 rows
    assert sh("U", 10, 2, 8, bogus, 8, bogus, 0, bogus) == 8
    assert sh("U", 0, 0, 0, bogus, 1, bogus, 1, bogus) == 0
    red = lambda *a: xs.symv_reduce(kind, *a, stream=0)        # noqa: E731
    assert red(-1, 2, one, bogus, 4, zero, bogus, 1) == 1
    assert red(4, 0, one, bogus, 4, zero, bogus, 1) == 2
    assert red(4, 2, one, bogus, 3, zero, bogus, 1) == 5
    assert red(4, 2, one, bogus, 4, zero, bogus, 0) == 8
    assert red(0, 2, one, bogus, 1, zero, bogus, 1) == 0
    assert red(4, 2, zero, bogus, 4, one, bogus, 1) == 0        # alpha 0, beta 1: nothing


def test_shard_bounds_split_evenly():
    """panel boundaries: start at 0, end at n, nondecreasing, inner ones on
    multiples of 16 columns (or n), and each panel within a few columns' worth of
    elements of an even share of the stored triangle"""
    for uplo in "UL":
        for n in (0, 1, 15, 16, 100, 1000, 4097, 32768, 100003):
            for N in (1, 2, 3, 5, 8, 64):
                b = xs.xsymv_shard_bounds(uplo, n, N)
                assert len(b) == N + 1 and b[0] == 0 and b[-1] == n
                assert all(b[r] <= b[r + 1] for r in range(N))
                assert all(v % 16 == 0 or v == n for v in b[1:-1])
                if n == 0:
                    continue
                j = np.arange(n, dtype=np.int64)
                pref = np.concatenate([[0], np.cumsum(j + 1 if uplo == "U" else n - j)])
                share = pref[-1] / N
                for r in range(N):
                    got = pref[b[r + 1]] - pref[b[r]]
                    assert abs(got - share) <= 16 * n + 1, (uplo, n, N, r, got, share)
    with pytest.raises(xs.XsymvError):
        xs.xsymv_shard_bounds("Q", 10, 2)
    with pytest.raises(xs.XsymvError):
        xs.xsymv_shard_bounds("U", 10, 0)


def test_unit_forms_probe_argument_errors_on_host(lib):
    """checked before any device work: an empty call succeeds, a negative
    count or a missing buffer is refused"""
    import symmetric_matrix_vector_gb300 as xs

    assert xs.xsymv_probe_unit_forms(0, 0, 0, 0) == 0
    assert xs.xsymv_probe_unit_forms(0, 0, 0, -1) == -4
    assert xs.xsymv_probe_unit_forms(0, 0, 0, 5) == -4
