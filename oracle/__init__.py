"""CPU oracle for xSYMV / xHEMV — test infrastructure, not part of the library.

Plain single-threaded C (``oracle.c``), compiled here with gcc into
``oracle/_build/liboracle.so`` and called through ctypes on numpy arrays.  It
follows "CUDA-xSYMV の実装と評価" (Implementation and evaluation of
CUDA-xSYMV, IPSJ 2014-HPC-146): equation (1) and the three-part sequential
algorithm of §2.1 (figure "Sequential SYMV kernel algorithm"), with a
higher-precision accumulator (binary64 for s/c, binary128 for d/z/w).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  It shares no code with the CUDA library.

Array conventions (numpy, host memory):
  * ``A`` has shape ``(n, lda)`` for s/d/c/z and ``(n, lda, 2)`` for w; row
    ``j`` of the numpy array is column ``j`` of the matrix, so the memory is
    column-major with leading dimension ``lda``.
  * ``x`` / ``y`` are 1-D (w: ``(m, 2)``) arrays holding a strided vector;
    ``incx`` / ``incy`` follow reference-BLAS rules (negative = reversed).
  * dtypes: s float32, d float64, c complex64, z complex128, w float64 pairs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_DEFAULT_LIB = os.path.join(_BUILD_DIR, "liboracle.so")

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]

_DTYPES = {"s": np.float32, "d": np.float64, "c": np.complex64, "z": np.complex128, "w": np.float64}


def build(source: str = SOURCE, out: str = _DEFAULT_LIB, force: bool = False) -> str:
    """Compile ``source`` (default: oracle.c) into the shared library ``out``."""
    header = os.path.join(_HERE, "oracle.h")
    if not force and os.path.exists(out):
        newest = max(os.path.getmtime(source), os.path.getmtime(header))
        if os.path.getmtime(out) >= newest:
            return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", *CFLAGS, "-I", _HERE, source, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


_dptr = ctypes.POINTER(ctypes.c_double)


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    return ctypes.c_void_p(a.ctypes.data)


class Oracle:
    """ctypes handle on one build of the oracle library."""

    def __init__(self, path: str):
        self.path = path
        lib = ctypes.CDLL(path)
        i, c, v = ctypes.c_int, ctypes.c_char, ctypes.c_void_p
        for name in ("oracle_ssymv",):
            fn = getattr(lib, name)
            fn.argtypes = [c, i, ctypes.c_float, v, i, v, i, ctypes.c_float, v, i, v, v]
            fn.restype = i
        lib.oracle_dsymv.argtypes = [c, i, ctypes.c_double, v, i, v, i, ctypes.c_double, v, i, v, v]
        lib.oracle_dsymv.restype = i
        for name in ("oracle_chemv", "oracle_zhemv", "oracle_wsymv"):
            fn = getattr(lib, name)
            fn.argtypes = [c, i, v, v, i, v, i, v, v, i, v, v]
            fn.restype = i
        lib.oracle_rows.argtypes = [c, c, i, v, v, i, v, i, v, v, i, i, v, v, v, v]
        lib.oracle_rows.restype = i
        lib.oracle_gemv_rows.argtypes = [c, i, v, v, i, v, i, v, v, i, i, v, v, v, v]
        lib.oracle_gemv_rows.restype = i
        lib.oracle_quad_mant_dig.restype = i
        self.lib = lib

    # ------------------------------------------------------------------
    def symv(self, kind, uplo, n, alpha, A, lda, x, incx, beta, y, incy):
        """Run the three-part algorithm.

        Returns ``(info, y_out, ref_hi, ref_lo)``: the BLAS info code, y
        rounded once to its type (a new array; the input is not modified),
        and the unrounded accumulator as a double pair (complex: interleaved
        re, im; shape ``(n,)`` or ``(n, 2)``).
        """
        kind = kind.lower()
        dt = _DTYPES[kind]
        A = np.ascontiguousarray(A, dtype=dt)
        x = np.ascontiguousarray(x, dtype=dt)
        y_out = np.array(y, dtype=dt, copy=True, order="C")
        nn = max(n, 0)
        width = 2 if kind in "cz" else 1
        ref_hi = np.zeros(nn * width, dtype=np.float64)
        ref_lo = np.zeros(nn * width, dtype=np.float64)
        u = uplo.encode() if isinstance(uplo, str) else uplo
        if kind == "s":
            info = self.lib.oracle_ssymv(u, n, float(alpha), _ptr(A), lda, _ptr(x), incx,
                                         float(beta), _ptr(y_out), incy, _ptr(ref_hi), _ptr(ref_lo))
        elif kind == "d":
            info = self.lib.oracle_dsymv(u, n, float(alpha), _ptr(A), lda, _ptr(x), incx,
                                         float(beta), _ptr(y_out), incy, _ptr(ref_hi), _ptr(ref_lo))
        else:
            sdt = np.float32 if kind == "c" else np.float64
            al = np.array(_pair(alpha, kind), dtype=sdt)
            be = np.array(_pair(beta, kind), dtype=sdt)
            fn = {"c": self.lib.oracle_chemv, "z": self.lib.oracle_zhemv, "w": self.lib.oracle_wsymv}[kind]
            info = fn(u, n, _ptr(al), _ptr(A), lda, _ptr(x), incx, _ptr(be), _ptr(y_out), incy,
                      _ptr(ref_hi), _ptr(ref_lo))
        if width == 2:
            ref_hi = ref_hi.reshape(nn, 2)
            ref_lo = ref_lo.reshape(nn, 2)
        return info, y_out, ref_hi, ref_lo

    def rows(self, kind, uplo, n, alpha, A, lda, x, incx, beta, y0, incy, rows):
        """Rows of y by the definition on the mirrored matrix.

        Returns ``(info, ref_hi, ref_lo, denom)`` for the row indices in
        ``rows``; ``denom`` is |alpha| * sum_j |A(i,j)| |x_j| + |beta| |y_i|.
        """
        kind = kind.lower()
        dt = _DTYPES[kind]
        A = np.ascontiguousarray(A, dtype=dt)
        x = np.ascontiguousarray(x, dtype=dt)
        y0 = np.ascontiguousarray(y0, dtype=dt)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        width = 2 if kind in "cz" else 1
        ref_hi = np.zeros(len(rows) * width, dtype=np.float64)
        ref_lo = np.zeros(len(rows) * width, dtype=np.float64)
        denom = np.zeros(len(rows), dtype=np.float64)
        al = np.array(_scalar_as_doubles(alpha, kind), dtype=np.float64)
        be = np.array(_scalar_as_doubles(beta, kind), dtype=np.float64)
        u = uplo.encode() if isinstance(uplo, str) else uplo
        info = self.lib.oracle_rows(kind.encode(), u, n, _ptr(al), _ptr(A), lda, _ptr(x), incx,
                                    _ptr(be), _ptr(y0), incy, len(rows), _ptr(rows),
                                    _ptr(ref_hi), _ptr(ref_lo), _ptr(denom))
        if width == 2:
            ref_hi = ref_hi.reshape(-1, 2)
            ref_lo = ref_lo.reshape(-1, 2)
        return info, ref_hi, ref_lo, denom

    def gemv_rows(self, kind, n, alpha, A, lda, x, incx, beta, y0, incy, rows):
        """Rows of the general product y := alpha*A*x + beta*y (all n*n
        elements of A read; kind 's' or 'd').

        Returns ``(info, ref_hi, ref_lo, denom)`` for the row indices in
        ``rows``; ``denom`` is |alpha| * sum_j |A(i,j)| |x_j| + |beta| |y_i|.
        """
        kind = kind.lower()
        dt = _DTYPES[kind]
        A = np.ascontiguousarray(A, dtype=dt)
        x = np.ascontiguousarray(x, dtype=dt)
        y0 = np.ascontiguousarray(y0, dtype=dt)
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        ref_hi = np.zeros(len(rows), dtype=np.float64)
        ref_lo = np.zeros(len(rows), dtype=np.float64)
        denom = np.zeros(len(rows), dtype=np.float64)
        al = np.array(_scalar_as_doubles(alpha, kind), dtype=np.float64)
        be = np.array(_scalar_as_doubles(beta, kind), dtype=np.float64)
        info = self.lib.oracle_gemv_rows(kind.encode(), n, _ptr(al), _ptr(A), lda, _ptr(x), incx,
                                         _ptr(be), _ptr(y0), incy, len(rows), _ptr(rows),
                                         _ptr(ref_hi), _ptr(ref_lo), _ptr(denom))
        return info, ref_hi, ref_lo, denom

    def quad_mant_dig(self) -> int:
        return self.lib.oracle_quad_mant_dig()


def _pair(s, kind):
    """alpha/beta as the two numbers the C entry expects (re, im) or (hi, lo)."""
    if kind == "w":
        if isinstance(s, (tuple, list, np.ndarray)):
            return (float(s[0]), float(s[1]))
        return (float(s), 0.0)
    s = complex(s)
    return (s.real, s.imag)


def _scalar_as_doubles(s, kind):
    if kind == "s":
        return (float(np.float32(s)), 0.0)
    if kind == "d":
        return (float(s), 0.0)
    if kind == "c":
        s = complex(s)
        return (float(np.float32(s.real)), float(np.float32(s.imag)))
    return _pair(s, kind)


_lock = threading.Lock()
_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from ``oracle.c`` (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
        return _default


def symv(*args, **kw):
    return get().symv(*args, **kw)


def rows(*args, **kw):
    return get().rows(*args, **kw)


def gemv_rows(*args, **kw):
    return get().gemv_rows(*args, **kw)
