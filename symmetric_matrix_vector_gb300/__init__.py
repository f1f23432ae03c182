"""xSYMV / xHEMV on NVIDIA GB300: y := alpha*A*x + beta*y for a symmetric or
Hermitian A of which only one triangle is stored and read.

A thin ctypes binding over the C ABI of ``include/xsymv.h`` (libxsymv.so,
built in-tree by ``_build.build()``).  The functions keep the C names and
argument order; they only marshal arguments: device pointers may be given as
integers or as CUDA tensors (anything with ``data_ptr()``), scalars as Python
numbers (complex for c/z, a (hi, lo) pair for w).  Every computation runs in
the library's CUDA kernels; there is no CPU path.  Each call is enqueued on
``stream`` (default: torch's current CUDA stream when torch is loaded, else
the legacy default stream).

Status codes are returned as ints (0 = success); ``check()`` turns a
non-zero status into an ``XsymvError``.
"""
from __future__ import annotations

import ctypes
import os
import sys
import threading

from . import _build

__all__ = [
    "xsymv_s", "xsymv_d", "xhemv_c", "xhemv_z", "xsymv_w", "symv",
    "xsymv_set_stream", "xsymv_get_stream", "xsymv_status_string", "xsymv_last_cuda_error",
    "xsymv_timing_enable", "xsymv_timing_read", "xsymv_launch_count",
    "xsymv_variant_count", "xsymv_variant_name", "xsymv_set_variant", "xsymv_selected_variant",
    "xsymv_workspace_bytes", "XsymvError", "check", "load", "library_path", "ENTRY_POINTS",
    "xsymv_s_host", "xsymv_d_host", "xhemv_c_host", "xhemv_z_host", "xsymv_w_host", "symv_host",
    "xsymv_host_traffic", "xsymv_sync_status", "xsymv_set_wait_limit", "xsymv_test_stall",
    "xsymv_test_set_call_number",
    "xsymv_probe_peaks", "xsymv_probe_unit_forms", "xgemv_s", "xgemv_d", "gemv", "xgemv_variant_count",
    "xgemv_variant_name", "xgemv_set_variant", "xgemv_selected_variant",
    "ELEM_BYTES_BY_KIND", "SHARD_ENTRY_POINTS", "REDUCE_ENTRY_POINTS", "symv_shard", "symv_reduce", "xsymv_shard_bounds",
    "xsymv_s_shard", "xsymv_d_shard", "xhemv_c_shard", "xhemv_z_shard", "xsymv_w_shard",
    "xsymv_s_reduce", "xsymv_d_reduce", "xhemv_c_reduce", "xhemv_z_reduce", "xsymv_w_reduce",
]

ENTRY_POINTS = {"s": "xsymv_s", "d": "xsymv_d", "c": "xhemv_c", "z": "xhemv_z", "w": "xsymv_w"}
ELEM_BYTES_BY_KIND = {"s": 4, "d": 8, "c": 8, "z": 16, "w": 16}
SHARD_ENTRY_POINTS = {k: v + "_shard" for k, v in ENTRY_POINTS.items()}
REDUCE_ENTRY_POINTS = {k: v + "_reduce" for k, v in ENTRY_POINTS.items()}


class C32(ctypes.Structure):
    _fields_ = [("re", ctypes.c_float), ("im", ctypes.c_float)]


class C64(ctypes.Structure):
    _fields_ = [("re", ctypes.c_double), ("im", ctypes.c_double)]


class DD(ctypes.Structure):
    _fields_ = [("hi", ctypes.c_double), ("lo", ctypes.c_double)]


class XsymvError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("xsymv status %d: %s" % (status, message))
        self.status = status


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIBPATH


def load():
    """The loaded libxsymv.so.  Raises if it has not been built: there is no
    fallback implementation."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = _build.LIBPATH
        if not os.path.exists(path):
            raise RuntimeError("libxsymv.so is not built (run __graft_entry__.build() or "
                               "python -m symmetric_matrix_vector_gb300._build)")
        lib = ctypes.CDLL(path)
        c_char, c_int, vp = ctypes.c_char, ctypes.c_int, ctypes.c_void_p
        scal = {"s": ctypes.c_float, "d": ctypes.c_double, "c": C32, "z": C64, "w": DD}
        for k, name in ENTRY_POINTS.items():
            for nm in (name, name + "_host"):
                fn = getattr(lib, nm)
                fn.argtypes = [c_char, c_int, scal[k], vp, c_int, vp, c_int, scal[k], vp, c_int]
                fn.restype = c_int
        for k in ENTRY_POINTS:
            fn = getattr(lib, SHARD_ENTRY_POINTS[k])
            fn.argtypes = [c_char, c_int, c_int, c_int, vp, c_int, vp, c_int, vp]
            fn.restype = c_int
            fn = getattr(lib, REDUCE_ENTRY_POINTS[k])
            fn.argtypes = [c_int, c_int, scal[k], vp, ctypes.c_longlong, scal[k], vp, c_int]
            fn.restype = c_int
        lib.xsymv_shard_bounds.argtypes = [c_char, c_int, c_int, ctypes.POINTER(c_int)]
        lib.xsymv_shard_bounds.restype = c_int
        lib.xsymv_host_traffic.argtypes = [ctypes.POINTER(ctypes.c_longlong)] * 2
        lib.xsymv_host_traffic.restype = c_int
        lib.xsymv_sync_status.restype = c_int
        lib.xsymv_probe_peaks.argtypes = [ctypes.POINTER(ctypes.c_double)] * 4
        lib.xsymv_probe_peaks.restype = c_int
        lib.xsymv_probe_unit_forms.argtypes = [vp, vp, vp, ctypes.c_longlong]
        lib.xsymv_probe_unit_forms.restype = c_int
        lib.xsymv_set_wait_limit.argtypes = [ctypes.c_ulonglong]
        lib.xsymv_set_wait_limit.restype = c_int
        lib.xsymv_test_stall.argtypes = [c_int]
        lib.xsymv_test_stall.restype = c_int
        lib.xsymv_test_set_call_number.argtypes = [c_int]
        lib.xsymv_test_set_call_number.restype = c_int
        lib.xsymv_set_stream.argtypes = [vp]
        lib.xsymv_set_stream.restype = c_int
        lib.xsymv_get_stream.restype = vp
        lib.xsymv_status_string.argtypes = [c_int]
        lib.xsymv_status_string.restype = ctypes.c_char_p
        lib.xsymv_last_cuda_error.restype = c_int
        lib.xsymv_timing_enable.argtypes = [c_int]
        lib.xsymv_timing_enable.restype = c_int
        lib.xsymv_timing_read.argtypes = [ctypes.POINTER(c_int), ctypes.POINTER(ctypes.c_double),
                                          ctypes.POINTER(ctypes.c_double)]
        lib.xsymv_timing_read.restype = c_int
        lib.xsymv_launch_count.restype = ctypes.c_longlong
        lib.xsymv_variant_count.argtypes = [c_char]
        lib.xsymv_variant_count.restype = c_int
        lib.xsymv_variant_name.argtypes = [c_char, c_int]
        lib.xsymv_variant_name.restype = ctypes.c_char_p
        lib.xsymv_set_variant.argtypes = [c_char, c_int]
        lib.xsymv_set_variant.restype = c_int
        lib.xsymv_selected_variant.argtypes = [c_char, c_char, c_int]
        lib.xsymv_selected_variant.restype = c_int
        lib.xsymv_workspace_bytes.argtypes = [c_char, c_char, c_int]
        lib.xsymv_workspace_bytes.restype = ctypes.c_longlong
        for k in ("s", "d"):
            fn = getattr(lib, "xgemv_" + k)
            fn.argtypes = [c_int, scal[k], vp, c_int, vp, c_int, scal[k], vp, c_int]
            fn.restype = c_int
        lib.xgemv_variant_count.argtypes = [c_char]
        lib.xgemv_variant_count.restype = c_int
        lib.xgemv_variant_name.argtypes = [c_char, c_int]
        lib.xgemv_variant_name.restype = ctypes.c_char_p
        lib.xgemv_set_variant.argtypes = [c_char, c_int]
        lib.xgemv_set_variant.restype = c_int
        lib.xgemv_selected_variant.argtypes = [c_char]
        lib.xgemv_selected_variant.restype = c_int
        _lib = lib
        return lib


# ------------------------------------------------------------- marshalling --

def _ptr(a) -> int:
    if a is None:
        return 0
    if isinstance(a, int):
        return a
    if hasattr(a, "data_ptr"):
        if hasattr(a, "is_cuda") and not a.is_cuda:
            raise ValueError("xsymv needs device memory; got a CPU tensor")
        return a.data_ptr()
    raise TypeError("expected a device pointer (int) or a CUDA tensor, got %r" % type(a))


def _scalar(kind: str, v):
    if kind == "s" or kind == "d":     # ctypes converts a float to the declared type
        return float(v)
    if kind == "c":
        v = complex(v)
        return C32(v.real, v.imag)
    if kind == "z":
        v = complex(v)
        return C64(v.real, v.imag)
    if isinstance(v, (tuple, list)):
        return DD(float(v[0]), float(v[1]))
    return DD(float(v), 0.0)


def _uplo(u) -> bytes:
    if isinstance(u, bytes):
        return u
    return str(u).encode()[:1] or b"?"


_cuda_ok = None          # torch's CUDA availability, asked once


def _torch_stream():
    """torch's current CUDA stream on the current device, as an address
    (None when torch is not loaded or has no GPU)"""
    global _cuda_ok
    torch = sys.modules.get("torch")
    if torch is None:
        return None
    if _cuda_ok is None:
        _cuda_ok = bool(torch.cuda.is_available())
    if not _cuda_ok:
        return None
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:
        return raw(torch._C._cuda_getDevice())
    return torch.cuda.current_stream().cuda_stream


_stream_set = [None]    # the stream last handed to xsymv_set_stream from here


def _use_stream(lib, stream):
    s = _torch_stream() if stream is None else (stream if isinstance(stream, int) else
                                                getattr(stream, "cuda_stream", stream))
    s = s or 0
    if s != _stream_set[0]:
        lib.xsymv_set_stream(s)
        _stream_set[0] = s


def _host_ptr(a) -> int:
    if a is None:
        return 0
    if isinstance(a, int):
        return a
    if hasattr(a, "data_ptr"):
        return a.data_ptr()
    if hasattr(a, "ctypes"):                      # numpy array
        return a.ctypes.data
    raise TypeError("expected a host pointer, a numpy array or a tensor, got %r" % type(a))


def _call(kind, uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream, host=False):
    lib = _lib if _lib is not None else load()
    _use_stream(lib, stream)
    fn = getattr(lib, ENTRY_POINTS[kind] + ("_host" if host else ""))
    cv = _host_ptr if host else _ptr
    return fn(_uplo(uplo), int(n), _scalar(kind, alpha), cv(A), int(lda), cv(x), int(incx),
              _scalar(kind, beta), cv(y), int(incy))


def xsymv_s(uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream=None) -> int:
    return _call("s", uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream)


def xsymv_d(uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream=None) -> int:
    return _call("d", uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream)


def xhemv_c(uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream=None) -> int:
    return _call("c", uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream)


def xhemv_z(uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream=None) -> int:
    return _call("z", uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream)


def xsymv_w(uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream=None) -> int:
    return _call("w", uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream)


def symv(kind, uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream=None) -> int:
    """Dispatch on kind ('s', 'd', 'c', 'z', 'w') to the matching entry point."""
    return _call(kind.lower(), uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream)


def xsymv_s_host(uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream=None) -> int:
    return _call("s", uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream, host=True)


def xsymv_d_host(uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream=None) -> int:
    return _call("d", uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream, host=True)


def xhemv_c_host(uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream=None) -> int:
    return _call("c", uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream, host=True)


def xhemv_z_host(uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream=None) -> int:
    return _call("z", uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream, host=True)


def xsymv_w_host(uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream=None) -> int:
    return _call("w", uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream, host=True)


def symv_host(kind, uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream=None) -> int:
    """Host-buffer variant of ``symv``: A, x, y are host arrays (numpy arrays,
    CPU tensors or raw addresses); y holds the result on return."""
    return _call(kind.lower(), uplo, n, alpha, A, lda, x, incx, beta, y, incy, stream, host=True)


# ------------------------------------------- the block-column split -------

def xsymv_shard_bounds(uplo, n, nparts):
    """Column boundaries [b_0 = 0, ..., b_nparts = n] of an even split of the
    stored triangle into nparts panels (panel r: columns b_r .. b_{r+1}-1).
    Host only.  Raises XsymvError on a bad argument."""
    nparts = int(nparts)
    if nparts < 1:
        raise XsymvError(3, "invalid argument 3 (nparts): must be >= 1")
    out = (ctypes.c_int * (nparts + 1))()
    check(load().xsymv_shard_bounds(_uplo(uplo), int(n), nparts, out))
    return list(out)


def symv_shard(kind, uplo, n, col_begin, col_end, A, lda, x, incx, partial, stream=None) -> int:
    """One shard of the block-column split: the panel of stored columns
    col_begin .. col_end-1 (A: the panel alone, device memory) writes its
    n-element partial vector to ``partial`` (device).  See include/xsymv.h."""
    kind = kind.lower()
    lib = load()
    _set_stream(lib, stream)
    return getattr(lib, SHARD_ENTRY_POINTS[kind])(
        _uplo(uplo), int(n), int(col_begin), int(col_end), ctypes.c_void_p(_ptr(A)), int(lda),
        ctypes.c_void_p(_ptr(x)), int(incx), ctypes.c_void_p(_ptr(partial)))


def symv_reduce(kind, n, nparts, alpha, partials, ldp, beta, y, incy, stream=None) -> int:
    """y := alpha * (sum of the nparts partial vectors, in rank order) + beta * y
    (partial r at partials + r*ldp elements; device memory)."""
    kind = kind.lower()
    lib = load()
    _set_stream(lib, stream)
    return getattr(lib, REDUCE_ENTRY_POINTS[kind])(
        int(n), int(nparts), _scalar(kind, alpha), ctypes.c_void_p(_ptr(partials)), int(ldp),
        _scalar(kind, beta), ctypes.c_void_p(_ptr(y)), int(incy))


def _shard_fn(kind):
    def f(uplo, n, col_begin, col_end, A, lda, x, incx, partial, stream=None):
        return symv_shard(kind, uplo, n, col_begin, col_end, A, lda, x, incx, partial, stream)
    f.__name__ = SHARD_ENTRY_POINTS[kind]
    return f


def _reduce_fn(kind):
    def f(n, nparts, alpha, partials, ldp, beta, y, incy, stream=None):
        return symv_reduce(kind, n, nparts, alpha, partials, ldp, beta, y, incy, stream)
    f.__name__ = REDUCE_ENTRY_POINTS[kind]
    return f


xsymv_s_shard, xsymv_d_shard, xhemv_c_shard, xhemv_z_shard, xsymv_w_shard = (
    _shard_fn(k) for k in "sdczw")
xsymv_s_reduce, xsymv_d_reduce, xhemv_c_reduce, xhemv_z_reduce, xsymv_w_reduce = (
    _reduce_fn(k) for k in "sdczw")


def xsymv_host_traffic():
    """(host-to-device bytes, device-to-host bytes) of the last host call"""
    h, d = ctypes.c_longlong(0), ctypes.c_longlong(0)
    check(load().xsymv_host_traffic(ctypes.byref(h), ctypes.byref(d)))
    return h.value, d.value


def xsymv_sync_status() -> int:
    """Wait for the current stream; XSYMV_ERR_TIMEOUT (-6) if its latest call
    gave up on a bounded wait (its y was set to NaN), else 0."""
    return load().xsymv_sync_status()


def xsymv_set_wait_limit(ns: int) -> int:
    return load().xsymv_set_wait_limit(int(ns))


def xsymv_test_stall(on: bool) -> int:
    return load().xsymv_test_stall(1 if on else 0)


def xsymv_test_set_call_number(number: int) -> int:
    return load().xsymv_test_set_call_number(int(number))


def xsymv_probe_peaks():
    """Measured now: dict of copy_gbs, read_gbs, fp64_tflops, fp32_tflops."""
    v = [ctypes.c_double(0) for _ in range(4)]
    check(load().xsymv_probe_peaks(*[ctypes.byref(x) for x in v]))
    return dict(zip(("copy_gbs", "read_gbs", "fp64_tflops", "fp32_tflops"), (x.value for x in v)))


def xsymv_probe_unit_forms(a, b, out, n: int, stream=None) -> int:
    """out[6i:6i+6] = a+b, a-b, a*b (plain instructions), then the same in the
    fused multiply-add form the DD kernels use; device tensors of doubles."""
    lib = load()
    _use_stream(lib, stream)
    return lib.xsymv_probe_unit_forms(_ptr(a), _ptr(b), _ptr(out), int(n))


def xsymv_set_stream(stream) -> int:
    s = int(stream or 0)
    _stream_set[0] = s
    return load().xsymv_set_stream(s)


def xsymv_get_stream() -> int:
    return load().xsymv_get_stream() or 0


def xsymv_status_string(status: int) -> str:
    return load().xsymv_status_string(int(status)).decode()


def xsymv_last_cuda_error() -> int:
    return load().xsymv_last_cuda_error()


def check(status: int) -> None:
    if status != 0:
        raise XsymvError(status, xsymv_status_string(status))


def xsymv_timing_enable(on: bool) -> int:
    return load().xsymv_timing_enable(1 if on else 0)


def xsymv_timing_read():
    """(calls, main-kernel ms summed, whole-call ms summed); clears the record."""
    calls, m, c = ctypes.c_int(0), ctypes.c_double(0), ctypes.c_double(0)
    st = load().xsymv_timing_read(ctypes.byref(calls), ctypes.byref(m), ctypes.byref(c))
    check(st)
    return calls.value, m.value, c.value


def xsymv_launch_count() -> int:
    return load().xsymv_launch_count()


def xsymv_variant_count(kind: str) -> int:
    return load().xsymv_variant_count(kind.encode())


def xsymv_variant_name(kind: str, index: int):
    r = load().xsymv_variant_name(kind.encode(), int(index))
    return r.decode() if r else None


def xsymv_set_variant(kind: str, index: int) -> int:
    return load().xsymv_set_variant(kind.encode(), int(index))


def xsymv_selected_variant(kind: str, uplo: str, n: int) -> int:
    return load().xsymv_selected_variant(kind.encode(), _uplo(uplo), int(n))


def xsymv_workspace_bytes(kind: str, uplo: str, n: int) -> int:
    return load().xsymv_workspace_bytes(kind.encode(), _uplo(uplo), int(n))


# ------------------------------------------- the general product (GEMV) --

def _set_stream(lib, stream):
    _use_stream(lib, stream)


def gemv(kind, n, alpha, A, lda, x, incx, beta, y, incy, stream=None) -> int:
    """y := alpha*A*x + beta*y for a general n-by-n A (kind 's' or 'd'),
    device memory, on the SYMV kernels' loader (xgemv_s / xgemv_d)."""
    kind = kind.lower()
    if kind not in ("s", "d"):
        raise ValueError("gemv kind must be 's' or 'd'")
    lib = load()
    _set_stream(lib, stream)
    return getattr(lib, "xgemv_" + kind)(int(n), _scalar(kind, alpha), ctypes.c_void_p(_ptr(A)),
                                         int(lda), ctypes.c_void_p(_ptr(x)), int(incx),
                                         _scalar(kind, beta), ctypes.c_void_p(_ptr(y)), int(incy))


def xgemv_s(n, alpha, A, lda, x, incx, beta, y, incy, stream=None) -> int:
    return gemv("s", n, alpha, A, lda, x, incx, beta, y, incy, stream)


def xgemv_d(n, alpha, A, lda, x, incx, beta, y, incy, stream=None) -> int:
    return gemv("d", n, alpha, A, lda, x, incx, beta, y, incy, stream)


def xgemv_variant_count(kind: str) -> int:
    return load().xgemv_variant_count(kind.encode())


def xgemv_variant_name(kind: str, index: int):
    r = load().xgemv_variant_name(kind.encode(), int(index))
    return r.decode() if r else None


def xgemv_set_variant(kind: str, index: int) -> int:
    return load().xgemv_set_variant(kind.encode(), int(index))


def xgemv_selected_variant(kind: str) -> int:
    return load().xgemv_selected_variant(kind.encode())
