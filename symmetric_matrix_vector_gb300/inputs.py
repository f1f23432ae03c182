"""Seeded synthetic inputs for xSYMV / xHEMV.

This module only draws random numbers and lays them out; it holds none of the
SYMV arithmetic.  Tests, the benchmark and the smoke check generate one
problem here and hand the same arrays to both the CUDA library and the CPU
oracle.

Layout (host numpy arrays, BLAS column-major):
  * ``A`` has shape ``(n, lda)`` (``(n, lda, 2)`` for double-double); numpy
    row ``j`` is matrix column ``j``, so ``A[j, i]`` is A(i, j).
  * Everything outside the stored triangle — the other triangle, the rows
    ``n..lda-1`` of each column, and for Hermitian matrices the imaginary
    part of the diagonal — is filled with NaN, so a kernel that uses any of
    it in its arithmetic produces NaN.
  * ``x`` / ``y`` are strided vectors of ``1 + (n-1)*|inc|`` elements whose
    gap elements are NaN.

The random stream is numpy's PCG64 seeded with the workload's seed; values
are drawn column by column in the order A, x, y.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

KINDS = ("s", "d", "c", "z", "w")
DTYPES = {"s": np.float32, "d": np.float64, "c": np.complex64, "z": np.complex128, "w": np.float64}
REAL_DTYPES = {"s": np.float32, "d": np.float64, "c": np.float32, "z": np.float64, "w": np.float64}
ELEM_BYTES = {"s": 4, "d": 8, "c": 8, "z": 16, "w": 16}


@dataclass
class Problem:
    """One SYMV/HEMV call: ``y := alpha*A*x + beta*y``."""

    kind: str
    uplo: str
    n: int
    lda: int
    alpha: object
    beta: object
    A: np.ndarray
    x: np.ndarray
    y: np.ndarray
    incx: int = 1
    incy: int = 1
    seed: int = 0
    name: str = ""
    notes: dict = field(default_factory=dict)

    @property
    def elem_bytes(self) -> int:
        return ELEM_BYTES[self.kind]


def _draw(rng: np.random.Generator, shape, dist: str, kind: str) -> np.ndarray:
    """Real array of ``shape`` in the working precision of ``kind``."""
    rdt = REAL_DTYPES[kind]
    if dist == "uniform":
        a = rng.random(shape, dtype=rdt)
        a *= 2
        a -= 1
        return a
    if dist == "normal":
        return rng.standard_normal(shape, dtype=rdt)
    raise ValueError(dist)


def _values(rng, count: int, dist: str, kind: str) -> np.ndarray:
    """``count`` scalars of ``kind``: complex draws re then im per element;
    double-double draws hi, then lo = hi * 2^-53 * U(-1, 1)."""
    if kind in ("s", "d"):
        return _draw(rng, (count,), dist, kind)
    if kind in ("c", "z"):
        ri = _draw(rng, (count, 2), dist, kind)
        return ri.view(DTYPES[kind]).reshape(count)
    hi = _draw(rng, (count,), dist, kind)
    lo = hi * np.ldexp(1.0, -53) * _draw(rng, (count,), "uniform", kind)
    return np.stack([hi, lo], axis=-1)


def _nan_of(kind: str):
    if kind in ("c", "z"):
        return complex(np.nan, np.nan)
    return np.nan


def _strided(v: np.ndarray, inc: int, kind: str) -> np.ndarray:
    """Place logical vector ``v`` with stride ``inc`` (BLAS), NaN in the gaps."""
    n = v.shape[0]
    m = 1 + (n - 1) * abs(inc) if n > 0 else 1
    out = np.empty((m,) + v.shape[1:], dtype=v.dtype)
    out[...] = np.nan if kind != "c" and kind != "z" else _nan_of(kind)
    idx = np.arange(n) * abs(inc)
    if inc < 0:
        idx = idx[::-1]
    out[idx] = v
    return out


def make_problem(kind: str, uplo: str, n: int, *, lda: int | None = None, alpha=1.0, beta=0.0,
                 dist: str = "uniform", diag_shift: float = 0.0, seed: int = 0,
                 incx: int = 1, incy: int = 1, name: str = "",
                 column_chunk: int = 2048) -> Problem:
    """Dense random problem with only the ``uplo`` triangle meaningful.

    The stored triangle (diagonal included) gets i.i.d. ``dist`` values;
    ``diag_shift`` is added to the real part of every diagonal element.
    Hermitian kinds (c, z) get a NaN imaginary part on the diagonal.
    """
    kind = kind.lower()
    uplo = uplo.upper()
    if kind not in KINDS or uplo not in ("U", "L"):
        raise ValueError((kind, uplo))
    lda = max(1, n) if lda is None else lda
    rng = np.random.default_rng(seed)
    shape = (n, lda) + ((2,) if kind == "w" else ())
    A = np.empty(shape, dtype=DTYPES[kind])
    nan = _nan_of(kind)
    # draw column by column (in chunks) so memory stays bounded at large n
    for j0 in range(0, n, column_chunk):
        j1 = min(n, j0 + column_chunk)
        cnt = (j1 - j0) * lda
        block = _values(rng, cnt, dist, kind).reshape((j1 - j0, lda) + A.shape[2:])
        A[j0:j1] = block
    for j in range(n):
        col = A[j]
        if uplo == "U":
            col[j + 1:] = nan            # strictly lower part and padding rows
        else:
            col[:j] = nan                # strictly upper part
            col[n:] = nan                # padding rows
        if diag_shift:
            if kind == "w":
                col[j, 0] += diag_shift
            else:
                col[j] += diag_shift
        if kind in ("c", "z"):
            col[j] = complex(col[j].real, np.nan)
    xv = _values(rng, n, dist, kind)
    yv = _values(rng, n, dist, kind)
    x = _strided(xv, incx, kind)
    y = _strided(yv, incy, kind)
    return Problem(kind=kind, uplo=uplo, n=n, lda=lda, alpha=alpha, beta=beta, A=A, x=x, y=y,
                   incx=incx, incy=incy, seed=seed, name=name)


def make_general(kind: str, n: int, *, lda: int | None = None, alpha=1.0, beta=0.0,
                 dist: str = "uniform", seed: int = 0, incx: int = 1, incy: int = 1,
                 name: str = "", column_chunk: int = 2048) -> Problem:
    """Dense random unsymmetric n-by-n problem for the general product
    (kind 's' or 'd'): every element of the n-by-n matrix gets an i.i.d.
    ``dist`` value, the padding rows n..lda-1 NaN.  ``uplo`` is "G"."""
    kind = kind.lower()
    if kind not in ("s", "d"):
        raise ValueError(kind)
    lda = max(1, n) if lda is None else lda
    rng = np.random.default_rng(seed)
    A = np.empty((n, lda), dtype=DTYPES[kind])
    for j0 in range(0, n, column_chunk):
        j1 = min(n, j0 + column_chunk)
        A[j0:j1] = _values(rng, (j1 - j0) * lda, dist, kind).reshape(j1 - j0, lda)
    A[:, n:] = np.nan
    x = _strided(_values(rng, n, dist, kind), incx, kind)
    y = _strided(_values(rng, n, dist, kind), incy, kind)
    return Problem(kind=kind, uplo="G", n=n, lda=lda, alpha=alpha, beta=beta, A=A, x=x, y=y,
                   incx=incx, incy=incy, seed=seed, name=name)


# ---------------------------------------------------------------------------
# The five workloads of the CUDA-xSYMV evaluation, restated at GB300 sizes
# ---------------------------------------------------------------------------

SSYMV_SWEEP = tuple(range(4096, 32768 + 1, 4096))


def workload(name: str, n: int | None = None, **over) -> Problem:
    """Named synthetic workloads.

    ssymv_small  SSYMV n=1024, L, lda=n; U(-1,1); alpha=1.25, beta=0.5; seed 0
    ssymv_sweep  SSYMV n in 4096..32768 (step 4096), U, lda=n+32; U(-1,1);
                 alpha=1, beta=0; seed n
    dsymv        DSYMV n=24576, L, lda=n; N(0,1) with diagonal +4;
                 alpha=-0.75, beta=2; seed 7
    chemv/zhemv  n=16384, U, lda=n; U(-1,1) re and im, diagonal imag NaN;
                 alpha=(1,0.5), beta=(0.5,-0.25); seed 11
    wsymv        double-double n=8192, L, lda=n; hi U(-1,1),
                 lo = hi*2^-53*U(-1,1); alpha=beta=(1,0); seed 13
    ``n`` overrides the size (the sweep's seed stays n); other keyword
    arguments override ``make_problem`` parameters.
    """
    if name == "ssymv_small":
        nn = n or 1024
        kw = dict(kind="s", uplo="L", n=nn, lda=nn, alpha=1.25, beta=0.5, seed=0)
    elif name == "ssymv_sweep":
        nn = n or 32768
        kw = dict(kind="s", uplo="U", n=nn, lda=nn + 32, alpha=1.0, beta=0.0, seed=nn)
    elif name == "dsymv":
        nn = n or 24576
        kw = dict(kind="d", uplo="L", n=nn, lda=nn, alpha=-0.75, beta=2.0, dist="normal",
                  diag_shift=4.0, seed=7)
    elif name in ("chemv", "zhemv"):
        nn = n or 16384
        kw = dict(kind=name[0], uplo="U", n=nn, lda=nn, alpha=complex(1.0, 0.5),
                  beta=complex(0.5, -0.25), seed=11)
    elif name == "wsymv":
        nn = n or 8192
        kw = dict(kind="w", uplo="L", n=nn, lda=nn, alpha=(1.0, 0.0), beta=(1.0, 0.0), seed=13)
    else:
        raise KeyError(name)
    kw.update(over)
    return make_problem(name=name, **kw)


WORKLOADS = ("ssymv_small", "ssymv_sweep", "dsymv", "chemv", "zhemv", "wsymv")


# ---------------------------------------------------------------------------
# the same recipe drawn on the GPU (torch's Philox generator), for benchmarks
# ---------------------------------------------------------------------------

def device_problem(kind: str, uplo: str, n: int, *, lda: int | None = None, alpha=1.0, beta=0.0,
                   dist: str = "uniform", diag_shift: float = 0.0, seed: int = 0,
                   device: str = "cuda"):
    """Dense random problem on the device, contiguous x and y (inc = 1).

    Same layout and sentinels as ``make_problem`` (NaN outside the stored
    triangle, in the padding rows and in Hermitian diagonal imaginary parts);
    the random stream is torch's CUDA generator seeded with ``seed``, so the
    values differ from the host recipe's.  Returns a dict with tensors ``A``
    (shape (n, lda), or (n, lda, 2) for w), ``x``, ``y`` and the scalars.
    """
    import torch

    kind = kind.lower()
    uplo = uplo.upper()
    lda = max(1, n) if lda is None else lda
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    rdt = {"s": torch.float32, "d": torch.float64, "c": torch.float32, "z": torch.float64,
           "w": torch.float64}[kind]
    width = {"s": 1, "d": 1, "c": 2, "z": 2, "w": 2}[kind]

    def draw(shape):
        if dist == "uniform":
            return torch.rand(shape, generator=g, device=device, dtype=rdt).mul_(2).sub_(1)
        return torch.randn(shape, generator=g, device=device, dtype=rdt)

    def values(count):
        if kind in ("s", "d"):
            return draw((count,))
        if kind in ("c", "z"):
            return draw((count, 2))
        hi = draw((count,))
        lo = hi * (2.0 ** -53) * (torch.rand((count,), generator=g, device=device,
                                             dtype=rdt) * 2 - 1)
        return torch.stack([hi, lo], dim=-1)

    A = values(n * lda).reshape(n, lda, *(() if width == 1 else (2,)))
    rows = torch.arange(lda, device=device)[None, :]
    cols = torch.arange(n, device=device)[:, None]
    unused = (rows > cols) if uplo == "U" else ((rows < cols) | (rows >= n))
    if width == 1:
        A.masked_fill_(unused, float("nan"))
    else:
        A.masked_fill_(unused[..., None], float("nan"))
    idx = torch.arange(n, device=device)
    if diag_shift:
        if width == 1:
            A[idx, idx] += diag_shift
        else:
            A[idx, idx, 0] += diag_shift
    if kind in ("c", "z"):
        A[idx, idx, 1] = float("nan")
    return dict(kind=kind, uplo=uplo, n=n, lda=lda, alpha=alpha, beta=beta, A=A.contiguous(),
                x=values(n).contiguous(), y=values(n).contiguous())


def device_general(kind: str, n: int, *, lda: int | None = None, alpha=1.0, beta=0.0,
                   dist: str = "uniform", seed: int = 0, device: str = "cuda"):
    """Dense random unsymmetric problem on the device for the general product
    (kind 's' or 'd'), contiguous x and y; NaN in the padding rows only."""
    import torch

    kind = kind.lower()
    lda = max(1, n) if lda is None else lda
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    dt = {"s": torch.float32, "d": torch.float64}[kind]

    def draw(shape):
        if dist == "uniform":
            return torch.rand(shape, generator=g, device=device, dtype=dt).mul_(2).sub_(1)
        return torch.randn(shape, generator=g, device=device, dtype=dt)

    A = draw((n, lda))
    A[:, n:] = float("nan")
    return dict(kind=kind, uplo="G", n=n, lda=lda, alpha=alpha, beta=beta, A=A.contiguous(),
                x=draw((n,)).contiguous(), y=draw((n,)).contiguous())
