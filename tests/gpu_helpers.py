"""Helpers for the GPU parity tests: move a Problem's arrays to the device as
raw bytes, run one C-ABI call, and measure the componentwise error against
the CPU oracle, normalised by |alpha|*(|A||x|)_i + |beta|*|y_i|."""
from __future__ import annotations

import numpy as np

# componentwise tolerances (|y - y_ref| / (|alpha| |A||x| + |beta| |y|))
TOL = {"s": 5e-5, "c": 5e-5, "d": 1e-13, "z": 1e-13, "w": 1e-28}


def to_device(arr: np.ndarray):
    import torch

    flat = np.ascontiguousarray(arr).reshape(-1).view(np.uint8)
    return torch.from_numpy(flat).cuda()


def from_device(t, like: np.ndarray) -> np.ndarray:
    return t.cpu().numpy().view(like.dtype).reshape(like.shape)


class DeviceProblem:
    """A Problem's A, x and y resident on the GPU (A and x read-only)."""

    def __init__(self, p):
        self.p = p
        self.A = to_device(p.A)
        self.x = to_device(p.x)
        self.y0 = to_device(p.y)

    def run(self, alpha=None, beta=None, y=None, lda=None, A=None, stream=None):
        import symmetric_matrix_vector_gb300 as xs

        p = self.p
        yd = self.y0.clone() if y is None else y
        st = xs.symv(p.kind, p.uplo, p.n, p.alpha if alpha is None else alpha,
                     self.A if A is None else A, p.lda if lda is None else lda, self.x, p.incx,
                     p.beta if beta is None else beta, yd, p.incy, stream=stream)
        return st, yd


def logical(kind: str, v: np.ndarray, n: int, inc: int) -> np.ndarray:
    """the n logical elements of a strided vector (BLAS indexing)"""
    idx = np.arange(n) * abs(inc)
    if inc < 0:
        idx = idx[::-1]
    return v[idx]


def errors(o, p, y_gpu: np.ndarray, rows=None, alpha=None, beta=None):
    """componentwise normalised error of the GPU result for the given rows
    (all rows by default); returns (err array, rows)"""
    n = p.n
    rows = np.arange(n) if rows is None else np.asarray(rows, dtype=np.int64)
    al = p.alpha if alpha is None else alpha
    be = p.beta if beta is None else beta
    info, hi, lo, den = o.rows(p.kind, p.uplo, n, al, p.A, p.lda, p.x, p.incx, be, p.y, p.incy,
                               rows)
    assert info == 0, info
    yl = logical(p.kind, y_gpu, n, p.incy)[rows]
    k = p.kind
    with np.errstate(invalid="ignore", divide="ignore"):
        if k == "w":
            d = (yl[:, 0] - hi) + (yl[:, 1] - lo)
            err = np.abs(d)
        elif k in ("c", "z"):
            dr = (yl.real.astype(np.float64) - hi[:, 0]) - lo[:, 0]
            di = (yl.imag.astype(np.float64) - hi[:, 1]) - lo[:, 1]
            err = np.hypot(dr, di)
        else:
            err = np.abs((yl.astype(np.float64) - hi) - lo)
        rel = np.where(den > 0, err / np.where(den > 0, den, 1.0), err)
    rel[~np.isfinite(rel)] = np.inf
    return rel, rows


def sample_rows(n: int, NB_list=(32, 64, 128, 256), count: int = 192, seed: int = 0):
    """row indices: both ends, every tile boundary +-1 for the given tile
    edges (capped), and a seeded random sample"""
    rng = np.random.default_rng(seed)
    s = {0, 1, n - 1, n - 2, n // 2}
    for nb in NB_list:
        for b in range(0, n, nb * max(1, (n // nb) // 16)):
            for d in (-1, 0, 1):
                if 0 <= b + d < n:
                    s.add(b + d)
    s.update(rng.choice(n, size=min(count, n), replace=False).tolist())
    return np.array(sorted(r for r in s if 0 <= r < n), dtype=np.int64)
