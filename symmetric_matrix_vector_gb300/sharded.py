"""One xSYMV / xHEMV call split across ranks by block columns.

The report builds on Level-2 BLAS for multi-GPU systems (its reference [7],
KBLAS, cited in §1 of "CUDA-xSYMV の実装と評価", IPSJ 2014-HPC-146) without
describing a split of its own.  The reading taken here: the stored triangle
is cut into panels of consecutive columns holding about equal numbers of
stored elements (``xsymv_shard_bounds``); rank r keeps only its panel in its
own GPU's memory, streams it once with the ``*_shard`` entry point and gets
a full-length partial vector (the row terms of its elements and the column
terms of its columns).  The partial vectors are gathered as plain copies (an
all-gather: rank r's vector lands in row r) and added in rank order by the
``*_reduce`` kernel, which also applies alpha and beta, so every rank ends
with the same, run-to-run identical y.

This module is host-side plumbing only: it slices panels out of a full
matrix held in a tensor, gathers through ``torch.distributed`` and calls the
library's entry points.  Every arithmetic step runs in the CUDA kernels.
"""
from __future__ import annotations

from . import ELEM_BYTES_BY_KIND, check, symv_reduce, symv_shard, xsymv_shard_bounds


def panel_rows(uplo: str, n: int, c0: int, c1: int):
    """(first row, row count) a panel of columns c0 .. c1-1 stores: rows
    0 .. c1-1 for upper storage, c0 .. n-1 for lower."""
    if str(uplo).upper().startswith("U"):
        return 0, c1
    return c0, n - c0


def split(uplo: str, n: int, world: int):
    """[(c0, c1)] per rank: the panels of an even split of the stored triangle."""
    b = xsymv_shard_bounds(uplo, n, world)
    return [(b[r], b[r + 1]) for r in range(world)]


def extract_panel(torch, A, kind: str, uplo: str, n: int, lda: int, c0: int, c1: int,
                  pad: int = 0):
    """A device copy of the panel of columns c0 .. c1-1 out of the full
    column-major matrix ``A`` (a tensor of raw elements, n columns of lda
    elements; complex and double-double elements as pairs of reals), in the
    layout the shard entry points take: leading dimension = panel rows + pad
    (rounded up to 16 bytes).  Returns (panel, ldp)."""
    r0, rows = panel_rows(uplo, n, c0, c1)
    per = ELEM_BYTES_BY_KIND[kind] // A.element_size()     # tensor elements per matrix element
    step = max(1, 16 // ELEM_BYTES_BY_KIND[kind])
    ldp = max(1, rows + pad)
    ldp = (ldp + step - 1) // step * step
    cols = max(0, c1 - c0)
    M = A.reshape(-1)[: n * lda * per].view(n, lda * per)
    panel = torch.zeros((max(cols, 1), ldp * per), dtype=A.dtype, device=A.device)
    if cols:
        panel[:cols, : rows * per] = M[c0:c1, r0 * per:(r0 + rows) * per]
    return panel, ldp


def gather_in_rank_order(torch, dist, partial, world: int):
    """All ranks' partial vectors, rank r's in row r (plain copies)."""
    out = torch.empty((world,) + tuple(partial.shape), dtype=partial.dtype, device=partial.device)
    if world == 1:
        out[0].copy_(partial)
        return out
    if partial.is_cuda:
        dist.all_gather_into_tensor(out, partial.contiguous())
    else:
        parts = list(out.unbind(0))
        dist.all_gather(parts, partial.contiguous())
    return out


class ShardedSymv:
    """One rank's share of y := alpha*A*x + beta*y split by block columns.

    panel: this rank's panel (device tensor, layout of ``extract_panel``);
    x: all of x on this rank's device.  step() runs the shard, gathers the
    partial vectors in rank order and reduces them into y (every rank)."""

    def __init__(self, torch, dist, kind, uplo, n, c0, c1, panel, ldp, x, incx, world):
        self.torch, self.dist = torch, dist
        self.kind, self.uplo, self.n = kind, uplo, n
        self.c0, self.c1, self.panel, self.ldp = c0, c1, panel, ldp
        self.x, self.incx, self.world = x, incx, world
        per = ELEM_BYTES_BY_KIND[kind] // x.element_size()
        self.partial = torch.empty(n * per, dtype=x.dtype, device=x.device)

    def step(self, alpha, beta, y, incy):
        check(symv_shard(self.kind, self.uplo, self.n, self.c0, self.c1, self.panel, self.ldp,
                         self.x, self.incx, self.partial))
        parts = gather_in_rank_order(self.torch, self.dist, self.partial, self.world)
        check(symv_reduce(self.kind, self.n, self.world, alpha, parts, self.n, beta, y, incy))
        return y
