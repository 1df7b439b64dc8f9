"""One fused call over a matrix whose rows are split across ranks, one GPU each.

The pattern's ``X^T (v * (X y))`` is a sum over the rows of X ("On optimizing machine
learning workloads via kernel fusion", abstract: the generic pattern): with t_i =
v_i (x_i . y), it equals sum_i t_i x_i. So a split of X into row blocks X_g (and v into
the matching v_g), with y on every rank, needs exactly one exchange:

1. each rank computes its partial w_g = X_g^T (v_g * (X_g y)) with one fused call at
   alpha = 1, beta = 0 and no z (the kernels of ``fxtx_dense_*`` / ``fxtx_csr_*``);
2. one all-reduce (sum) of the n-vector w_g across the ranks;
3. every rank applies out = alpha * w + beta * z with ``fxtx_epilogue_*``.

A CSR block keeps its rows' entries and a row_ptr rebased to start at 0. Blocks are
balanced by rows (dense) or by equal shares of nnz + 8 * rows (CSR, the weight the
single-device partition of the CSR kernels also uses). The device work is the library's
kernels; this module only partitions, slices and calls ``torch.distributed``.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Any, Callable, Optional

import numpy as np

from . import _lib

CSR_ROW_COST = 8  # nnz-equivalent cost of one row in the CSR partition


def row_bounds(m: int, world: int, row_ptr=None, row_cost: int = CSR_ROW_COST) -> list[int]:
    """Row boundaries 0 = r_0 <= r_1 <= ... <= r_world = m of `world` blocks.

    Dense (row_ptr None): equal row counts. CSR: block g starts at the first row i with
    row_ptr[i] + row_cost * i >= g * (nnz + row_cost * m) / world.
    """
    if m < 0 or world < 1:
        raise ValueError("row_bounds: m >= 0 and world >= 1")
    if row_ptr is None:
        return [m * g // world for g in range(world + 1)]
    rp = _host_int64(row_ptr)
    if rp.shape[0] != m + 1:
        raise ValueError("row_bounds: row_ptr must hold m + 1 entries")
    cost = rp + row_cost * np.arange(m + 1, dtype=np.int64)
    total = int(cost[-1])
    targets = [total * g // world for g in range(1, world)]
    inner = [int(np.searchsorted(cost, t, side="left")) for t in targets]
    return [0] + [min(max(r, 0), m) for r in inner] + [m]


def _host_int64(a) -> np.ndarray:
    if hasattr(a, "detach"):  # a torch tensor, on any device
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int64)


@dataclass
class RowShard:
    """The rows [r0, r1) of X held by one rank, with the matching slice of v."""

    kind: str  # "dense" or "csr"
    n: int
    r0: int
    r1: int
    v: Any = None
    X: Any = None  # dense: the (r1 - r0, n) row block
    row_ptr: Any = None  # CSR: r1 - r0 + 1 offsets rebased to 0
    col_idx: Any = None
    vals: Any = None

    @property
    def rows(self) -> int:
        return self.r1 - self.r0


def shard_dense(X, v, bounds: list[int], rank: int) -> RowShard:
    """Rank `rank`'s row block of a dense X (numpy array or torch tensor) and of v."""
    r0, r1 = bounds[rank], bounds[rank + 1]
    return RowShard("dense", int(X.shape[1]), r0, r1, v=None if v is None else v[r0:r1], X=X[r0:r1])


def shard_csr(row_ptr, col_idx, vals, v, n: int, bounds: list[int], rank: int) -> RowShard:
    """Rank `rank`'s row block of a CSR X: row_ptr[r0 .. r1] rebased to 0, and the entries
    row_ptr[r0] .. row_ptr[r1] - 1 of col_idx and vals (numpy arrays or torch tensors)."""
    r0, r1 = bounds[rank], bounds[rank + 1]
    s, e = int(row_ptr[r0]), int(row_ptr[r1])
    rp = row_ptr[r0:r1 + 1] - s
    return RowShard("csr", n, r0, r1, v=None if v is None else v[r0:r1], row_ptr=rp, col_idx=col_idx[s:e],
                    vals=vals[s:e])


def partial(shard: RowShard, y, stream=None):
    """w_g = X_g^T (v_g * (X_g y)): one fused call on the rank's rows, alpha = 1, beta = 0."""
    if shard.kind == "dense":
        return _lib.dense(shard.X, y, shard.v, 1.0, 0.0, None, stream=stream)
    return _lib.csr(shard.row_ptr, shard.col_idx, shard.vals, y, shard.n, shard.v, 1.0, 0.0, None, stream=stream)


def reduce_and_finish(w, alpha: float, beta: float, z=None, group=None,
                      epilogue: Optional[Callable] = None):
    """Sums the ranks' partials in place (one all-reduce of n values) and returns
    alpha * w + beta * z, written over w."""
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(w, op=dist.ReduceOp.SUM, group=group)
    if epilogue is None:
        return _lib.epilogue(w, alpha, beta, z, out=w)
    return epilogue(w, alpha, beta, z)


def sharded_call(shard: RowShard, y, alpha: float, beta: float, z=None, group=None,
                 partial_fn: Optional[Callable] = None, epilogue: Optional[Callable] = None):
    """out = alpha * X^T (v * (X y)) + beta * z for the whole X, on every rank.

    `partial_fn(shard, y)` and `epilogue(w, alpha, beta, z)` default to the library's
    GPU calls (``partial`` and ``fxtx_epilogue_*``)."""
    w = (partial_fn or partial)(shard, y)
    return reduce_and_finish(w, alpha, beta, z, group, epilogue)
