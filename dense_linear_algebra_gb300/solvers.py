"""Whole ML algorithms whose inner loop is the fused pattern.

"On optimizing machine learning workloads via kernel fusion" (abstract) closes by
applying the fused kernel inside an entire ML algorithm. The two here are the
textbook consumers of ``alpha * X^T (v * (X p)) + beta * z``:

* ``ridge_cg``: least squares with an L2 penalty, ``min ||X w - b||^2 + lam ||w||^2``,
  solved by conjugate gradients on ``(X^T X + lam I) w = X^T b``. Every operator
  application ``X^T (X p) + lam p`` is ONE fused call (v = 1, z = p, beta = lam).
* ``ridge_cg_multi``: the same for k targets at once (block CG); every iteration applies
  the operator to all k search directions in ONE multi-vector call, one pass over X.
* ``logistic_newton_cg``: L2-regularised logistic regression by Newton's method;
  each Newton step solves ``(X^T D X + lam I) d = -g`` by conjugate gradients, where
  every Hessian-vector product ``X^T (D * (X p)) + lam p`` is ONE fused call with
  v = D = mu (1 - mu).

X may be dense (a 2-D CUDA tensor) or CSR (a tuple ``(row_ptr, col_idx, vals, n)``).
The few operations outside the pattern (``X^T b`` once, and per Newton step the
margins ``X w`` and the gradient ``X^T (mu - b)``) are plain matrix-vector products
done by torch (for CSR X on torch CSR copies built once per solve); vector updates on
n-vectors are torch operations as well.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from . import _lib


def _is_csr(X) -> bool:
    return isinstance(X, tuple)


def _shape(X):
    if _is_csr(X):
        row_ptr, _, vals, n = X
        return row_ptr.shape[0] - 1, n, vals.dtype, vals.device
    return X.shape[0], X.shape[1], X.dtype, X.device


def fused(X, p, v, alpha: float, beta: float, z, out=None):
    """alpha * X^T (v * (X p)) + beta * z, dense or CSR."""
    if _is_csr(X):
        row_ptr, col_idx, vals, n = X
        return _lib.csr(row_ptr, col_idx, vals, p, n, v, alpha, beta, z, out=out)
    return _lib.dense(X, p, v, alpha, beta, z, out=out)


def _torch_csr(X):
    row_ptr, col_idx, vals, n = X
    return torch.sparse_csr_tensor(row_ptr, col_idx.to(torch.int64), vals, size=(row_ptr.shape[0] - 1, n))


class TorchOps:
    """X w and X^T r outside the pattern (torch). For CSR X the torch CSR tensor and its
    transposed copy are built once, when the operator is made, not per product."""

    def __init__(self, X):
        if _is_csr(X):
            self.A = _torch_csr(X)
            self.AT = self.A.t().to_sparse_csr()
        else:
            self.A, self.AT = X, X.t()

    def matvec(self, w):
        return torch.mv(self.A, w)

    def rmatvec(self, r):
        return torch.mv(self.AT, r)


def matvec(X, w):
    """X w (outside the pattern; torch)."""
    return TorchOps(X).matvec(w) if _is_csr(X) else torch.mv(X, w)


def rmatvec(X, r):
    """X^T r (outside the pattern; torch)."""
    return TorchOps(X).rmatvec(r) if _is_csr(X) else torch.mv(X.t(), r)


@dataclass
class CGInfo:
    iterations: int = 0
    residual: float = 0.0
    converged: bool = False
    history: list = field(default_factory=list)


def cg(apply, rhs, tol: float = 1e-6, max_iter: int = 100, x0=None, check_every: int = 1):
    """Conjugate gradients for the symmetric positive definite operator `apply` (one fused call each).

    The residual is read back to the host (a synchronisation) every `check_every`
    iterations and at the last one; between checks the iterations queue on the
    stream back to back.
    """
    x = torch.zeros_like(rhs) if x0 is None else x0.clone()
    r = rhs - apply(x) if x0 is not None else rhs.clone()
    p = r.clone()
    rs = torch.dot(r, r)
    bnorm = float(torch.linalg.vector_norm(rhs))
    info = CGInfo()
    if bnorm == 0.0:
        info.converged = True
        return x, info
    for k in range(max_iter):
        q = apply(p)
        pq = torch.dot(p, q)
        # once the residual is exactly zero, stop moving (no 0/0 on the device)
        a = torch.where(pq > 0, rs / torch.where(pq > 0, pq, torch.ones_like(pq)), torch.zeros_like(pq))
        x.add_(a * p)
        r.sub_(a * q)
        rs_new = torch.dot(r, r)
        info.iterations = k + 1
        if (k + 1) % check_every == 0 or k + 1 == max_iter:
            res = float(torch.sqrt(rs_new)) / bnorm
            info.residual = res
            info.history.append(res)
            if res <= tol:
                info.converged = True
                break
        p.mul_(torch.where(rs > 0, rs_new / torch.where(rs > 0, rs, torch.ones_like(rs)), torch.zeros_like(rs))).add_(r)
        rs = rs_new
    return x, info


def ridge_cg(X, b, lam: float, tol: float = 1e-6, max_iter: int = 200):
    """Ridge regression by CG: each iteration applies X^T (X p) + lam p in one fused call."""
    m, n, dt, dev = _shape(X)
    rhs = rmatvec(X, b)
    return cg(lambda p: fused(X, p, None, 1.0, lam, p), rhs, tol=tol, max_iter=max_iter)


def fused_multi(X, P, V, alpha: float, beta: float, Z, out=None):
    """alpha * X^T (V * (X P)) + beta * Z for k right-hand sides (dense X): one pass over X."""
    return _lib.dense_multi(X, P, V, alpha, beta, Z, out=out)


def cg_block(apply, rhs, tol: float = 1e-6, max_iter: int = 100, check_every: int = 1):
    """k independent conjugate-gradient solves in lockstep, one per column of `rhs` (n, k).

    `apply` maps an (n, k) block to the operator applied to each column, so one call
    serves all k solves. Each column has its own step sizes; a column whose residual
    reaches zero stops moving. Converged when every column's relative residual is <= tol.
    """
    x = torch.zeros_like(rhs)
    r = rhs.clone()
    p = r.clone()
    rs = (r * r).sum(dim=0)
    bnorm = torch.linalg.vector_norm(rhs, dim=0)
    info = CGInfo()
    safe_b = torch.where(bnorm > 0, bnorm, torch.ones_like(bnorm))
    if float(bnorm.max()) == 0.0:
        info.converged = True
        return x, info
    for k in range(max_iter):
        q = apply(p)
        pq = (p * q).sum(dim=0)
        a = torch.where(pq > 0, rs / torch.where(pq > 0, pq, torch.ones_like(pq)), torch.zeros_like(pq))
        x.add_(a * p)
        r.sub_(a * q)
        rs_new = (r * r).sum(dim=0)
        info.iterations = k + 1
        if (k + 1) % check_every == 0 or k + 1 == max_iter:
            res = float((torch.sqrt(rs_new) / safe_b).max())
            info.residual = res
            info.history.append(res)
            if res <= tol:
                info.converged = True
                break
        b = torch.where(rs > 0, rs_new / torch.where(rs > 0, rs, torch.ones_like(rs)), torch.zeros_like(rs))
        p.mul_(b).add_(r)
        rs = rs_new
    return x, info


def ridge_cg_multi(X, B, lam: float, tol: float = 1e-6, max_iter: int = 200):
    """Ridge regression for k targets at once (B is (m, k)): block CG in which every
    iteration applies X^T (X P) + lam P to all k directions in one multi-vector call."""
    rhs = torch.mm(X.t(), B).contiguous()
    return cg_block(lambda P: fused_multi(X, P.contiguous(), None, 1.0, lam, P.contiguous()), rhs, tol=tol,
                    max_iter=max_iter)


@dataclass
class NewtonInfo:
    newton_steps: int = 0
    cg_iterations: int = 0
    grad_norm: float = 0.0
    converged: bool = False


def logistic_newton_cg(X, labels, lam: float, newton_steps: int = 20, tol: float = 1e-6, cg_tol: float = 1e-4,
                       cg_max: int = 100):
    """L2 logistic regression (labels in {0, 1}) by Newton-CG.

    Minimises sum_i log(1 + exp(x_i . w)) - b_i (x_i . w) + lam / 2 ||w||^2. Each Hessian-vector
    product X^T (D * (X p)) + lam p, D = mu (1 - mu), is one fused call with v = D.
    """
    m, n, dt, dev = _shape(X)
    ops = TorchOps(X)  # the margins' and the gradient's products; CSR copies built once per solve
    w = torch.zeros(n, dtype=dt, device=dev)
    info = NewtonInfo()
    g0 = None
    for step in range(newton_steps):
        mu = torch.sigmoid(ops.matvec(w))
        g = ops.rmatvec(mu - labels) + lam * w
        gn = float(torch.linalg.vector_norm(g))
        if g0 is None:
            g0 = max(gn, 1e-300)
        info.grad_norm = gn
        if gn <= tol * g0:
            info.converged = True
            break
        D = (mu * (1.0 - mu)).contiguous()
        d, ci = cg(lambda p: fused(X, p, D, 1.0, lam, p), -g, tol=cg_tol, max_iter=cg_max)
        w.add_(d)
        info.newton_steps = step + 1
        info.cg_iterations += ci.iterations
    return w, info
