"""Whole ML algorithms on the fused pattern: ridge regression by CG and logistic
regression by Newton-CG, checked against float64 numpy solutions of the same
problems (direct solves on the CPU)."""
import numpy as np
import pytest
import torch

import inputgen
from dense_linear_algebra_gb300 import solvers
from _util import dense_to_csr


def test_cg_on_cpu_operator():
    """The CG driver alone (no GPU): an SPD matrix applied by torch."""
    rng = np.random.default_rng(0)
    A = rng.standard_normal((30, 30))
    A = torch.from_numpy(A @ A.T + 30 * np.eye(30))
    b = torch.from_numpy(rng.standard_normal(30))
    x, info = solvers.cg(lambda p: A @ p, b, tol=1e-12, max_iter=200)
    assert info.converged
    assert np.allclose(x.numpy(), np.linalg.solve(A.numpy(), b.numpy()), rtol=1e-9, atol=1e-10)


def test_cg_block_on_cpu_operator():
    """The block CG driver alone (no GPU): k columns, an SPD matrix applied by torch."""
    rng = np.random.default_rng(1)
    A = rng.standard_normal((25, 25))
    A = torch.from_numpy(A @ A.T + 25 * np.eye(25))
    B = torch.from_numpy(rng.standard_normal((25, 4)))
    B[:, 2] = 0.0  # a zero right-hand side stays at zero
    x, info = solvers.cg_block(lambda P: A @ P, B, tol=1e-12, max_iter=200)
    assert info.converged
    assert np.allclose(x.numpy(), np.linalg.solve(A.numpy(), B.numpy()), rtol=1e-9, atol=1e-10)
    assert np.all(x.numpy()[:, 2] == 0.0)


def _ridge_ref(X, b, lam):
    return np.linalg.solve(X.T @ X + lam * np.eye(X.shape[1]), X.T @ b)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,m,n,rtol", [(np.float64, 3000, 24, 1e-9), (np.float32, 200_000, 32, 2e-3)])
def test_ridge_cg_dense(dtype, m, n, rtol):
    X = inputgen.normal(3, 1, (m, n), np.float64)
    w_true = inputgen.normal(3, 2, n, np.float64)
    b = X @ w_true + 0.1 * inputgen.normal(3, 3, m, np.float64)
    lam = 0.5
    ref = _ridge_ref(X, b, lam)
    Xd = torch.from_numpy(X.astype(dtype)).cuda()
    bd = torch.from_numpy(b.astype(dtype)).cuda()
    w, info = solvers.ridge_cg(Xd, bd, lam, tol=1e-10 if dtype == np.float64 else 1e-5, max_iter=200)
    assert info.iterations <= 3 * n
    assert np.linalg.norm(w.cpu().numpy() - ref) <= rtol * np.linalg.norm(ref)


@pytest.mark.gpu
@pytest.mark.parametrize("dtype,rtol", [(np.float64, 1e-9), (np.float32, 2e-3)])
def test_ridge_cg_multi(dtype, rtol):
    """k = 6 targets solved together with the multi-vector operator match six direct solves."""
    m, n, k = 20_000, 32, 6
    X = inputgen.normal(4, 1, (m, n), np.float64)
    W = inputgen.normal(4, 2, (n, k), np.float64)
    B = X @ W + 0.1 * inputgen.normal(4, 3, (m, k), np.float64)
    lam = 0.5
    ref = np.linalg.solve(X.T @ X + lam * np.eye(n), X.T @ B)
    Xd = torch.from_numpy(X.astype(dtype)).cuda()
    Bd = torch.from_numpy(B.astype(dtype)).cuda()
    w, info = solvers.ridge_cg_multi(Xd, Bd, lam, tol=1e-10 if dtype == np.float64 else 1e-5, max_iter=200)
    assert info.iterations <= 3 * n
    assert np.linalg.norm(w.cpu().numpy() - ref) <= rtol * np.linalg.norm(ref)


@pytest.mark.gpu
def test_ridge_cg_csr():
    rng = np.random.default_rng(7)
    m, n = 6000, 150
    X = rng.standard_normal((m, n))
    X[rng.random((m, n)) < 0.85] = 0.0
    b = rng.standard_normal(m)
    lam = 1.0
    ref = _ridge_ref(X, b, lam)
    rp, ci, vals = dense_to_csr(X)
    Xc = (torch.from_numpy(rp).cuda(), torch.from_numpy(ci).cuda(), torch.from_numpy(vals).cuda(), n)
    w, info = solvers.ridge_cg(Xc, torch.from_numpy(b).cuda(), lam, tol=1e-11, max_iter=500)
    assert info.converged
    assert np.linalg.norm(w.cpu().numpy() - ref) <= 1e-8 * np.linalg.norm(ref)


def _logistic_ref(X, y, lam, steps=50):
    w = np.zeros(X.shape[1])
    for _ in range(steps):
        mu = 1.0 / (1.0 + np.exp(-(X @ w)))
        g = X.T @ (mu - y) + lam * w
        H = X.T @ ((mu * (1 - mu))[:, None] * X) + lam * np.eye(X.shape[1])
        w = w - np.linalg.solve(H, g)
        if np.linalg.norm(g) < 1e-13:
            break
    return w


@pytest.mark.gpu
@pytest.mark.parametrize("sparse", [False, True])
def test_logistic_newton_cg(sparse):
    rng = np.random.default_rng(11)
    m, n = 5000, 12
    X = rng.standard_normal((m, n))
    if sparse:
        X[rng.random((m, n)) < 0.5] = 0.0
    w_true = rng.standard_normal(n)
    y = (rng.random(m) < 1.0 / (1.0 + np.exp(-(X @ w_true)))).astype(np.float64)
    lam = 2.0
    ref = _logistic_ref(X, y, lam)
    if sparse:
        rp, ci, vals = dense_to_csr(X)
        Xd = (torch.from_numpy(rp).cuda(), torch.from_numpy(ci).cuda(), torch.from_numpy(vals).cuda(), n)
    else:
        Xd = torch.from_numpy(X).cuda()
    w, info = solvers.logistic_newton_cg(Xd, torch.from_numpy(y).cuda(), lam, newton_steps=30, tol=1e-10,
                                         cg_tol=1e-12, cg_max=200)
    assert info.converged
    assert np.linalg.norm(w.cpu().numpy() - ref) <= 1e-7 * np.linalg.norm(ref)
