"""Parity of the dense CUDA path against the oracle, element by element.

Bound: |gpu_j - ref_j| <= c * S_j with S_j = |alpha| sum_i |t_i| |X_ij| + |beta z_j|,
c = 1e-12 (fp64) or 2e-5 (fp32); integer-valued inputs must match bitwise.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import dense_linear_algebra_gb300 as fx
import inputgen
import oracle
from _gpu import DeviceProblem, run_problem, to_dev
from _util import assert_within_bound, rel_for

pytestmark = pytest.mark.gpu


def make_dense(dtype, m, n, ld=None, seed=1, with_v=True, with_z=True, alpha=1.25, beta=-0.75, ints=False):
    ld = n if ld is None else ld
    dt = np.dtype(dtype).type
    if ints:
        X = inputgen.integers(seed, 1, (m, ld), -2, 2, dt)
        y = inputgen.integers(seed, 2, n, -2, 2, dt)
        v = inputgen.integers(seed, 3, m, -2, 2, dt) if with_v else None
        z = inputgen.integers(seed, 4, n, -2, 2, dt) if with_z else None
    else:
        X = inputgen.uniform(seed, 1, (m, ld), -1.0, 1.0, dt)
        y = inputgen.uniform(seed, 2, n, -1.0, 1.0, dt)
        v = inputgen.uniform(seed, 3, m, -1.0, 1.0, dt) if with_v else None
        z = inputgen.uniform(seed, 4, n, -1.0, 1.0, dt) if with_z else None
    return inputgen.Problem(f"dense_{m}x{n}_ld{ld}", "dense", dt, m, n, alpha, beta, y=y, v=v, z=z, X=X, ld=ld)


def check(p, acc="ld"):
    got = run_problem(p)
    ref, S = oracle.solve(p, acc=acc)
    assert_within_bound(got, ref, S, rel_for(p.dtype), p.name)
    return got, ref


def test_dense_small_workload():
    """dense f64 1000 x 64, U[-1,1], alpha=1.5, beta=0.5, seed 0."""
    check(inputgen.dense_small())


@pytest.mark.parametrize("variant", ["a", "b", "c"])
def test_dense_tall_recipe_scaled(variant):
    """The tall-skinny f32 recipe (N(0,1) X, v U[0.1,2]) at 300,000 rows."""
    check(inputgen.dense_tall(m=300_000, variant=variant))


def test_dense_wide_recipe_scaled():
    """The wide f64 recipe at 400 x 3000 (wide kernel: rows longer than 256 fp64)."""
    check(inputgen.dense_wide(m=400, n=3000))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("n", [1, 2, 3, 4, 7, 8, 12, 16, 31, 32, 33, 48, 64, 100, 128, 255, 256, 257, 384, 512, 513, 1031])
def test_shapes(dtype, n):
    for m in (1, 37, 2049):
        check(make_dense(dtype, m, n, seed=n + m))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("n,ld", [(32, 36), (32, 40), (64, 72), (30, 32), (5, 9), (600, 608), (16, 4096)])
def test_leading_dimension(dtype, n, ld):
    check(make_dense(dtype, 1500, n, ld=ld, seed=ld))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_unaligned_base(dtype):
    """X starting one element past a 16-byte boundary takes the direct-load path."""
    p = make_dense(dtype, 3000, 32, seed=9)
    ref, S = oracle.solve(p)
    Xbig = torch.zeros(p.m * p.n + 1, dtype=torch.float32 if dtype == np.float32 else torch.float64, device="cuda")
    Xbig[1:] = to_dev(p.X.ravel())
    X = Xbig[1:].view(p.m, p.n)
    assert X.data_ptr() % 16 != 0
    out = fx.dense(X, to_dev(p.y), to_dev(p.v), p.alpha, p.beta, to_dev(p.z))
    assert_within_bound(out.cpu().numpy(), ref, S, rel_for(dtype))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("with_v,with_z,beta", [(True, True, -0.75), (False, False, 0.0), (True, False, 0.0),
                                                (False, True, 2.0)])
def test_instantiations(dtype, with_v, with_z, beta):
    check(make_dense(dtype, 5000, 32, with_v=with_v, with_z=with_z, beta=beta, seed=3))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("m,n", [(50_000, 32), (20_000, 64), (3000, 200), (300, 2000)])
def test_integer_inputs_are_exact(dtype, m, n):
    """Integer X, y, v, z with |out| < 2^24: any summation order is exact, so bitwise equality."""
    p = make_dense(dtype, m, n, ints=True, alpha=2.0, beta=-1.0, seed=m)
    got = run_problem(p)
    ref, _ = oracle.solve(p)
    assert np.abs(ref).max() < 2 ** 24
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("dtype", [torch.float32, torch.float64])
def test_empty_and_degenerate(dtype):
    dev = "cuda"
    n = 10
    z = torch.arange(n, dtype=dtype, device=dev)
    y = torch.ones(n, dtype=dtype, device=dev)
    # m = 0: out = beta z
    out = fx.dense(torch.empty(0, n, dtype=dtype, device=dev), y, None, 3.0, -2.0, z)
    assert torch.equal(out, -2.0 * z)
    out = fx.dense(torch.empty(0, n, dtype=dtype, device=dev), y, None, 3.0, 1.0, None)
    assert torch.equal(out, torch.zeros_like(z))
    # n = 0: nothing happens
    out = fx.dense(torch.empty(4, 0, dtype=dtype, device=dev), torch.empty(0, dtype=dtype, device=dev))
    assert out.shape == (0,)
    # beta = 0: z is not read (NaN stays out)
    X = torch.rand(100, n, dtype=dtype, device=dev)
    zn = torch.full((n,), float("nan"), dtype=dtype, device=dev)
    a = fx.dense(X, y, None, 1.0, 0.0, zn)
    b = fx.dense(X, y, None, 1.0, 0.0, None)
    assert torch.equal(a, b) and torch.isfinite(a).all()
    # alpha = 0: out = beta z exactly
    out = fx.dense(X, y, None, 0.0, 2.0, z)
    assert torch.equal(out, 2.0 * z)
    # out aliasing z (in place)
    ref = fx.dense(X, y, None, 1.5, 0.5, z.clone())
    zz = z.clone()
    fx.dense(X, y, None, 1.5, 0.5, zz, out=zz)
    assert torch.equal(zz, ref)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_deterministic(dtype):
    """The dense reduction is fixed-order: repeated calls, on two streams, agree bitwise."""
    p = make_dense(dtype, 200_000, 32, seed=11)
    dp = DeviceProblem(p)
    a = dp.run().clone()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        b = dp.run(stream=s)
    s.synchronize()
    c = dp.run()
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(a, c)


@pytest.mark.parametrize("dtype,n,C", [(np.float64, 64, 100.0), (np.float64, 3000, 100.0),
                                        (np.float32, 256, 30.0), (np.float32, 2000, 30.0)])
def test_dot_cancellation(dtype, n, C):
    """Rows nearly orthogonal to y: sum_j |x_ij y_j| / |x_i . y| is about C (median).

    The bound scales with |t_i| = |v_i x_i . y|, not with sum_j |x_ij y_j|, so each dot
    must stay accurate relative to its cancelled value. fp64 in working precision
    meets it at this cancellation; fp32 needs the compensated dot for long rows.
    (Cancellation by ~1e9 would defeat any dot computed in working precision.)
    """
    m = 2000
    rng = np.random.default_rng(5)
    X0 = rng.uniform(-1, 1, (m, n))
    y = rng.uniform(-1, 1, n)
    X0 -= np.outer(X0 @ y / (y @ y), y)  # every row orthogonal to y ...
    r = rng.uniform(-1, 1, (m, n))
    a = np.median(np.abs(X0) @ np.abs(y)) / C / np.median(np.abs(r @ y))
    X = (X0 + a * r).astype(dtype)  # ... plus a residual that sets the dot
    y = y.astype(dtype)
    c = np.median(np.abs(X.astype(np.float64)) @ np.abs(y) / np.abs(X.astype(np.float64) @ y))
    assert 0.5 * C < c < 2 * C, c
    p = inputgen.Problem("cancel", "dense", dtype, m, n, 1.0, 0.0, y=y, v=None, z=None, X=X, ld=n)
    check(p)


@pytest.mark.slow
@pytest.mark.parametrize("variant", ["a", "b", "c"])
def test_full_size_tall(variant):
    """16,000,000 x 32 fp32 as benchmarked: every output column (n = 32) against the oracle.

    The oracle runs with its double accumulator here: its own error, at most about
    m * 2^-53 * S_j = 2e-9 * S_j, is far inside the fp32 bound.
    """
    check(inputgen.dense_tall(variant=variant), acc="d")


@pytest.mark.slow
def test_full_size_wide_sampled():
    """20,000 x 20,000 fp64: 48 sampled columns (including both ends) against the oracle."""
    p = inputgen.dense_wide()
    got = run_problem(p)
    cols = np.unique(np.concatenate([[0, 1, p.n - 1], np.random.default_rng(0).integers(0, p.n, 45)]))
    ref, S = oracle.solve(p, cols=cols)
    assert_within_bound(got[cols], ref, S, 1e-12, "dense_wide")


def test_allocation_failure_is_reported():
    """FXTX_FAIL_ALLOC=1 makes the workspace allocation fail on the host: the call returns
    FXTX_ERR_ALLOC without launching, and the next call (hook off) works."""
    import os

    X = torch.rand(1000, 32, device="cuda")
    y = torch.rand(32, device="cuda")
    os.environ["FXTX_FAIL_ALLOC"] = "1"
    try:
        with pytest.raises(fx.FxtxError) as ei:
            fx.dense(X, y)
        assert ei.value.status == fx.FXTX_ERR_ALLOC
    finally:
        del os.environ["FXTX_FAIL_ALLOC"]
    out = fx.dense(X, y)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all() and fx.device_error() == fx.FXTX_OK


def test_allocation_failure_is_reported_by_every_entry():
    """The same hook through the multi-vector and CSR entry points, and through a tuned call
    (a candidate whose workspace cannot be had is skipped; the call then reports the failure)."""
    import os

    X = torch.rand(2000, 32, device="cuda")
    Y = torch.rand(32, 4, device="cuda")
    rp = torch.arange(0, 2001 * 5, 5, dtype=torch.int64, device="cuda")
    ci = (torch.arange(2000 * 5, device="cuda") % 32).to(torch.int32)
    va = torch.rand(2000 * 5, device="cuda")
    y = torch.rand(32, device="cuda")
    mode = fx.autotune_mode()
    os.environ["FXTX_FAIL_ALLOC"] = "1"
    try:
        for tuned in (0, 1):
            fx.autotune(tuned)
            fx.autotune_clear()
            for call in (lambda: fx.dense_multi(X, Y), lambda: fx.csr(rp, ci, va, y, 32), lambda: fx.dense(X, y)):
                with pytest.raises(fx.FxtxError) as ei:
                    call()
                assert ei.value.status == fx.FXTX_ERR_ALLOC
            assert fx.autotune_entries() == 0
    finally:
        del os.environ["FXTX_FAIL_ALLOC"]
        fx.autotune_clear()
        fx.autotune(mode)
    out = fx.dense_multi(X, Y)
    o2 = fx.csr(rp, ci, va, y, 32)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all() and torch.isfinite(o2).all() and fx.device_error() == fx.FXTX_OK
