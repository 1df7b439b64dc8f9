"""Parity of the CSR CUDA path against the oracle, element by element, and the
device-side structure check."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import dense_linear_algebra_gb300 as fx
import inputgen
import oracle
from _gpu import run_problem, to_dev
from _util import assert_within_bound, dense_to_csr, rel_for

pytestmark = pytest.mark.gpu


def make_csr(dtype, lens, n, seed=1, zipf=0.0, with_v=True, with_z=True, alpha=1.25, beta=-0.75, ints=False):
    dt = np.dtype(dtype).type
    lens = np.asarray(lens, dtype=np.int64)
    m = lens.shape[0]
    rp = inputgen.row_ptr_from_lengths(lens)
    col = inputgen.csr_columns(seed, n, rp, zipf)
    nnz = int(rp[-1])
    if ints:
        vals = inputgen.integers(seed, 1, nnz, -2, 2, dt)
        y = inputgen.integers(seed, 2, n, -2, 2, dt)
        v = inputgen.integers(seed, 3, m, -2, 2, dt) if with_v else None
        z = inputgen.integers(seed, 4, n, -2, 2, dt) if with_z else None
    else:
        vals = inputgen.uniform(seed, 1, nnz, -1.0, 1.0, dt)
        y = inputgen.uniform(seed, 2, n, -1.0, 1.0, dt)
        v = inputgen.uniform(seed, 3, m, -1.0, 1.0, dt) if with_v else None
        z = inputgen.uniform(seed, 4, n, -1.0, 1.0, dt) if with_z else None
    return inputgen.Problem(f"csr_{m}x{n}", "csr", dt, m, n, alpha, beta, y=y, v=v, z=z, row_ptr=rp, col_idx=col,
                            vals=vals)


def check(p, acc="ld"):
    got = run_problem(p)
    ref, S = oracle.solve(p, acc=acc)
    assert_within_bound(got, ref, S, rel_for(p.dtype), p.name)
    return got, ref


def test_csr_uniform_recipe_scaled():
    """Poisson(50) distinct uniform columns, f64, n = 10,000, at 40,000 rows."""
    check(inputgen.csr_uniform(m=40_000))


def test_csr_powerlaw_recipe_scaled():
    """Zipf row lengths (mean 100, long rows up to 5,000), Zipf(1.1) columns over 100,000, f32."""
    check(inputgen.csr_powerlaw(m=20_000, n=100_000, cap=5_000))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("L", [0, 1, 2, 3, 5, 8, 16, 17, 33, 63, 64, 65, 128, 255, 256, 257, 1000, 2048, 2049, 4097,
                               8193])
def test_uniform_row_lengths(dtype, L):
    """Every row of the same length: short / medium / long bins and their boundaries."""
    n = max(8000, L)
    m = 3000 if L <= 256 else 200
    check(make_csr(dtype, np.full(m, L), n, seed=L))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_very_long_rows_every_bucket(dtype):
    """Rows in every long-row length bucket, up to beyond 64K entries (the last bucket),
    among short rows, so that the longest-first claim order spans all six buckets."""
    lens = np.full(4000, 7)
    lens[[5, 700, 1500, 2200, 3000, 3100, 3999]] = [2100, 5000, 9000, 17000, 33000, 70000, 100000]
    check(make_csr(dtype, lens, 120_000, seed=9))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_mixed_lengths_and_empty_rows(dtype):
    rng = np.random.default_rng(3)
    lens = rng.choice([0, 0, 1, 3, 20, 90, 300, 2000], size=5000)
    check(make_csr(dtype, lens, 5000, seed=4))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_columns_outside_shared_window(dtype):
    """n far larger than the shared-memory column window: most scatters go to global atomics."""
    rng = np.random.default_rng(6)
    lens = rng.integers(0, 400, 4000)
    check(make_csr(dtype, lens, 300_000, seed=6))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_hot_column(dtype):
    """Every row hits column 0 and a few neighbours (Zipf 2.0 columns): contention on one address."""
    lens = np.full(20_000, 12)
    check(make_csr(dtype, lens, 50_000, seed=8, zipf=2.0))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_full_row_and_single_row(dtype):
    n = 3000
    check(make_csr(dtype, [n], n, seed=2))
    check(make_csr(dtype, [n, 0, n, 1], n, seed=3))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_duplicates_and_unsorted(dtype):
    """Repeated (i, j) entries add; column order inside a row is free."""
    rng = np.random.default_rng(10)
    m, n = 2000, 500
    lens = rng.integers(0, 60, m)
    rp = inputgen.row_ptr_from_lengths(lens)
    nnz = int(rp[-1])
    col = rng.integers(0, n, nnz).astype(np.int32)  # repeats allowed, unsorted
    dt = np.dtype(dtype).type
    p = inputgen.Problem("dups", "csr", dt, m, n, 0.5, 2.0, y=rng.uniform(-1, 1, n).astype(dt),
                         v=rng.uniform(-1, 1, m).astype(dt), z=rng.uniform(-1, 1, n).astype(dt), row_ptr=rp,
                         col_idx=col, vals=rng.uniform(-1, 1, nnz).astype(dt))
    check(p)


@pytest.mark.parametrize("L", [40, 200, 700, 3000])
def test_row_dots_that_cancel(L):
    """Rows whose entries cancel to a small dot: the first half +a_k (integers in [64, 128)), the
    second half -a_k + e_k with e_k a few units of 2^-17 (all exact in fp32), y = 1. Partial sums
    reach thousands while the dot is ~1e-3, so a row's segments (across lanes, packed batches
    or warps) must be summed without losing the small remainder: the bound is relative to |t_i|."""
    m, n = 3000, 4 * L
    lens = np.full(m, L, dtype=np.int64)
    rp = inputgen.row_ptr_from_lengths(lens)
    col = inputgen.csr_columns(5, n, rp, 0.0)
    half = L // 2
    a = (64.0 + (np.arange(m * half) % 61)).reshape(m, half)
    e = ((np.arange(m * half) % 7) + 1).reshape(m, half) * 2.0 ** -17
    vals = np.concatenate([a, -a + e], axis=1).astype(np.float32)
    assert np.array_equal(vals[:, half:2 * half].astype(np.float64), -a + e)
    if L % 2:
        vals = np.concatenate([vals, np.zeros((m, 1), np.float32)], axis=1)
    p = inputgen.Problem(f"csr_cancel_{L}", "csr", np.float32, m, n, 1.0, 0.0, y=np.ones(n, np.float32),
                         v=None, z=None, row_ptr=rp, col_idx=col, vals=vals.ravel())
    check(p)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_integer_inputs_are_exact(dtype):
    rng = np.random.default_rng(12)
    lens = rng.choice([1, 4, 40, 200, 700], size=6000)
    p = make_csr(dtype, lens, 20_000, seed=12, ints=True, alpha=2.0, beta=-1.0)
    got = run_problem(p)
    ref, _ = oracle.solve(p)
    assert np.abs(ref).max() < 2 ** 24
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_dense_and_csr_agree(dtype):
    """The same matrix through both paths."""
    rng = np.random.default_rng(13)
    m, n = 3000, 32
    X = rng.uniform(-1, 1, (m, n)).astype(dtype)
    X[rng.random((m, n)) < 0.6] = 0
    y = rng.uniform(-1, 1, n).astype(dtype)
    v = rng.uniform(-1, 1, m).astype(dtype)
    z = rng.uniform(-1, 1, n).astype(dtype)
    rp, ci, vals = dense_to_csr(X)
    ref, S = oracle.dense(X, y, v, 1.5, -0.5, z)
    d = fx.dense(to_dev(X), to_dev(y), to_dev(v), 1.5, -0.5, to_dev(z)).cpu().numpy()
    c = fx.csr(to_dev(rp), to_dev(ci), to_dev(vals), to_dev(y), n, to_dev(v), 1.5, -0.5, to_dev(z)).cpu().numpy()
    assert_within_bound(d, ref, S, rel_for(dtype))
    assert_within_bound(c, ref, S, rel_for(dtype))


@pytest.mark.parametrize("dtype", [torch.float32, torch.float64])
def test_empty_structures(dtype):
    dev = "cuda"
    n = 7
    z = torch.arange(n, dtype=dtype, device=dev)
    y = torch.ones(n, dtype=dtype, device=dev)
    e32 = torch.empty(0, dtype=torch.int32, device=dev)
    ev = torch.empty(0, dtype=dtype, device=dev)
    # m = 0
    out = fx.csr(torch.zeros(1, dtype=torch.int64, device=dev), e32, ev, y, n, None, 2.0, 3.0, z)
    assert torch.equal(out, 3.0 * z)
    # nnz = 0 with rows
    out = fx.csr(torch.zeros(6, dtype=torch.int64, device=dev), e32, ev, y, n, torch.ones(5, dtype=dtype, device=dev),
                 2.0, 0.0, z)
    assert torch.equal(out, torch.zeros_like(z))


def test_validate():
    dev = "cuda"
    rp = torch.tensor([0, 2, 3, 3], dtype=torch.int64, device=dev)
    ci = torch.tensor([0, 4, 2], dtype=torch.int32, device=dev)
    assert fx.csr_validate(rp, ci, 5)
    assert not fx.csr_validate(rp, ci, 4)  # column 4 out of range
    assert not fx.csr_validate(torch.tensor([0, 2, 1, 3], dtype=torch.int64, device=dev), ci, 5)  # decreasing
    assert not fx.csr_validate(torch.tensor([1, 2, 3, 3], dtype=torch.int64, device=dev), ci, 5)  # row_ptr[0] != 0
    assert not fx.csr_validate(torch.tensor([0, 2, 3, 4], dtype=torch.int64, device=dev), ci, 5)  # row_ptr[m] != nnz
    bad = torch.tensor([0, -1, 2], dtype=torch.int32, device=dev)
    assert not fx.csr_validate(rp, bad, 5)
    p = inputgen.csr_powerlaw(m=5000, n=20_000, cap=2000)
    assert fx.csr_validate(to_dev(p.row_ptr), to_dev(p.col_idx), p.n)


@pytest.mark.slow
def test_full_size_csr_uniform():
    """CSR f64 4,000,000 x 10,000 (~2e8 nnz) as configured, every column against the oracle."""
    check(inputgen.csr_uniform())


@pytest.mark.slow
def test_full_size_csr_powerlaw():
    """CSR f32 2,000,000 x 1,000,000 power-law (2e8 nnz), every column against the oracle.

    The oracle's double accumulator is used; its own error (well under 1e-9 * S_j) is
    far inside the fp32 bound.
    """
    check(inputgen.csr_powerlaw(), acc="d")
