"""The fp64 scatter's double-word arithmetic across magnitudes (GPU against the oracle).

The fp64 kernels keep the row dot in fp64 and form the scatter's products t_i * X_ij as
pairs of fp32 values built from the fp64 bits. That representation holds values of
magnitude 2^-50 .. 2^51 exactly enough; products of anything else (and NaN, infinity) take
fp64 atomics instead. These cases cover entries spread over 2^40, entries far outside the
double-word range in whole rows and in single entries, and non-finite values, for the
wide dense kernel and the CSR kernels.
"""
from __future__ import annotations

import numpy as np
import pytest

import inputgen
import oracle
from _gpu import run_problem
from _util import assert_within_bound, dense_to_csr

pytestmark = pytest.mark.gpu

REL = 1e-12


def _spread(rng, shape, lo, hi):
    """sign * 2^U[lo, hi] * U[1, 2): magnitudes spread over hi - lo binades."""
    return rng.choice([-1.0, 1.0], shape) * np.exp2(rng.uniform(lo, hi, shape)) * rng.uniform(1.0, 2.0, shape)


def _dense(X, y, v, z, alpha=0.7, beta=0.3):
    m, n = X.shape
    return inputgen.Problem(f"dense_{m}x{n}", "dense", np.float64, m, n, alpha, beta, y=y, v=v, z=z, X=X, ld=n)


def _csr_of(p):
    rp, ci, vals = dense_to_csr(p.X[:, : p.n])
    return inputgen.Problem(p.name + "_csr", "csr", np.float64, p.m, p.n, p.alpha, p.beta, y=p.y, v=p.v, z=p.z,
                            row_ptr=rp, col_idx=ci, vals=vals)


def _sparse(rng, X, keep):
    return np.where(rng.random(X.shape) < keep, X, 0.0)


def _check(p):
    got = run_problem(p)
    ref, S = oracle.solve(p)
    fin = np.isfinite(ref)
    assert np.array_equal(np.isnan(got), np.isnan(ref)), p.name
    assert np.array_equal(got[np.isinf(ref)], ref[np.isinf(ref)]), p.name
    assert_within_bound(got[fin], ref[fin], S[fin], REL, p.name)


@pytest.mark.parametrize("kind", ["wide", "csr"])
def test_entries_spread_over_2_40(kind):
    rng = np.random.default_rng(21)
    m, n = 300, 3000
    X = _spread(rng, (m, n), -20, 20)
    p = _dense(X, rng.uniform(-1, 1, n), rng.uniform(-1, 1, m), rng.uniform(-1, 1, n))
    if kind == "csr":
        p.X = _sparse(rng, p.X, 0.05)
        p = _csr_of(p)
    _check(p)


@pytest.mark.parametrize("kind", ["wide", "csr"])
def test_scales_outside_the_double_word_range(kind):
    """Whole rows of 1e-30 or 1e30 (their t_i leave the double-word range), rows of 1e-8
    whose t_i does, and single entries of 2^-60 / 2^60 in ordinary rows."""
    rng = np.random.default_rng(22)
    m, n = 256, 2600
    X = rng.uniform(-1, 1, (m, n))
    X[3] *= 1e-30
    X[10] *= 1e30
    X[17] *= 1e-8  # t ~ 1e-16 * n: below 2^-50
    X[rng.integers(0, m, 40), rng.integers(0, n, 40)] = 2.0 ** -60
    X[rng.integers(0, m, 40), rng.integers(0, n, 40)] = -(2.0 ** 60)
    p = _dense(X, rng.uniform(-1, 1, n), rng.uniform(-1, 1, m), rng.uniform(-1, 1, n))
    if kind == "csr":
        p.X = _sparse(rng, p.X, 0.1)
        p.X[10, ::7] = 1e30  # keep the huge row populated
        p = _csr_of(p)
    _check(p)


@pytest.mark.parametrize("bad", ["inf", "nan"])
@pytest.mark.parametrize("kind", ["wide", "csr"])
def test_non_finite_entries_propagate(kind, bad):
    """One infinite entry makes its row's t_i infinite: every column then holds +-inf, with
    the sign of that row's entry. One NaN entry makes every column NaN."""
    rng = np.random.default_rng(23)
    m, n = 200, 2100
    X = rng.uniform(-1, 1, (m, n))
    X[5, 7] = np.inf if bad == "inf" else np.nan
    p = _dense(X, rng.uniform(0.5, 1, n), rng.uniform(0.5, 1, m), rng.uniform(-1, 1, n))
    if kind == "csr":
        p = _csr_of(p)
    _check(p)


def test_integer_sums_beyond_2_24_stay_exact():
    """Integer products whose column sums pass 2^24 (where a single fp32 stops being exact):
    the double-word sums keep them exact, so the result matches the oracle bitwise."""
    rng = np.random.default_rng(24)
    m, n = 4000, 2500
    X = rng.integers(-300, 301, (m, n)).astype(np.float64)
    y = rng.integers(-3, 4, n).astype(np.float64)
    v = rng.integers(1, 4, m).astype(np.float64)
    p = _dense(X, y, v, None, alpha=1.0, beta=0.0)
    got = run_problem(p)
    ref, _ = oracle.solve(p)
    assert np.abs(ref).max() > 2 ** 24
    assert np.array_equal(got, ref)
