"""Pins for the CPU oracle: each check ties it to something other than itself.

The pattern is out = alpha * X^T (v * (X y)) + beta * z ("On optimizing machine
learning workloads via kernel fusion", abstract). The pins are:

* a worked example computed by hand from that definition (tests/golden);
* closed forms: X^T (X y) = (X^T X) y through a separately formed Gram matrix, and
  y . out = alpha * sum_i v_i (x_i . y)^2 + beta * y . z;
* linearity in alpha, beta and v, invariance under a joint row permutation of X and
  v, equivariance under a column permutation of X, y and z;
* exact rational brute force (Python Fractions) on tiny integer inputs, including
  every sparsity pattern of a 3x3 and a 2x4 matrix;
* dense and CSR forms of one matrix agreeing bitwise, and duplicate CSR entries
  summing;
* the textbook composition X.T @ (X @ y) from numpy;
* the instantiations' special cases (m = 0, n = 0, v absent, z absent, beta = 0
  with z unread);
* for the multi-vector instantiation (k right-hand sides), exact rational arithmetic
  over the matrix form and the numpy matrix composition, with its own planted mistakes.

``test_planted_mistakes`` compiles altered copies of the oracle (a dropped term, a
wrong sign, a transposed index, an off-by-one row range, ...) and checks that every
one of them fails at least one pin.
"""
from __future__ import annotations

import json
import os
from fractions import Fraction

import numpy as np
import pytest

import inputgen
import oracle
from _util import dense_to_csr

HERE = os.path.dirname(os.path.abspath(__file__))
GOLDEN = os.path.join(HERE, "golden", "worked_example_3x2.json")


def _close(a, b, scale, rel=1e-13):
    return np.all(np.abs(np.asarray(a) - np.asarray(b)) <= rel * np.asarray(scale))


def _absscale(X, y, v, alpha, beta, z):
    """|alpha| |X|^T (|v| |X| |y|) + |beta z|: bounds every rounding error of any order."""
    aX = np.abs(X)
    vv = np.ones(X.shape[0]) if v is None else np.abs(v)
    s = abs(alpha) * aX.T @ (vv * (aX @ np.abs(y)))
    if z is not None and beta != 0:
        s = s + np.abs(beta * z)
    return s


def _exact(Xq, yq, vq, alpha, beta, zq):
    """Exact rational value of the pattern, written as a double sum over (i, k)."""
    m = len(Xq)
    n = len(yq)
    out = []
    for j in range(n):
        acc = Fraction(0)
        for i in range(m):
            vi = Fraction(1) if vq is None else vq[i]
            for k in range(n):
                acc += Xq[i][j] * vi * Xq[i][k] * yq[k]
        o = Fraction(alpha) * acc
        if zq is not None and beta != 0:
            o += Fraction(beta) * zq[j]
        out.append(o)
    return out


def _frac(a):
    return [Fraction(float(x)) for x in np.ravel(a)]


# ----------------------------------------------------------------------------- pins
def pin_worked_example(lib):
    g = json.load(open(GOLDEN))
    for dt in (np.float32, np.float64):
        X = np.array(g["X"], dtype=dt)
        y = np.array(g["y"], dtype=dt)
        v = np.array(g["v"], dtype=dt)
        z = np.array(g["z"], dtype=dt)
        for acc in ("ld", "d"):
            out, S = oracle.dense(X, y, v, g["alpha"], g["beta"], z, acc=acc, lib=lib)
            assert np.array_equal(out, g["out"]), (dt, acc, out)
            out, _ = oracle.dense(X, y, None, 1.0, 0.0, None, acc=acc, lib=lib)
            assert np.array_equal(out, g["instantiation_XtXy"]["out"]), (dt, acc, out)
            out, _ = oracle.dense(X, y, v, 1.0, 0.0, z, acc=acc, lib=lib)
            assert np.array_equal(out, g["instantiation_Xt_v_Xy"]["out"]), (dt, acc, out)
            rp, ci, vals = dense_to_csr(X)
            out, _ = oracle.csr(rp, ci, vals, y, v, g["alpha"], g["beta"], z, 2, acc=acc, lib=lib)
            assert np.array_equal(out, g["out"]), ("csr", dt, acc, out)


def pin_gram_identity(lib):
    rng = np.random.default_rng(1)
    for m, n in ((40, 7), (7, 40), (1, 5), (33, 33)):
        X = rng.uniform(-1, 1, (m, n))
        y = rng.uniform(-1, 1, n)
        G = X.T @ X  # Gram matrix formed on its own, then applied to y
        ref = G @ y
        out, S = oracle.dense(X, y, None, 1.0, 0.0, None, lib=lib)
        assert _close(out, ref, _absscale(X, y, None, 1.0, 0.0, None)), (m, n)
        rp, ci, vals = dense_to_csr(X)
        out, S = oracle.csr(rp, ci, vals, y, None, 1.0, 0.0, None, n, lib=lib)
        assert _close(out, ref, _absscale(X, y, None, 1.0, 0.0, None)), ("csr", m, n)


def pin_quadratic_form(lib):
    rng = np.random.default_rng(2)
    for m, n in ((50, 9), (9, 50)):
        X = rng.uniform(-1, 1, (m, n))
        y = rng.uniform(-1, 1, n)
        v = rng.uniform(-2, 2, m)
        z = rng.uniform(-1, 1, n)
        alpha, beta = 1.75, -0.625
        u = X @ y
        rhs = alpha * np.sum(v * u * u) + beta * np.dot(y, z)
        scale = abs(alpha) * np.sum(np.abs(v) * (np.abs(X) @ np.abs(y)) ** 2) + abs(beta) * np.abs(y) @ np.abs(z)
        out, _ = oracle.dense(X, y, v, alpha, beta, z, lib=lib)
        assert abs(np.dot(y, out) - rhs) <= 1e-13 * scale
        rp, ci, vals = dense_to_csr(X)
        out, _ = oracle.csr(rp, ci, vals, y, v, alpha, beta, z, n, lib=lib)
        assert abs(np.dot(y, out) - rhs) <= 1e-13 * scale


def pin_linearity_and_permutations(lib):
    rng = np.random.default_rng(3)
    m, n = 30, 11
    X = rng.uniform(-1, 1, (m, n))
    y = rng.uniform(-1, 1, n)
    v1 = rng.uniform(-1, 1, m)
    v2 = rng.uniform(-1, 1, m)
    z = rng.uniform(-1, 1, n)
    sc = _absscale(X, y, np.abs(v1) + np.abs(v2), 3.0, 2.0, z)
    base, _ = oracle.dense(X, y, v1, 1.0, 0.0, None, lib=lib)
    # alpha and beta enter linearly
    out, _ = oracle.dense(X, y, v1, 3.0, 2.0, z, lib=lib)
    assert _close(out, 3.0 * base + 2.0 * z, sc)
    # v enters linearly
    o1, _ = oracle.dense(X, y, v1, 1.0, 0.0, None, lib=lib)
    o2, _ = oracle.dense(X, y, v2, 1.0, 0.0, None, lib=lib)
    o12, _ = oracle.dense(X, y, v1 + v2, 1.0, 0.0, None, lib=lib)
    assert _close(o12, o1 + o2, sc)
    # joint row permutation of X and v changes nothing
    p = rng.permutation(m)
    op, _ = oracle.dense(X[p], y, v1[p], 1.0, 0.0, None, lib=lib)
    assert _close(op, base, sc)
    # a column permutation of X, y, z permutes out
    q = rng.permutation(n)
    ref, _ = oracle.dense(X, y, v1, 3.0, 2.0, z, lib=lib)
    oq, _ = oracle.dense(np.ascontiguousarray(X[:, q]), y[q], v1, 3.0, 2.0, z[q], lib=lib)
    assert _close(oq, ref[q], sc[q])
    # the same through CSR, with an unsorted column order inside rows
    rp, ci, vals = dense_to_csr(X)
    for i in range(m):
        a, b = rp[i], rp[i + 1]
        r = rng.permutation(b - a)
        ci[a:b] = ci[a:b][r]
        vals[a:b] = vals[a:b][r]
    oc, _ = oracle.csr(rp, ci, vals, y, v1, 3.0, 2.0, z, n, lib=lib)
    assert _close(oc, ref, sc)


def pin_exact_bruteforce(lib):
    rng = np.random.default_rng(4)
    for trial in range(60):
        m = int(rng.integers(1, 5))
        n = int(rng.integers(1, 5))
        X = rng.integers(-2, 3, (m, n)).astype(np.float64)
        y = rng.integers(-2, 3, n).astype(np.float64)
        v = rng.integers(-2, 3, m).astype(np.float64) if trial % 3 else None
        z = rng.integers(-2, 3, n).astype(np.float64) if trial % 2 else None
        alpha = [1.0, -1.0, 2.0, -2.0, 0.5, -0.5][trial % 6]
        beta = [0.0, 1.0, -1.0, 2.0, -0.5][trial % 5]
        Xq = [[Fraction(float(X[i, j])) for j in range(n)] for i in range(m)]
        ref = _exact(Xq, _frac(y), None if v is None else _frac(v), alpha, beta, None if z is None else _frac(z))
        for dt in (np.float32, np.float64):
            c = lambda a: None if a is None else a.astype(dt)
            for acc in ("ld", "d"):
                out, _ = oracle.dense(c(X), c(y), c(v), alpha, beta, c(z), acc=acc, lib=lib)
                assert [Fraction(float(o)) for o in out] == ref, (trial, dt, acc)
                rp, ci, vals = dense_to_csr(c(X))
                out, _ = oracle.csr(rp, ci, vals, c(y), c(v), alpha, beta, c(z), n, acc=acc, lib=lib)
                assert [Fraction(float(o)) for o in out] == ref, ("csr", trial, dt, acc)


def _pattern_check(lib, m, n):
    vals3 = np.array([-1.0, 1.0, 2.0])
    y = np.array([1.0, -2.0, 2.0, -1.0][:n])
    v = np.array([2.0, -1.0, 1.0][:m])
    z = np.array([1.0, 2.0, -1.0, 2.0][:n])
    for pat in range(1 << (m * n)):
        X = np.zeros((m, n))
        for b in range(m * n):
            if pat >> b & 1:
                X[b // n, b % n] = vals3[(b + pat) % 3]
        Xq = [[Fraction(X[i, j]) for j in range(n)] for i in range(m)]
        ref = _exact(Xq, _frac(y), _frac(v), -0.5, 2.0, _frac(z))
        rp, ci, vv = dense_to_csr(X)
        out, _ = oracle.csr(rp, ci, vv, y, v, -0.5, 2.0, z, n, lib=lib)
        assert [Fraction(o) for o in out] == ref, (m, n, pat)
        out, _ = oracle.dense(X, y, v, -0.5, 2.0, z, lib=lib)
        assert [Fraction(o) for o in out] == ref, ("dense", m, n, pat)


def pin_all_patterns(lib):
    _pattern_check(lib, 3, 3)
    _pattern_check(lib, 2, 4)


def pin_dense_equals_csr(lib):
    rng = np.random.default_rng(5)
    m, n = 60, 17
    X = rng.uniform(-1, 1, (m, n))
    X[rng.random((m, n)) < 0.7] = 0.0
    X[3, :] = 0.0  # an empty row
    y = rng.uniform(-1, 1, n)
    v = rng.uniform(-1, 1, m)
    z = rng.uniform(-1, 1, n)
    ref, S = oracle.dense(X, y, v, 1.25, 0.5, z, lib=lib)
    for keep in (False, True):
        rp, ci, vals = dense_to_csr(X, keep_zeros=keep)
        out, S2 = oracle.csr(rp, ci, vals, y, v, 1.25, 0.5, z, n, lib=lib)
        assert np.array_equal(out, ref), keep
        assert np.array_equal(S, S2), keep
    # duplicates add: split each integer entry into two exactly representable parts
    Xi = rng.integers(-4, 5, (m, n)).astype(np.float64)
    Xi[rng.random((m, n)) < 0.5] = 0.0
    yi = rng.integers(-3, 4, n).astype(np.float64)
    vi = rng.integers(-3, 4, m).astype(np.float64)
    ref, _ = oracle.dense(Xi, yi, vi, 2.0, -1.0, z, lib=lib)
    rp, ci, vals = dense_to_csr(Xi)
    rows = np.repeat(np.arange(m), np.diff(rp))
    half = np.floor(vals / 2)
    rows2 = np.concatenate([rows, rows])
    ci2 = np.concatenate([ci, ci])
    vals2 = np.concatenate([half, vals - half])
    order = np.lexsort((np.arange(rows2.size), rows2))
    rp2 = np.zeros(m + 1, dtype=np.int64)
    rp2[1:] = np.cumsum(np.bincount(rows2, minlength=m))
    out, _ = oracle.csr(rp2, ci2[order], vals2[order], yi, vi, 2.0, -1.0, z, n, lib=lib)
    assert np.array_equal(out, ref)


def pin_library_composition(lib):
    rng = np.random.default_rng(6)
    for m, n in ((200, 13), (13, 200), (64, 64)):
        X = rng.standard_normal((m, n))
        y = rng.standard_normal(n)
        ref = X.T @ (X @ y)
        out, S = oracle.dense(X, y, None, 1.0, 0.0, None, lib=lib)
        assert _close(out, ref, _absscale(X, y, None, 1.0, 0.0, None)), (m, n)
        v = rng.uniform(0.1, 2.0, m)
        z = rng.standard_normal(n)
        ref = 2.0 * (X.T @ (v * (X @ y))) - z
        out, S = oracle.dense(X, y, v, 2.0, -1.0, z, lib=lib)
        assert _close(out, ref, _absscale(X, y, v, 2.0, -1.0, z)), (m, n)
        # S is the bound's scale: |alpha| |X|^T |t| + |beta z|, with t = v * (X y)
        t = v * (X @ y)
        assert _close(S, 2.0 * (np.abs(X).T @ np.abs(t)) + np.abs(z), np.abs(S) + 1.0)


def pin_special_cases(lib):
    rng = np.random.default_rng(7)
    n = 5
    z = rng.uniform(-1, 1, n)
    y = rng.uniform(-1, 1, n)
    # m = 0: out = beta z
    out, S = oracle.dense(np.zeros((0, n)), y, np.zeros(0), 2.0, -3.0, z, lib=lib)
    assert np.array_equal(out, -3.0 * z) and np.array_equal(S, 3.0 * np.abs(z))
    out, _ = oracle.csr(np.zeros(1, np.int64), np.zeros(0, np.int32), np.zeros(0), y, None, 2.0, -3.0, z, n, lib=lib)
    assert np.array_equal(out, -3.0 * z)
    # m = 0 without z: zeros
    out, _ = oracle.dense(np.zeros((0, n)), y, None, 2.0, 1.0, None, lib=lib)
    assert np.array_equal(out, np.zeros(n))
    # n = 0: nothing to compute
    out, _ = oracle.dense(np.zeros((4, 0)), np.zeros(0), np.ones(4), 1.0, 1.0, np.zeros(0), lib=lib)
    assert out.shape == (0,)
    # beta = 0: z is not read, so a NaN there does not reach out
    X = rng.uniform(-1, 1, (6, n))
    znan = np.full(n, np.nan)
    ref, _ = oracle.dense(X, y, None, 1.0, 0.0, None, lib=lib)
    out, _ = oracle.dense(X, y, None, 1.0, 0.0, znan, lib=lib)
    assert np.array_equal(out, ref)
    rp, ci, vals = dense_to_csr(X)
    out, _ = oracle.csr(rp, ci, vals, y, None, 1.0, 0.0, znan, n, lib=lib)
    assert np.array_equal(out, ref)
    # alpha = 0: out = beta z exactly
    out, _ = oracle.dense(X, y, np.ones(6), 0.0, 2.0, z, lib=lib)
    assert np.array_equal(out, 2.0 * z)
    # v absent is v = 1
    a, _ = oracle.dense(X, y, None, 1.5, 0.0, None, lib=lib)
    b, _ = oracle.dense(X, y, np.ones(6), 1.5, 0.0, None, lib=lib)
    assert np.array_equal(a, b)
    # sampled columns equal the full computation
    full, Sf = oracle.dense(X, y, rng.uniform(-1, 1, 6), 1.5, 0.5, z, lib=lib)
    vv = rng.uniform(-1, 1, 6)
    full, Sf = oracle.dense(X, y, vv, 1.5, 0.5, z, lib=lib)
    cols = np.array([4, 0, 2])
    part, Sp = oracle.dense(X, y, vv, 1.5, 0.5, z, cols=cols, lib=lib)
    assert np.array_equal(part, full[cols]) and np.array_equal(Sp, Sf[cols])
    # leading dimension: padding columns are ignored
    Xp = np.concatenate([X, np.full((6, 3), np.nan)], axis=1)
    a, _ = oracle.dense(Xp, y, vv, 1.5, 0.5, z, n=n, lib=lib)
    assert np.array_equal(a, full)
    # malformed CSR is refused
    with pytest.raises(ValueError):
        oracle.csr(np.array([0, 2, 1], np.int64), np.zeros(1, np.int32), np.zeros(1), y, None, 1.0, 0.0, None, n, lib=lib)
    with pytest.raises(ValueError):
        oracle.csr(np.array([0, 1], np.int64), np.array([n], np.int32), np.zeros(1), y, None, 1.0, 0.0, None, n, lib=lib)
    # row_ptr must start at 0 and end at nnz, even when it is non-decreasing and every column is in range
    with pytest.raises(ValueError):
        oracle.csr(np.array([1, 2], np.int64), np.zeros(2, np.int32), np.ones(2), y, None, 1.0, 0.0, None, n, lib=lib)
    with pytest.raises(ValueError):
        oracle.csr(np.array([0, 1, 1], np.int64), np.zeros(2, np.int32), np.ones(2), y, None, 1.0, 0.0, None, n,
                   lib=lib)
    assert not oracle.csr_is_valid(np.array([0, 1, 1], np.int64), np.zeros(2, np.int32), n, lib=lib)
    assert oracle.csr_is_valid(np.array([0, 1, 2], np.int64), np.zeros(2, np.int32), n, lib=lib)


PINS = [pin_worked_example, pin_gram_identity, pin_quadratic_form, pin_linearity_and_permutations,
        pin_exact_bruteforce, pin_all_patterns, pin_dense_equals_csr, pin_library_composition,
        pin_special_cases]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(oracle._load())


def test_accumulators_agree_on_workload_recipe():
    """The double and long double variants agree within the fp64 bound on the small dense workload."""
    p = inputgen.dense_small()
    a, S = oracle.solve(p, acc="ld")
    b, _ = oracle.solve(p, acc="d")
    assert np.all(np.abs(a - b) <= 1e-12 * S)
    assert np.all(S > 0)


# ---------------------------------------------------------------------------------------------
# The multi-vector instantiation OUT = alpha * X^T (V * (X Y)) + beta * Z ("On optimizing
# machine learning workloads via kernel fusion", abstract: the pattern and its
# instantiations, here with k right-hand sides at once).
# ---------------------------------------------------------------------------------------------
def _exact_multi(Xq, Yq, Vq, alpha, beta, Zq):
    """Exact rational OUT over the whole matrix, written out as row sums and column sums."""
    m, n, k = len(Xq), len(Yq), len(Yq[0]) if Yq else 0
    a, b = Fraction(alpha), Fraction(beta)
    T = [[sum((Xq[i][j] * Yq[j][c] for j in range(n)), Fraction(0)) for c in range(k)] for i in range(m)]
    if Vq is not None:
        T = [[T[i][c] * (Vq[i][c] if isinstance(Vq[i], list) else Vq[i]) for c in range(k)] for i in range(m)]
    out = []
    for j in range(n):
        row = []
        for c in range(k):
            w = sum((Xq[i][j] * T[i][c] for i in range(m)), Fraction(0))
            row.append(a * w + (b * Zq[j][c] if Zq is not None and beta != 0 else Fraction(0)))
        out.append(row)
    return out


def _fracm(A):
    return None if A is None else [[Fraction(float(x)) for x in row] for row in A] if A.ndim == 2 else _frac(A)


def pin_multi_exact(lib, fn=None):
    """Tiny integer inputs: the multi-vector oracle equals exact rational arithmetic for
    full (m, k) weights, one shared weight vector, and no weights."""
    fn = fn or oracle.dense_multi
    rng = np.random.default_rng(21)
    for (m, n, k) in ((4, 3, 2), (5, 2, 3), (1, 4, 4), (3, 3, 1)):
        X = rng.integers(-3, 4, (m, n)).astype(np.float64)
        Y = rng.integers(-3, 4, (n, k)).astype(np.float64)
        Z = rng.integers(-3, 4, (n, k)).astype(np.float64)
        for V in (rng.integers(-2, 3, (m, k)).astype(np.float64), rng.integers(-2, 3, m).astype(np.float64), None):
            ref = _exact_multi(_fracm(X), _fracm(Y), None if V is None else _fracm(V), -1.5, 2.0, _fracm(Z))
            out, _ = fn(X, Y, V, -1.5, 2.0, Z, lib=lib)
            assert out.shape == (n, k)
            assert [[Fraction(o) for o in row] for row in out] == ref, (m, n, k, None if V is None else V.ndim)


def pin_multi_library(lib, fn=None):
    """The matrix form from numpy, and the bound's scale per (column, right-hand side)."""
    fn = fn or oracle.dense_multi
    rng = np.random.default_rng(22)
    m, n, k = 300, 11, 5
    X = rng.standard_normal((m, n))
    Y = rng.standard_normal((n, k))
    V = rng.uniform(0.1, 2.0, (m, k))
    Z = rng.standard_normal((n, k))
    T = V * (X @ Y)
    ref = 0.75 * (X.T @ T) + 0.5 * Z
    out, S = fn(X, Y, V, 0.75, 0.5, Z, lib=lib)
    scale = 0.75 * (np.abs(X).T @ (np.abs(V) * (np.abs(X) @ np.abs(Y)))) + 0.5 * np.abs(Z)
    assert np.all(np.abs(out - ref) <= 1e-13 * scale)
    assert np.allclose(S, 0.75 * (np.abs(X).T @ np.abs(T)) + 0.5 * np.abs(Z), rtol=1e-12)
    # one shared v is the same as that v repeated in every column
    v = rng.uniform(0.1, 2.0, m)
    a, _ = fn(X, Y, v, 0.75, 0.5, Z, lib=lib)
    b, _ = fn(X, Y, np.repeat(v[:, None], k, axis=1), 0.75, 0.5, Z, lib=lib)
    assert np.array_equal(a, b)
    # k = 1 is the single-vector pattern; sampled columns equal the full computation
    one, _ = oracle.dense(X, Y[:, 2].copy(), V[:, 2].copy(), 0.75, 0.5, Z[:, 2].copy(), lib=lib)
    c1, _ = fn(X, Y[:, 2:3], V[:, 2:3], 0.75, 0.5, Z[:, 2:3], lib=lib)
    assert np.array_equal(c1[:, 0], one) and np.array_equal(out[:, 2], one)
    cols = np.array([7, 0, 3])
    part, Sp = fn(X, Y, V, 0.75, 0.5, Z, cols=cols, lib=lib)
    assert np.array_equal(part, out[cols]) and np.array_equal(Sp, S[cols])
    # the right-hand sides do not interact: permuting Y's columns (with V and Z) permutes OUT's
    perm = np.array([3, 1, 4, 0, 2])
    pout, _ = fn(X, Y[:, perm], V[:, perm], 0.75, 0.5, Z[:, perm], lib=lib)
    assert np.array_equal(pout, out[:, perm])
    # beta = 0 leaves Z unread
    a, _ = fn(X, Y, V, 0.75, 0.0, np.full((n, k), np.nan), lib=lib)
    b, _ = fn(X, Y, V, 0.75, 0.0, None, lib=lib)
    assert np.array_equal(a, b)


MULTI_PINS = [pin_multi_exact, pin_multi_library]


@pytest.mark.parametrize("pin", MULTI_PINS, ids=lambda f: f.__name__)
def test_multi_pin(pin):
    pin(oracle._load())


# Planted mistakes in the multi-vector wrapper: (description, exact text, replacement).
MULTI_MUTANTS = [
    ("every right-hand side reads Y's first column", "np.ascontiguousarray(Y[:, c])", "np.ascontiguousarray(Y[:, 0])"),
    ("weights taken from the wrong column", "np.ascontiguousarray(V[:, c])", "np.ascontiguousarray(V[:, -1 - c])"),
    ("Z's columns shifted", "zc = None if Z is None else np.ascontiguousarray(Z[:, c])",
     "zc = None if Z is None else np.ascontiguousarray(Z[:, (c + 1) % k])"),
    ("shared weights ignored", "if V is None or V.ndim == 1:\n        return V", "if V is None or V.ndim == 1:\n        return None"),
]


@pytest.mark.parametrize("mutant", MULTI_MUTANTS, ids=lambda m: m[0])
def test_multi_planted_mistakes(mutant):
    """An altered multi-vector oracle must fail at least one of its pins."""
    import inspect
    import textwrap
    desc, old, new = mutant
    src = textwrap.dedent(inspect.getsource(oracle._vcol)) + "\n" + textwrap.dedent(inspect.getsource(oracle.dense_multi))
    assert old in src, f"mutation target for '{desc}' not found in the oracle source"
    ns = dict(vars(oracle))
    exec(compile(src.replace(old, new), "<mutant>", "exec"), ns)
    failures = []
    for pin in MULTI_PINS:
        try:
            pin(oracle._load(), fn=ns["dense_multi"])
        except (AssertionError, ValueError):
            failures.append(pin.__name__)
    assert failures, f"mutant '{desc}' passed every pin"


# Each entry: (description, exact text in fxtx_oracle.c, replacement, occurrence count to replace)
MUTANTS = [
    ("v dropped", "acc_t vi = v ? at(v, dtype, i) : (acc_t)1;", "acc_t vi = 1;"),
    ("dot uses transposed index", "u += at(X, dtype, i * ld + j) * at(y, dtype, j);",
     "u += at(X, dtype, j * ld + i) * at(y, dtype, j);"),
    ("beta sign flipped", "o += (acc_t)beta * at(z, dtype, j);", "o -= (acc_t)beta * at(z, dtype, j);"),
    ("alpha dropped", "acc_t o = (acc_t)alpha * w[k];", "acc_t o = w[k];"),
    ("scatter uses y instead of t", "w[j] += at(X, dtype, i * ld + j) * t[i];",
     "w[j] += at(X, dtype, i * ld + j) * at(y, dtype, j);"),
    ("CSR row starts one late", "for (int64_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) u +=",
     "for (int64_t k = row_ptr[i] + 1; k < row_ptr[i + 1]; ++k) u +="),
    ("CSR scatter to wrong column", "int64_t j = col_idx[k];", "int64_t j = (col_idx[k] + 1) % n;"),
    ("z read when beta is zero", "int use_z = (z != NULL && beta != 0.0);", "int use_z = (z != NULL);"),
    ("dot drops the last column", "for (int64_t j = 0; j < n; ++j) u +=", "for (int64_t j = 0; j + 1 < n; ++j) u +="),
    ("S omits beta z", "sj += fabs(beta * atd(z, dtype, j));", "sj += 0;"),
    ("CSR row_ptr ends unchecked", "if (row_ptr[0] != 0 || row_ptr[m] != nnz) return ORACLE_BAD_CSR;", ""),
    ("CSR row_ptr end checked only", "if (row_ptr[0] != 0 || row_ptr[m] != nnz) return ORACLE_BAD_CSR;",
     "if (row_ptr[m] != nnz) return ORACLE_BAD_CSR;"),
]


@pytest.mark.parametrize("mutant", MUTANTS, ids=lambda m: m[0])
def test_planted_mistakes(mutant, tmp_path):
    """An altered oracle must fail at least one pin."""
    desc, old, new = mutant
    src = open(os.path.join(os.path.dirname(oracle.__file__), "fxtx_oracle.c")).read()
    assert old in src, f"mutation target for '{desc}' not found in the oracle source"
    msrc = tmp_path / "mutant.c"
    msrc.write_text(src.replace(old, new))
    so = str(tmp_path / "libmutant.so")
    oracle.compile_oracle(str(msrc), so)
    lib = oracle.bind(so)
    failures = []
    for pin in PINS:
        try:
            pin(lib)
        except (AssertionError, ValueError, pytest.fail.Exception):  # pytest.raises that saw no error fails so
            failures.append(pin.__name__)
    assert failures, f"mutant '{desc}' passed every pin"
