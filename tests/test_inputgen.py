"""The seeded input generator: determinism, structure validity and distribution shape."""
import numpy as np

import inputgen
import oracle


def test_deterministic_and_stream_separated():
    a = inputgen.uniform(0, 1, 1000, -1.0, 1.0)
    b = inputgen.uniform(0, 1, 1000, -1.0, 1.0)
    c = inputgen.uniform(0, 2, 1000, -1.0, 1.0)
    d = inputgen.uniform(1, 1, 1000, -1.0, 1.0)
    assert np.array_equal(a, b)
    assert not np.array_equal(a, c) and not np.array_equal(a, d)
    assert a.min() >= -1.0 and a.max() < 1.0
    # a prefix of a longer draw is the shorter draw (counter-based)
    assert np.array_equal(inputgen.uniform(0, 1, 10, -1.0, 1.0), a[:10])
    f = inputgen.uniform(0, 1, 1000, -1.0, 1.0, np.float32)
    assert np.array_equal(f, a.astype(np.float32))


def test_moments():
    x = inputgen.normal(3, 1, 200_000)
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    u = inputgen.uniform(3, 2, 200_000, 0.1, 2.0)
    assert abs(u.mean() - 1.05) < 0.01
    k = inputgen.integers(3, 4, 100_000, -2, 2)
    assert set(np.unique(k)) == {-2.0, -1.0, 0.0, 1.0, 2.0}


def test_csr_uniform_recipe_small():
    p = inputgen.csr_uniform(m=20_000, n=1_000, lam=50.0)
    lens = np.diff(p.row_ptr)
    assert abs(lens.mean() - 50.0) < 0.5
    assert abs(lens.var() - 50.0) < 3.0  # Poisson: variance equals the mean
    assert oracle.csr_is_valid(p.row_ptr, p.col_idx, p.n)
    for i in (0, 7, 19_999):
        c = p.col_idx[p.row_ptr[i]:p.row_ptr[i + 1]]
        assert np.all(np.diff(c) > 0)  # distinct and sorted


def test_csr_powerlaw_recipe_small():
    p = inputgen.csr_powerlaw(m=20_000, n=50_000, mean_len=100.0, cap=5_000)
    lens = np.diff(p.row_ptr)
    assert abs(lens.mean() - 100.0) < 1.0
    assert lens.max() <= 5_000 and lens.min() >= 1
    assert oracle.csr_is_valid(p.row_ptr, p.col_idx, p.n)
    # Zipf(1.1) columns with column = rank - 1: column 0 is the most frequent, and
    # with distinct columns per row it appears in nearly every row of length >= 20
    counts = np.bincount(p.col_idx, minlength=p.n)
    assert counts.argmax() == 0
    assert counts[0] > counts[100] > counts[10_000]
    rows = np.repeat(np.arange(p.m), lens)
    assert np.all(np.diff(p.col_idx)[np.diff(rows) == 0] > 0)


def test_workload_shapes_small():
    p = inputgen.dense_tall(m=1000, n=32, variant="b")
    assert p.X.shape == (1000, 32) and p.X.dtype == np.float32 and p.alpha == 2.0 and p.beta == -1.0
    assert inputgen.dense_tall(m=10, variant="c").v is None
    assert inputgen.dense_tall(m=10, variant="a").z is None
    p = inputgen.dense_small()
    assert p.ideal_bytes() == 1000 * 64 * 8 + 64 * 8 * 3 + 1000 * 8
    p = inputgen.dense_multi(m=100, n=32, k=8)
    assert p.y.shape == (32, 8) and p.z.shape == (32, 8) and p.v.shape == (100, 8)
    assert p.ideal_bytes() == 100 * 32 * 4 + 2 * 32 * 8 * 4 + 100 * 8 * 4 + 32 * 8 * 4
    assert inputgen.dense_multi(m=10, k=3, v_mode="shared").v.shape == (10,)
    assert inputgen.dense_multi(m=10, k=3, v_mode="none").v is None
    q = inputgen.dense_multi(m=100, n=32, k=8)
    assert np.array_equal(p.X, q.X) and np.array_equal(p.y, q.y) and np.array_equal(p.v, q.v)
