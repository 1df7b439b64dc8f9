"""The multi-vector instantiation OUT = alpha * X^T (V * (X Y)) + beta * Z (k right-hand
sides in one pass over X) against the oracle, column by column, with the bound of the
single-vector pattern per (column, right-hand side): fp32 2e-5 * S, fp64 1e-12 * S."""
import numpy as np
import pytest
import torch

import dense_linear_algebra_gb300 as fx
import inputgen
import oracle
from _util import assert_within_bound

pytestmark = pytest.mark.gpu

TOL = {np.float32: 2e-5, np.float64: 1e-12}


def make(m, n, k, dtype, v_mode="full", seed=1, ld=None, alpha=1.25, beta=-0.75, with_z=True):
    ld = n if ld is None else ld
    X = inputgen.uniform(seed, 1, (m, ld), -1.0, 1.0, dtype)
    Y = inputgen.uniform(seed, 2, (n, k), -1.0, 1.0, dtype)
    Z = inputgen.uniform(seed, 4, (n, k), -1.0, 1.0, dtype) if with_z else None
    if v_mode == "full":
        V = inputgen.uniform(seed, 3, (m, k), -1.0, 1.0, dtype)
    elif v_mode == "shared":
        V = inputgen.uniform(seed, 3, m, -1.0, 1.0, dtype)
    else:
        V = None
    return inputgen.Problem(f"multi_{m}x{n}x{k}_{v_mode}_ld{ld}", "dense", dtype, m, n, alpha, beta, y=Y, v=V, z=Z,
                            X=X, ld=ld)


def dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run(p, out=None):
    X = dev(p.X)[:, : p.n]
    got = fx.dense_multi(X, dev(p.y), dev(p.v), p.alpha, p.beta, dev(p.z), out=out)
    torch.cuda.synchronize()
    assert fx.device_error() == fx.FXTX_OK
    return got.cpu().numpy().astype(np.float64)


def check(p, got=None):
    got = run(p) if got is None else got
    ref, S = oracle.dense_multi(p.X, p.y, p.v, p.alpha, p.beta, p.z, n=p.n)
    assert got.shape == ref.shape
    assert_within_bound(got.ravel(), ref.ravel(), S.ravel(), TOL[p.dtype], p.name)


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("n", [1, 5, 16, 17, 32, 33, 64, 65, 100, 128, 200, 256, 512])
def test_shapes(dtype, n):
    if n * np.dtype(dtype).itemsize > 2048:
        pytest.skip("rows above 2 KB are not taken")
    for m, k in ((1, 3), (37, 8), (3001, 5)):
        check(make(m, n, k, dtype, seed=n + m))


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
@pytest.mark.parametrize("k", [1, 2, 3, 4, 7, 8, 16, 31, 32, 33, 64, 70])
def test_right_hand_sides(dtype, k):
    check(make(5000, 32, k, dtype, seed=k))


@pytest.mark.parametrize("v_mode", ["full", "shared", "none"])
@pytest.mark.parametrize("n,k", [(32, 8), (128, 4), (20, 32)])
def test_weight_modes(v_mode, n, k):
    for dtype in (np.float32, np.float64):
        check(make(4000, n, k, dtype, v_mode=v_mode, seed=n * k))


@pytest.mark.parametrize("n,ld", [(32, 33), (32, 40), (30, 32), (100, 101), (256, 264)])
def test_leading_dimension(n, ld):
    """Padded rows; odd pitches take the plain-load staging."""
    for dtype in (np.float32, np.float64):
        if n * np.dtype(dtype).itemsize <= 2048:
            check(make(3000, n, 6, dtype, ld=ld, seed=ld))


def test_unaligned_x_takes_plain_loads():
    p = make(3000, 32, 8, np.float32, seed=5)
    ref, S = oracle.dense_multi(p.X, p.y, p.v, p.alpha, p.beta, p.z)
    big = torch.zeros(p.m * p.n + 1, dtype=torch.float32, device="cuda")
    big[1:] = torch.from_numpy(p.X.ravel()).cuda()
    X = big[1:].view(p.m, p.n)  # 4-byte offset: no tensor copies
    got = fx.dense_multi(X, dev(p.y), dev(p.v), p.alpha, p.beta, dev(p.z)).cpu().numpy()
    assert_within_bound(got.ravel(), ref.ravel(), S.ravel(), 2e-5)


def test_edge_cases():
    # m == 0: OUT = beta Z; beta == 0: Z not read (NaN there does not reach OUT); k == 0 / n == 0: no-ops
    p = make(0, 24, 5, np.float64, seed=2)
    check(p)
    p = make(500, 24, 5, np.float64, seed=3, beta=0.0)
    ref, S = oracle.dense_multi(p.X, p.y, p.v, p.alpha, 0.0, None)
    got = fx.dense_multi(dev(p.X), dev(p.y), dev(p.v), p.alpha, 0.0, torch.full((24, 5), float("nan"),
                                                                                 dtype=torch.float64, device="cuda"))
    assert_within_bound(got.cpu().numpy().ravel(), ref.ravel(), S.ravel(), 1e-12)
    p = make(500, 24, 5, np.float64, seed=3, with_z=False)
    check(p)
    e = torch.empty((24, 0), dtype=torch.float64, device="cuda")
    assert fx.dense_multi(dev(p.X), e, None, 1.0, 0.0, None).shape == (24, 0)
    # rows above 2 KB are refused
    with pytest.raises(fx.FxtxError) as ei:
        fx.dense_multi(torch.zeros(4, 600, device="cuda"), torch.zeros(600, 2, device="cuda"))
    assert ei.value.status == fx.FXTX_ERR_UNSUPPORTED


def test_in_place_and_column_slices():
    """OUT may be Z; Y, V, Z and OUT may be column slices of wider matrices."""
    p = make(4000, 32, 6, np.float32, seed=8)
    ref, S = oracle.dense_multi(p.X, p.y, p.v, p.alpha, p.beta, p.z)
    Zd = dev(p.z)
    fx.dense_multi(dev(p.X), dev(p.y), dev(p.v), p.alpha, p.beta, Zd, out=Zd)
    assert_within_bound(Zd.cpu().numpy().ravel(), ref.ravel(), S.ravel(), 2e-5)
    Yw = torch.zeros(32, 11, device="cuda")
    Yw[:, 2:8] = dev(p.y)
    Vw = torch.zeros(4000, 9, device="cuda")
    Vw[:, 1:7] = dev(p.v)
    Zw = torch.zeros(32, 10, device="cuda")
    Zw[:, 3:9] = dev(p.z)
    Ow = torch.full((32, 13), 7.0, device="cuda")
    fx.dense_multi(dev(p.X), Yw[:, 2:8], Vw[:, 1:7], p.alpha, p.beta, Zw[:, 3:9], out=Ow[:, 4:10])
    got = Ow.cpu().numpy()
    assert_within_bound(got[:, 4:10].astype(np.float64).ravel(), ref.ravel(), S.ravel(), 2e-5)
    assert np.all(got[:, :4] == 7.0) and np.all(got[:, 10:] == 7.0)


def test_integer_inputs_are_exact():
    """Small integers: every partial sum is exact in fp32, so OUT equals the exact value."""
    m, n, k = 20_000, 32, 8
    X = inputgen.integers(3, 1, (m, n), -2, 2, np.float32)
    Y = inputgen.integers(3, 2, (n, k), -2, 2, np.float32)
    V = inputgen.integers(3, 3, (m, k), -2, 2, np.float32)
    Z = inputgen.integers(3, 4, (n, k), -2, 2, np.float32)
    ref, _ = oracle.dense_multi(X, Y, V, 2.0, -1.0, Z)
    assert np.abs(ref).max() < 2 ** 24
    got = fx.dense_multi(dev(X), dev(Y), dev(V), 2.0, -1.0, dev(Z)).cpu().numpy()
    assert np.array_equal(got.astype(np.float64), ref)


def test_deterministic_and_matches_single_vector_calls():
    p = make(100_000, 32, 8, np.float32, seed=4)
    a = run(p)
    b = run(p)
    assert np.array_equal(a, b)
    # each right-hand side through the single-vector entry point, within the same bound
    ref, S = oracle.dense_multi(p.X, p.y, p.v, p.alpha, p.beta, p.z)
    Xd = dev(p.X)
    for c in range(p.y.shape[1]):
        one = fx.dense(Xd, dev(p.y[:, c]), dev(p.v[:, c]), p.alpha, p.beta, dev(p.z[:, c])).cpu().numpy()
        assert_within_bound(one.astype(np.float64), ref[:, c], S[:, c], 2e-5)
        assert_within_bound(a[:, c], ref[:, c], S[:, c], 2e-5)


@pytest.mark.parametrize("v_mode", ["full", "shared"])
def test_tall_recipe_scaled(v_mode):
    check(inputgen.dense_multi(m=400_000, n=32, k=8, v_mode=v_mode))


@pytest.mark.slow
def test_full_size_workload_sampled():
    """The benchmark's multi-vector workload (16,000,000 x 32, k = 8, fp32) in its launch
    configuration, checked on sampled columns of OUT (each needs every row's dots)."""
    p = inputgen.dense_multi()
    got = run(p)
    cols = np.array([0, 7, 13, 31])
    ref, S = oracle.dense_multi(p.X, p.y, p.v, p.alpha, p.beta, p.z, cols=cols)
    assert_within_bound(got[cols].ravel(), ref.ravel(), S.ravel(), 2e-5)
