"""The tensor-core form of the multi-vector instantiation (fp32 X of at most 32 columns,
8 or more right-hand sides; both products on tcgen05 with three-term bfloat16 splits)
against the oracle, within the fp32 bound 2e-5 * S per (column, right-hand side): ragged
tiles, every weight mode and its staging (tensor copies or plain loads), several passes,
magnitudes far from 1, and the CUDA-core kernel for the same shapes."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

import dense_linear_algebra_gb300 as fx
import inputgen
import oracle
from _util import assert_within_bound

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def make(m, n, k, v_mode="full", seed=1, xscale=1.0, yscale=1.0, alpha=1.25, beta=-0.75):
    X = inputgen.uniform(seed, 1, (m, n), -1.0, 1.0, np.float32) * np.float32(xscale)
    Y = inputgen.uniform(seed, 2, (n, k), -1.0, 1.0, np.float32) * np.float32(yscale)
    Z = inputgen.uniform(seed, 4, (n, k), -1.0, 1.0, np.float32)
    V = {"full": lambda: inputgen.uniform(seed, 3, (m, k), 0.1, 2.0, np.float32),
         "shared": lambda: inputgen.uniform(seed, 3, m, 0.1, 2.0, np.float32),
         "none": lambda: None}[v_mode]()
    return X, Y, V, Z, alpha, beta


def dev(a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check(X, Y, V, Z, alpha, beta, got=None, what=""):
    if got is None:
        got = fx.dense_multi(dev(X), dev(Y), dev(V), alpha, beta, dev(Z))
        torch.cuda.synchronize()
        assert fx.device_error() == fx.FXTX_OK
        got = got.cpu().numpy()
    ref, S = oracle.dense_multi(X, Y, V, alpha, beta, Z)
    assert_within_bound(got.astype(np.float64).ravel(), ref.ravel(), S.ravel(), 2e-5, what)


@pytest.mark.parametrize("k", [8, 12, 16, 24, 32, 40, 64])
def test_plan_takes_tensor_cores(k):
    d = fx.multi_plan_describe("f32", 1_000_000, 32, k, "full")
    assert "tc=1" in d, d


@pytest.mark.parametrize("k", [8, 16, 32])
@pytest.mark.parametrize("m", [1, 127, 128, 129, 1000, 19_457, 300_001])
def test_ragged_rows(m, k):
    """Tiles of 128 rows: a single short tile, exactly one, one plus a row, ragged tails,
    and ranges of many tiles per CTA."""
    check(*make(m, 32, k, seed=m + k), what=f"m={m} k={k}")


@pytest.mark.parametrize("n", [1, 7, 16, 31, 32])
@pytest.mark.parametrize("k", [8, 9, 16, 17, 32])
def test_columns_and_partial_passes(n, k):
    """X narrower than the 32-column tile (the copy fills the rest with zeros) and passes
    with fewer right-hand sides than the kernel's width. X is a column slice of a matrix
    whose pitch is a multiple of 16 bytes, so the tensor copies (and the tensor cores) take
    it; with the pitch n itself, rows of 1, 7 or 31 values go to the CUDA-core kernel."""
    X, Y, V, Z, alpha, beta = make(20_000, n, k, seed=n * 100 + k)
    ld = (n + 3) // 4 * 4
    assert "tc=1" in fx.multi_plan_describe("f32", X.shape[0], n, k, "full", ld)
    Xp = torch.zeros(X.shape[0], ld, device="cuda")
    Xp[:, :n] = dev(X)
    got = fx.dense_multi(Xp[:, :n], dev(Y), dev(V), alpha, beta, dev(Z))
    torch.cuda.synchronize()
    assert fx.device_error() == fx.FXTX_OK
    check(X, Y, V, Z, alpha, beta, got=got.cpu().numpy(), what=f"n={n} ld={ld} k={k}")
    if n % 4:
        assert "tc=0" in fx.multi_plan_describe("f32", X.shape[0], n, k, "full", n)
        check(X, Y, V, Z, alpha, beta, what=f"n={n} ld={n} k={k} (CUDA cores)")


@pytest.mark.parametrize("v_mode", ["full", "shared", "none"])
@pytest.mark.parametrize("k", [8, 16, 32])
def test_weight_modes(v_mode, k):
    check(*make(50_000, 32, k, v_mode=v_mode, seed=k), what=f"{v_mode} k={k}")


@pytest.mark.parametrize("k", [8, 32])
def test_weights_by_plain_loads(k):
    """V whose address or pitch rules out tensor copies is read with plain loads."""
    X, Y, V, Z, alpha, beta = make(30_000, 32, k, seed=11)
    ref, S = oracle.dense_multi(X, Y, V, alpha, beta, Z)
    # 4-byte offset (an m x k view at an unaligned address)
    big = torch.zeros(V.size + 1, dtype=torch.float32, device="cuda")
    big[1:] = torch.from_numpy(V.ravel()).cuda()
    got = fx.dense_multi(dev(X), dev(Y), big[1:].view(V.shape), alpha, beta, dev(Z)).cpu().numpy()
    assert_within_bound(got.astype(np.float64).ravel(), ref.ravel(), S.ravel(), 2e-5)
    # pitch of k + 1 floats (not a multiple of 16 bytes)
    wide = torch.zeros(V.shape[0], k + 1, dtype=torch.float32, device="cuda")
    wide[:, :k] = dev(V)
    got = fx.dense_multi(dev(X), dev(Y), wide[:, :k], alpha, beta, dev(Z)).cpu().numpy()
    assert_within_bound(got.astype(np.float64).ravel(), ref.ravel(), S.ravel(), 2e-5)
    # a shared m-vector at an unaligned address
    Vs = inputgen.uniform(12, 3, V.shape[0], 0.1, 2.0, np.float32)
    ref, S = oracle.dense_multi(X, Y, Vs, alpha, beta, Z)
    big = torch.zeros(Vs.size + 1, dtype=torch.float32, device="cuda")
    big[1:] = torch.from_numpy(Vs).cuda()
    got = fx.dense_multi(dev(X), dev(Y), big[1:], alpha, beta, dev(Z)).cpu().numpy()
    assert_within_bound(got.astype(np.float64).ravel(), ref.ravel(), S.ravel(), 2e-5)


@pytest.mark.parametrize("xscale,yscale", [(1e-12, 1.0), (1e12, 1e-3), (3e-8, 5e7), (1.0, 1e-25)])
def test_magnitudes(xscale, yscale):
    """The split carries fp32's exponent range: inputs far from 1 (every product and term
    still a normal fp32 number) keep the relative bound. beta = 0, so S is the scatter's
    own scale."""
    check(*make(40_000, 32, 16, seed=21, xscale=xscale, yscale=yscale, beta=0.0), what=f"x*{xscale} y*{yscale}")


def test_cancelling_dots():
    """Rows whose dots partly cancel (x_i . y_0 a tenth of its typical size): the dots'
    error stays at an fp32 dot's, so the bound relative to S (built from the cancelled t_i)
    still holds."""
    m, n, k = 40_000, 32, 8
    rng = inputgen.uniform(31, 1, (m, n), -1.0, 1.0, np.float64)
    Y = inputgen.uniform(31, 2, (n, k), -1.0, 1.0, np.float64)
    # shrink column 0's dot tenfold: remove 90 % of X's component along Y[:, 0]
    y0 = Y[:, 0] / np.linalg.norm(Y[:, 0])
    X = (rng - 0.9 * np.outer(rng @ y0, y0)).astype(np.float32)
    V = inputgen.uniform(31, 3, (m, k), 0.1, 2.0, np.float32)
    Z = inputgen.uniform(31, 4, (n, k), -1.0, 1.0, np.float32)
    check(X, Y.astype(np.float32), V, Z, 1.0, 0.5, what="cancelling")


def test_in_place_deterministic_and_slices():
    X, Y, V, Z, alpha, beta = make(70_000, 32, 16, seed=41)
    ref, S = oracle.dense_multi(X, Y, V, alpha, beta, Z)
    Zd = dev(Z)
    fx.dense_multi(dev(X), dev(Y), dev(V), alpha, beta, Zd, out=Zd)
    a = Zd.cpu().numpy()
    assert_within_bound(a.astype(np.float64).ravel(), ref.ravel(), S.ravel(), 2e-5)
    b = fx.dense_multi(dev(X), dev(Y), dev(V), alpha, beta, dev(Z)).cpu().numpy()
    assert np.array_equal(a, b)  # fixed reduction order: repeat calls agree bit for bit
    Yw = torch.zeros(32, 21, device="cuda")
    Yw[:, 3:19] = dev(Y)
    Vw = torch.zeros(70_000, 20, device="cuda")
    Vw[:, 4:20] = dev(V)  # 16-byte aligned slice, pitch 80 bytes: tensor copies
    Ow = torch.full((32, 24), 7.0, device="cuda")
    fx.dense_multi(dev(X), Yw[:, 3:19], Vw[:, 4:20], alpha, beta, dev(Z), out=Ow[:, 2:18])
    got = Ow.cpu().numpy()
    assert_within_bound(got[:, 2:18].astype(np.float64).ravel(), ref.ravel(), S.ravel(), 2e-5)
    assert np.all(got[:, :2] == 7.0) and np.all(got[:, 18:] == 7.0)


def test_integer_inputs_are_exact():
    """Small integers: every term split is exact (one bfloat16 term each) and every partial
    sum is an integer below 2^24, so OUT is exact."""
    m, n, k = 30_000, 32, 16
    X = inputgen.integers(5, 1, (m, n), -2, 2, np.float32)
    Y = inputgen.integers(5, 2, (n, k), -2, 2, np.float32)
    V = inputgen.integers(5, 3, (m, k), -2, 2, np.float32)
    Z = inputgen.integers(5, 4, (n, k), -2, 2, np.float32)
    ref, _ = oracle.dense_multi(X, Y, V, 2.0, -1.0, Z)
    assert np.abs(ref).max() < 2 ** 24
    got = fx.dense_multi(dev(X), dev(Y), dev(V), 2.0, -1.0, dev(Z)).cpu().numpy()
    assert np.array_equal(got.astype(np.float64), ref)


_CHILD = r"""
import json, sys
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
import dense_linear_algebra_gb300 as fx, inputgen
m, n, k = 60_000, 32, 16
X = inputgen.uniform(51, 1, (m, n), -1.0, 1.0, np.float32)
Y = inputgen.uniform(51, 2, (n, k), -1.0, 1.0, np.float32)
V = inputgen.uniform(51, 3, (m, k), 0.1, 2.0, np.float32)
Z = inputgen.uniform(51, 4, (n, k), -1.0, 1.0, np.float32)
d = lambda a: torch.from_numpy(a).cuda()
out = fx.dense_multi(d(X), d(Y), d(V), 1.5, 0.25, d(Z)).cpu().numpy()
print(json.dumps({"plan": fx.multi_plan_describe("f32", m, n, k, "full"), "out": out.ravel().tolist()}))
"""


def test_cuda_core_kernel_for_the_same_shapes():
    """FXTX_MULTI_TC=0 keeps these shapes on the CUDA-core kernel: both kernels meet the bound."""
    env = dict(os.environ, FXTX_MULTI_TC="0")
    r = subprocess.run([sys.executable, "-c", _CHILD, ROOT], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert "tc=0" in res["plan"]
    m, n, k = 60_000, 32, 16
    X = inputgen.uniform(51, 1, (m, n), -1.0, 1.0, np.float32)
    Y = inputgen.uniform(51, 2, (n, k), -1.0, 1.0, np.float32)
    V = inputgen.uniform(51, 3, (m, k), 0.1, 2.0, np.float32)
    Z = inputgen.uniform(51, 4, (n, k), -1.0, 1.0, np.float32)
    ref, S = oracle.dense_multi(X, Y, V, 1.5, 0.25, Z)
    cuda_core = np.array(res["out"], dtype=np.float64)
    assert_within_bound(cuda_core, ref.ravel(), S.ravel(), 2e-5, "CUDA-core kernel")
    assert "tc=1" in fx.multi_plan_describe("f32", m, n, k, "full")
    check(X, Y, V, Z, 1.5, 0.25, what="tensor-core kernel")


@pytest.mark.slow
@pytest.mark.parametrize("k", [16, 32])
def test_full_size_sampled(k):
    """16,000,000 x 32 rows with k = 16 and 32 in the benchmark's launch configuration,
    checked on sampled columns of OUT for two of the right-hand sides (the oracle's cost is
    per right-hand side)."""
    p = inputgen.dense_multi(k=k)
    got = fx.dense_multi(dev(p.X), dev(p.y), dev(p.v), p.alpha, p.beta, dev(p.z)).cpu().numpy()
    assert fx.device_error() == fx.FXTX_OK
    cols, rhs = np.array([0, 9, 22, 31]), [1, k - 1]
    ref, S = oracle.dense_multi(p.X, p.y[:, rhs], p.v[:, rhs], p.alpha, p.beta, p.z[:, rhs], cols=cols)
    assert_within_bound(got[np.ix_(cols, rhs)].astype(np.float64).ravel(), ref.ravel(), S.ravel(), 2e-5)
