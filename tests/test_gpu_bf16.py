"""X stored as bfloat16 (NEXT-3: half the bytes of the dominant stream), fp32 vectors and
fp32 arithmetic. The oracle sees the same numbers: X's float32 values are bfloat16-
representable, so the device copy in bfloat16 holds them exactly. Bound: 2e-5 * S_j."""
import numpy as np
import pytest
import torch

import dense_linear_algebra_gb300 as fx
import inputgen
import oracle
from _gpu import run_problem
from _util import assert_within_bound

pytestmark = pytest.mark.gpu


def make_bf16(m, n, ld=None, seed=1, with_v=True, with_z=True, alpha=1.25, beta=-0.75, ints=False):
    ld = n if ld is None else ld
    if ints:
        X = inputgen.integers(seed, 1, (m, ld), -2, 2, np.float32)
        y = inputgen.integers(seed, 2, n, -2, 2, np.float32)
        v = inputgen.integers(seed, 3, m, -2, 2, np.float32) if with_v else None
        z = inputgen.integers(seed, 4, n, -2, 2, np.float32) if with_z else None
    else:
        X = inputgen.round_to_bf16(inputgen.uniform(seed, 1, (m, ld), -1.0, 1.0, np.float32))
        y = inputgen.uniform(seed, 2, n, -1.0, 1.0, np.float32)
        v = inputgen.uniform(seed, 3, m, -1.0, 1.0, np.float32) if with_v else None
        z = inputgen.uniform(seed, 4, n, -1.0, 1.0, np.float32) if with_z else None
    return inputgen.Problem(f"bf16_{m}x{n}_ld{ld}", "dense", np.float32, m, n, alpha, beta, y=y, v=v, z=z, X=X,
                            ld=ld, x_store="bf16")


def check(p, acc="ld"):
    got = run_problem(p)
    ref, S = oracle.solve(p, acc=acc)
    assert_within_bound(got, ref, S, 2e-5, p.name)


@pytest.mark.parametrize("n", [1, 8, 16, 31, 32, 33, 48, 64, 100, 128, 200, 256, 500, 512])
def test_shapes(n):
    for m in (1, 37, 3001):
        check(make_bf16(m, n, seed=n + m))


@pytest.mark.parametrize("n,ld", [(32, 40), (64, 72), (30, 32), (100, 104), (256, 264)])
def test_leading_dimension(n, ld):
    check(make_bf16(2000, n, ld=ld, seed=ld))


@pytest.mark.parametrize("variant", ["a", "b", "c"])
def test_tall_recipe_scaled(variant):
    check(inputgen.dense_tall(m=300_000, variant=variant, x_store="bf16"))


@pytest.mark.parametrize("m,n", [(50_000, 32), (3000, 256)])
def test_integer_inputs_are_exact(m, n):
    p = make_bf16(m, n, ints=True, alpha=2.0, beta=-1.0, seed=m)
    got = run_problem(p)
    ref, _ = oracle.solve(p)
    assert np.abs(ref).max() < 2 ** 24
    assert np.array_equal(got, ref)


def test_unaligned_and_too_wide():
    p = make_bf16(3000, 32, seed=5)
    ref, S = oracle.solve(p)
    big = torch.zeros(p.m * p.n + 1, dtype=torch.bfloat16, device="cuda")
    big[1:] = torch.from_numpy(p.X.ravel()).cuda().to(torch.bfloat16)
    X = big[1:].view(p.m, p.n)  # 2-byte offset: the direct-load path
    out = fx.dense(X, torch.from_numpy(p.y).cuda(), torch.from_numpy(p.v).cuda(), p.alpha, p.beta,
                   torch.from_numpy(p.z).cuda())
    assert_within_bound(out.cpu().numpy(), ref, S, 2e-5)
    with pytest.raises(fx.FxtxError) as ei:
        fx.dense(torch.zeros(4, 600, dtype=torch.bfloat16, device="cuda"), torch.zeros(600, device="cuda"))
    assert ei.value.status == fx.FXTX_ERR_UNSUPPORTED


def test_matches_fp32_path_on_same_values():
    """The same (bfloat16-representable) X through the fp32 and bfloat16 entry points."""
    p = make_bf16(100_000, 32, seed=9)
    Xf = torch.from_numpy(p.X).cuda()
    args = (torch.from_numpy(p.y).cuda(), torch.from_numpy(p.v).cuda(), p.alpha, p.beta, torch.from_numpy(p.z).cuda())
    a = fx.dense(Xf, *args)
    b = fx.dense(Xf.to(torch.bfloat16), *args)
    ref, S = oracle.solve(p)
    assert_within_bound(a.cpu().numpy(), ref, S, 2e-5)
    assert_within_bound(b.cpu().numpy(), ref, S, 2e-5)


@pytest.mark.slow
def test_full_size_tall_bf16():
    """16,000,000 x 32 with X in bfloat16, every column against the oracle (double accumulator)."""
    check(inputgen.dense_tall(variant="b", x_store="bf16"), acc="d")
