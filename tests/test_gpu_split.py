"""The row-sharded split on one GPU: the blocks' partials w_g come from the fused
kernels (alpha = 1, beta = 0), are summed (standing in for the all-reduce of a
multi-GPU run; the blocks run one after another, never waiting on each other) and
finished by the epilogue kernel. The result must meet the oracle's bound for the
whole matrix."""
import numpy as np
import pytest
import torch

import dense_linear_algebra_gb300 as fx
import inputgen
import oracle
from _gpu import to_dev
from _util import assert_within_bound, rel_for
from dense_linear_algebra_gb300 import distributed as sp

pytestmark = pytest.mark.gpu


def _split_on_one_gpu(p, world):
    y, v, z = to_dev(p.y), to_dev(p.v), to_dev(p.z)
    if p.kind == "dense":
        X = to_dev(p.X)[:, : p.n]
        b = sp.row_bounds(p.m, world)
        shards = [sp.shard_dense(X, v, b, g) for g in range(world)]
    else:
        rp, ci, vals = to_dev(p.row_ptr), to_dev(p.col_idx), to_dev(p.vals)
        b = sp.row_bounds(p.m, world, p.row_ptr)
        shards = [sp.shard_csr(rp, ci, vals, v, p.n, b, g) for g in range(world)]
    w = None
    for s in shards:
        part = sp.partial(s, y)
        w = part if w is None else w + part
    out = sp.reduce_and_finish(w, p.alpha, p.beta, z)
    torch.cuda.synchronize()
    assert fx.device_error() == fx.FXTX_OK
    return out.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("world", [1, 2, 3, 8])
@pytest.mark.parametrize("make", [
    lambda: inputgen.dense_tall(m=300_001, variant="b"),
    lambda: inputgen.dense_small(m=5_000),
    lambda: inputgen.dense_wide(m=257, n=3_000),
    lambda: inputgen.csr_uniform(m=40_000, n=2_000, lam=30.0),
    lambda: inputgen.csr_powerlaw(m=30_000, n=20_000),
], ids=["dense_f32", "dense_f64", "wide_f64", "csr_f64", "csr_f32_powerlaw"])
def test_split_matches_oracle(make, world):
    p = make()
    got = _split_on_one_gpu(p, world)
    ref, S = oracle.solve(p)
    # a few extra roundings (each block's partial, their sum) on top of one call's bound
    assert_within_bound(got, ref, S, 2 * rel_for(p.dtype), f"{p.name} split in {world}")


@pytest.mark.parametrize("dtype", [np.float32, np.float64])
def test_epilogue_kernel(dtype):
    rng = np.random.default_rng(11)
    n = 100_003
    w = rng.standard_normal(n).astype(dtype)
    z = rng.standard_normal(n).astype(dtype)
    for alpha, beta, use_z in [(1.5, -0.25, True), (2.0, 0.0, True), (0.7, 3.0, False), (0.0, 1.0, True)]:
        out = fx.epilogue(to_dev(w), alpha, beta, to_dev(z) if use_z else None)
        torch.cuda.synchronize()
        a, b = float(np.asarray(alpha, dtype)), float(np.asarray(beta, dtype))
        ref = a * w.astype(np.float64) + (b * z.astype(np.float64) if use_z and beta != 0 else 0.0)
        got = out.cpu().numpy().astype(np.float64)
        # a few roundings in the working type on either side (an fp64 FMA may fuse the sum)
        tol = 2 * np.finfo(dtype).eps * (np.abs(a * w) + np.abs(b * z)) + 1e-300
        assert np.all(np.abs(got - ref) <= tol)
    # in place, z not read at beta = 0 (a NaN there does not reach out)
    wd = to_dev(w)
    zn = torch.full((n,), float("nan"), dtype=wd.dtype, device="cuda")
    fx.epilogue(wd, 2.0, 0.0, zn, out=wd)
    torch.cuda.synchronize()
    assert np.array_equal(wd.cpu().numpy(), (2.0 * w.astype(np.float64)).astype(dtype))


def test_epilogue_rejects_bad_arguments():
    w = torch.zeros(8, dtype=torch.float32, device="cuda")
    assert fx.fxtx_epilogue_f32(-1, w.data_ptr(), 1.0, 0.0, None, w.data_ptr(), None) == fx.FXTX_ERR_INVALID_ARG
    assert fx.fxtx_epilogue_f32(8, None, 1.0, 0.0, None, w.data_ptr(), None) == fx.FXTX_ERR_INVALID_ARG
    assert fx.fxtx_epilogue_f64(0, None, 1.0, 0.0, None, None, None) == fx.FXTX_OK
    with pytest.raises(ValueError):
        fx.epilogue(w, 1.0, 1.0, torch.zeros(8, dtype=torch.float64, device="cuda"))
