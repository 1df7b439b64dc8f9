"""The row-sharded split without a GPU: the row partition, the CSR rebase, and the
sum of the ranks' partials on two and three gloo ranks. Each rank's partial
w_g = X_g^T (v_g * (X_g y)) comes from the oracle here (test-side only); the ranks
sum them with one all-reduce and finish with alpha * w + beta * z. On integer-valued
inputs every partial and every sum is exact, so the split must equal the unsplit
oracle bitwise; on real-valued inputs it must meet the fp64 bound."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import inputgen
import oracle
from _util import assert_within_bound, dense_to_csr
from dense_linear_algebra_gb300 import distributed as sp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.mark.parametrize("m,world", [(10, 3), (7, 7), (3, 5), (0, 2), (1000, 8)])
def test_dense_bounds_cover_every_row_once(m, world):
    b = sp.row_bounds(m, world)
    assert b[0] == 0 and b[-1] == m and len(b) == world + 1
    assert all(b[g] <= b[g + 1] for g in range(world))
    sizes = np.diff(b)
    assert sizes.max() - sizes.min() <= 1


def test_csr_bounds_balance_entries():
    p = inputgen.csr_powerlaw(m=20_000, n=5_000)
    for world in (2, 3, 8):
        b = sp.row_bounds(p.m, world, p.row_ptr)
        assert b[0] == 0 and b[-1] == p.m and all(b[g] <= b[g + 1] for g in range(world))
        cost = p.row_ptr + sp.CSR_ROW_COST * np.arange(p.m + 1)
        share = np.diff(cost[b])
        longest = int(np.diff(p.row_ptr).max()) + sp.CSR_ROW_COST
        # every block is within one row of an equal share of nnz + 8 * rows
        assert np.all(np.abs(share - cost[-1] / world) <= longest)


def test_csr_bounds_with_empty_rows_and_more_ranks_than_rows():
    rp = np.array([0, 0, 0, 5, 5], np.int64)
    b = sp.row_bounds(4, 6, rp)
    assert b[0] == 0 and b[-1] == 4 and all(b[g] <= b[g + 1] for g in range(6))
    with pytest.raises(ValueError):
        sp.row_bounds(3, 2, rp)


def test_csr_rebase_reassembles_the_matrix():
    p = inputgen.csr_uniform(m=3_001, n=700, lam=9.0)
    b = sp.row_bounds(p.m, 4, p.row_ptr)
    shards = [sp.shard_csr(p.row_ptr, p.col_idx, p.vals, p.v, p.n, b, g) for g in range(4)]
    for s in shards:
        assert s.row_ptr[0] == 0 and s.row_ptr[-1] == s.col_idx.shape[0] == s.vals.shape[0]
        assert s.row_ptr.shape[0] == s.rows + 1 and s.v.shape[0] == s.rows
    assert np.array_equal(np.concatenate([s.col_idx for s in shards]), p.col_idx)
    assert np.array_equal(np.concatenate([s.vals for s in shards]), p.vals)
    assert np.array_equal(np.concatenate([s.v for s in shards]), p.v)
    lens = np.concatenate([np.diff(s.row_ptr) for s in shards])
    assert np.array_equal(lens, np.diff(p.row_ptr))


def _integer_problem(kind, m=300, n=40, seed=3):
    rng = np.random.default_rng(seed)
    X = rng.integers(-2, 3, (m, n)).astype(np.float64)
    X[rng.random((m, n)) < 0.6] = 0.0
    X[5] = 0.0  # an empty row
    y = rng.integers(-2, 3, n).astype(np.float64)
    v = rng.integers(-2, 3, m).astype(np.float64)
    z = rng.integers(-2, 3, n).astype(np.float64)
    return X, y, v, z


def _oracle_partial(shard, y):
    """The rank's w_g from the oracle (alpha = 1, beta = 0)."""
    if shard.kind == "dense":
        w, _ = oracle.dense(shard.X, y, shard.v, 1.0, 0.0, None)
    else:
        w, _ = oracle.csr(shard.row_ptr, shard.col_idx, shard.vals, y, shard.v, 1.0, 0.0, None, shard.n)
    return torch.from_numpy(w)


def _cpu_epilogue(w, alpha, beta, z):
    return alpha * w + (beta * torch.from_numpy(z) if z is not None and beta != 0 else 0.0)


@pytest.mark.parametrize("kind", ["dense", "csr"])
@pytest.mark.parametrize("world", [1, 2, 5])
def test_sum_of_block_partials_is_the_pattern(kind, world):
    """Single process: the partials of all blocks, summed and finished, equal the unsplit oracle."""
    X, y, v, z = _integer_problem(kind)
    alpha, beta = 2.0, -0.5
    ref, _ = oracle.dense(X, y, v, alpha, beta, z)
    if kind == "dense":
        b = sp.row_bounds(X.shape[0], world)
        shards = [sp.shard_dense(X, v, b, g) for g in range(world)]
    else:
        rp, ci, vals = dense_to_csr(X)
        b = sp.row_bounds(X.shape[0], world, rp)
        shards = [sp.shard_csr(rp, ci, vals, v, X.shape[1], b, g) for g in range(world)]
    w = sum(_oracle_partial(s, y) for s in shards)
    out = _cpu_epilogue(w, alpha, beta, z).numpy()
    assert np.array_equal(out, ref)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, kind, exact, results):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        if exact:
            X, y, v, z = _integer_problem(kind)
            alpha, beta = 2.0, -0.5
            rp = ci = vals = None
            if kind == "csr":
                rp, ci, vals = dense_to_csr(X)
        else:
            p = inputgen.csr_uniform(m=5_000, n=300, lam=12.0) if kind == "csr" else inputgen.dense_small(m=999)
            y, v, z, alpha, beta = p.y, p.v, p.z, p.alpha, p.beta
            X = p.X[:, : p.n] if kind == "dense" else None
            rp, ci, vals = (p.row_ptr, p.col_idx, p.vals) if kind == "csr" else (None, None, None)
        m = X.shape[0] if X is not None else rp.shape[0] - 1
        n = y.shape[0]
        if kind == "dense":
            shard = sp.shard_dense(X, v, sp.row_bounds(m, world), rank)
        else:
            shard = sp.shard_csr(rp, ci, vals, v, n, sp.row_bounds(m, world, rp), rank)
        out = sp.sharded_call(shard, y, alpha, beta, z, partial_fn=_oracle_partial, epilogue=_cpu_epilogue)
        if kind == "dense":
            ref, S = oracle.dense(X, y, v, alpha, beta, z)
        else:
            ref, S = oracle.csr(rp, ci, vals, y, v, alpha, beta, z, n)
        results[rank] = (out.numpy(), ref, S, shard.rows)
    finally:
        dist.barrier()
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("kind", ["dense", "csr"])
@pytest.mark.parametrize("exact", [True, False], ids=["integer", "real"])
def test_gloo_ranks_reproduce_the_unsplit_call(world, kind, exact):
    mgr = mp.Manager()
    results = mgr.dict()
    mp.spawn(_rank, args=(world, _free_port(), kind, exact, results), nprocs=world, join=True)
    rows = 0
    for rank in range(world):
        out, ref, S, r = results[rank]
        rows += r
        if exact:
            assert np.array_equal(out, ref), f"rank {rank}: the split differs from the unsplit oracle"
        else:
            assert_within_bound(out, ref, S, 1e-12, f"rank {rank}")
    m = 300 if exact else (5_000 if kind == "csr" else 999)
    assert rows == m
