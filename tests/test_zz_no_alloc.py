"""fxtx_dense_f32_noalloc: the dense fp32 call for callers that cannot allocate device
memory while they run (their memory belongs to another allocator, or their loop
forbids allocation after start-up). It keeps its scratch in one library-wide
device array instead of the stream-ordered pool.

Collected last on purpose, and written to pass both alone in a fresh process and
after every other test: the first call on the device performs the one-time look-up
of the scratch array's address.
"""
import numpy as np
import pytest
import torch

import dense_linear_algebra_gb300 as fx
import inputgen
import oracle
from _gpu import DeviceProblem
from _util import assert_within_bound

pytestmark = pytest.mark.gpu

SCRATCH = 1 << 20  # FXTX_NOALLOC_SCRATCH_BYTES


def _noalloc(dp, out):
    p = dp.p
    X = dp.X
    stream = torch.cuda.current_stream().cuda_stream
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    return fx.fxtx_dense_f32_noalloc(p.m, p.n, X.data_ptr(), X.stride(0), ptr(dp.y), ptr(dp.v), p.alpha, p.beta,
                                     ptr(dp.z), out.data_ptr(), stream)


def _check_two_calls(p):
    """Two calls in a row (sharing the scratch array) against the oracle, and against the allocating entry."""
    dp = DeviceProblem(p)
    ref, S = oracle.solve(p, acc="d")
    alloc = dp.run().cpu().numpy().astype(np.float64)
    for call in range(2):
        out = torch.full((p.n,), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(dp, out) == fx.FXTX_OK
        torch.cuda.synchronize()
        got = out.cpu().numpy().astype(np.float64)
        assert_within_bound(got, ref, S, 2e-5, f"noalloc call {call} against the oracle")
        assert_within_bound(got, alloc, S, 4e-5, f"noalloc call {call} against fxtx_dense_f32")
    assert fx.device_error() == fx.FXTX_OK


@pytest.mark.parametrize("m,n,variant", [(1_000_000, 32, "b"), (200_000, 32, "c"), (50_000, 100, "a")])
def test_noalloc_matches_oracle(m, n, variant):
    _check_two_calls(inputgen.dense_tall(m=m, n=n, variant=variant))


def test_noalloc_capped_grid_matches_oracle():
    """Rows of 500 columns with pitch 501 take the direct-load narrow kernel, whose planned grid holds
    more CTA partials than the scratch array: the entry point caps the grid to fit."""
    m, n, ld = 200_000, 500, 501
    X = inputgen.normal(0, 1, (m, ld), np.float32)
    p = inputgen.Problem("dense_f32_%dx%d_ld%d" % (m, n, ld), "dense", np.float32, m, n, 2.0, -1.0,
                         X=X, ld=ld, y=inputgen.normal(0, 2, n, np.float32),
                         v=inputgen.uniform(0, 3, m, 0.1, 2.0, np.float32), z=inputgen.normal(0, 4, n, np.float32))
    plan = dict(kv.split("=") for kv in fx.plan_describe("dense", "f32", m, n, 0, ld).split()[1:] if "=" in kv)
    assert plan["kind"] == "narrow_direct"
    assert int(plan["ctas"]) * n * 8 > SCRATCH - 256, "the planned grid must exceed the scratch, so the cap fires"
    _check_two_calls(p)


def test_noalloc_rejects_rows_beyond_its_scratch():
    X = torch.zeros(8, 600, dtype=torch.float32, device="cuda")
    y = torch.zeros(600, dtype=torch.float32, device="cuda")
    out = torch.zeros(600, dtype=torch.float32, device="cuda")
    rc = fx.fxtx_dense_f32_noalloc(8, 600, X.data_ptr(), 600, y.data_ptr(), None, 1.0, 0.0, None, out.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    assert rc == fx.FXTX_ERR_TOO_LARGE
    assert "FXTX_ERR_TOO_LARGE" in fx.fxtx_status_string(rc)
