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


def _noalloc(dp, out):
    p = dp.p
    X = dp.X
    stream = torch.cuda.current_stream().cuda_stream
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    return fx.fxtx_dense_f32_noalloc(p.m, p.n, X.data_ptr(), X.stride(0), ptr(dp.y), ptr(dp.v), p.alpha, p.beta,
                                     ptr(dp.z), out.data_ptr(), stream)


@pytest.mark.parametrize("m,n,variant", [(1_000_000, 32, "b"), (200_000, 32, "c"), (50_000, 100, "a")])
def test_noalloc_matches_allocating_entry_point(m, n, variant):
    p = inputgen.dense_tall(m=m, n=n, variant=variant)
    dp = DeviceProblem(p)
    ref = dp.run().cpu().numpy().astype(np.float64)  # the allocating entry point
    _, S = oracle.solve(p, acc="d")
    for call in range(2):  # two calls in a row share the same scratch array
        out = torch.full((p.n,), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(dp, out) == fx.FXTX_OK
        torch.cuda.synchronize()
        got = out.cpu().numpy().astype(np.float64)
        assert_within_bound(got, ref, S, 2e-5, f"noalloc call {call}")


def test_noalloc_rejects_rows_beyond_its_scratch():
    X = torch.zeros(8, 600, dtype=torch.float32, device="cuda")
    y = torch.zeros(600, dtype=torch.float32, device="cuda")
    out = torch.zeros(600, dtype=torch.float32, device="cuda")
    rc = fx.fxtx_dense_f32_noalloc(8, 600, X.data_ptr(), 600, y.data_ptr(), None, 1.0, 0.0, None, out.data_ptr(),
                                   torch.cuda.current_stream().cuda_stream)
    assert rc == fx.FXTX_ERR_TOO_LARGE
    assert "FXTX_ERR_TOO_LARGE" in fx.fxtx_status_string(rc)
