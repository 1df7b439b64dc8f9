"""The data-aware CSR plan on the GPU: the per-call device-side placement of the shared
windows, the analysed (host-sampled) plan, and their parity with the oracle on a
power-law matrix whose hot columns sit mid-range."""
import numpy as np
import pytest
import torch

import dense_linear_algebra_gb300 as fx
import inputgen
import oracle
from _gpu import DeviceProblem
from _util import assert_within_bound, rel_for

pytestmark = pytest.mark.gpu


def _run(dp):
    out = dp.run()
    torch.cuda.synchronize()
    assert fx.device_error() == fx.FXTX_OK
    return out.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("offset", [0, 333_333, 990_000])
@pytest.mark.parametrize("analysed", [False, True], ids=["device_placement", "analysed"])
def test_rotated_powerlaw_parity(offset, analysed):
    p = inputgen.csr_powerlaw(m=150_000, n=1_000_000, col_offset=offset)
    dp = DeviceProblem(p)
    fx.csr_analysis_clear()
    if analysed:
        st = fx.csr_analyze(dp.row_ptr, dp.col_idx, p.n, "f32")
        assert st["window_c0"] <= offset < st["window_c0"] + st["window_len"] or offset == 0
    ref, S = oracle.solve(p)
    assert_within_bound(_run(dp), ref, S, rel_for(p.dtype), f"{p.name} analysed={analysed}")
    fx.csr_analysis_clear()


def test_device_sample_equals_host_sample():
    """fxtx_csr_analyze gathers its sample on the device; the host model samples the same
    positions of host arrays: the statistics must agree exactly."""
    for p, dt in ((inputgen.csr_powerlaw(m=120_000, n=700_000, col_offset=123_456), "f32"),
                  (inputgen.csr_uniform(m=300_000, n=10_000), "f64"),
                  (inputgen.csr_uniform(m=3_000, n=500, lam=4.0), "f64")):
        dp = DeviceProblem(p)
        dev = fx.csr_analyze(dp.row_ptr, dp.col_idx, p.n, dt)
        _, host = fx.csr_plan_describe_host(p.row_ptr, p.col_idx, p.n, dt)
        assert dev == host, (p.name, dev, host)
    fx.csr_analysis_clear()


@pytest.mark.parametrize("make", [
    lambda: inputgen.csr_uniform(m=200_000, n=10_000),
    lambda: inputgen.csr_uniform(m=100_000, n=300_000, lam=30.0),
], ids=["uniform_f64_whole_window", "uniform_f64_wide"])
def test_analysed_fp64_parity(make):
    p = make()
    dp = DeviceProblem(p)
    fx.csr_analysis_clear()
    fx.csr_analyze(dp.row_ptr, dp.col_idx, p.n, "f64")
    ref, S = oracle.solve(p)
    assert_within_bound(_run(dp), ref, S, rel_for(p.dtype), p.name)
    fx.csr_analysis_clear()
    assert_within_bound(_run(dp), ref, S, rel_for(p.dtype), p.name + " (analysis cleared)")


def test_analyze_edge_cases():
    rp = torch.zeros(1, dtype=torch.int64, device="cuda")
    ci = torch.zeros(0, dtype=torch.int32, device="cuda")
    st = fx.csr_analyze(rp, ci, 5, "f32")
    assert st["row_samples"] == 0 and st["col_samples"] == 0
    rp = torch.tensor([0, 2, 2, 5], dtype=torch.int64, device="cuda")
    ci = torch.tensor([0, 4, 1, 2, 3], dtype=torch.int32, device="cuda")
    st = fx.csr_analyze(rp, ci, 5, "f32")
    assert st["row_samples"] == 3 and st["col_samples"] == 5 and st["max_sampled_row_len"] == 3
    with pytest.raises(ValueError):
        fx.csr_analyze(rp.to(torch.int32), ci, 5)
    fx.csr_analysis_clear()
