"""The launch model's candidates and the autotune cache, without a GPU: candidate lists,
the mode switch, and the cache file's round trip and validation."""
import os

import pytest

import dense_linear_algebra_gb300 as fx


@pytest.fixture(autouse=True)
def _restore():
    mode = fx.autotune_mode()
    yield
    fx.autotune_clear()
    fx.autotune(mode)


@pytest.mark.parametrize("args", [("dense", "f32", 16_000_000, 32), ("dense", "f64", 1000, 64),
                                  ("dense", "f64", 20_000, 20_000), ("csr", "f32", 2_000_000, 1_000_000, 200_000_000),
                                  ("csr", "f64", 4_000_000, 10_000, 200_000_000)])
def test_candidates_start_with_the_model_and_fit(args):
    c = fx.autotune_candidates(*args)
    assert c[0] == fx.plan_describe(*args)
    assert len(c) == len(set(c)) and len(c) >= 2
    for d in c:
        f = dict(kv.split("=") for kv in d.split()[1:] if "=" in kv)
        assert int(f["smem"]) <= 227 * 1024
        assert float(f["est_us"]) > 0


def test_model_estimates_are_rooflines():
    """The tall fp32 workload: 2.112 GB at 99 % of 6.8 TB/s plus the fixed call cost."""
    d = fx.plan_describe("dense", "f32", 16_000_000, 32)
    est = float(dict(kv.split("=") for kv in d.split()[1:])["est_us"])
    assert abs(est - (2_112_000_384 / (6.8e12 * 0.99) * 1e6 + 4.0)) < 1.0
    # the fp64 wide workload is bound by its 8e8 fp64 FMAs at 2 per SM and clock (70 % of that rate)
    d = fx.plan_describe("dense", "f64", 20_000, 20_000)
    est = float(dict(kv.split("=") for kv in d.split()[1:])["est_us"])
    assert abs(est - (2 * 20_000 ** 2 / (2 * 152 * 2.07e9 * 0.7) * 1e6 + 4.0)) < 1.0


def test_csr_fp64_estimate_is_fma_bound():
    """The uniform fp64 CSR workload: 4e8 fp64 FMAs at 45 % of 2 per SM and clock."""
    d = fx.plan_describe("csr", "f64", 4_000_000, 10_000, 200_000_000)
    est = float(dict(kv.split("=") for kv in d.split()[1:] if "=" in kv)["est_us"])
    assert abs(est - (2 * 200_000_000 / (2 * 152 * 2.07e9 * 0.45) * 1e6 + 4.0)) < 1.0


def test_mode_switch():
    fx.autotune(1)
    assert fx.autotune_mode() == 1
    fx.autotune(0)
    assert fx.autotune_mode() == 0
    with pytest.raises(fx.FxtxError):
        fx.autotune(2)


def test_cache_file_round_trip(tmp_path):
    src = tmp_path / "tune.txt"
    src.write_text("# comment\n0 4 16000000 32 0 32 3 152 2 6 301.250 330.900\n"
                   "1 8 4000000 10000 200000000 0 0 152 1 3 1500.000 1063.400\n")
    fx.autotune_load(str(src))
    assert fx.autotune_entries() == 2
    out = tmp_path / "out.txt"
    fx.autotune_save(str(out))
    lines = [ln for ln in out.read_text().splitlines() if not ln.startswith("#")]
    assert sorted(lines) == sorted(["0 4 16000000 32 0 32 3 152 2 6 301.250 330.900",
                                    "1 8 4000000 10000 200000000 0 0 152 1 3 1500.000 1063.400"])
    fx.autotune_clear()
    assert fx.autotune_entries() == 0


@pytest.mark.parametrize("bad", ["0 4 100 32 0 32 3 152 7 6 1.0 1.0\n",       # choice >= candidates
                                 "2 4 100 32 0 32 3 152 0 6 1.0 1.0\n",       # unknown kind
                                 "0 4 100 32 0 32 3 152 0 6 1.0\n",           # a field short
                                 "0 4 100 32 0 32 3 152 0 6 1.0 1.0 9\n",     # a field too many
                                 "0 4 -5 32 0 32 3 152 0 6 1.0 1.0\n"])      # negative size
def test_malformed_cache_file_is_refused(tmp_path, bad):
    good = tmp_path / "good.txt"
    good.write_text("0 4 16000000 32 0 32 3 152 2 6 301.250 330.900\n")
    fx.autotune_load(str(good))
    f = tmp_path / "bad.txt"
    f.write_text(bad)
    with pytest.raises(fx.FxtxError):
        fx.autotune_load(str(f))
    assert fx.autotune_entries() == 1  # unchanged
    with pytest.raises(fx.FxtxError):
        fx.autotune_load(str(tmp_path / "missing.txt"))
