"""The C ABI without a GPU: the library loads, exports every declared entry point,
rejects bad arguments before touching a device, and its launch model picks the
expected variants."""
import ctypes
import os
import re

import pytest

import dense_linear_algebra_gb300 as fx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(fxtx_\w+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported():
    names = _declared()
    assert "fxtx_dense_f32" in names and "fxtx_csr_f64" in names
    lib = ctypes.CDLL(fx.library_path)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings():
    for code in range(7):
        s = fx.fxtx_status_string(code)
        assert s.startswith("FXTX_")
    assert "unknown" in fx.fxtx_status_string(99)


def test_invalid_arguments_rejected_on_host():
    # negative sizes, ld < n, missing pointers: refused before any device work
    assert fx.fxtx_dense_f32(-1, 4, None, 4, None, None, 1.0, 0.0, None, None, None) == fx.FXTX_ERR_INVALID_ARG
    assert fx.fxtx_dense_f64(4, 8, 16, 4, 16, None, 1.0, 0.0, None, 16, None) == fx.FXTX_ERR_INVALID_ARG
    assert fx.fxtx_dense_f64(4, 8, None, 8, 16, None, 1.0, 0.0, None, 16, None) == fx.FXTX_ERR_INVALID_ARG
    assert fx.fxtx_dense_f32(4, 8, 16, 8, None, None, 1.0, 0.0, None, 16, None) == fx.FXTX_ERR_INVALID_ARG
    assert fx.fxtx_csr_f32(4, 8, -1, None, None, None, None, None, 1.0, 0.0, None, None, None) == fx.FXTX_ERR_INVALID_ARG
    assert fx.fxtx_csr_f64(4, 8, 3, 16, None, 16, 16, None, 1.0, 0.0, None, 16, None) == fx.FXTX_ERR_INVALID_ARG
    assert fx.fxtx_csr_f64(4, 8, 0, None, None, None, 16, None, 1.0, 0.0, None, 16, None) == fx.FXTX_ERR_INVALID_ARG
    # n == 0 is a no-op that succeeds without a device
    assert fx.fxtx_dense_f32(5, 0, None, 1, None, None, 1.0, 0.0, None, None, None) == fx.FXTX_OK
    assert fx.fxtx_csr_f32(5, 0, 0, None, None, None, None, None, 1.0, 0.0, None, None, None) == fx.FXTX_OK
    # an empty CSR structure without row_ptr is valid
    assert fx.fxtx_csr_validate(0, 3, 0, None, None, None) == fx.FXTX_OK
    assert fx.fxtx_csr_validate(0, 3, 2, None, None, None) == fx.FXTX_ERR_BAD_CSR


def test_no_device_is_reported_as_unsupported():
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert fx.fxtx_dense_f32(4, 8, 16, 8, 16, None, 1.0, 0.0, None, 16, None) == fx.FXTX_ERR_UNSUPPORTED


@pytest.mark.parametrize(
    "args,expect",
    [
        (("dense", "f32", 16_000_000, 32), "kind=tile_tma lanes_per_row=2 chunks_per_lane=4 rows_per_tile=64"),
        (("dense", "f64", 1000, 64), "kind=tile_tma lanes_per_row=8 chunks_per_lane=4 rows_per_tile=16"),
        (("dense", "f32", 1000, 512), "kind=tile_tma lanes_per_row=32 chunks_per_lane=4 rows_per_tile=8"),
        (("dense", "f32", 1000, 8), "kind=tile_tma lanes_per_row=1 chunks_per_lane=4 rows_per_tile=128"),
        (("dense", "f32", 1000, 16), "box=64"),
        (("dense", "f32", 1000, 4), "kind=narrow_tma lanes_per_row=1 chunks_per_lane=1 rows_per_tile=32"),
        (("dense", "f64", 20_000, 20_000), "kind=wide"),
        (("dense", "f32", 10, 3), "kind=narrow_direct"),
        (("dense", "f32", 0, 3), "kind=empty_rows"),
        (("csr", "f64", 4_000_000, 10_000, 200_000_000), "csr group_lanes=8 pack_k=4 pack_cap=128 warp_cap=1024 ctas=152"),
        (("csr", "f32", 2_000_000, 1_000_000, 200_000_000), "window=[0,+"),
    ],
)
def test_launch_model(args, expect):
    desc = fx.plan_describe(*args)
    assert expect in desc, desc


def test_launch_model_grid_and_smem_limits():
    d = fx.plan_describe("dense", "f32", 16_000_000, 32)
    fields = dict(kv.split("=") for kv in d.split()[1:])
    # one CTA per SM; at least 128 KB of X in flight per SM; within the shared-memory limit
    assert int(fields["ctas"]) == 152 and int(fields["warps"]) * int(fields["stages"]) * 8192 >= 128 * 1024
    assert int(fields["smem"]) <= 227 * 1024
    d = fx.plan_describe("dense", "f32", 100, 32)  # few rows: a CTA per few tiles
    fields = dict(kv.split("=") for kv in d.split()[1:])
    assert int(fields["ctas"]) == 1
