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


def test_binding_rejects_host_tensors():
    """The torch binding hands only device pointers to the library: host tensors, wrong
    dtypes and wrong lengths are refused in Python, before any C call."""
    import torch

    X, y = torch.zeros(8, 4), torch.zeros(4)
    with pytest.raises(ValueError):
        fx.dense(X, y)
    with pytest.raises(ValueError):
        fx.dense_multi(X, torch.zeros(4, 2))
    rp, ci, va = torch.zeros(9, dtype=torch.int64), torch.zeros(0, dtype=torch.int32), torch.zeros(0)
    with pytest.raises(ValueError):
        fx.csr(rp, ci, va, y, 4)
    with pytest.raises(ValueError):
        fx.csr_validate(rp, ci, 4)
    with pytest.raises(ValueError):
        fx.csr(rp.view(3, 3), ci, va, y, 4)


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
        (("csr", "f64", 4_000_000, 10_000, 200_000_000), "csr group_lanes=4 group_entries=16 pack_k=4 pack_cap=128 warp_cap=2048 ctas=152"),
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


@pytest.mark.parametrize(
    "args,expect",
    [
        (("f32", 16_000_000, 32, 8), "tma=1 tc=1 blocks=1 kb=8 passes=1 rows_per_tile=128 stages=6 warps=20 ctas=152"),
        (("f32", 16_000_000, 32, 4), "tma=1 tc=0 blocks=1 kb=4 passes=1 rows_per_tile=64"),
        (("f32", 16_000_000, 32, 16), "tc=1 blocks=1 kb=16 passes=1"),
        (("f64", 16_000_000, 32, 8), "tc=0"),
        (("f32", 1000, 33, 8), "tc=0"),
        (("f32", 16_000_000, 32, 1), "kb=1 passes=1 rows_per_tile=32 stages=6"),
        (("f32", 16_000_000, 32, 40), "kb=32 passes=2"),
        (("f32", 1000, 32, 3), "kb=4 passes=1"),
        (("f64", 1000, 128, 8, "shared"), "blocks=8 kb=4 passes=2 rows_per_tile=8"),
        (("f32", 1000, 512, 8, "none"), "blocks=16 kb=2 passes=4 rows_per_tile=8 stages=3 warps=4"),
        (("f32", 1000, 513, 8), "ok=0"),
        (("f64", 0, 17, 8), "tma=0"),
        (("f32", 1000, 32, 8, "full", 33), "tma=0 tc=0 blocks=1 kb=8"),
    ],
)
def test_multi_launch_model(args, expect):
    desc = fx.multi_plan_describe(*args)
    assert expect in desc, desc


def test_multi_plans_fit_shared_memory():
    """Every shape the multi-vector entry takes plans within the 227 KB per-CTA limit,
    with at least two pipeline stages when tensor copies stage X."""
    for dt, elem in (("f32", 4), ("f64", 8)):
        for n in (1, 16, 17, 32, 33, 64, 65, 128, 129, 256, 257, 512):
            if n * elem > 2048:
                continue
            for k in (1, 3, 8, 16, 32, 33, 100):
                for vm in ("none", "shared", "full"):
                    f = dict(kv.split("=") for kv in fx.multi_plan_describe(dt, 10**6, n, k, vm).split()[1:])
                    assert f["ok"] == "1" and int(f["smem"]) <= 227 * 1024, (dt, n, k, vm, f)
                    tma = (n * elem) % 16 == 0  # ld = n: a 16-byte pitch is needed for tensor copies
                    assert f["tma"] == ("1" if tma else "0") and int(f["stages"]) >= (2 if tma else 1)
                    kb = int(f["kb"])
                    assert kb & (kb - 1) == 0 and kb * int(f["blocks"]) <= 32
                    assert int(f["passes"]) == -(-k // kb)


def test_multi_invalid_arguments_rejected_on_host():
    m32 = fx.fxtx_dense_multi_f32
    assert m32(-1, 4, 2, None, 4, None, 2, None, 0, 1.0, 0.0, None, 0, None, 2, None) == fx.FXTX_ERR_INVALID_ARG
    assert m32(4, 4, 2, 16, 4, 16, 1, None, 0, 1.0, 0.0, None, 0, 16, 2, None) == fx.FXTX_ERR_INVALID_ARG  # ldy < k
    assert m32(4, 4, 2, 16, 4, 16, 2, None, 0, 1.0, 0.0, None, 0, 16, 1, None) == fx.FXTX_ERR_INVALID_ARG  # ldo < k
    assert m32(4, 4, 2, 16, 4, 16, 2, 16, 1, 1.0, 0.0, None, 0, 16, 2, None) == fx.FXTX_ERR_INVALID_ARG  # 0 < ldv < k
    assert m32(4, 4, 2, 16, 4, 16, 2, None, 0, 1.0, 1.0, 16, 1, 16, 2, None) == fx.FXTX_ERR_INVALID_ARG  # ldz < k
    assert fx.fxtx_dense_multi_f64(4, 8, 2, None, 8, 16, 2, None, 0, 1.0, 0.0, None, 0, 16, 2, None) == fx.FXTX_ERR_INVALID_ARG
    assert m32(4, 0, 2, None, 1, None, 2, None, 0, 1.0, 0.0, None, 0, None, 2, None) == fx.FXTX_OK  # n == 0
    assert m32(4, 4, 0, None, 4, None, 0, None, 0, 1.0, 0.0, None, 0, None, 0, None) == fx.FXTX_OK  # k == 0


def test_multi_tensor_core_estimate():
    """The tensor-core form's estimate: never below the HBM time of its bytes (X and an m x k
    V once, at 6.8 TB/s), and rising with the right-hand sides a pass takes."""
    est = {}
    for k in (8, 16, 32):
        f = dict(kv.split("=") for kv in fx.multi_plan_describe("f32", 16_000_000, 32, k, "full").split()[1:])
        assert f["tc"] == "1"
        est[k] = float(f["est_us"])
        hbm_us = (16_000_000 * 32 * 4 + 16_000_000 * k * 4) / 6.8e12 * 1e6
        assert est[k] >= hbm_us, (k, est[k], hbm_us)
    assert est[8] < est[16] < est[32]


@pytest.mark.parametrize("args,tc", [
    (("f32", 1_000_000, 32, 7), "0"), (("f32", 1_000_000, 32, 8), "1"),
    (("f32", 1_000_000, 33, 8), "0"), (("f32", 1_000_000, 4, 8), "1"), (("f32", 1_000_000, 1, 8), "0"),
    (("f64", 1_000_000, 16, 8), "0"), (("f32", 1_000_000, 32, 100), "1"),
    (("f32", 1_000_000, 32, 8, "full", 33), "0"),  # a pitch tensor copies cannot take
])
def test_multi_tensor_core_choice(args, tc):
    f = dict(kv.split("=") for kv in fx.multi_plan_describe(*args).split()[1:])
    assert f["tc"] == tc, (args, f)


def test_multi_tensor_core_switch():
    """FXTX_MULTI_TC=0, read when the library first plans such a call, keeps the shapes the
    tensor cores would take on the CUDA-core kernel."""
    import subprocess
    import sys

    code = ("import dense_linear_algebra_gb300 as fx; "
            "print(fx.multi_plan_describe('f32', 1000000, 32, 8, 'full'))")
    env = dict(os.environ, FXTX_MULTI_TC="0")
    out = subprocess.run([sys.executable, "-c", code], env=env, cwd=ROOT, capture_output=True, text=True,
                         timeout=300)
    assert out.returncode == 0, out.stderr
    assert " tc=0 " in out.stdout, out.stdout
