"""ctypes binding over libfusedxtx's C ABI (argument marshalling only)."""
from __future__ import annotations

import contextlib
import ctypes
import os

from . import build as _build

FXTX_OK = 0
FXTX_ERR_INVALID_ARG = 1
FXTX_ERR_UNSUPPORTED = 2
FXTX_ERR_CUDA = 3
FXTX_ERR_ALLOC = 4
FXTX_ERR_BAD_CSR = 5
FXTX_ERR_TIMEOUT = 6
FXTX_ERR_TOO_LARGE = 7


class CsrStats(ctypes.Structure):
    """fxtx_csr_stats_t: sampled characteristics of a CSR matrix and the plan figures they lead to."""

    _fields_ = [("row_samples", ctypes.c_int64), ("col_samples", ctypes.c_int64),
                ("mean_row_len", ctypes.c_double), ("cv_row_len", ctypes.c_double),
                ("p50_row_len", ctypes.c_int64), ("p75_row_len", ctypes.c_int64), ("p90_row_len", ctypes.c_int64),
                ("max_sampled_row_len", ctypes.c_int64), ("long_row_share", ctypes.c_double),
                ("window_c0", ctypes.c_int64), ("window_len", ctypes.c_int64),
                ("y_c0", ctypes.c_int64), ("y_len", ctypes.c_int64),
                ("window_hit_share", ctypes.c_double), ("y_hit_share", ctypes.c_double),
                ("group_lanes", ctypes.c_int32), ("group_entries", ctypes.c_int32)]

    def as_dict(self) -> dict:
        return {name: getattr(self, name) for name, _ in self._fields_}


def _load() -> ctypes.CDLL:
    path = _build.LIB
    if not os.path.exists(path) or _build._stale():
        try:
            _build.build()
        except Exception as e:  # no silent fallback: the library is the product
            raise ImportError(f"libfusedxtx could not be built or loaded from {path}: {e}") from e
    lib = ctypes.CDLL(path)
    i32, i64, f32, f64, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double, ctypes.c_void_p
    lib.fxtx_dense_f32.argtypes = [i64, i64, vp, i64, vp, vp, f32, f32, vp, vp, vp]
    lib.fxtx_dense_f64.argtypes = [i64, i64, vp, i64, vp, vp, f64, f64, vp, vp, vp]
    lib.fxtx_dense_f32_noalloc.argtypes = [i64, i64, vp, i64, vp, vp, f32, f32, vp, vp, vp]
    lib.fxtx_dense_bf16.argtypes = [i64, i64, vp, i64, vp, vp, f32, f32, vp, vp, vp]
    lib.fxtx_dense_multi_f32.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, f32, f32, vp, i64, vp, i64, vp]
    lib.fxtx_dense_multi_f64.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, f64, f64, vp, i64, vp, i64, vp]
    lib.fxtx_csr_f32.argtypes = [i64, i64, i64, vp, vp, vp, vp, vp, f32, f32, vp, vp, vp]
    lib.fxtx_csr_f64.argtypes = [i64, i64, i64, vp, vp, vp, vp, vp, f64, f64, vp, vp, vp]
    lib.fxtx_csr_validate.argtypes = [i64, i64, i64, vp, vp, vp]
    lib.fxtx_csr_analyze.argtypes = [i32, i64, i64, i64, vp, vp, vp, ctypes.POINTER(CsrStats)]
    lib.fxtx_csr_analysis_clear.argtypes = []
    lib.fxtx_csr_plan_describe_host.argtypes = [i32, i64, i64, i64, vp, vp, ctypes.POINTER(CsrStats),
                                                ctypes.c_char_p, i64]
    lib.fxtx_epilogue_f32.argtypes = [i64, vp, f32, f32, vp, vp, vp]
    lib.fxtx_epilogue_f64.argtypes = [i64, vp, f64, f64, vp, vp, vp]
    lib.fxtx_device_error.argtypes = [vp]
    lib.fxtx_status_string.argtypes = [i32]
    lib.fxtx_status_string.restype = ctypes.c_char_p
    lib.fxtx_plan_describe.argtypes = [i32, i32, i64, i64, i64, i64, ctypes.c_char_p, i64]
    lib.fxtx_multi_plan_describe.argtypes = [i32, i64, i64, i64, i64, i32, ctypes.c_char_p, i64]
    lib.fxtx_autotune_set.argtypes = [i32]
    lib.fxtx_autotune_get.argtypes = []
    lib.fxtx_autotune_entries.argtypes = []
    lib.fxtx_autotune_entries.restype = i64
    lib.fxtx_autotune_clear.argtypes = []
    lib.fxtx_autotune_save.argtypes = [ctypes.c_char_p]
    lib.fxtx_autotune_load.argtypes = [ctypes.c_char_p]
    lib.fxtx_autotune_candidates.argtypes = [i32, i32, i64, i64, i64, i64, ctypes.c_char_p, i64]
    for name in ("fxtx_dense_f32", "fxtx_dense_f64", "fxtx_dense_f32_noalloc", "fxtx_dense_bf16", "fxtx_dense_multi_f32",
                 "fxtx_dense_multi_f64", "fxtx_csr_f32", "fxtx_csr_f64", "fxtx_csr_validate", "fxtx_device_error",
                 "fxtx_epilogue_f32", "fxtx_epilogue_f64", "fxtx_csr_analyze", "fxtx_csr_analysis_clear",
                 "fxtx_csr_plan_describe_host",
                 "fxtx_plan_describe", "fxtx_multi_plan_describe", "fxtx_autotune_set", "fxtx_autotune_get",
                 "fxtx_autotune_clear", "fxtx_autotune_save", "fxtx_autotune_load", "fxtx_autotune_candidates"):
        getattr(lib, name).restype = i32
    return lib


_lib = _load()
library_path = _build.LIB

fxtx_dense_f32 = _lib.fxtx_dense_f32
fxtx_dense_f64 = _lib.fxtx_dense_f64
fxtx_dense_f32_noalloc = _lib.fxtx_dense_f32_noalloc
fxtx_dense_bf16 = _lib.fxtx_dense_bf16
fxtx_dense_multi_f32 = _lib.fxtx_dense_multi_f32
fxtx_dense_multi_f64 = _lib.fxtx_dense_multi_f64
fxtx_csr_f32 = _lib.fxtx_csr_f32
fxtx_csr_f64 = _lib.fxtx_csr_f64
fxtx_csr_validate = _lib.fxtx_csr_validate
fxtx_csr_analyze = _lib.fxtx_csr_analyze
fxtx_csr_analysis_clear = _lib.fxtx_csr_analysis_clear
fxtx_csr_plan_describe_host = _lib.fxtx_csr_plan_describe_host
fxtx_epilogue_f32 = _lib.fxtx_epilogue_f32
fxtx_epilogue_f64 = _lib.fxtx_epilogue_f64
fxtx_device_error = _lib.fxtx_device_error
fxtx_plan_describe = _lib.fxtx_plan_describe
fxtx_multi_plan_describe = _lib.fxtx_multi_plan_describe
fxtx_autotune_set = _lib.fxtx_autotune_set
fxtx_autotune_get = _lib.fxtx_autotune_get
fxtx_autotune_entries = _lib.fxtx_autotune_entries
fxtx_autotune_clear = _lib.fxtx_autotune_clear
fxtx_autotune_save = _lib.fxtx_autotune_save
fxtx_autotune_load = _lib.fxtx_autotune_load
fxtx_autotune_candidates = _lib.fxtx_autotune_candidates


def fxtx_status_string(status: int) -> str:
    return _lib.fxtx_status_string(int(status)).decode()


class FxtxError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__(f"{where}: {fxtx_status_string(status)}" if where else fxtx_status_string(status))


def _check(status: int, where: str) -> None:
    if status != FXTX_OK:
        raise FxtxError(status, where)


def plan_describe(kind: str, dtype: str, m: int, n: int, nnz: int = 0, ld: int | None = None) -> str:
    """The launch plan the analytical model picks (host only)."""
    buf = ctypes.create_string_buffer(512)
    _check(fxtx_plan_describe(1 if kind == "csr" else 0, 1 if dtype in ("f64", "float64") else 0, m, n, nnz,
                              n if ld is None else ld, buf, 512), "fxtx_plan_describe")
    return buf.value.decode()


def multi_plan_describe(dtype: str, m: int, n: int, k: int, v_mode: str = "full", ld: int | None = None) -> str:
    """The launch plan of a multi-vector call (host only); v_mode "none", "shared" or "full"."""
    buf = ctypes.create_string_buffer(512)
    vm = {"none": 0, "shared": 1, "full": 2}[v_mode]
    _check(fxtx_multi_plan_describe(1 if dtype in ("f64", "float64") else 0, m, n, k, n if ld is None else ld, vm,
                                    buf, 512), "fxtx_multi_plan_describe")
    return buf.value.decode()


def autotune(mode: int) -> None:
    """0: the launch model picks (default); 1: time the model's candidates once per call shape and cache the fastest."""
    _check(fxtx_autotune_set(int(mode)), "fxtx_autotune_set")


def autotune_mode() -> int:
    return int(fxtx_autotune_get())


def autotune_entries() -> int:
    return int(fxtx_autotune_entries())


def autotune_clear() -> None:
    _check(fxtx_autotune_clear(), "fxtx_autotune_clear")


def autotune_save(path: str) -> None:
    _check(fxtx_autotune_save(os.fsencode(path)), "fxtx_autotune_save")


def autotune_load(path: str) -> None:
    _check(fxtx_autotune_load(os.fsencode(path)), "fxtx_autotune_load")


def autotune_candidates(kind: str, dtype: str, m: int, n: int, nnz: int = 0, ld: int | None = None) -> list[str]:
    """The candidate launches the tuner times for a shape, the model's plan first (host only)."""
    buf = ctypes.create_string_buffer(4096)
    _check(fxtx_autotune_candidates(1 if kind == "csr" else 0, 1 if dtype in ("f64", "float64") else 0, m, n, nnz,
                                    n if ld is None else ld, buf, 4096), "fxtx_autotune_candidates")
    return buf.value.decode().split("\n")


# ---------------------------------------------------------------------------- torch tensors
def _torch():
    import torch

    return torch


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream, device):
    torch = _torch()
    if stream is None:
        return torch.cuda.current_stream(device).cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _on(dev_index):
    """The calls run on the current device: make it the tensors' device for the call."""
    torch = _torch()
    return torch.cuda.device(dev_index) if torch.cuda.current_device() != dev_index else contextlib.nullcontext()


def _vec(t, dtype, length, name, dev_index):
    if t is None:
        return None
    if (t.dtype is not dtype or not t.is_cuda or t.get_device() != dev_index or t.dim() != 1
            or t.shape[0] != length or (length > 1 and t.stride(0) != 1)):
        raise ValueError(f"{name}: expected a contiguous {dtype} vector of length {length} on cuda:{dev_index}")
    return t


def dense(X, y, v=None, alpha: float = 1.0, beta: float = 0.0, z=None, out=None, stream=None):
    """out = alpha * X^T (v * (X y)) + beta * z for a row-major CUDA tensor X (m, n), X.stride(1) == 1.

    X may be float32, float64 or bfloat16; for bfloat16 X the vectors are float32 and the
    arithmetic is fp32.

    ``v=None`` means v = 1; ``z=None`` (or beta = 0) drops the beta z term. A column slice of a
    wider matrix is accepted: its row stride is passed as the leading dimension.
    """
    torch = _torch()
    if X.dim() != 2 or (X.shape[0] > 1 and X.shape[1] > 1 and X.stride(1) != 1) or not X.is_cuda:
        raise ValueError("X: expected a 2-D CUDA tensor with unit column stride")
    m, n = X.shape
    ld = X.stride(0) if m > 1 else max(n, 1)
    # bfloat16 X computes in fp32: y, v, z and out are float32
    dt, di = (torch.float32 if X.dtype == torch.bfloat16 else X.dtype), X.get_device()
    y = _vec(y, dt, n, "y", di)
    v = _vec(v, dt, m, "v", di)
    z = _vec(z, dt, n, "z", di)
    if out is None:
        out = torch.empty(n, dtype=dt, device=X.device)
    _vec(out, dt, n, "out", di)
    if X.dtype == torch.bfloat16:
        fn = fxtx_dense_bf16
    elif dt == torch.float32:
        fn = fxtx_dense_f32
    elif dt == torch.float64:
        fn = fxtx_dense_f64
    else:
        raise TypeError(f"unsupported dtype {dt}")
    with _on(di):
        rc = fn(m, n, _ptr(X), ld, _ptr(y), _ptr(v), alpha, beta, _ptr(z), _ptr(out), _stream(stream, X.device))
    _check(rc, "fxtx_dense")
    return out


def _rows(t, dtype, shape, name, dev_index):
    """A 2-D row-major CUDA tensor (unit column stride); returns its row stride."""
    if (t.dtype is not dtype or not t.is_cuda or t.get_device() != dev_index or t.dim() != 2
            or tuple(t.shape) != tuple(shape) or (shape[0] > 0 and shape[1] > 1 and t.stride(1) != 1)):
        raise ValueError(f"{name}: expected a row-major {dtype} tensor of shape {tuple(shape)} on cuda:{dev_index}")
    return t.stride(0) if shape[0] > 1 else max(shape[1], 1)


def dense_multi(X, Y, V=None, alpha: float = 1.0, beta: float = 0.0, Z=None, out=None, stream=None):
    """OUT = alpha * X^T (V * (X Y)) + beta * Z for k right-hand sides in one pass over X.

    X (m, n) as in ``dense`` (float32 or float64); Y (n, k), Z (n, k) and ``out`` (n, k)
    row-major. ``V`` is None (weights 1), an m-vector shared by every right-hand side,
    or an (m, k) row-major matrix. Column slices with unit column stride are accepted.
    """
    torch = _torch()
    if X.dim() != 2 or (X.shape[0] > 1 and X.shape[1] > 1 and X.stride(1) != 1) or not X.is_cuda:
        raise ValueError("X: expected a 2-D CUDA tensor with unit column stride")
    m, n = X.shape
    ld = X.stride(0) if m > 1 else max(n, 1)
    dt, di = X.dtype, X.get_device()
    if Y.dim() != 2:
        raise ValueError("Y: expected a 2-D tensor (n, k)")
    k = Y.shape[1]
    ldy = _rows(Y, dt, (n, k), "Y", di)
    if V is None:
        ldv = 0
    elif V.dim() == 1:
        _vec(V, dt, m, "V", di)
        ldv = 0
    else:
        ldv = _rows(V, dt, (m, k), "V", di)
        ldv = max(ldv, k)
    ldz = 0 if Z is None else _rows(Z, dt, (n, k), "Z", di)
    if out is None:
        out = torch.empty((n, k), dtype=dt, device=X.device)
    ldo = _rows(out, dt, (n, k), "out", di)
    if dt == torch.float32:
        fn = fxtx_dense_multi_f32
    elif dt == torch.float64:
        fn = fxtx_dense_multi_f64
    else:
        raise TypeError(f"unsupported dtype {dt}")
    with _on(di):
        rc = fn(m, n, k, _ptr(X), ld, _ptr(Y), max(ldy, k), _ptr(V), ldv, alpha, beta, _ptr(Z),
                max(ldz, k) if Z is not None else 0, _ptr(out), max(ldo, k), _stream(stream, X.device))
    _check(rc, "fxtx_dense_multi")
    return out


def csr(row_ptr, col_idx, vals, y, n: int, v=None, alpha: float = 1.0, beta: float = 0.0, z=None, out=None,
        stream=None):
    """The same pattern for CSR X: int64 row_ptr (m + 1), int32 col_idx and vals (nnz), n columns."""
    torch = _torch()
    if row_ptr.dim() != 1 or row_ptr.shape[0] < 1 or vals.dim() != 1 or not vals.is_cuda:
        raise ValueError("row_ptr (m + 1) and vals (nnz) must be 1-D, vals a CUDA tensor")
    m = row_ptr.shape[0] - 1
    nnz = vals.shape[0]
    dt, dev = vals.dtype, vals.device
    di = vals.get_device()
    _vec(row_ptr, torch.int64, m + 1, "row_ptr", di)
    _vec(col_idx, torch.int32, nnz, "col_idx", di)
    _vec(vals, dt, nnz, "vals", di)
    y = _vec(y, dt, n, "y", di)
    v = _vec(v, dt, m, "v", di)
    z = _vec(z, dt, n, "z", di)
    if out is None:
        out = torch.empty(n, dtype=dt, device=dev)
    _vec(out, dt, n, "out", di)
    if dt == torch.float32:
        fn = fxtx_csr_f32
    elif dt == torch.float64:
        fn = fxtx_csr_f64
    else:
        raise TypeError(f"unsupported dtype {dt}")
    with _on(di):
        rc = fn(m, n, nnz, _ptr(row_ptr), _ptr(col_idx), _ptr(vals), _ptr(y), _ptr(v), alpha, beta, _ptr(z), _ptr(out),
                _stream(stream, dev))
    _check(rc, "fxtx_csr")
    return out


def epilogue(w, alpha: float = 1.0, beta: float = 0.0, z=None, out=None, stream=None):
    """out = alpha * w + beta * z on the GPU (the last step of a row-sharded call, after the
    partials w_g = X_g^T (v_g * (X_g y)) of the row blocks are summed). ``z=None`` or beta = 0
    drops the beta z term; ``out`` may be ``w`` or ``z``."""
    torch = _torch()
    if w.dim() != 1 or not w.is_cuda:
        raise ValueError("w: expected a 1-D CUDA tensor")
    n, dt, di = w.shape[0], w.dtype, w.get_device()
    _vec(w, dt, n, "w", di)
    z = _vec(z, dt, n, "z", di)
    if out is None:
        out = torch.empty(n, dtype=dt, device=w.device)
    _vec(out, dt, n, "out", di)
    if dt == torch.float32:
        fn = fxtx_epilogue_f32
    elif dt == torch.float64:
        fn = fxtx_epilogue_f64
    else:
        raise TypeError(f"unsupported dtype {dt}")
    with _on(di):
        rc = fn(n, _ptr(w), alpha, beta, _ptr(z), _ptr(out), _stream(stream, w.device))
    _check(rc, "fxtx_epilogue")
    return out


def csr_analyze(row_ptr, col_idx, n: int, dtype: str = "f32", stream=None) -> dict:
    """Samples a CSR matrix on its GPU and records the statistics for later ``csr`` calls on
    the same tensors (see fxtx_csr_analyze). Returns the statistics and plan figures for
    values of `dtype` ("f32" or "f64"). Synchronous."""
    torch = _torch()
    if (row_ptr.dim() != 1 or row_ptr.shape[0] < 1 or col_idx.dim() != 1 or not row_ptr.is_cuda
            or not col_idx.is_cuda):
        raise ValueError("row_ptr (m + 1) and col_idx (nnz) must be 1-D CUDA tensors")
    di = row_ptr.get_device()
    _vec(row_ptr, torch.int64, row_ptr.shape[0], "row_ptr", di)
    _vec(col_idx, torch.int32, col_idx.shape[0], "col_idx", di)
    st = CsrStats()
    with _on(di):
        rc = fxtx_csr_analyze(1 if dtype in ("f64", "float64") else 0, row_ptr.shape[0] - 1, n, col_idx.shape[0],
                              _ptr(row_ptr), _ptr(col_idx), _stream(stream, row_ptr.device), ctypes.byref(st))
    _check(rc, "fxtx_csr_analyze")
    return st.as_dict()


def csr_analysis_clear() -> None:
    _check(fxtx_csr_analysis_clear(), "fxtx_csr_analysis_clear")


def csr_plan_describe_host(row_ptr, col_idx, n: int, dtype: str = "f32") -> tuple[str, dict]:
    """The plan the model picks for a CSR matrix given as host (numpy) arrays, from its sampled
    statistics; host only. Returns (description, statistics)."""
    import numpy as np

    rp = np.ascontiguousarray(row_ptr, dtype=np.int64)
    ci = np.ascontiguousarray(col_idx, dtype=np.int32)
    buf = ctypes.create_string_buffer(768)
    st = CsrStats()
    _check(fxtx_csr_plan_describe_host(1 if dtype in ("f64", "float64") else 0, rp.shape[0] - 1, n, ci.shape[0],
                                       rp.ctypes.data if rp.size else None, ci.ctypes.data if ci.size else None,
                                       ctypes.byref(st), buf, 768), "fxtx_csr_plan_describe_host")
    return buf.value.decode(), st.as_dict()


def csr_validate(row_ptr, col_idx, n: int, stream=None) -> bool:
    """True if the CSR structure is well formed (synchronous device check)."""
    torch = _torch()
    if row_ptr.dim() != 1 or row_ptr.shape[0] < 1 or not row_ptr.is_cuda or col_idx.dim() != 1:
        raise ValueError("row_ptr (m + 1) and col_idx (nnz) must be 1-D CUDA tensors")
    m, di = row_ptr.shape[0] - 1, row_ptr.get_device()
    _vec(row_ptr, torch.int64, m + 1, "row_ptr", di)
    _vec(col_idx, torch.int32, col_idx.shape[0], "col_idx", di)
    with _on(di):
        rc = fxtx_csr_validate(m, n, col_idx.shape[0], _ptr(row_ptr), _ptr(col_idx), _stream(stream, row_ptr.device))
    if rc == FXTX_ERR_BAD_CSR:
        return False
    _check(rc, "fxtx_csr_validate")
    return True


def device_error(stream=None) -> int:
    """Reads and clears the device-side error word (FXTX_OK or FXTX_ERR_TIMEOUT)."""
    torch = _torch()
    st = _stream(stream, torch.device("cuda", torch.cuda.current_device()))
    return fxtx_device_error(st)
