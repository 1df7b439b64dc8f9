"""Seeded synthetic inputs for the fused pattern ``alpha * X^T (v * (X y)) + beta * z``.

This package draws numbers and sparsity structures only; it holds none of the
pattern's arithmetic. The CPU oracle (``oracle/``) and the CUDA library are both fed
from the arrays built here, so they see identical bits.

Streams per problem (one key each, derived from the seed): 0 structure, 1 X / vals,
2 y, 3 v, 4 z. The workloads are the five of the kernel-fusion paper's setting as
restated for this library:

* ``dense_small``     dense f64 1000 x 64, everything U[-1, 1], alpha=1.5, beta=0.5
* ``dense_tall``      dense f32 16,000,000 x 32, X, y, z ~ N(0, 1), v ~ U[0.1, 2]
                      (variant "a": alpha=1, beta=0, no z; "b": alpha=2, beta=-1 with z;
                      "c": v=1, alpha=1, beta=0, i.e. X^T X y)
* ``dense_wide``      dense f64 20,000 x 20,000, everything U[-1, 1], alpha=0.7, beta=0.3
* ``csr_uniform``     CSR f64 4,000,000 x 10,000, Poisson(50) distinct uniform columns
                      per row, everything U[-1, 1], alpha=beta=1
* ``csr_powerlaw``    CSR f32 2,000,000 x 1,000,000, row lengths Zipf(1.5) scaled to a
                      mean of 100 and capped at 50,000, columns Zipf(1.1) over ranks with
                      column = rank - 1; vals, y ~ N(0, 1), v ~ U[0, 1], no z,
                      alpha=1, beta=0

Every constructor takes smaller sizes too, keeping the recipe, for tests.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "inputgen.c")
_LIB_PATH = os.path.join(_HERE, "libinputgen.so")
_lib = None

STRUCTURE, XSTREAM, YSTREAM, VSTREAM, ZSTREAM = 0, 1, 2, 3, 4


def build(force: bool = False) -> str:
    """Compile ``libinputgen.so`` next to its source (gcc, OpenMP)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = f"{_LIB_PATH}.{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        i64, u64, dbl, vp = ctypes.c_int64, ctypes.c_uint64, ctypes.c_double, ctypes.c_void_p
        for nm in ("ig_fill_uniform_f64", "ig_fill_uniform_f32"):
            getattr(lib, nm).argtypes = [u64, u64, i64, dbl, dbl, vp]
        for nm in ("ig_fill_normal_f64", "ig_fill_normal_f32"):
            getattr(lib, nm).argtypes = [u64, u64, i64, vp]
        for nm in ("ig_fill_int_f64", "ig_fill_int_f32"):
            getattr(lib, nm).argtypes = [u64, u64, i64, i64, i64, vp]
        lib.ig_poisson_lengths.argtypes = [u64, u64, i64, dbl, i64, vp]
        lib.ig_zipf_lengths.argtypes = [u64, u64, i64, dbl, i64, i64, i64, vp]
        lib.ig_zipf_lengths.restype = dbl
        lib.ig_fill_csr_cols.argtypes = [u64, u64, i64, i64, dbl, vp, vp]
        lib.ig_fill_csr_cols.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def uniform(seed: int, stream: int, shape, a: float, b: float, dtype=np.float64) -> np.ndarray:
    out = np.empty(shape, dtype=dtype)
    fn = _load().ig_fill_uniform_f64 if out.dtype == np.float64 else _load().ig_fill_uniform_f32
    fn(seed, stream, out.size, a, b, _ptr(out))
    return out


def normal(seed: int, stream: int, shape, dtype=np.float64) -> np.ndarray:
    out = np.empty(shape, dtype=dtype)
    fn = _load().ig_fill_normal_f64 if out.dtype == np.float64 else _load().ig_fill_normal_f32
    fn(seed, stream, out.size, _ptr(out))
    return out


def integers(seed: int, stream: int, shape, lo: int, hi: int, dtype=np.float64) -> np.ndarray:
    """Integer values uniform in [lo, hi], stored as floating point."""
    out = np.empty(shape, dtype=dtype)
    fn = _load().ig_fill_int_f64 if out.dtype == np.float64 else _load().ig_fill_int_f32
    fn(seed, stream, out.size, lo, hi, _ptr(out))
    return out


def round_to_bf16(a: np.ndarray) -> np.ndarray:
    """float32 values rounded to the nearest bfloat16 (ties to even), kept as float32.

    Every result is exactly representable in bfloat16, so a device copy in bfloat16 and
    the float32 array hold the same numbers.
    """
    bits = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)
    rounded = (bits + np.uint32(0x7FFF) + ((bits >> np.uint32(16)) & np.uint32(1))) & np.uint32(0xFFFF0000)
    return rounded.view(np.float32)


def poisson_lengths(seed: int, m: int, lam: float, cap: int) -> np.ndarray:
    lens = np.empty(m, dtype=np.int64)
    _load().ig_poisson_lengths(seed, STRUCTURE, m, lam, cap, _ptr(lens))
    return lens


def zipf_lengths(seed: int, m: int, s: float, kmax: int, target_nnz: int, cap: int):
    lens = np.empty(m, dtype=np.int64)
    c = _load().ig_zipf_lengths(seed, STRUCTURE, m, s, kmax, target_nnz, cap, _ptr(lens))
    if c < 0:
        raise MemoryError("ig_zipf_lengths failed")
    return lens, c


def csr_columns(seed: int, n: int, row_ptr: np.ndarray, zipf_s: float = 0.0) -> np.ndarray:
    """Distinct, sorted column indices per row (uniform, or Zipf over rank = col + 1)."""
    m = row_ptr.shape[0] - 1
    col = np.empty(int(row_ptr[-1]), dtype=np.int32)
    rc = _load().ig_fill_csr_cols(seed, STRUCTURE + 100, m, n, zipf_s, _ptr(row_ptr), _ptr(col))
    if rc != 0:
        raise ValueError("csr_columns: a row is longer than n, or out of memory")
    return col


def row_ptr_from_lengths(lens: np.ndarray) -> np.ndarray:
    rp = np.zeros(lens.shape[0] + 1, dtype=np.int64)
    np.cumsum(lens, out=rp[1:])
    return rp


@dataclass
class Problem:
    """One instance of the pattern: inputs, scalars and a name. X is (m, ld) dense or CSR."""

    name: str
    kind: str  # "dense" or "csr"
    dtype: type
    m: int
    n: int
    alpha: float
    beta: float
    y: np.ndarray
    v: Optional[np.ndarray]
    z: Optional[np.ndarray]
    X: Optional[np.ndarray] = None  # dense: shape (m, ld), the first n columns are the matrix
    ld: int = 0
    row_ptr: Optional[np.ndarray] = None
    col_idx: Optional[np.ndarray] = None
    vals: Optional[np.ndarray] = None
    info: dict = field(default_factory=dict)
    x_store: str = ""  # "bf16": X holds bfloat16-representable values, stored on the device as bfloat16

    @property
    def nnz(self) -> int:
        return int(self.row_ptr[-1]) if self.kind == "csr" else self.m * self.n

    @property
    def itemsize(self) -> int:
        return np.dtype(self.dtype).itemsize

    def ideal_bytes(self) -> int:
        """Algorithmic bytes: X once, y, v (if given), z (if read), out once."""
        s = self.itemsize
        b = 2 * self.y.size * s  # y, out (n, or n x k for several right-hand sides)
        if self.v is not None:
            b += self.v.size * s
        if self.z is not None and self.beta != 0.0:
            b += self.z.size * s
        if self.kind == "dense":
            b += self.m * self.n * (2 if self.x_store == "bf16" else s)
        else:
            b += self.nnz * (s + 4) + (self.m + 1) * 8
        return b


def dense_small(seed: int = 0, m: int = 1000, n: int = 64) -> Problem:
    d = np.float64
    return Problem("dense_f64_%dx%d" % (m, n), "dense", d, m, n, 1.5, 0.5,
                   X=uniform(seed, XSTREAM, (m, n), -1.0, 1.0, d), ld=n,
                   y=uniform(seed, YSTREAM, n, -1.0, 1.0, d),
                   v=uniform(seed, VSTREAM, m, -1.0, 1.0, d),
                   z=uniform(seed, ZSTREAM, n, -1.0, 1.0, d))


def dense_tall(seed: int = 0, m: int = 16_000_000, n: int = 32, variant: str = "b", x_store: str = "") -> Problem:
    d = np.float32
    X = normal(seed, XSTREAM, (m, n), d)
    if x_store == "bf16":
        p = dense_tall(seed, m=1, n=n, variant=variant)  # the vectors and scalars of the same recipe
        p.X = round_to_bf16(X)
        p.m = m
        p.v = None if p.v is None else uniform(seed, VSTREAM, m, 0.1, 2.0, d)
        p.x_store = "bf16"
        p.name = p.name.replace("dense_f32_1x", "dense_bf16_%dx" % m)
        return p
    y = normal(seed, YSTREAM, n, d)
    v = uniform(seed, VSTREAM, m, 0.1, 2.0, d)
    if variant == "a":
        return Problem("dense_f32_%dx%d_a" % (m, n), "dense", d, m, n, 1.0, 0.0, X=X, ld=n, y=y, v=v, z=None)
    if variant == "b":
        z = normal(seed, ZSTREAM, n, d)
        return Problem("dense_f32_%dx%d_b" % (m, n), "dense", d, m, n, 2.0, -1.0, X=X, ld=n, y=y, v=v, z=z)
    if variant == "c":
        return Problem("dense_f32_%dx%d_c" % (m, n), "dense", d, m, n, 1.0, 0.0, X=X, ld=n, y=y, v=None, z=None)
    raise ValueError(variant)


def dense_multi(seed: int = 0, m: int = 16_000_000, n: int = 32, k: int = 8, dtype=np.float32,
                v_mode: str = "full") -> Problem:
    """Several right-hand sides on the tall-skinny recipe: Y (n, k) and Z (n, k) N(0,1);
    V U[0.1, 2] either (m, k) ("full"), one m-vector shared by all k ("shared"), or
    absent ("none"); alpha = 2, beta = -1."""
    d = dtype
    X = normal(seed, XSTREAM, (m, n), d)
    Y = normal(seed, YSTREAM, (n, k), d)
    Z = normal(seed, ZSTREAM, (n, k), d)
    if v_mode == "full":
        V = uniform(seed, VSTREAM, (m, k), 0.1, 2.0, d)
    elif v_mode == "shared":
        V = uniform(seed, VSTREAM, m, 0.1, 2.0, d)
    elif v_mode == "none":
        V = None
    else:
        raise ValueError(v_mode)
    tag = "f32" if d == np.float32 else "f64"
    return Problem("dense_multi_%s_%dx%dx%d_%s" % (tag, m, n, k, v_mode), "dense", d, m, n, 2.0, -1.0,
                   X=X, ld=n, y=Y, v=V, z=Z)


def dense_wide(seed: int = 0, m: int = 20_000, n: int = 20_000) -> Problem:
    d = np.float64
    return Problem("dense_f64_%dx%d" % (m, n), "dense", d, m, n, 0.7, 0.3,
                   X=uniform(seed, XSTREAM, (m, n), -1.0, 1.0, d), ld=n,
                   y=uniform(seed, YSTREAM, n, -1.0, 1.0, d),
                   v=uniform(seed, VSTREAM, m, -1.0, 1.0, d),
                   z=uniform(seed, ZSTREAM, n, -1.0, 1.0, d))


def csr_uniform(seed: int = 0, m: int = 4_000_000, n: int = 10_000, lam: float = 50.0) -> Problem:
    d = np.float64
    lens = poisson_lengths(seed, m, lam, n)
    rp = row_ptr_from_lengths(lens)
    col = csr_columns(seed, n, rp, 0.0)
    nnz = int(rp[-1])
    return Problem("csr_f64_%dx%d_uniform" % (m, n), "csr", d, m, n, 1.0, 1.0,
                   row_ptr=rp, col_idx=col, vals=uniform(seed, XSTREAM, nnz, -1.0, 1.0, d),
                   y=uniform(seed, YSTREAM, n, -1.0, 1.0, d),
                   v=uniform(seed, VSTREAM, m, -1.0, 1.0, d),
                   z=uniform(seed, ZSTREAM, n, -1.0, 1.0, d),
                   info={"nnz": nnz, "max_row": int(lens.max(initial=0))})


def csr_powerlaw(seed: int = 0, m: int = 2_000_000, n: int = 1_000_000, mean_len: float = 100.0,
                 cap: int = 50_000, len_s: float = 1.5, col_s: float = 1.1, col_offset: int = 0) -> Problem:
    """Zipf row lengths and Zipf-skewed columns (rank r at column r - 1). ``col_offset``
    rotates every column index by that many places (mod n), so the hottest columns sit
    at [col_offset, ...) instead of [0, ...); the rows stay sorted up to the wrap."""
    d = np.float32
    cap = min(cap, n)
    lens, c = zipf_lengths(seed, m, len_s, cap, int(round(mean_len * m)), cap)
    rp = row_ptr_from_lengths(lens)
    col = csr_columns(seed, n, rp, col_s)
    if col_offset:
        col = ((col.astype(np.int64) + col_offset) % n).astype(np.int32)
    nnz = int(rp[-1])
    mu = lens.mean() if m else 0.0
    name = "csr_f32_%dx%d_powerlaw" % (m, n) + ("_rot%d" % col_offset if col_offset else "")
    return Problem(name, "csr", d, m, n, 1.0, 0.0,
                   row_ptr=rp, col_idx=col, vals=normal(seed, XSTREAM, nnz, d),
                   y=normal(seed, YSTREAM, n, d),
                   v=uniform(seed, VSTREAM, m, 0.0, 1.0, d), z=None,
                   info={"nnz": nnz, "scale_c": c, "max_row": int(lens.max(initial=0)),
                         "cv": float(lens.std() / mu) if mu else 0.0})


WORKLOADS = {
    "dense_small": dense_small,
    "dense_tall": dense_tall,
    "dense_wide": dense_wide,
    "csr_uniform": csr_uniform,
    "csr_powerlaw": csr_powerlaw,
}
