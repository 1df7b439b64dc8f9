"""CPU oracle for ``out = alpha * X^T (v * (X y)) + beta * z``.

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may import this package; the library itself never does, and it
shares no code with the CUDA path.

The arithmetic lives in ``fxtx_oracle.c`` (plain C, four naive loops following the
pattern in "On optimizing machine learning workloads via kernel fusion", abstract).
It is compiled twice into ``liboracle.so``: with a ``long double`` accumulator
(``acc="ld"``, used for checking) and with a ``double`` accumulator (``acc="d"``,
the timed CPU baseline). Both return the output and the per-column error scale
``S_j = |alpha| sum_i |t_i| |X_ij| + |beta z_j|``.

``dense_multi`` is the multi-vector instantiation ``OUT = alpha * X^T (V * (X Y)) +
beta * Z`` with k right-hand sides: column by column, the single-vector oracle.

Parity: every function here is pinned by ``tests/test_oracle.py`` (worked example,
closed-form identities, exact arithmetic on tiny inputs, dense-vs-CSR, a library
composition and planted-mistake checks). Nothing is left unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fxtx_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None

F32, F64 = 0, 1
_STATUS = {0: "ok", -1: "out of memory", -2: "malformed CSR structure", -3: "bad argument"}


def compile_oracle(src: str, out_path: str) -> None:
    """Compile one oracle source into a shared library holding both accumulator variants."""
    tmpdir = os.path.dirname(out_path)
    objs = []
    for acc, suffix in (("long double", "ld"), ("double", "d")):
        obj = os.path.join(tmpdir, f".oracle_{suffix}.{os.getpid()}.o")
        subprocess.check_call(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-c", src, "-o", obj,
                               f"-DORACLE_ACC={acc}", f"-DORACLE_SUFFIX={suffix}"])
        objs.append(obj)
    tmp = f"{out_path}.{os.getpid()}.tmp"
    subprocess.check_call(["gcc", "-shared", "-o", tmp] + objs + ["-lm"])
    for o in objs:
        os.remove(o)
    os.replace(tmp, out_path)


def build(force: bool = False) -> str:
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        compile_oracle(_SRC, _LIB_PATH)
    return _LIB_PATH


def bind(path: str):
    """Load an oracle shared library and declare its signatures."""
    lib = ctypes.CDLL(path)
    i32, i64, dbl, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
    for sfx in ("ld", "d"):
        f = getattr(lib, "oracle_dense_" + sfx)
        f.argtypes = [i32, i64, i64, vp, i64, vp, vp, dbl, dbl, vp, i64, vp, vp, vp]
        f.restype = i32
        f = getattr(lib, "oracle_csr_" + sfx)
        f.argtypes = [i32, i64, i64, i64, vp, vp, vp, vp, vp, dbl, dbl, vp, vp, vp]
        f.restype = i32
        f = getattr(lib, "oracle_csr_check_" + sfx)
        f.argtypes = [i64, i64, i64, vp, vp]
        f.restype = i32
    return lib


def _load():
    global _lib
    if _lib is None:
        build()
        _lib = bind(_LIB_PATH)
    return _lib


def _dt(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.float64:
        return F64
    raise TypeError(f"oracle takes float32 or float64 arrays, got {a.dtype}")


def _p(a):
    return None if a is None else a.ctypes.data


def _check(rc: int) -> None:
    if rc != 0:
        raise ValueError(f"oracle: {_STATUS.get(rc, rc)}")


def _vec(a, dtype, length, name):
    if a is None:
        return None
    a = np.ascontiguousarray(a)
    if a.dtype != dtype or a.shape != (length,):
        raise ValueError(f"{name}: expected {dtype} of shape ({length},), got {a.dtype} {a.shape}")
    return a


def dense(X: np.ndarray, y, v, alpha: float, beta: float, z, n: int | None = None, cols=None,
          acc: str = "ld", lib=None):
    """Oracle for dense X given as an (m, ld) C-contiguous array whose first n columns are X.

    Returns (out, S) as float64 arrays, over all n columns or over ``cols``.
    """
    lib = lib or _load()
    X = np.ascontiguousarray(X)
    m, ld = X.shape
    n = ld if n is None else n
    dt = X.dtype
    y = _vec(y, dt, n, "y")
    v = _vec(v, dt, m, "v")
    z = _vec(z, dt, n, "z")
    if cols is not None:
        cols = np.ascontiguousarray(cols, dtype=np.int64)
        nout = cols.shape[0]
    else:
        nout = n
    out = np.empty(nout, dtype=np.float64)
    S = np.empty(nout, dtype=np.float64)
    fn = getattr(lib, "oracle_dense_" + acc)
    _check(fn(_dt(X), m, n, _p(X), ld, _p(y), _p(v), float(alpha), float(beta), _p(z),
              nout if cols is not None else 0, _p(cols), _p(out), _p(S)))
    return out, S


def csr(row_ptr, col_idx, vals, y, v, alpha: float, beta: float, z, n: int, acc: str = "ld", lib=None):
    """Oracle for CSR X (int64 row_ptr, int32 col_idx). Returns (out, S) over all n columns."""
    lib = lib or _load()
    row_ptr = np.ascontiguousarray(row_ptr, dtype=np.int64)
    col_idx = np.ascontiguousarray(col_idx, dtype=np.int32)
    vals = np.ascontiguousarray(vals)
    m = row_ptr.shape[0] - 1
    nnz = vals.shape[0]
    dt = vals.dtype
    y = _vec(y, dt, n, "y")
    v = _vec(v, dt, m, "v")
    z = _vec(z, dt, n, "z")
    if col_idx.shape[0] != nnz:
        raise ValueError("col_idx and vals differ in length")
    out = np.empty(n, dtype=np.float64)
    S = np.empty(n, dtype=np.float64)
    fn = getattr(lib, "oracle_csr_" + acc)
    _check(fn(_dt(vals), m, n, nnz, _p(row_ptr), _p(col_idx), _p(vals), _p(y), _p(v),
              float(alpha), float(beta), _p(z), _p(out), _p(S)))
    return out, S


def csr_is_valid(row_ptr, col_idx, n: int, lib=None) -> bool:
    lib = lib or _load()
    row_ptr = np.ascontiguousarray(row_ptr, dtype=np.int64)
    col_idx = np.ascontiguousarray(col_idx, dtype=np.int32)
    m = row_ptr.shape[0] - 1
    return lib.oracle_csr_check_ld(m, n, col_idx.shape[0], _p(row_ptr), _p(col_idx)) == 0


def _vcol(V, c):
    """Column c of the row weights: None (all ones), one shared m-vector, or an (m, k) matrix."""
    if V is None or V.ndim == 1:
        return V
    return np.ascontiguousarray(V[:, c])


def dense_multi(X: np.ndarray, Y: np.ndarray, V, alpha: float, beta: float, Z, n: int | None = None, cols=None,
                acc: str = "ld", lib=None):
    """Oracle for the multi-vector instantiation ``OUT = alpha * X^T (V * (X Y)) + beta * Z``.

    Y is (n, k); V is None (all ones), an m-vector shared by every right-hand side, or
    an (m, k) matrix; Z is None or (n, k). The k right-hand sides do not interact: each
    column c of OUT is the single-vector pattern with y = Y[:, c], v = V[:, c] (or the
    shared v) and z = Z[:, c], computed by ``dense``. Returns (OUT, S), each (nout, k).
    """
    X = np.ascontiguousarray(X)
    n = X.shape[1] if n is None else n
    if Y.ndim != 2 or Y.shape[0] != n:
        raise ValueError(f"Y: expected shape ({n}, k), got {Y.shape}")
    k = Y.shape[1]
    if V is not None and V.ndim == 2 and V.shape != (X.shape[0], k):
        raise ValueError(f"V: expected shape ({X.shape[0]}, {k}), got {V.shape}")
    if Z is not None and Z.shape != (n, k):
        raise ValueError(f"Z: expected shape ({n}, {k}), got {Z.shape}")
    nout = n if cols is None else len(cols)
    OUT = np.empty((nout, k), dtype=np.float64)
    S = np.empty((nout, k), dtype=np.float64)
    for c in range(k):
        zc = None if Z is None else np.ascontiguousarray(Z[:, c])
        OUT[:, c], S[:, c] = dense(X, np.ascontiguousarray(Y[:, c]), _vcol(V, c), alpha, beta, zc, n=n, cols=cols,
                                   acc=acc, lib=lib)
    return OUT, S


def solve(p, cols=None, acc: str = "ld", lib=None):
    """Oracle for an ``inputgen.Problem``."""
    if p.kind == "dense" and p.y.ndim == 2:
        return dense_multi(p.X, p.y, p.v, p.alpha, p.beta, p.z, n=p.n, cols=cols, acc=acc, lib=lib)
    if p.kind == "dense":
        return dense(p.X, p.y, p.v, p.alpha, p.beta, p.z, n=p.n, cols=cols, acc=acc, lib=lib)
    if cols is not None:
        out, S = csr(p.row_ptr, p.col_idx, p.vals, p.y, p.v, p.alpha, p.beta, p.z, p.n, acc=acc, lib=lib)
        return out[cols], S[cols]
    return csr(p.row_ptr, p.col_idx, p.vals, p.y, p.v, p.alpha, p.beta, p.z, p.n, acc=acc, lib=lib)
