"""Helpers shared by the tests: tolerance checks and small matrix builders."""
from __future__ import annotations

import numpy as np

# |result_j - ref_j| <= REL[dtype] * S_j, S_j = |alpha| sum_i |t_i| |X_ij| + |beta z_j|
REL = {np.dtype(np.float64): 1e-12, np.dtype(np.float32): 2e-5}


def rel_for(dtype) -> float:
    return REL[np.dtype(dtype)]


def within_bound(got, ref, S, rel) -> np.ndarray:
    got = np.asarray(got, dtype=np.float64)
    return np.abs(got - np.asarray(ref)) <= rel * np.asarray(S)


def assert_within_bound(got, ref, S, rel, what=""):
    ok = within_bound(got, ref, S, rel)
    if not ok.all():
        bad = np.flatnonzero(~ok)
        j = bad[0]
        ratio = np.abs(np.asarray(got, np.float64) - ref) / np.where(S > 0, S, np.inf)
        raise AssertionError(
            f"{what}: {bad.size} of {ok.size} outputs outside {rel:g}*S; first j={j}: got {got[j]!r} "
            f"ref {ref[j]!r} S {S[j]!r}; worst |err|/S = {np.nanmax(ratio):.3g}")


def dense_to_csr(X: np.ndarray, keep_zeros: bool = False):
    """CSR (int64 row_ptr, int32 col_idx, vals) of a dense (m, n) array, columns ascending."""
    m, n = X.shape
    mask = np.ones_like(X, dtype=bool) if keep_zeros else (X != 0)
    rows, cols = np.nonzero(mask)
    row_ptr = np.zeros(m + 1, dtype=np.int64)
    np.add.at(row_ptr, rows + 1, 1)
    row_ptr = np.cumsum(row_ptr)
    return row_ptr, cols.astype(np.int32), X[rows, cols].copy()
