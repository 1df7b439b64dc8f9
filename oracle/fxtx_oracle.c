/*
 * fxtx_oracle.c — CPU oracle for the fused pattern
 *
 *     out = alpha * X^T (v .* (X y)) + beta * z
 *
 * as defined in "On optimizing machine learning workloads via kernel fusion",
 * abstract (the generic pattern and its instantiations). X is m x n, y and z
 * have n entries, v has m entries and multiplies element-wise.
 *
 * TEST INFRASTRUCTURE ONLY. Tests, the smoke check and the CPU-baseline leg of
 * the benchmark use this file; the library never does. It shares no code, header
 * or constant with the CUDA path.
 *
 * The definition is written out as four separate naive loops, in the order the
 * pattern reads from the inside out:
 *   1. u_i = sum_j X_ij * y_j              (j ascending)
 *   2. t_i = v_i * u_i                     (v absent: v_i = 1)
 *   3. w_j = sum_i X_ij * t_i              (i ascending)
 *   4. out_j = alpha * w_j + beta * z_j    (z absent or beta == 0: no z term, z unread)
 * Every input is converted to the accumulator type before it is multiplied. The
 * accumulator type is chosen at compile time: `long double` for checking
 * (suffix _ld) and `double` for the timed CPU baseline (suffix _d).
 *
 * Alongside out it returns the error scale
 *     S_j = |alpha| * sum_i |t_i| * |X_ij| + |beta * z_j|
 * in double, against which results computed in another summation order are
 * checked.
 *
 * Sparse X is CSR: row_ptr (int64, m+1 entries, row_ptr[0] = 0, non-decreasing,
 * row_ptr[m] = nnz), col_idx (int32, 0 <= col < n) and vals. Column order inside
 * a row is free and repeated (i, j) entries add, because the matrix they stand
 * for is their sum. Empty rows give u_i = 0.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

#ifndef ORACLE_ACC
#define ORACLE_ACC long double
#endif
#ifndef ORACLE_SUFFIX
#define ORACLE_SUFFIX ld
#endif

typedef ORACLE_ACC acc_t;

#define ORACLE_CAT2(a, b) a##_##b
#define ORACLE_CAT(a, b) ORACLE_CAT2(a, b)
#define ORACLE_NAME(f) ORACLE_CAT(f, ORACLE_SUFFIX)

/* element type of the floating-point arrays */
enum { ORACLE_F32 = 0, ORACLE_F64 = 1 };

/* status codes */
enum { ORACLE_OK = 0, ORACLE_NOMEM = -1, ORACLE_BAD_CSR = -2, ORACLE_BAD_ARG = -3 };

static acc_t at(const void* p, int dtype, int64_t k) {
  if (dtype == ORACLE_F32) return (acc_t)((const float*)p)[k];
  return (acc_t)((const double*)p)[k];
}

static double atd(const void* p, int dtype, int64_t k) {
  if (dtype == ORACLE_F32) return (double)((const float*)p)[k];
  return ((const double*)p)[k];
}

/*
 * Dense X, row-major with leading dimension ld (entry (i, j) at X[i * ld + j]).
 * If cols is NULL, out and S receive all n columns; otherwise they receive the
 * ncols columns listed in cols (each 0 <= cols[k] < n), in that order. Step 3
 * then runs only over the listed columns, so sampled outputs of a large X cost
 * one pass for the dots plus m per listed column.
 */
int ORACLE_NAME(oracle_dense)(int dtype, int64_t m, int64_t n, const void* X, int64_t ld,
                              const void* y, const void* v, double alpha, double beta,
                              const void* z, int64_t ncols, const int64_t* cols,
                              double* out, double* S) {
  if (m < 0 || n < 0 || (m > 0 && n > 0 && ld < n)) return ORACLE_BAD_ARG;
  int64_t nout = cols ? ncols : n;
  int use_z = (z != NULL && beta != 0.0);
  acc_t* t = (acc_t*)malloc((size_t)(m > 0 ? m : 1) * sizeof(acc_t));
  if (!t) return ORACLE_NOMEM;

  /* step 1 and step 2: u_i = sum_j X_ij y_j, then t_i = v_i u_i */
  for (int64_t i = 0; i < m; ++i) {
    acc_t u = 0;
    for (int64_t j = 0; j < n; ++j) u += at(X, dtype, i * ld + j) * at(y, dtype, j);
    acc_t vi = v ? at(v, dtype, i) : (acc_t)1;
    t[i] = vi * u;
  }

  /* step 3: w_j = sum_i X_ij t_i, i ascending for every j */
  acc_t* w = (acc_t*)calloc((size_t)(nout > 0 ? nout : 1), sizeof(acc_t));
  double* s = (double*)calloc((size_t)(nout > 0 ? nout : 1), sizeof(double));
  if (!w || !s) { free(t); free(w); free(s); return ORACLE_NOMEM; }
  if (cols == NULL) {
    for (int64_t i = 0; i < m; ++i)
      for (int64_t j = 0; j < n; ++j) {
        w[j] += at(X, dtype, i * ld + j) * t[i];
        s[j] += fabs((double)t[i]) * fabs(atd(X, dtype, i * ld + j));
      }
  } else {
    for (int64_t k = 0; k < ncols; ++k) {
      int64_t j = cols[k];
      if (j < 0 || j >= n) { free(t); free(w); free(s); return ORACLE_BAD_ARG; }
      for (int64_t i = 0; i < m; ++i) {
        w[k] += at(X, dtype, i * ld + j) * t[i];
        s[k] += fabs((double)t[i]) * fabs(atd(X, dtype, i * ld + j));
      }
    }
  }

  /* step 4: out_j = alpha w_j + beta z_j */
  for (int64_t k = 0; k < nout; ++k) {
    int64_t j = cols ? cols[k] : k;
    acc_t o = (acc_t)alpha * w[k];
    double sj = fabs(alpha) * s[k];
    if (use_z) {
      o += (acc_t)beta * at(z, dtype, j);
      sj += fabs(beta * atd(z, dtype, j));
    }
    out[k] = (double)o;
    if (S) S[k] = sj;
  }
  free(t); free(w); free(s);
  return ORACLE_OK;
}

/* 0 if the CSR structure is well formed, else ORACLE_BAD_CSR. */
int ORACLE_NAME(oracle_csr_check)(int64_t m, int64_t n, int64_t nnz, const int64_t* row_ptr,
                                  const int32_t* col_idx) {
  if (m < 0 || n < 0 || nnz < 0) return ORACLE_BAD_ARG;
  if (row_ptr[0] != 0 || row_ptr[m] != nnz) return ORACLE_BAD_CSR;
  for (int64_t i = 0; i < m; ++i)
    if (row_ptr[i + 1] < row_ptr[i]) return ORACLE_BAD_CSR;
  for (int64_t k = 0; k < nnz; ++k)
    if (col_idx[k] < 0 || (int64_t)col_idx[k] >= n) return ORACLE_BAD_CSR;
  return ORACLE_OK;
}

/* CSR X; out and S receive all n columns. */
int ORACLE_NAME(oracle_csr)(int dtype, int64_t m, int64_t n, int64_t nnz, const int64_t* row_ptr,
                            const int32_t* col_idx, const void* vals, const void* y,
                            const void* v, double alpha, double beta, const void* z,
                            double* out, double* S) {
  int rc = ORACLE_NAME(oracle_csr_check)(m, n, nnz, row_ptr, col_idx);
  if (rc != ORACLE_OK) return rc;
  int use_z = (z != NULL && beta != 0.0);
  acc_t* t = (acc_t*)malloc((size_t)(m > 0 ? m : 1) * sizeof(acc_t));
  acc_t* w = (acc_t*)calloc((size_t)(n > 0 ? n : 1), sizeof(acc_t));
  double* s = (double*)calloc((size_t)(n > 0 ? n : 1), sizeof(double));
  if (!t || !w || !s) { free(t); free(w); free(s); return ORACLE_NOMEM; }

  /* step 1 and step 2: u_i = sum over the row's entries of vals_k y_{col_k}; t_i = v_i u_i */
  for (int64_t i = 0; i < m; ++i) {
    acc_t u = 0;
    for (int64_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) u += at(vals, dtype, k) * at(y, dtype, col_idx[k]);
    acc_t vi = v ? at(v, dtype, i) : (acc_t)1;
    t[i] = vi * u;
  }

  /* step 3: w_j = sum_i X_ij t_i, rows in ascending order */
  for (int64_t i = 0; i < m; ++i)
    for (int64_t k = row_ptr[i]; k < row_ptr[i + 1]; ++k) {
      int64_t j = col_idx[k];
      w[j] += at(vals, dtype, k) * t[i];
      s[j] += fabs((double)t[i]) * fabs(atd(vals, dtype, k));
    }

  /* step 4: out_j = alpha w_j + beta z_j */
  for (int64_t j = 0; j < n; ++j) {
    acc_t o = (acc_t)alpha * w[j];
    double sj = fabs(alpha) * s[j];
    if (use_z) {
      o += (acc_t)beta * at(z, dtype, j);
      sj += fabs(beta * atd(z, dtype, j));
    }
    out[j] = (double)o;
    if (S) S[j] = sj;
  }
  free(t); free(w); free(s);
  return ORACLE_OK;
}
