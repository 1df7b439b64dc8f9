/*
 * fxtx.h — libfusedxtx: the fused pattern
 *
 *     out = alpha * X^T (v .* (X y)) + beta * z
 *
 * and its instantiations, from "On optimizing machine learning workloads via
 * kernel fusion", abstract (the generic pattern; a fused GPU kernel for sparse
 * and dense X that reads X once; coarsening and hierarchical aggregation of
 * partial results; an analytical model choosing launch parameters).
 *
 * Shapes: X is m x n, y, z and out have n entries, v has m entries and scales
 * element-wise. The instantiations are selected by NULL arguments:
 *   v == NULL                 v_i = 1            (X^T X y when alpha = 1, beta = 0)
 *   z == NULL or beta == 0    no beta z term, and z is not read
 *
 * Memory: every pointer argument is a DEVICE pointer owned by the caller, and
 * `stream` is a cudaStream_t (NULL for the legacy default stream). Calls are
 * asynchronous with respect to the host, like cuBLAS: they return after the
 * work is enqueued on `stream`, and errors of execution surface at the caller's
 * next synchronisation (and through fxtx_device_error). The one exception is the
 * first call of a shape with autotuning switched on (fxtx_autotune_set), which
 * times its candidates and synchronises `stream`. The library allocates only
 * transient workspace, with cudaMallocAsync on `stream` and freed with
 * cudaFreeAsync on the same stream; besides the opt-in autotune cache it keeps no
 * global state between calls, so concurrent calls on different streams are safe.
 *
 * Aliasing: out may equal z (in place). Any other overlap of out with an input
 * is undefined.
 *
 * Arithmetic: fp32 entry points compute in fp32 with compensated accumulation of
 * column partials and an fp64 final reduction; fp64 entry points compute in
 * fp64. The result matches the exact value within
 *     |out_j - exact_j| <= c * S_j,  S_j = |alpha| sum_i |t_i| |X_ij| + |beta z_j|,
 * t_i = v_i (x_i . y), with c = 2e-5 (fp32) or 1e-12 (fp64).
 */
#ifndef FXTX_H
#define FXTX_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FXTX_OK = 0,
  FXTX_ERR_INVALID_ARG = 1, /* a size is negative, ld < n, or a required pointer is NULL */
  FXTX_ERR_UNSUPPORTED = 2, /* no compute capability 10.3 device is current, or a shape an entry does not take */
  FXTX_ERR_CUDA = 3,        /* a CUDA runtime call failed while enqueueing (launch, allocation) */
  FXTX_ERR_ALLOC = 4,       /* workspace allocation failed */
  FXTX_ERR_BAD_CSR = 5,     /* fxtx_csr_validate found a malformed structure */
  FXTX_ERR_TIMEOUT = 6,     /* a kernel gave up a bounded wait (reported by fxtx_device_error) */
  FXTX_ERR_TOO_LARGE = 7    /* the problem needs more scratch than fxtx_dense_f32_noalloc holds */
} fxtx_status_t;

/*
 * Dense X, row-major: entry (i, j) at X[i * ld + j], ld >= max(1, n).
 *
 * m, n >= 0. X may be NULL only when m == 0 or n == 0; y and out must be non-NULL
 * when n > 0. When m == 0, out = beta * z (or 0). When n == 0 the call does
 * nothing and returns FXTX_OK.
 *
 * Any alignment and any ld are accepted. When X is 16-byte aligned and
 * ld * sizeof(T) and n * sizeof(T) are multiples of 16, X is staged through
 * shared memory by bulk asynchronous copies; otherwise a direct-load variant
 * runs. The result is the same within the bound above.
 *
 * The column reduction of the dense kernels is deterministic: repeated calls
 * with the same arguments give bitwise-identical out.
 */
fxtx_status_t fxtx_dense_f32(int64_t m, int64_t n, const float* X, int64_t ld, const float* y,
                             const float* v, float alpha, float beta, const float* z, float* out,
                             void* stream);
fxtx_status_t fxtx_dense_f64(int64_t m, int64_t n, const double* X, int64_t ld, const double* y,
                             const double* v, double alpha, double beta, const double* z, double* out,
                             void* stream);

/*
 * Dense X stored as bfloat16 (the upper 16 bits of an IEEE binary32, given as
 * uint16_t), with y, v, z and out in fp32 and all arithmetic in fp32 as in
 * fxtx_dense_f32 (each bfloat16 widens exactly). Reading X in bfloat16 halves the
 * bytes of the dominant stream. Shapes: n <= 512. Rows of at least 64 bytes with
 * X 16-byte aligned and ld * 2 a multiple of 16 take the tensor-copied tile
 * kernel; others a direct-load kernel. n > 512 returns FXTX_ERR_UNSUPPORTED.
 * Arguments, ownership and the bound are otherwise those of fxtx_dense_f32.
 */
fxtx_status_t fxtx_dense_bf16(int64_t m, int64_t n, const uint16_t* X, int64_t ld, const float* y,
                              const float* v, float alpha, float beta, const float* z, float* out,
                              void* stream);

/*
 * Multi-vector instantiation: k right-hand sides in one pass over dense X.
 * ("On optimizing machine learning workloads via kernel fusion", abstract: the
 * fused pattern and its instantiations, here with k vectors y at once.)
 *
 *     OUT[:, c] = alpha * X^T (V[:, c] * (X Y[:, c])) + beta * Z[:, c],  c = 0 .. k-1
 *
 * X as in fxtx_dense_f32 (m x n, row pitch ld >= n). Y, Z and OUT are n x k,
 * row-major: entry (j, c) at Y[j * ldy + c], Z[j * ldz + c], OUT[j * ldo + c],
 * with ldy, ldz, ldo >= k. V holds the row weights:
 *   V == NULL          all weights 1;
 *   ldv == 0           V is one m-vector, V[i], shared by every right-hand side;
 *   ldv >= k           V is m x k, entry (i, c) at V[i * ldv + c].
 * Z is read only when beta != 0 (it may then be NULL). OUT may equal Z with
 * ldo == ldz (in place); any other overlap of OUT with an input is undefined.
 *
 * Shapes: rows of at most 2 KB (n <= 512 in fp32, n <= 256 in fp64); wider
 * rows return FXTX_ERR_UNSUPPORTED. Each pass over X takes up to 32 / b
 * right-hand sides, b = the row's 128-byte blocks rounded up to a power of
 * two (32 for n <= 32 fp32 or n <= 16 fp64); larger k runs ceil(k / that)
 * passes. X 16-byte aligned with ld * sizeof(T) a multiple of 16 is staged by
 * tensor copies; otherwise by plain loads. m, n, k >= 0; n == 0 or k == 0 does
 * nothing; m == 0 gives OUT = beta * Z (or 0).
 *
 * fp32 with n <= 32, k >= 8 and tensor-copied X runs both products on the tensor
 * cores (8, 16 or 32 right-hand sides a pass): X, Y and each row's v * (x_i . Y)
 * are split into three bfloat16 terms whose products are summed in fp32, which
 * keeps the same bound for inputs of magnitude below 3.39e38 (larger ones round
 * to infinity as bfloat16). The environment variable FXTX_MULTI_TC set to "0"
 * when the library first plans such a call keeps those shapes on the CUDA cores.
 *
 * Each column c meets the bound of fxtx_dense_f32 / _f64 with its own
 * S_jc = |alpha| sum_i |t_ic| |X_ij| + |beta Z_jc|, t_ic = V_ic (x_i . Y[:, c]).
 * Workspace, streams, determinism and errors are those of fxtx_dense_f32.
 */
fxtx_status_t fxtx_dense_multi_f32(int64_t m, int64_t n, int64_t k, const float* X, int64_t ld, const float* Y,
                                   int64_t ldy, const float* V, int64_t ldv, float alpha, float beta, const float* Z,
                                   int64_t ldz, float* OUT, int64_t ldo, void* stream);
fxtx_status_t fxtx_dense_multi_f64(int64_t m, int64_t n, int64_t k, const double* X, int64_t ld, const double* Y,
                                   int64_t ldy, const double* V, int64_t ldv, double alpha, double beta,
                                   const double* Z, int64_t ldz, double* OUT, int64_t ldo, void* stream);

/*
 * fxtx_dense_f32 without any device allocation at call time. (The paper has no
 * counterpart: this entry point exists for callers that cannot allocate.)
 *
 * For callers that must not allocate device memory while they run: code whose
 * device memory belongs to another allocator or runtime, real-time loops that
 * allow no allocation after start-up, or paths that must not touch the stream-
 * ordered memory pool. Arguments and results are those of fxtx_dense_f32.
 *
 * Scratch: one library-wide device array of FXTX_NOALLOC_SCRATCH_BYTES (1 MiB),
 * which every GPU that loads the library holds until the process exits. The
 * first call on a device (with that device current) looks up the array's address
 * and caches it; make that first call before any stream capture. A later call
 * that finds a different context current on the device (after cudaDeviceReset,
 * which reloads the library's device code at a new address) looks it up again.
 * No call allocates or frees memory.
 *
 * Limits: rows of at most 512 fp32 columns (the narrow kernel); n > 512 returns
 * FXTX_ERR_TOO_LARGE. The grid is capped so that the per-CTA partials fit the
 * array.
 *
 * Concurrency: all calls on a device share the array, which keeps the last
 * call's contents (the part that must start at zero is cleared on `stream`
 * before each launch). Calls whose executions overlap on the GPU race on it and
 * give wrong results: order them on one stream or with events.
 */
#define FXTX_NOALLOC_SCRATCH_BYTES (1u << 20)
fxtx_status_t fxtx_dense_f32_noalloc(int64_t m, int64_t n, const float* X, int64_t ld, const float* y,
                                     const float* v, float alpha, float beta, const float* z, float* out,
                                     void* stream);

/*
 * CSR X: row_ptr (int64, m + 1 entries), col_idx (int32, nnz entries), vals
 * (nnz entries). The structure must satisfy row_ptr[0] = 0, row_ptr
 * non-decreasing, row_ptr[m] = nnz and 0 <= col_idx[k] < n; it is NOT checked
 * on this path (see fxtx_csr_validate). Column order inside a row is free and
 * repeated (i, j) entries add. row_ptr, col_idx and vals may be NULL only when
 * m == 0 (row_ptr) or nnz == 0 (col_idx, vals).
 *
 * The scatter into out uses atomic additions, so the order of the column sums,
 * and with it the last bits of out, may differ between calls.
 */
fxtx_status_t fxtx_csr_f32(int64_t m, int64_t n, int64_t nnz, const int64_t* row_ptr,
                           const int32_t* col_idx, const float* vals, const float* y, const float* v,
                           float alpha, float beta, const float* z, float* out, void* stream);
fxtx_status_t fxtx_csr_f64(int64_t m, int64_t n, int64_t nnz, const int64_t* row_ptr,
                           const int32_t* col_idx, const double* vals, const double* y,
                           const double* v, double alpha, double beta, const double* z, double* out,
                           void* stream);

/*
 * The epilogue of a row-sharded call: out = alpha * w + beta * z.
 * ("On optimizing machine learning workloads via kernel fusion", abstract: the
 * generic pattern, whose X^T (v * (X y)) is a sum over the rows of X.)
 *
 * Row sharding: split X by rows into blocks X_g (for CSR, the row_ptr range of the
 * block rebased to start at 0, with its col_idx and vals entries) and v into the
 * matching v_g. Each device computes its partial w_g = X_g^T (v_g * (X_g y)) with
 * the fused entry points above at alpha = 1, beta = 0, z = NULL; the partials are
 * summed across devices (one all-reduce of n values); this call then applies
 * alpha * w + beta * z once. The result meets the bound of a single call up to
 * the rounding of the partials and of their sum (a few units of the working
 * precision times S_j).
 *
 * n >= 0 (n == 0 does nothing); w and out are device pointers of n entries, z of
 * n entries or NULL. z is read only when z != NULL and beta != 0. out may equal w
 * or z (element j is read before it is written); other overlaps are undefined.
 * Asynchronous on `stream`; allocates nothing.
 */
fxtx_status_t fxtx_epilogue_f32(int64_t n, const float* w, float alpha, float beta, const float* z, float* out,
                                void* stream);
fxtx_status_t fxtx_epilogue_f64(int64_t n, const double* w, double alpha, double beta, const double* z, double* out,
                                void* stream);

/*
 * Input-data characteristics of a CSR matrix, read by the launch model ("On
 * optimizing machine learning workloads via kernel fusion", abstract: the
 * analytical model considers input data characteristics and the GPU's resources).
 * All figures come from a strided sample of 8,192 row lengths and 8,192 column
 * indices (positions spread evenly over the rows and over the entries).
 */
typedef struct {
  int64_t row_samples, col_samples;  /* sampled rows and entries (min(m or nnz, 8192)) */
  double mean_row_len, cv_row_len;   /* sampled row lengths: mean and coefficient of variation */
  int64_t p50_row_len, p75_row_len, p90_row_len, max_sampled_row_len;
  double long_row_share;             /* length-weighted share of sampled rows over 2,048 entries */
  int64_t window_c0, window_len;     /* the columns the plan accumulates in shared memory */
  int64_t y_c0, y_len;               /* the entries of y the plan copies to shared memory */
  double window_hit_share, y_hit_share; /* sampled column indices falling in each */
  int32_t group_lanes, group_entries;   /* fp64 lane groups (0 for fp32: packed batches) */
} fxtx_csr_stats_t;

/*
 * Samples a CSR matrix on the device (row_ptr, col_idx: device pointers, as for
 * fxtx_csr_f32/_f64) and records the statistics for later calls on the same
 * matrix: a fxtx_csr_f32/_f64 call whose (current device, row_ptr, col_idx, m, n,
 * nnz) match an analysed matrix plans from them (the fp64 lane groups are sized to
 * the sampled 75th-percentile row, the shared-memory split between the scatter
 * window and the copy of y is chosen, and both are placed, from the sampled
 * columns). Without an analysis every call places the two windows itself, on the
 * device, from its own sample of col_idx, so the call stays asynchronous. The
 * statistics steer launch parameters only, never results; analyse again after
 * changing a matrix in place, or clear. Synchronous on `stream` (one small kernel
 * and two copies of 64 KB and 32 KB). is_f64 selects the element size the returned
 * plan figures are for; `stats` may be NULL. Up to 64 analyses are kept (the oldest
 * is dropped). Errors: FXTX_ERR_INVALID_ARG (sizes, NULL structure), FXTX_ERR_ALLOC,
 * FXTX_ERR_CUDA, FXTX_ERR_UNSUPPORTED.
 */
fxtx_status_t fxtx_csr_analyze(int is_f64, int64_t m, int64_t n, int64_t nnz, const int64_t* row_ptr,
                               const int32_t* col_idx, void* stream, fxtx_csr_stats_t* stats);
/* Forgets every analysis. */
fxtx_status_t fxtx_csr_analysis_clear(void);

/*
 * The plan the model picks for a CSR matrix given as HOST arrays (row_ptr: m + 1
 * entries, col_idx: nnz entries), from the same sample positions as
 * fxtx_csr_analyze. Host only, no device needed (without a GB300 current it plans
 * for 152 SMs and 227 KB of shared memory). Writes the statistics to `stats` (may
 * be NULL) and a NUL-terminated description of at most `cap` bytes to `buf` (may
 * be NULL).
 */
fxtx_status_t fxtx_csr_plan_describe_host(int is_f64, int64_t m, int64_t n, int64_t nnz, const int64_t* row_ptr,
                                          const int32_t* col_idx, fxtx_csr_stats_t* stats, char* buf, int64_t cap);

/*
 * Checks a CSR structure on the device (row_ptr[0] == 0, non-decreasing,
 * row_ptr[m] == nnz, 0 <= col_idx < n). Synchronous: it waits for `stream`.
 * Returns FXTX_OK or FXTX_ERR_BAD_CSR (or an argument/CUDA error).
 */
fxtx_status_t fxtx_csr_validate(int64_t m, int64_t n, int64_t nnz, const int64_t* row_ptr,
                                const int32_t* col_idx, void* stream);

/*
 * Reads and clears the device-side error word of the current device: FXTX_OK,
 * or FXTX_ERR_TIMEOUT when a kernel abandoned a bounded wait since the last
 * read (its output is then invalid). Synchronous on `stream`.
 */
fxtx_status_t fxtx_device_error(void* stream);

/* A static string naming a status code. */
const char* fxtx_status_string(fxtx_status_t status);

/*
 * The launch plan the analytical model picks for a dense or CSR call, for
 * logging and tests. Host only; nothing is launched. For CSR this is the plan
 * from the shape alone (m, n, nnz): the window placement is then left to each
 * call's device-side sample ("placement=device"); fxtx_csr_plan_describe_host
 * gives the plan that sampled statistics lead to. Writes a NUL-terminated
 * description of at most `cap` bytes into `buf` and returns FXTX_OK.
 */
fxtx_status_t fxtx_plan_describe(int is_csr, int is_f64, int64_t m, int64_t n, int64_t nnz,
                                  int64_t ld, char* buf, int64_t cap);

/*
 * One-shot autotuning of the launch model ("On optimizing machine learning workloads
 * via kernel fusion", abstract: the analytical model for launch parameters; the model
 * picks by default). With mode 1, the first dense or CSR call of each shape (m, n,
 * nnz, ld, element type, alignment class and SM count) runs each of the model's
 * candidate launches once to warm up and three times timed, on the caller's stream,
 * and caches the fastest; that call synchronises the stream and leaves the result of
 * the chosen launch in out. The timed runs write to a scratch vector of n elements
 * (cudaMallocAsync on the stream; if it cannot be had, the call takes the model's plan
 * untimed), so out may equal z on that call too. Later calls of the shape, and calls
 * during stream capture, launch without timing (the model's plan when the shape is not
 * cached). The cache is process-wide and thread-safe. The initial mode is 1 when the
 * environment variable FXTX_AUTOTUNE is "1", else 0. The multi-vector and no-allocation
 * entry points always take the model's plan.
 *
 * fxtx_autotune_set: mode 0 or 1 (else FXTX_ERR_INVALID_ARG). fxtx_autotune_save /
 * _load: a text file, one cached shape per line ("kind elem m n nnz ld flags sm_count
 * choice candidates best_us model_us", '#' lines ignored); load replaces the cache and
 * returns FXTX_ERR_INVALID_ARG, leaving it unchanged, for a missing file or a
 * malformed line. fxtx_autotune_candidates writes the candidate plans of a shape, the
 * model's first, one per line, as fxtx_plan_describe does (host only).
 */
fxtx_status_t fxtx_autotune_set(int mode);
int fxtx_autotune_get(void);
int64_t fxtx_autotune_entries(void);
fxtx_status_t fxtx_autotune_clear(void);
fxtx_status_t fxtx_autotune_save(const char* path);
fxtx_status_t fxtx_autotune_load(const char* path);
fxtx_status_t fxtx_autotune_candidates(int is_csr, int is_f64, int64_t m, int64_t n, int64_t nnz, int64_t ld,
                                       char* buf, int64_t cap);

/*
 * The launch plan of a multi-vector call (fxtx_dense_multi_*), for logging and
 * tests: v_mode 0 = no weights, 1 = one shared m-vector, 2 = an m x k matrix.
 * Host only; writes a NUL-terminated description of at most `cap` bytes.
 */
fxtx_status_t fxtx_multi_plan_describe(int is_f64, int64_t m, int64_t n, int64_t k, int64_t ld, int v_mode, char* buf,
                                       int64_t cap);

#ifdef __cplusplus
}
#endif

#endif /* FXTX_H */
