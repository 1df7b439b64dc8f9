// kernels.h — argument blocks and launchers of the fused kernels (host-visible).
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "plan.h"

namespace fxtx {

// One dense call. T is the compute type of y, v, z and out; TX the storage type of X
// (T itself, or bfloat16 with T = float). alpha and beta are carried in double.
template <typename T, typename TX = T>
struct DenseArgs {
  int64_t m = 0, n = 0, ld = 0;
  const TX* X = nullptr;
  const T* y = nullptr;
  const T* v = nullptr;  // NULL: v_i = 1
  const T* z = nullptr;  // read only when use_z
  T* out = nullptr;
  double alpha = 1.0, beta = 0.0;
  bool use_z = false;
  double* ws = nullptr;         // [ctas][n] column partials of each CTA
  unsigned* ticket = nullptr;   // arrival counter of the last-CTA reduction, zero at launch
  int64_t tiles = 0;            // ceil(m / rows_per_tile)
};

template <typename T>
cudaError_t launch_dense(const DensePlan& p, const DenseArgs<T>& a, cudaStream_t st);

// X stored as bfloat16, computed in fp32 (tile kernel, or the direct-load narrow kernel).
cudaError_t launch_dense_bf16(const DensePlan& p, const DenseArgs<float, __nv_bfloat16>& a, cudaStream_t st);

// One CSR call. alpha is folded into t_i; out is pre-set to beta z (or 0) by the
// prologue and then receives atomic additions.
template <typename T>
struct CsrArgs {
  int64_t m = 0, n = 0, nnz = 0;
  const int64_t* row_ptr = nullptr;
  const int32_t* col_idx = nullptr;
  const T* vals = nullptr;
  const T* y = nullptr;
  const T* v = nullptr;
  const T* z = nullptr;
  T* out = nullptr;
  double alpha = 1.0, beta = 0.0;
  bool use_z = false;
  int64_t* part = nullptr;       // [ctas + 1] row partition of the row-group kernel
  int64_t* queue = nullptr;      // [buckets][queue_cap] rows deferred to the long-row kernel, by length
  int64_t queue_cap = 0;
  int64_t* med_queue = nullptr;  // [med_cap] rows too long for the row kernel's batches, taken one warp each
  int64_t med_cap = 0;
  // [0] long-row claims, [1 .. buckets] bucket lengths, [buckets + 1] row windows handed out,
  // [8], [9] the window starts, [10] medium rows queued, [11] medium rows claimed
  unsigned long long* counters = nullptr;
};

template <typename T>
cudaError_t launch_csr(const CsrPlan& p, const CsrArgs<T>& a, cudaStream_t st);

cudaError_t launch_csr_validate(int64_t m, int64_t n, int64_t nnz, const int64_t* row_ptr,
                                const int32_t* col_idx, int* flag, cudaStream_t st);

// Gathers the model's strided sample: kCsrSamples row lengths into lens and column indices
// into cols (the first min(m, kCsrSamples) and min(nnz, kCsrSamples) entries are written).
cudaError_t launch_csr_sample(int64_t m, int64_t nnz, const int64_t* row_ptr, const int32_t* col_idx, int64_t* lens,
                              int32_t* cols, cudaStream_t st);

// out = alpha * w + beta * z (z read only when use_z): the epilogue of a row-sharded call,
// applied once after the devices' partials are summed.
template <typename T>
cudaError_t launch_epilogue(int64_t n, const T* w, double alpha, double beta, const T* z, bool use_z, T* out,
                            int sm_count, cudaStream_t st);

// Read and clear the device-side error word of each kernel file (synchronous;
// -1 if the read itself failed).
int take_dense_device_error();
int take_csr_device_error();

// Ensures a kernel may use `bytes` of dynamic shared memory on the current device.
cudaError_t ensure_smem(const void* kernel, size_t bytes);

}  // namespace fxtx
