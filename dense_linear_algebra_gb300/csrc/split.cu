// split.cu — the epilogue of a row-sharded call:
//     out = alpha * w + beta * z
// The pattern is a sum over rows ("On optimizing machine learning workloads via
// kernel fusion", abstract: X^T (v * (X y)) = sum_i t_i x_i), so a matrix split
// by rows across devices gives each device a partial w_g = X_g^T (v_g * (X_g y))
// (a fused call with alpha = 1, beta = 0 on its rows); after the partials are
// summed across devices this kernel applies the epilogue once. It is the same
// epilogue the fused kernels apply in their last step, in fp64 and rounded once.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace fxtx {

template <typename T>
__global__ void __launch_bounds__(256) epilogue_kernel(int64_t n, const T* w, double alpha, double beta, const T* z,
                                                       bool use_z, T* out) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += stride) {
    double o = alpha * (double)w[j];
    if (use_z) o += beta * (double)z[j];
    out[j] = (T)o;
  }
}

template <typename T>
cudaError_t launch_epilogue(int64_t n, const T* w, double alpha, double beta, const T* z, bool use_z, T* out,
                            int sm_count, cudaStream_t st) {
  if (n == 0) return cudaSuccess;
  const int64_t blocks = std::min<int64_t>((n + 255) / 256, (int64_t)std::max(sm_count, 1) * 8);
  epilogue_kernel<T><<<(unsigned)blocks, 256, 0, st>>>(n, w, alpha, beta, z, use_z, out);
  return cudaGetLastError();
}

template cudaError_t launch_epilogue<float>(int64_t, const float*, double, double, const float*, bool, float*, int,
                                            cudaStream_t);
template cudaError_t launch_epilogue<double>(int64_t, const double*, double, double, const double*, bool, double*,
                                             int, cudaStream_t);

}  // namespace fxtx
