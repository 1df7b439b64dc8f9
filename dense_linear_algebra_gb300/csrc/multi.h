// multi.h — the multi-vector instantiation: k right-hand sides in one pass over X.
//
//   OUT = alpha * X^T (V ⊙ (X Y)) + beta * Z,   Y, Z, OUT: n x k row-major;
//   V: m x k row-major, one m-vector shared by all k columns (ldv = 0), or absent.
//
// "On optimizing machine learning workloads via kernel fusion" (abstract) names the
// fused pattern and its instantiations; with k right-hand sides, one read of X serves
// k products.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "plan.h"

namespace fxtx {

// One pass over X for kb right-hand sides (columns c0 .. c0 + kb of Y, V, Z and OUT;
// the pointers below already point at column c0).
template <typename T>
struct MultiArgs {
  int64_t m = 0, n = 0, ld = 0;
  const T* X = nullptr;
  const T* Y = nullptr;
  int64_t ldy = 0;
  const T* V = nullptr;  // NULL: all weights 1
  int64_t ldv = 0;       // 0: V is one m-vector shared by every right-hand side
  const T* Z = nullptr;  // read only when use_z
  int64_t ldz = 0;
  T* OUT = nullptr;
  int64_t ldo = 0;
  int kb = 0;            // right-hand sides of this pass (<= the kernel's KB)
  double alpha = 1.0, beta = 0.0;
  bool use_z = false;
  double* ws = nullptr;        // [ctas][n * KB] partials of each CTA
  unsigned* ticket = nullptr;  // arrival counter of the last-CTA reduction, zero at launch
  int64_t tiles = 0;           // ceil(m / rows per tile), set by the launcher for the pass's kernel
};

// Launch shape of one multi-vector call. A call of k right-hand sides runs
// ceil(k / kb_max) passes; the last one may take fewer.
struct MultiPlan {
  bool ok = false;      // false: the shape is not taken (n * elem > 2 KB)
  bool tma = false;     // X staged by tensor copies (else by plain loads)
  int nb = 0;           // 128-byte blocks per row (1, 2, 4, 8, 16)
  int kb_max = 0;       // right-hand sides per pass (a power of two, 32 / nb at most)
  int passes = 0;
  int rows_per_tile = 0;  // of a kb_max-wide pass (a narrower last pass may take taller tiles)
  int stages = 0;
  int warps = 0;
  int ctas = 0;
  size_t smem = 0;
  size_t ws_bytes = 0;  // per-CTA partials of the widest pass, plus the ticket
  double est_us = 0.0;  // the model's estimate of the call (all passes)
  bool tc = false;      // fp32, n <= 32, k >= 8: X^T T on the tensor cores (multi_tc.cu)
};

MultiPlan plan_multi(const DeviceInfo& dev, int64_t m, int64_t n, int64_t k, int elem, bool tma_ok, bool full_v,
                     bool has_v);

// The right-hand sides the pass starting at column c0 takes.
int multi_pass_kb(const MultiPlan& p, int64_t k, int64_t c0);

template <typename T>
cudaError_t launch_multi(const MultiPlan& p, const MultiArgs<T>& a, cudaStream_t st);

// The tensor-core form (fp32 X of at most 32 columns, kb_max = 8, 16 or 32 right-hand sides
// a pass): its dynamic shared memory, its X pipeline depth, and its launcher.
size_t multi_tc_smem(int kb);
int multi_tc_stages(int kb);
int multi_tc_warps(int kb);
cudaError_t launch_multi_tc(const MultiPlan& p, const MultiArgs<float>& a, cudaStream_t st);

int describe_multi(const MultiPlan& p, char* buf, size_t cap);

// Reads and clears the device-side error word of the multi-vector kernels (synchronous).
int take_multi_device_error();

}  // namespace fxtx
