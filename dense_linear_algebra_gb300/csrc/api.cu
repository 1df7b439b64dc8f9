// api.cu — the C ABI of libfusedxtx (declared in include/fxtx.h): argument
// checks, the launch plan, transient workspace and the launches, all enqueued
// on the caller's stream.
#include <cstdio>
#include <cstdlib>
#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "fxtx.h"
#include "kernels.h"
#include "multi.h"
#include "plan.h"
#include "tune.h"

namespace fxtx {
namespace {

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
std::once_flag g_dev_once[kMaxDevices];

// Properties of the current device, queried once per device.
fxtx_status_t current_device(const DeviceInfo** out) {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) {
    cudaGetLastError();
    return FXTX_ERR_UNSUPPORTED;
  }
  std::call_once(g_dev_once[d], [d] {
    DeviceInfo& di = g_dev[d];
    di.device = d;
    cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, d);
    cudaDeviceGetAttribute(&di.cc_major, cudaDevAttrComputeCapabilityMajor, d);
    cudaDeviceGetAttribute(&di.cc_minor, cudaDevAttrComputeCapabilityMinor, d);
    cudaDeviceGetAttribute(&di.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
    cudaDeviceGetAttribute(&di.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, d);
    cudaGetLastError();
  });
  const DeviceInfo& di = g_dev[d];
  if (di.cc_major != 10 || di.cc_minor != 3 || di.sm_count <= 0) return FXTX_ERR_UNSUPPORTED;
  *out = &di;
  return FXTX_OK;
}

bool log_enabled() {
  static const bool on = [] {
    const char* s = getenv("FXTX_LOG");
    return s && s[0] && s[0] != '0';
  }();
  return on;
}

// Test hook: FXTX_FAIL_ALLOC=1 makes every workspace allocation fail (host side).
bool fail_alloc() {
  const char* s = getenv("FXTX_FAIL_ALLOC");
  return s && s[0] == '1';
}

fxtx_status_t alloc_ws(void** p, size_t bytes, cudaStream_t st) {
  *p = nullptr;
  if (bytes == 0) return FXTX_OK;
  if (fail_alloc()) return FXTX_ERR_ALLOC;
  if (cudaMallocAsync(p, bytes, st) != cudaSuccess) {
    cudaGetLastError();
    *p = nullptr;
    return FXTX_ERR_ALLOC;
  }
  return FXTX_OK;
}

// Sampled statistics of analysed CSR matrices (fxtx_csr_analyze), keyed by device,
// structure pointers and sizes. They steer launch parameters only, never results.
struct Analysis {
  int dev;
  const void* row_ptr;
  const void* col_idx;
  int64_t m, n, nnz;
  CsrStats stats;
};
constexpr size_t kMaxAnalyses = 64;
std::mutex g_an_mu;
std::vector<Analysis> g_an;  // most recent last

bool find_analysis(int dev, const void* rp, const void* ci, int64_t m, int64_t n, int64_t nnz, CsrStats* out) {
  std::lock_guard<std::mutex> lock(g_an_mu);
  for (auto it = g_an.rbegin(); it != g_an.rend(); ++it)
    if (it->dev == dev && it->row_ptr == rp && it->col_idx == ci && it->m == m && it->n == n && it->nnz == nnz) {
      *out = it->stats;
      return true;
    }
  return false;
}

void store_analysis(const Analysis& a) {
  std::lock_guard<std::mutex> lock(g_an_mu);
  for (auto it = g_an.begin(); it != g_an.end(); ++it)
    if (it->dev == a.dev && it->row_ptr == a.row_ptr && it->col_idx == a.col_idx && it->m == a.m && it->n == a.n &&
        it->nnz == a.nnz) {
      g_an.erase(it);
      break;
    }
  if (g_an.size() >= kMaxAnalyses) g_an.erase(g_an.begin());
  g_an.push_back(a);
}

template <typename T>
bool aligned16(const T* p) {
  return (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

// Compute type of the vectors for X stored as TX (bfloat16 X computes in fp32).
template <typename TX>
struct DenseT {
  using T = TX;
};
template <>
struct DenseT<__nv_bfloat16> {
  using T = float;
};

// One dense launch with its own transient workspace (the column partials and the
// ticket of the last-CTA reduction).
template <typename TX>
fxtx_status_t run_dense(const DensePlan& plan, DenseArgs<typename DenseT<TX>::T, TX> a, cudaStream_t st) {
  a.tiles = plan.rows_per_tile > 0 ? (a.m + plan.rows_per_tile - 1) / plan.rows_per_tile : 0;
  void* ws = nullptr;
  fxtx_status_t s = alloc_ws(&ws, plan.ws_bytes, st);
  if (s != FXTX_OK) return s;
  if (ws) {
    a.ws = static_cast<double*>(ws);
    a.ticket = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + plan.ws_bytes - 128);
    const cudaError_t e = cudaMemsetAsync(a.ticket, 0, sizeof(unsigned), st);
    if (e != cudaSuccess) {
      cudaGetLastError();
      cudaFreeAsync(ws, st);
      return FXTX_ERR_CUDA;
    }
  }
  cudaError_t e;
  if constexpr (sizeof(TX) == 2)
    e = launch_dense_bf16(plan, a, st);
  else
    e = launch_dense<TX>(plan, a, st);
  if (ws) cudaFreeAsync(ws, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FXTX_ERR_CUDA;
  }
  return FXTX_OK;
}

// One CSR call (prologue, row kernel, long-row kernel) with its own workspace.
template <typename T>
fxtx_status_t run_csr(const CsrPlan& plan, CsrArgs<T> a, cudaStream_t st) {
  void* ws = nullptr;
  fxtx_status_t s = alloc_ws(&ws, plan.ws_bytes, st);
  if (s != FXTX_OK) return s;
  char* w = static_cast<char*>(ws);
  const size_t part_bytes = ((size_t)(plan.ctas + 1) * 8 + 127) / 128 * 128;
  const size_t queue_bytes =
      ((size_t)csr_long_buckets() * (size_t)std::max<int64_t>(plan.queue_cap, 1) * 8 + 127) / 128 * 128;
  a.part = reinterpret_cast<int64_t*>(w);
  a.queue = reinterpret_cast<int64_t*>(w + part_bytes);
  a.queue_cap = plan.queue_cap;
  a.med_queue = reinterpret_cast<int64_t*>(w + part_bytes + queue_bytes);
  a.med_cap = plan.med_cap;
  a.counters = reinterpret_cast<unsigned long long*>(w + plan.ws_bytes - 128);
  cudaError_t e = launch_csr<T>(plan, a, st);
  cudaFreeAsync(ws, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FXTX_ERR_CUDA;
  }
  return FXTX_OK;
}

// The candidate to launch for `key`: the model's plan (index 0) unless autotuning is on.
// On a cache miss outside stream capture, every candidate runs once to warm up and
// then three times between events on the caller's stream (so the call synchronises),
// and the fastest is cached. `run(plan, o)` enqueues one complete call with a
// candidate, writing to `o` instead of out when `o` is not NULL: the timed runs write
// to a scratch vector of `out_bytes`, so out keeps its value (and z, which out may
// equal, is read unchanged by every run).
template <typename P, typename Run>
int choose(const TuneKey& key, const std::vector<P>& cands, Run run, size_t out_bytes, cudaStream_t st) {
  if (cands.size() < 2 || tune_mode() == 0) return 0;
  int choice = 0;
  if (tune_lookup(key, &choice)) return choice < (int)cands.size() ? choice : 0;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
    cudaGetLastError();
    return 0;
  }
  void* scratch = nullptr;
  if (alloc_ws(&scratch, out_bytes, st) != FXTX_OK) return 0;
  cudaEvent_t e0, e1;
  if (cudaEventCreate(&e0) != cudaSuccess) {
    cudaGetLastError();
    cudaFreeAsync(scratch, st);
    return 0;
  }
  if (cudaEventCreate(&e1) != cudaSuccess) {
    cudaGetLastError();
    cudaEventDestroy(e0);
    cudaFreeAsync(scratch, st);
    return 0;
  }
  double best = 0.0;
  int bi = -1;
  for (int i = 0; i < (int)cands.size(); ++i) {
    if (run(cands[i], scratch) != FXTX_OK) continue;
    float t = 0.f, tmin = 0.f;
    bool ok = true;
    for (int rep = 0; rep < 3 && ok; ++rep) {
      ok = cudaEventRecord(e0, st) == cudaSuccess && run(cands[i], scratch) == FXTX_OK &&
           cudaEventRecord(e1, st) == cudaSuccess && cudaEventSynchronize(e1) == cudaSuccess &&
           cudaEventElapsedTime(&t, e0, e1) == cudaSuccess;
      if (ok && (rep == 0 || t < tmin)) tmin = t;
    }
    if (ok && (bi < 0 || tmin * 1e3 < best)) {
      best = tmin * 1e3;
      bi = i;
    }
  }
  cudaGetLastError();
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  cudaFreeAsync(scratch, st);
  cudaGetLastError();
  if (bi < 0) return 0;
  tune_store(key, bi, (int)cands.size(), best, cands[0].est_us);
  if (log_enabled())
    fprintf(stderr, "[fxtx] autotune kind=%d m=%lld n=%lld nnz=%lld: candidate %d of %d, %.1f us (model estimate %.1f us)\n",
            key.kind, (long long)key.m, (long long)key.n, (long long)key.nnz, bi, (int)cands.size(), best,
            cands[0].est_us);
  return bi;
}

template <typename TX>
fxtx_status_t dense_impl(int64_t m, int64_t n, const TX* X, int64_t ld, const typename DenseT<TX>::T* y,
                         const typename DenseT<TX>::T* v, typename DenseT<TX>::T alpha,
                         typename DenseT<TX>::T beta, const typename DenseT<TX>::T* z, typename DenseT<TX>::T* out,
                         void* stream) {
  using T = typename DenseT<TX>::T;
  if (m < 0 || n < 0) return FXTX_ERR_INVALID_ARG;
  if (n == 0) return FXTX_OK;
  if (ld < n || y == nullptr || out == nullptr) return FXTX_ERR_INVALID_ARG;
  if (m > 0 && X == nullptr) return FXTX_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  fxtx_status_t s = current_device(&dev);
  if (s != FXTX_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  const int elem = (int)sizeof(TX);
  const bool tile_ok = aligned16(X) && (ld * elem) % 16 == 0;
  // bfloat16 X takes the tile kernel or the direct-load narrow kernel only
  const bool tma_ok = elem != 2 && tile_ok && (n * elem) % 16 == 0;
  const DensePlan model = plan_dense(*dev, m, n, ld, elem, tma_ok, tile_ok);
  if (elem == 2 && (model.kind == DENSE_WIDE || model.kind == DENSE_NARROW_TMA)) return FXTX_ERR_UNSUPPORTED;

  DenseArgs<T, TX> a;
  a.m = m; a.n = n; a.ld = ld;
  a.X = X; a.y = y; a.v = v; a.z = z; a.out = out;
  a.alpha = (double)alpha; a.beta = (double)beta;
  a.use_z = (z != nullptr && beta != T(0));

  const std::vector<DensePlan> cands = dense_candidates(*dev, model, m, n, elem);
  TuneKey key;
  key.kind = 0; key.elem = elem; key.m = m; key.n = n; key.ld = ld;
  key.flags = (tile_ok ? 1 : 0) | (tma_ok ? 2 : 0);
  key.sm_count = dev->sm_count;
  auto run = [&](const DensePlan& p, void* o) {
    DenseArgs<T, TX> b = a;
    if (o) b.out = static_cast<T*>(o);
    return run_dense<TX>(p, b, st);
  };
  const DensePlan& plan = cands[choose(key, cands, run, (size_t)n * sizeof(T), st)];
  if (log_enabled()) {
    char buf[320];
    describe(plan, buf, sizeof buf);
    fprintf(stderr, "[fxtx] %s m=%lld n=%lld ld=%lld %s\n", elem == 2 ? "bf16" : "dense", (long long)m, (long long)n,
            (long long)ld, buf);
  }
  return run_dense<TX>(plan, a, st);
}

template <typename T>
fxtx_status_t csr_impl(int64_t m, int64_t n, int64_t nnz, const int64_t* row_ptr, const int32_t* col_idx,
                       const T* vals, const T* y, const T* v, T alpha, T beta, const T* z, T* out, void* stream) {
  if (m < 0 || n < 0 || nnz < 0) return FXTX_ERR_INVALID_ARG;
  if (n == 0) return FXTX_OK;
  if (n > INT32_MAX || y == nullptr || out == nullptr) return FXTX_ERR_INVALID_ARG;
  if (m > 0 && row_ptr == nullptr) return FXTX_ERR_INVALID_ARG;
  if (nnz > 0 && (col_idx == nullptr || vals == nullptr)) return FXTX_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  fxtx_status_t s = current_device(&dev);
  if (s != FXTX_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  CsrStats stats;
  const bool analysed = find_analysis(dev->device, row_ptr, col_idx, m, n, nnz, &stats);
  const CsrStats* sp = analysed ? &stats : nullptr;
  const CsrPlan model = plan_csr(*dev, m, n, nnz, (int)sizeof(T), sp);
  CsrArgs<T> a;
  a.m = m; a.n = n; a.nnz = nnz;
  a.row_ptr = row_ptr; a.col_idx = col_idx; a.vals = vals;
  a.y = y; a.v = v; a.z = z; a.out = out;
  a.alpha = (double)alpha; a.beta = (double)beta;
  a.use_z = (z != nullptr && beta != T(0));

  const std::vector<CsrPlan> cands = csr_candidates(*dev, model, m, n, nnz, (int)sizeof(T), sp);
  TuneKey key;
  key.kind = 1; key.elem = (int)sizeof(T); key.m = m; key.n = n; key.nnz = nnz;
  key.flags = analysed ? 1 : 0;
  key.sm_count = dev->sm_count;
  auto run = [&](const CsrPlan& p, void* o) {
    CsrArgs<T> b = a;
    if (o) b.out = static_cast<T*>(o);
    return run_csr<T>(p, b, st);
  };
  const CsrPlan& plan = cands[choose(key, cands, run, (size_t)n * sizeof(T), st)];
  if (log_enabled()) {
    char buf[512];
    describe(plan, buf, sizeof buf);
    fprintf(stderr, "[fxtx] m=%lld n=%lld nnz=%lld %s\n", (long long)m, (long long)n, (long long)nnz, buf);
  }
  return run_csr<T>(plan, a, st);
}

// k right-hand sides: ceil(k / kb) passes over X, each for kb of them.
template <typename T>
fxtx_status_t dense_multi_impl(int64_t m, int64_t n, int64_t k, const T* X, int64_t ld, const T* Y, int64_t ldy,
                               const T* V, int64_t ldv, T alpha, T beta, const T* Z, int64_t ldz, T* OUT,
                               int64_t ldo, void* stream) {
  if (m < 0 || n < 0 || k < 0) return FXTX_ERR_INVALID_ARG;
  if (n == 0 || k == 0) return FXTX_OK;
  if (ld < n || Y == nullptr || OUT == nullptr || ldy < k || ldo < k) return FXTX_ERR_INVALID_ARG;
  if (m > 0 && X == nullptr) return FXTX_ERR_INVALID_ARG;
  if (V != nullptr && ldv != 0 && ldv < k) return FXTX_ERR_INVALID_ARG;
  if (ldv < 0) return FXTX_ERR_INVALID_ARG;
  const bool use_z = Z != nullptr && beta != T(0);
  if (use_z && ldz < k) return FXTX_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  fxtx_status_t s = current_device(&dev);
  if (s != FXTX_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  const int elem = (int)sizeof(T);
  const bool tma_ok = aligned16(X) && (ld * elem) % 16 == 0;
  const MultiPlan plan = plan_multi(*dev, m, n, k, elem, tma_ok, V != nullptr && ldv != 0, V != nullptr);
  if (!plan.ok) return FXTX_ERR_UNSUPPORTED;
  if (log_enabled()) {
    char buf[256];
    describe_multi(plan, buf, sizeof buf);
    fprintf(stderr, "[fxtx] m=%lld n=%lld k=%lld ld=%lld %s\n", (long long)m, (long long)n, (long long)k,
            (long long)ld, buf);
  }

  void* ws = nullptr;
  s = alloc_ws(&ws, plan.ws_bytes, st);
  if (s != FXTX_OK) return s;
  MultiArgs<T> a;
  a.m = m; a.n = n; a.ld = ld; a.X = X;
  a.ldy = ldy; a.ldv = V != nullptr ? ldv : 0; a.ldz = ldz; a.ldo = ldo;
  a.alpha = (double)alpha; a.beta = (double)beta; a.use_z = use_z;
  a.ws = static_cast<double*>(ws);
  a.ticket = reinterpret_cast<unsigned*>(static_cast<char*>(ws) + plan.ws_bytes - 128);
  cudaError_t e = cudaMemsetAsync(a.ticket, 0, sizeof(unsigned), st);
  for (int64_t c0 = 0; c0 < k && e == cudaSuccess; c0 += a.kb) {
    a.kb = multi_pass_kb(plan, k, c0);
    a.Y = Y + c0;
    a.V = V == nullptr ? nullptr : (ldv != 0 ? V + c0 : V);
    a.Z = use_z ? Z + c0 : nullptr;
    a.OUT = OUT + c0;
    e = launch_multi<T>(plan, a, st);
  }
  cudaFreeAsync(ws, st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FXTX_ERR_CUDA;
  }
  return FXTX_OK;
}

template <typename T>
fxtx_status_t epilogue_impl(int64_t n, const T* w, T alpha, T beta, const T* z, T* out, void* stream) {
  if (n < 0) return FXTX_ERR_INVALID_ARG;
  if (n == 0) return FXTX_OK;
  if (w == nullptr || out == nullptr) return FXTX_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  fxtx_status_t s = current_device(&dev);
  if (s != FXTX_OK) return s;
  const bool use_z = z != nullptr && beta != T(0);
  if (launch_epilogue<T>(n, w, (double)alpha, (double)beta, z, use_z, out, dev->sm_count,
                         static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return FXTX_ERR_CUDA;
  }
  return FXTX_OK;
}

void fill_stats(const CsrStats& st, const CsrPlan& p, fxtx_csr_stats_t* out) {
  out->row_samples = st.row_samples;
  out->col_samples = st.col_samples;
  out->mean_row_len = st.mean_len;
  out->cv_row_len = st.cv_len;
  out->p50_row_len = st.p50_len;
  out->p75_row_len = st.p75_len;
  out->p90_row_len = st.p90_len;
  out->max_sampled_row_len = st.max_len;
  out->long_row_share = st.long_share;
  out->window_c0 = p.win_c0;
  out->window_len = p.win_len;
  out->y_c0 = p.y0;
  out->y_len = p.ylen;
  out->window_hit_share = p.win_hit;
  out->y_hit_share = p.y_hit;
  out->group_lanes = p.group_lpr;
  out->group_entries = p.group_kg;
}

const DeviceInfo* device_or_fallback(DeviceInfo* fallback) {
  const DeviceInfo* dev = nullptr;
  if (current_device(&dev) == FXTX_OK) return dev;
  // no GB300 current: a 152-SM device with 227 KB of shared memory per block
  fallback->sm_count = 152;
  fallback->cc_major = 10;
  fallback->cc_minor = 3;
  fallback->smem_optin = 232448;
  fallback->smem_per_sm = 233472;
  return fallback;
}

}  // namespace
}  // namespace fxtx

using namespace fxtx;

extern "C" {

fxtx_status_t fxtx_dense_f32(int64_t m, int64_t n, const float* X, int64_t ld, const float* y, const float* v,
                             float alpha, float beta, const float* z, float* out, void* stream) {
  return dense_impl<float>(m, n, X, ld, y, v, alpha, beta, z, out, stream);
}

fxtx_status_t fxtx_dense_f64(int64_t m, int64_t n, const double* X, int64_t ld, const double* y, const double* v,
                             double alpha, double beta, const double* z, double* out, void* stream) {
  return dense_impl<double>(m, n, X, ld, y, v, alpha, beta, z, out, stream);
}

fxtx_status_t fxtx_dense_bf16(int64_t m, int64_t n, const uint16_t* X, int64_t ld, const float* y, const float* v,
                              float alpha, float beta, const float* z, float* out, void* stream) {
  return dense_impl<__nv_bfloat16>(m, n, reinterpret_cast<const __nv_bfloat16*>(X), ld, y, v, alpha, beta, z, out,
                                   stream);
}

fxtx_status_t fxtx_dense_multi_f32(int64_t m, int64_t n, int64_t k, const float* X, int64_t ld, const float* Y,
                                   int64_t ldy, const float* V, int64_t ldv, float alpha, float beta, const float* Z,
                                   int64_t ldz, float* OUT, int64_t ldo, void* stream) {
  return dense_multi_impl<float>(m, n, k, X, ld, Y, ldy, V, ldv, alpha, beta, Z, ldz, OUT, ldo, stream);
}

fxtx_status_t fxtx_dense_multi_f64(int64_t m, int64_t n, int64_t k, const double* X, int64_t ld, const double* Y,
                                   int64_t ldy, const double* V, int64_t ldv, double alpha, double beta,
                                   const double* Z, int64_t ldz, double* OUT, int64_t ldo, void* stream) {
  return dense_multi_impl<double>(m, n, k, X, ld, Y, ldy, V, ldv, alpha, beta, Z, ldz, OUT, ldo, stream);
}

fxtx_status_t fxtx_csr_f32(int64_t m, int64_t n, int64_t nnz, const int64_t* row_ptr, const int32_t* col_idx,
                           const float* vals, const float* y, const float* v, float alpha, float beta, const float* z,
                           float* out, void* stream) {
  return csr_impl<float>(m, n, nnz, row_ptr, col_idx, vals, y, v, alpha, beta, z, out, stream);
}

fxtx_status_t fxtx_csr_f64(int64_t m, int64_t n, int64_t nnz, const int64_t* row_ptr, const int32_t* col_idx,
                           const double* vals, const double* y, const double* v, double alpha, double beta,
                           const double* z, double* out, void* stream) {
  return csr_impl<double>(m, n, nnz, row_ptr, col_idx, vals, y, v, alpha, beta, z, out, stream);
}

fxtx_status_t fxtx_epilogue_f32(int64_t n, const float* w, float alpha, float beta, const float* z, float* out,
                                void* stream) {
  return epilogue_impl<float>(n, w, alpha, beta, z, out, stream);
}

fxtx_status_t fxtx_epilogue_f64(int64_t n, const double* w, double alpha, double beta, const double* z, double* out,
                                void* stream) {
  return epilogue_impl<double>(n, w, alpha, beta, z, out, stream);
}

fxtx_status_t fxtx_csr_validate(int64_t m, int64_t n, int64_t nnz, const int64_t* row_ptr, const int32_t* col_idx,
                                void* stream) {
  if (m < 0 || n < 0 || nnz < 0) return FXTX_ERR_INVALID_ARG;
  if (m == 0 && row_ptr == nullptr) return nnz == 0 ? FXTX_OK : FXTX_ERR_BAD_CSR;
  if (row_ptr == nullptr || (nnz > 0 && col_idx == nullptr)) return FXTX_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  fxtx_status_t s = current_device(&dev);
  if (s != FXTX_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* flag = nullptr;
  s = alloc_ws(&flag, sizeof(int), st);
  if (s != FXTX_OK) return s;
  int host = 0;
  cudaError_t e = cudaMemsetAsync(flag, 0, sizeof(int), st);
  if (e == cudaSuccess) e = launch_csr_validate(m, n, nnz, row_ptr, col_idx, static_cast<int*>(flag), st);
  if (e == cudaSuccess) e = cudaMemcpyAsync(&host, flag, sizeof(int), cudaMemcpyDeviceToHost, st);
  cudaFreeAsync(flag, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return FXTX_ERR_CUDA;
  }
  return host ? FXTX_ERR_BAD_CSR : FXTX_OK;
}

fxtx_status_t fxtx_csr_analyze(int is_f64, int64_t m, int64_t n, int64_t nnz, const int64_t* row_ptr,
                               const int32_t* col_idx, void* stream, fxtx_csr_stats_t* stats) {
  if (m < 0 || n < 0 || nnz < 0 || n > INT32_MAX) return FXTX_ERR_INVALID_ARG;
  if ((m > 0 && row_ptr == nullptr) || (nnz > 0 && col_idx == nullptr)) return FXTX_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  fxtx_status_t s = current_device(&dev);
  if (s != FXTX_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  std::vector<int64_t> lens(kCsrSamples, 0);
  std::vector<int32_t> cols(kCsrSamples, 0);
  const int nl = (int)std::min<int64_t>(m, kCsrSamples), nc = (int)std::min<int64_t>(nnz, kCsrSamples);
  if (nl > 0 || nc > 0) {
    void* ws = nullptr;
    const size_t lb = (size_t)kCsrSamples * 8, cb = (size_t)kCsrSamples * 4;
    s = alloc_ws(&ws, lb + cb, st);
    if (s != FXTX_OK) return s;
    int64_t* dl = static_cast<int64_t*>(ws);
    int32_t* dc = reinterpret_cast<int32_t*>(static_cast<char*>(ws) + lb);
    cudaError_t e = launch_csr_sample(m, nnz, row_ptr, col_idx, dl, dc, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(lens.data(), dl, lb, cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(cols.data(), dc, cb, cudaMemcpyDeviceToHost, st);
    cudaFreeAsync(ws, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return FXTX_ERR_CUDA;
    }
  }
  Analysis an{dev->device, row_ptr, col_idx, m, n, nnz,
              csr_stats_from_samples(n, lens.data(), nl, cols.data(), nc, csr_warp_long())};
  store_analysis(an);
  if (stats) fill_stats(an.stats, plan_csr(*dev, m, n, nnz, is_f64 ? 8 : 4, &an.stats), stats);
  return FXTX_OK;
}

fxtx_status_t fxtx_csr_analysis_clear(void) {
  std::lock_guard<std::mutex> lock(g_an_mu);
  g_an.clear();
  return FXTX_OK;
}

fxtx_status_t fxtx_csr_plan_describe_host(int is_f64, int64_t m, int64_t n, int64_t nnz, const int64_t* row_ptr,
                                          const int32_t* col_idx, fxtx_csr_stats_t* stats, char* buf, int64_t cap) {
  if (m < 0 || n < 0 || nnz < 0 || (m > 0 && row_ptr == nullptr) || (nnz > 0 && col_idx == nullptr))
    return FXTX_ERR_INVALID_ARG;
  DeviceInfo fallback;
  const DeviceInfo* dev = device_or_fallback(&fallback);
  const CsrStats st = csr_stats_from_host(m, n, nnz, row_ptr, col_idx);
  const CsrPlan p = plan_csr(*dev, m, n, nnz, is_f64 ? 8 : 4, &st);
  if (stats) fill_stats(st, p, stats);
  if (buf != nullptr && cap > 0) describe(p, buf, (size_t)cap);
  return FXTX_OK;
}

fxtx_status_t fxtx_device_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return FXTX_ERR_CUDA;
  }
  const int a = take_dense_device_error();
  const int b = take_csr_device_error();
  const int c = take_multi_device_error();
  if (a < 0 || b < 0 || c < 0) {
    cudaGetLastError();
    return FXTX_ERR_CUDA;
  }
  return (a || b || c) ? FXTX_ERR_TIMEOUT : FXTX_OK;
}

const char* fxtx_status_string(fxtx_status_t status) {
  switch (status) {
    case FXTX_OK: return "FXTX_OK";
    case FXTX_ERR_INVALID_ARG: return "FXTX_ERR_INVALID_ARG: invalid argument";
    case FXTX_ERR_UNSUPPORTED:
      return "FXTX_ERR_UNSUPPORTED: no compute capability 10.3 device is current, or a shape this entry does not take";
    case FXTX_ERR_CUDA: return "FXTX_ERR_CUDA: a CUDA call failed while enqueueing";
    case FXTX_ERR_ALLOC: return "FXTX_ERR_ALLOC: workspace allocation failed";
    case FXTX_ERR_BAD_CSR: return "FXTX_ERR_BAD_CSR: malformed CSR structure";
    case FXTX_ERR_TIMEOUT: return "FXTX_ERR_TIMEOUT: a kernel abandoned a bounded wait";
    case FXTX_ERR_TOO_LARGE: return "FXTX_ERR_TOO_LARGE: the problem exceeds the no-allocation scratch (n <= 512)";
  }
  return "FXTX: unknown status";
}

fxtx_status_t fxtx_plan_describe(int is_csr, int is_f64, int64_t m, int64_t n, int64_t nnz, int64_t ld, char* buf,
                                 int64_t cap) {
  if (buf == nullptr || cap <= 0 || m < 0 || n < 0 || nnz < 0) return FXTX_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  DeviceInfo fallback;
  if (current_device(&dev) != FXTX_OK) {
    // no GB300 current: describe the plan for a 152-SM device with 227 KB shared memory
    fallback.sm_count = 152;
    fallback.cc_major = 10;
    fallback.cc_minor = 3;
    fallback.smem_optin = 232448;
    fallback.smem_per_sm = 233472;
    dev = &fallback;
  }
  const int elem = is_f64 ? 8 : 4;
  if (is_csr) {
    describe(plan_csr(*dev, m, n, nnz, elem), buf, (size_t)cap);
  } else {
    const int64_t l = ld < n ? n : ld;
    const bool tile_ok = (l * elem) % 16 == 0;
    describe(plan_dense(*dev, m, n, l, elem, tile_ok && (n * elem) % 16 == 0, tile_ok), buf, (size_t)cap);
  }
  return FXTX_OK;
}

fxtx_status_t fxtx_autotune_set(int mode) {
  if (mode != 0 && mode != 1) return FXTX_ERR_INVALID_ARG;
  tune_set_mode(mode);
  return FXTX_OK;
}

int fxtx_autotune_get(void) { return tune_mode(); }

int64_t fxtx_autotune_entries(void) { return tune_entries(); }

fxtx_status_t fxtx_autotune_clear(void) {
  tune_clear();
  return FXTX_OK;
}

fxtx_status_t fxtx_autotune_save(const char* path) {
  if (path == nullptr) return FXTX_ERR_INVALID_ARG;
  return tune_save(path) ? FXTX_OK : FXTX_ERR_INVALID_ARG;
}

fxtx_status_t fxtx_autotune_load(const char* path) {
  if (path == nullptr) return FXTX_ERR_INVALID_ARG;
  return tune_load(path) ? FXTX_OK : FXTX_ERR_INVALID_ARG;
}

fxtx_status_t fxtx_autotune_candidates(int is_csr, int is_f64, int64_t m, int64_t n, int64_t nnz, int64_t ld,
                                       char* buf, int64_t cap) {
  if (buf == nullptr || cap <= 0 || m < 0 || n < 0 || nnz < 0) return FXTX_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  DeviceInfo fallback;
  if (current_device(&dev) != FXTX_OK) {
    fallback.sm_count = 152;
    fallback.cc_major = 10;
    fallback.cc_minor = 3;
    fallback.smem_optin = 232448;
    fallback.smem_per_sm = 233472;
    dev = &fallback;
  }
  const int elem = is_f64 ? 8 : 4;
  size_t used = 0;
  buf[0] = '\0';
  auto put = [&](const char* line) {
    const int w = snprintf(buf + used, (size_t)cap - used, "%s%s", used ? "\n" : "", line);
    if (w > 0) used = std::min<size_t>((size_t)cap - 1, used + (size_t)w);
  };
  char line[512];
  if (is_csr) {
    for (const CsrPlan& p : csr_candidates(*dev, plan_csr(*dev, m, n, nnz, elem), m, n, nnz, elem)) {
      describe(p, line, sizeof line);
      put(line);
    }
  } else {
    const int64_t l = ld < n ? n : ld;
    const bool tile_ok = (l * elem) % 16 == 0;
    const DensePlan model = plan_dense(*dev, m, n, l, elem, tile_ok && (n * elem) % 16 == 0, tile_ok);
    for (const DensePlan& p : dense_candidates(*dev, model, m, n, elem)) {
      describe(p, line, sizeof line);
      put(line);
    }
  }
  return FXTX_OK;
}

fxtx_status_t fxtx_multi_plan_describe(int is_f64, int64_t m, int64_t n, int64_t k, int64_t ld, int v_mode, char* buf,
                                       int64_t cap) {
  if (buf == nullptr || cap <= 0 || m < 0 || n < 0 || k < 0 || v_mode < 0 || v_mode > 2) return FXTX_ERR_INVALID_ARG;
  const DeviceInfo* dev = nullptr;
  DeviceInfo fallback;
  if (current_device(&dev) != FXTX_OK) {
    fallback.sm_count = 152;
    fallback.cc_major = 10;
    fallback.cc_minor = 3;
    fallback.smem_optin = 232448;
    fallback.smem_per_sm = 233472;
    dev = &fallback;
  }
  const int elem = is_f64 ? 8 : 4;
  const int64_t l = ld < n ? n : ld;
  describe_multi(plan_multi(*dev, m, n, k, elem, (l * elem) % 16 == 0, v_mode == 2, v_mode != 0), buf, (size_t)cap);
  return FXTX_OK;
}

}  // extern "C"
