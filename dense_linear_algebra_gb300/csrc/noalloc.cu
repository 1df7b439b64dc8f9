// noalloc.cu — fxtx_dense_f32_noalloc: the dense fp32 call with no device
// allocation at call time.
//
// The regular entry points take their scratch (the per-CTA column partials and
// the arrival ticket of the final reduction) from cudaMallocAsync on the
// caller's stream. Some callers cannot allocate there: a caller whose device
// memory is owned by another allocator or runtime that must not be bypassed, a
// real-time loop under a no-allocation-after-start-up rule, or code paths that
// must not touch a memory pool at all. This entry point serves them. Its
// scratch is one file-scope device array of FXTX_NOALLOC_SCRATCH_BYTES, created
// when the library is loaded and held by every GPU that loads it until the
// process exits. The caller still passes every input and output.
//
// Set-up: the first call on a device, with that device current, looks up the
// array's device address (cudaGetSymbolAddress) and caches it for that device,
// together with the unique id of the device's current context. That first call
// should therefore come before any stream capture. Later calls compare the
// context id (one driver query, no allocation or synchronisation) and look the
// address up again only when the context has changed: after cudaDeviceReset, or
// a release and re-creation of the primary context, the library's device code is
// loaded anew and the array has a new address.
//
// Sharing: every call on a device uses the same array and finds it as the last
// call left it. The arrival ticket, which must start at zero, is cleared on the
// caller's stream before each launch. Calls whose executions overlap on the GPU
// (different streams, no ordering between them) race on the array and give
// wrong results; order them on one stream or with events.
#include <cuda.h>

#include <mutex>

#include "fxtx.h"
#include "kernels.h"
#include "plan.h"

namespace fxtx {
namespace {

constexpr size_t kScratchBytes = FXTX_NOALLOC_SCRATCH_BYTES;
constexpr size_t kTicketOffset = kScratchBytes - 256;  // the ticket lives in the last 256 bytes
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

struct NoallocDevice {
  std::once_flag once;
  std::mutex mu;                   // guards scratch and ctx_id
  unsigned char* scratch = nullptr;
  unsigned long long ctx_id = 0;   // unique id of the context the address belongs to
  DeviceInfo info;
};
NoallocDevice g_devs[kMaxDevices];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// The unique id of the calling thread's current context (0 if it cannot be had).
unsigned long long current_ctx_id() {
  static std::once_flag once;
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
    cudaGetLastError();
  });
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current == nullptr || get_id == nullptr || get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr ||
      get_id(ctx, &id) != CUDA_SUCCESS)
    return 0;
  return id;
}

// Device properties and the scratch address for the current device and context.
fxtx_status_t setup(NoallocDevice** out, unsigned char** scratch) {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) {
    cudaGetLastError();
    return FXTX_ERR_UNSUPPORTED;
  }
  NoallocDevice& nd = g_devs[d];
  std::call_once(nd.once, [&nd, d] {
    DeviceInfo& di = nd.info;
    di.device = d;
    cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, d);
    cudaDeviceGetAttribute(&di.cc_major, cudaDevAttrComputeCapabilityMajor, d);
    cudaDeviceGetAttribute(&di.cc_minor, cudaDevAttrComputeCapabilityMinor, d);
    cudaDeviceGetAttribute(&di.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, d);
    cudaDeviceGetAttribute(&di.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, d);
    cudaGetLastError();
  });
  if (nd.info.cc_major != 10 || nd.info.cc_minor != 3 || nd.info.sm_count <= 0) return FXTX_ERR_UNSUPPORTED;
  // the first cudaGetSymbolAddress on a device also makes its primary context current,
  // so the context id is read after it
  std::lock_guard<std::mutex> lock(nd.mu);
  const unsigned long long id = nd.scratch ? current_ctx_id() : 0;
  if (nd.scratch == nullptr || id == 0 || id != nd.ctx_id) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      nd.scratch = nullptr;
      return FXTX_ERR_CUDA;
    }
    nd.scratch = static_cast<unsigned char*>(p);
    nd.ctx_id = current_ctx_id();
  }
  *out = &nd;
  *scratch = nd.scratch;
  return FXTX_OK;
}

}  // namespace
}  // namespace fxtx

using namespace fxtx;

extern "C" fxtx_status_t fxtx_dense_f32_noalloc(int64_t m, int64_t n, const float* X, int64_t ld, const float* y,
                                                const float* v, float alpha, float beta, const float* z, float* out,
                                                void* stream) {
  if (m < 0 || n < 0) return FXTX_ERR_INVALID_ARG;
  if (n == 0) return FXTX_OK;
  if (ld < n || y == nullptr || out == nullptr) return FXTX_ERR_INVALID_ARG;
  if (m > 0 && X == nullptr) return FXTX_ERR_INVALID_ARG;
  NoallocDevice* nd = nullptr;
  unsigned char* scratch = nullptr;
  fxtx_status_t s = setup(&nd, &scratch);
  if (s != FXTX_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);

  const int elem = (int)sizeof(float);
  const bool tile_ok = (reinterpret_cast<uintptr_t>(X) & 15u) == 0 && (ld * elem) % 16 == 0;
  DensePlan plan = plan_dense(nd->info, m, n, ld, elem, tile_ok && (n * elem) % 16 == 0, tile_ok);
  if (plan.kind == DENSE_WIDE) return FXTX_ERR_TOO_LARGE;  // rows longer than the narrow kernels' 512 columns
  const bool partials = plan.kind == DENSE_NARROW_TMA || plan.kind == DENSE_NARROW_DIRECT || plan.kind == DENSE_TILE_TMA;
  if (partials) {
    // fit the per-CTA partials into the scratch array by capping the grid
    const int64_t max_ctas = (int64_t)(kTicketOffset / ((size_t)n * sizeof(double)));
    if (max_ctas < 1) return FXTX_ERR_TOO_LARGE;
    if (plan.ctas > max_ctas) plan.ctas = (int)max_ctas;
  }

  DenseArgs<float> a;
  a.m = m; a.n = n; a.ld = ld;
  a.X = X; a.y = y; a.v = v; a.z = z; a.out = out;
  a.alpha = (double)alpha; a.beta = (double)beta;
  a.use_z = (z != nullptr && beta != 0.0f);
  a.tiles = plan.rows_per_tile > 0 ? (m + plan.rows_per_tile - 1) / plan.rows_per_tile : 0;
  a.ws = reinterpret_cast<double*>(scratch);
  a.ticket = reinterpret_cast<unsigned*>(scratch + kTicketOffset);
  if (partials) {
    if (cudaMemsetAsync(a.ticket, 0, sizeof(unsigned), st) != cudaSuccess) {
      cudaGetLastError();
      return FXTX_ERR_CUDA;
    }
  }
  if (launch_dense<float>(plan, a, st) != cudaSuccess) {
    cudaGetLastError();
    return FXTX_ERR_CUDA;
  }
  return FXTX_OK;
}
