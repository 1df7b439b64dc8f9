// common.cuh — device helpers shared by the fused kernels: mbarrier and bulk
// asynchronous copy wrappers (inline PTX for sm_103a), bounded waits, warp
// reductions and the compensated (two-float) accumulator.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "fxtx.h"

namespace fxtx {

constexpr unsigned FULL_MASK = 0xffffffffu;

// Upper bound on polls of one mbarrier phase before a kernel gives up. Each poll
// is an mbarrier.try_wait, which itself suspends for a bounded time, so this is
// on the order of a second: far beyond any legitimate copy latency.
constexpr uint32_t WAIT_LIMIT = 1u << 22;

// Sticky device-side error word (FXTX_OK or FXTX_ERR_TIMEOUT). Each translation
// unit has its own copy (internal linkage, no relocatable device code); its
// host-side reader is take_device_error() below, which every kernel file
// exports under its own name for fxtx_device_error.
static __device__ int g_device_error = 0;

__device__ __forceinline__ void raise_error(int code) { atomicCAS(&g_device_error, 0, code); }

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Makes mbarrier initialisation visible to the asynchronous proxy (bulk copies).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Orders this thread's generic-proxy shared-memory accesses before later
// asynchronous-proxy accesses (a bulk copy that overwrites a consumed buffer).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

// One bulk copy global -> shared, completing `bytes` of transaction count on `bar`.
// dst and src must be 16-byte aligned and bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// One 2-D tiled tensor copy global -> shared (box at element coordinates x, y
// of the tensor map), completing its box bytes of transaction count on `bar`.
// x * sizeof(element) must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int x, int y, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
      "l"(tmap), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
      : "memory");
}

// L2 policy for data read exactly once: evict it first.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of `bar` to complete, polling at most WAIT_LIMIT
// times. Returns false (after raising FXTX_ERR_TIMEOUT) if it never did.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  for (uint32_t it = 0; it < WAIT_LIMIT; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  raise_error(FXTX_ERR_TIMEOUT);
  return false;
}

// Read-only, L1-allocating global load.
template <typename T>
__device__ __forceinline__ T ldg(const T* p) {
  return __ldg(p);
}

// Streaming global load that does not allocate in L1 (data read once).
__device__ __forceinline__ float ld_stream(const float* p) {
  float r;
  asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(r) : "l"(p));
  return r;
}
__device__ __forceinline__ double ld_stream(const double* p) {
  double r;
  asm volatile("ld.global.nc.L1::no_allocate.f64 %0, [%1];" : "=d"(r) : "l"(p));
  return r;
}
__device__ __forceinline__ int32_t ld_stream(const int32_t* p) {
  int32_t r;
  asm volatile("ld.global.nc.L1::no_allocate.s32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}

template <typename T>
__host__ __device__ __forceinline__ T tmin(T a, T b) {
  return a < b ? a : b;
}
template <typename T>
__host__ __device__ __forceinline__ T tmax(T a, T b) {
  return a < b ? b : a;
}

template <typename T>
__device__ __forceinline__ T shfl_xor(T x, int mask) {
  return __shfl_xor_sync(FULL_MASK, x, mask);
}

// Sum over aligned groups of W lanes (W a power of two, <= 32); every lane of a
// group receives the group's sum.
template <int W, typename T>
__device__ __forceinline__ T group_sum(T x) {
#pragma unroll
  for (int o = W / 2; o > 0; o >>= 1) x += shfl_xor(x, o);
  return x;
}

// Error-free transformation of a sum (Knuth's TwoSum): s + e == a + b exactly.
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
  s = __fadd_rn(a, b);
  float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// Dot-product accumulator. The plain form is one fused multiply-add per term.
// The compensated form (COMP, fp32 only) follows Ogita, Rump and Oishi,
// "Accurate sum and dot product" (SIAM J. Sci. Comput. 2005), algorithm Dot2:
// each product is split exactly into p + e (TwoProduct via FMA), p is added
// with TwoSum, and the two error terms are collected in c. The result is as
// accurate as if computed in twice the working precision and then rounded,
// which keeps long fp32 dots with heavy cancellation inside the fp32 bound.
template <typename T, bool COMP>
struct DotAcc {
  T s = T(0);
  __device__ __forceinline__ void add(T a, T b) { s = fma(a, b, s); }
  template <int W>
  __device__ __forceinline__ void group_reduce() {
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  }
  __device__ __forceinline__ T value() const { return s; }
  __device__ __forceinline__ double value_f64() const { return (double)s; }
};

template <>
struct DotAcc<float, true> {
  float s = 0.f, c = 0.f;
  __device__ __forceinline__ void add(float a, float b) {
    const float p = __fmul_rn(a, b);
    const float e = __fmaf_rn(a, b, -p);
    float t, q;
    two_sum(s, p, t, q);
    s = t;
    c = __fadd_rn(c, __fadd_rn(q, e));
  }
  template <int W>
  __device__ __forceinline__ void group_reduce() {
#pragma unroll
    for (int o = W / 2; o > 0; o >>= 1) {
      const float s2 = __shfl_xor_sync(0xffffffffu, s, o), c2 = __shfl_xor_sync(0xffffffffu, c, o);
      float t, q;
      two_sum(s, s2, t, q);
      s = t;
      c = __fadd_rn(__fadd_rn(c, c2), q);
    }
  }
  __device__ __forceinline__ float value() const { return __fadd_rn(s, c); }
  __device__ __forceinline__ double value_f64() const { return (double)s + (double)c; }
};

// Two-float accumulator: hi + lo carries about 48 bits. add() folds one float
// into it with TwoSum, so the accumulated rounding error stays near 2^-44
// relative to the sum of magnitudes however many values are folded in.
struct CompF32 {
  float hi = 0.f, lo = 0.f;
  __device__ __forceinline__ void add(float x) {
    float s, e;
    two_sum(hi, x, s, e);
    hi = s;
    lo = __fadd_rn(lo, e);
  }
  __device__ __forceinline__ double value() const { return (double)hi + (double)lo; }
};

// Plain fp64 accumulator with the same interface.
struct AccF64 {
  double s = 0.0;
  __device__ __forceinline__ void add(double x) { s += x; }
  __device__ __forceinline__ double value() const { return s; }
};

template <typename T>
struct OuterAcc;
template <>
struct OuterAcc<float> {
  using type = CompF32;
};
template <>
struct OuterAcc<double> {
  using type = AccF64;
};

// Reads and clears this translation unit's error word (synchronous).
static inline int take_device_error() {
  int v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int)) != cudaSuccess) return -1;
  if (v != 0 && cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess) return -1;
  return v;
}

template <typename T>
struct Vec16;  // the 16-byte vector of T
template <>
struct Vec16<float> {
  using type = float4;
  static constexpr int N = 4;
};
template <>
struct Vec16<double> {
  using type = double2;
  static constexpr int N = 2;
};

template <typename T>
__device__ __forceinline__ void unpack(const typename Vec16<T>::type& v, T* e);
template <>
__device__ __forceinline__ void unpack<float>(const float4& v, float* e) {
  e[0] = v.x; e[1] = v.y; e[2] = v.z; e[3] = v.w;
}
template <>
__device__ __forceinline__ void unpack<double>(const double2& v, double* e) {
  e[0] = v.x; e[1] = v.y;
}

}  // namespace fxtx
