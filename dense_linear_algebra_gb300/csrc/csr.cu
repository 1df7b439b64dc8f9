// csr.cu — fused kernels for CSR X:
//     out = alpha * X^T (v .* (X y)) + beta * z
// ("On optimizing machine learning workloads via kernel fusion", abstract: the
// fused kernel with its sparse specialisation, coarsening and hierarchical
// aggregation of partial results).
//
// A row's entries are loaded once into registers, used for the dot with y
// (gathered through the read-only cache), and reused for the scatter of
// t_i * vals into the output — X is not read twice. Rows are binned on the fly
// by length:
//   short  (<= lpr * 4)   a group of lpr lanes, entries in registers
//   medium (<= 256)       the whole warp, entries in registers
//   long  (> 256)         deferred to a queue and handled by a whole CTA in a
//                         second kernel (two passes, the second served by L2)
// Column partials are aggregated per CTA in a shared-memory window of columns
// and flushed with one atomic per column at the end; columns outside the
// window go straight to out with atomics. A prologue writes out = beta z and
// splits the rows among CTAs so that each gets an equal share of
// nnz + row_cost * rows; inside a CTA, warps take rows from a shared counter.
#include "common.cuh"
#include "kernels.h"

namespace fxtx {

namespace {

constexpr int KG = 4;  // entries per lane for short rows
constexpr int KW = 8;  // entries per lane for medium rows

template <typename T>
struct Window {
  T* acc;
  int64_t c0;
  int64_t len;
  T* out;
  __device__ __forceinline__ void add(int32_t col, T x) const {
    const uint64_t off = (uint64_t)((int64_t)col - c0);
    if (off < (uint64_t)len)
      atomicAdd(acc + off, x);
    else
      atomicAdd(out + col, x);
  }
};

template <typename T>
__device__ __forceinline__ void window_zero(T* acc, int64_t len) {
  for (int64_t j = threadIdx.x; j < len; j += blockDim.x) acc[j] = T(0);
}

template <typename T>
__device__ __forceinline__ void window_flush(const T* acc, int64_t c0, int64_t len, T* out) {
  for (int64_t j = threadIdx.x; j < len; j += blockDim.x) {
    const T x = acc[j];
    if (x != T(0)) atomicAdd(out + c0 + j, x);
  }
}

}  // namespace

int take_csr_device_error() { return take_device_error(); }

// out = beta z (or 0); row partition; counters.
template <typename T>
__global__ void csr_prologue_kernel(const CsrArgs<T> a, const int nparts, const int row_cost) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (int64_t j = tid; j < a.n; j += stride) a.out[j] = a.use_z ? (T)(a.beta * (double)a.z[j]) : T(0);
  const int64_t total = a.nnz + (int64_t)row_cost * a.m;
  for (int64_t p = tid; p <= nparts; p += stride) {
    int64_t r;
    if (p == 0) {
      r = 0;
    } else if (p == nparts) {
      r = a.m;
    } else {
      // first row i with row_ptr[i] + row_cost * i >= p * total / nparts
      const int64_t target = (int64_t)((__int128)total * p / nparts);
      int64_t lo = 0, hi = a.m;
      while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if (a.row_ptr[mid] + (int64_t)row_cost * mid < target) lo = mid + 1; else hi = mid;
      }
      r = lo;
    }
    a.part[p] = r;
  }
  if (tid == 0) {
    a.counters[0] = 0ull;
    a.counters[1] = 0ull;
  }
}

template <typename T, int LPR>
__global__ void __launch_bounds__(512) csr_rows_kernel(const CsrArgs<T> a, const int64_t win_c0, const int64_t win_len) {
  constexpr int G = 32 / LPR;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ unsigned long long s_next;
  T* wacc = reinterpret_cast<T*>(smem);
  const Window<T> win{wacc, win_c0, win_len, a.out};
  const int lane = threadIdx.x & 31;
  const int g = lane / LPR, q = lane % LPR;
  const int64_t rb = a.part[blockIdx.x], re = a.part[blockIdx.x + 1];
  const T alpha = (T)a.alpha;

  window_zero(wacc, win_len);
  if (threadIdx.x == 0) s_next = (unsigned long long)rb;
  __syncthreads();

  for (;;) {
    unsigned long long base = 0;
    if (lane == 0) base = atomicAdd(&s_next, (unsigned long long)G);
    base = __shfl_sync(FULL_MASK, base, 0);
    if ((int64_t)base >= re) break;
    const int64_t r = (int64_t)base + g;
    const bool has = r < re;
    const int64_t st = has ? a.row_ptr[r] : 0, en = has ? a.row_ptr[r + 1] : 0;
    const int64_t len = en - st;

    // short rows: one lane group, entries in registers
    const bool small = has && len <= LPR * KG;
    T val[KG];
    int32_t col[KG];
    T d = T(0);
#pragma unroll
    for (int k = 0; k < KG; ++k) {
      const int64_t idx = st + q + LPR * k;
      const bool ok = small && idx < en;
      val[k] = ok ? ldg(a.vals + idx) : T(0);
      col[k] = ok ? ldg(a.col_idx + idx) : -1;
      if (ok) d = fma(val[k], ldg(a.y + col[k]), d);
    }
    d = group_sum<LPR>(d);
    if (small) {
      const T vi = a.v ? ldg(a.v + r) : T(1);
      const T ts = alpha * (vi * d);
#pragma unroll
      for (int k = 0; k < KG; ++k)
        if (col[k] >= 0) win.add(col[k], ts * val[k]);
    }

    // medium rows: the whole warp, one row at a time
    unsigned mm = __ballot_sync(FULL_MASK, has && !small && len <= 32 * KW && q == 0);
    while (mm) {
      const int src = __ffs(mm) - 1;
      mm &= mm - 1;
      const int64_t rr = __shfl_sync(FULL_MASK, r, src);
      const int64_t s2 = __shfl_sync(FULL_MASK, st, src), e2 = __shfl_sync(FULL_MASK, en, src);
      T mv[KW];
      int32_t mc[KW];
      DotAcc<T, sizeof(T) == 4> mdot;
#pragma unroll
      for (int k = 0; k < KW; ++k) {
        const int64_t idx = s2 + lane + 32 * k;
        const bool ok = idx < e2;
        mv[k] = ok ? ldg(a.vals + idx) : T(0);
        mc[k] = ok ? ldg(a.col_idx + idx) : -1;
        if (ok) mdot.add(mv[k], ldg(a.y + mc[k]));
      }
      mdot.template group_reduce<32>();
      const T md = mdot.value();
      const T vi = a.v ? ldg(a.v + rr) : T(1);
      const T ts = alpha * (vi * md);
#pragma unroll
      for (int k = 0; k < KW; ++k)
        if (mc[k] >= 0) win.add(mc[k], ts * mv[k]);
    }

    // long rows: defer to the long-row kernel
    if (has && len > 32 * KW && q == 0) {
      const unsigned long long pos = atomicAdd(&a.counters[0], 1ull);
      a.queue[pos] = r;
    }
  }
  __syncthreads();
  window_flush(wacc, win_c0, win_len, a.out);
}

template <typename T>
__global__ void __launch_bounds__(512) csr_long_kernel(const CsrArgs<T> a, const int64_t win_c0, const int64_t win_len) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ long long s_row;
  __shared__ double s_red[16];
  __shared__ T s_t;
  T* wacc = reinterpret_cast<T*>(smem);
  const Window<T> win{wacc, win_c0, win_len, a.out};
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const T alpha = (T)a.alpha;

  window_zero(wacc, win_len);
  __syncthreads();
  const unsigned long long count = a.counters[0];
  for (;;) {
    if (threadIdx.x == 0) {
      const unsigned long long k = atomicAdd(&a.counters[1], 1ull);
      s_row = k < count ? (long long)a.queue[k] : -1ll;
    }
    __syncthreads();
    const int64_t r = s_row;
    if (r < 0) break;
    const int64_t st = a.row_ptr[r], en = a.row_ptr[r + 1];
    // pass 1: the dot
    DotAcc<T, sizeof(T) == 4> d;
    for (int64_t idx = st + threadIdx.x; idx < en; idx += blockDim.x) d.add(ldg(a.vals + idx), ldg(a.y + ldg(a.col_idx + idx)));
    d.template group_reduce<32>();
    if (lane == 0) s_red[warp] = d.value_f64();
    __syncthreads();
    if (threadIdx.x == 0) {
      double u = 0.0;
      for (int w = 0; w < nw; ++w) u += s_red[w];
      const T vi = a.v ? a.v[r] : T(1);
      s_t = alpha * (vi * (T)u);
    }
    __syncthreads();
    const T ts = s_t;
    // pass 2: the scatter, re-reading the row from L2
    for (int64_t idx = st + threadIdx.x; idx < en; idx += blockDim.x) win.add(ldg(a.col_idx + idx), ts * ldg(a.vals + idx));
    __syncthreads();  // s_row / s_red / s_t reuse
  }
  __syncthreads();
  window_flush(wacc, win_c0, win_len, a.out);
}

template <typename T, int LPR>
static cudaError_t launch_rows(const CsrPlan& p, const CsrArgs<T>& a, cudaStream_t st) {
  cudaError_t e = ensure_smem((const void*)csr_rows_kernel<T, LPR>, p.smem);
  if (e != cudaSuccess) return e;
  csr_rows_kernel<T, LPR><<<p.ctas, p.threads, p.smem, st>>>(a, p.win_c0, p.win_len);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_csr(const CsrPlan& p, const CsrArgs<T>& a, cudaStream_t st) {
  {
    const int64_t work = std::max<int64_t>(a.n, (int64_t)p.ctas + 1);
    const int blocks = (int)std::min<int64_t>((work + 255) / 256, 4096);
    csr_prologue_kernel<T><<<blocks, 256, 0, st>>>(a, p.ctas, p.row_cost);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (a.m == 0) return cudaSuccess;
  cudaError_t e;
  switch (p.lpr) {
    case 2: e = launch_rows<T, 2>(p, a, st); break;
    case 4: e = launch_rows<T, 4>(p, a, st); break;
    case 8: e = launch_rows<T, 8>(p, a, st); break;
    case 16: e = launch_rows<T, 16>(p, a, st); break;
    default: return cudaErrorInvalidConfiguration;
  }
  if (e != cudaSuccess) return e;
  e = ensure_smem((const void*)csr_long_kernel<T>, p.long_smem);
  if (e != cudaSuccess) return e;
  csr_long_kernel<T><<<p.long_ctas, p.long_threads, p.long_smem, st>>>(a, p.win_c0, p.win_len);
  return cudaGetLastError();
}

template cudaError_t launch_csr<float>(const CsrPlan&, const CsrArgs<float>&, cudaStream_t);
template cudaError_t launch_csr<double>(const CsrPlan&, const CsrArgs<double>&, cudaStream_t);

// Structure check: flag bit 1 set on any violation.
__global__ void csr_validate_kernel(int64_t m, int64_t n, int64_t nnz, const int64_t* row_ptr, const int32_t* col_idx,
                                    int* flag) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  bool bad = false;
  if (tid == 0) bad = (row_ptr[0] != 0) || (row_ptr[m] != nnz);
  for (int64_t i = tid; i < m; i += stride) bad |= row_ptr[i + 1] < row_ptr[i];
  for (int64_t k = tid; k < nnz; k += stride) bad |= (col_idx[k] < 0) || ((int64_t)col_idx[k] >= n);
  if (__any_sync(FULL_MASK, bad) && (threadIdx.x & 31) == 0) atomicOr(flag, 1);
}

cudaError_t launch_csr_validate(int64_t m, int64_t n, int64_t nnz, const int64_t* row_ptr, const int32_t* col_idx,
                                int* flag, cudaStream_t st) {
  const int64_t work = std::max<int64_t>(std::max<int64_t>(m, nnz), 1);
  const int blocks = (int)std::min<int64_t>((work + 255) / 256, 8192);
  csr_validate_kernel<<<blocks, 256, 0, st>>>(m, n, nnz, row_ptr, col_idx, flag);
  return cudaGetLastError();
}

}  // namespace fxtx
