// csr.cu — fused kernels for CSR X:
//     out = alpha * X^T (v .* (X y)) + beta * z
// ("On optimizing machine learning workloads via kernel fusion", abstract: the
// fused kernel with its sparse specialisation, coarsening and hierarchical
// aggregation of partial results).
//
// A row's entries are loaded once, used for the dot with y (gathered through
// the read-only cache) and reused for the scatter of t_i * vals into the
// output. Rows are binned on the fly by length:
//   short  (<= lpr * 4)   a group of lpr lanes, entries in registers
//   medium (<= 256)       the whole warp, entries in registers
//   long   (> 256)        deferred to a queue; a group of 8 warps takes each
//                         one in the long-row kernel (pass 1 forms the dot,
//                         pass 2 re-reads the row, from L2, for the scatter)
// Each CTA (one per SM, 1024 threads) accumulates scatters into a shared-
// memory window of columns and flushes it once with one atomic per column;
// columns outside the window go straight to out with atomics. fp64 window
// updates fold the product into the atomic itself (a CAS loop around one
// fused multiply-add), so each entry costs two fp64 operations: the dot's
// FMA and the scatter's.
// The prologue writes out = beta z and splits rows among CTAs by equal shares
// of nnz + row_cost * rows. Inside a CTA, warps take row batches in a static
// interleave, which lets each warp prefetch its next batch's row bounds and
// entries while it computes the current one.
#include "common.cuh"
#include "kernels.h"

namespace fxtx {

namespace {

constexpr int KG = 4;               // entries per lane for short rows
constexpr int KW = 8;               // entries per lane for medium rows
constexpr int LONG_UNROLL = 8;      // loads in flight per thread in the long-row kernel
constexpr int LONG_GROUP = 256;     // threads that share one long row
constexpr int CSR_THREADS = 1024;

// out_j += a * b, with out_j in shared memory (fp64: CAS loop around one FMA).
__device__ __forceinline__ void smem_fma_add(float* p, float a, float b) { atomicAdd(p, a * b); }
__device__ __forceinline__ void smem_fma_add(double* p, double a, double b) {
  unsigned long long* q = reinterpret_cast<unsigned long long*>(p);
  unsigned long long old = *q, assumed;
  do {
    assumed = old;
    old = atomicCAS(q, assumed, __double_as_longlong(fma(a, b, __longlong_as_double(assumed))));
  } while (old != assumed);
}

template <typename T>
struct Window {
  T* acc;
  int64_t c0;
  int64_t len;
  T* out;
  // out[col] += a * b, through the shared window when col falls inside it
  __device__ __forceinline__ void add(int32_t col, T a, T b) const {
    const uint64_t off = (uint64_t)((int64_t)col - c0);
    if (off < (uint64_t)len)
      smem_fma_add(acc + off, a, b);
    else
      atomicAdd(out + col, a * b);
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

// Named barrier over the `count` threads of one row group (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void group_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
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
__global__ void __launch_bounds__(CSR_THREADS, 1)
    csr_rows_kernel(const CsrArgs<T> a, const int64_t win_c0, const int64_t win_len) {
  constexpr int G = 32 / LPR;  // rows per warp batch
  extern __shared__ __align__(128) unsigned char smem[];
  T* wacc = reinterpret_cast<T*>(smem);
  const Window<T> win{wacc, win_c0, win_len, a.out};
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int g = lane / LPR, q = lane % LPR;
  const int64_t rb = a.part[blockIdx.x], re = a.part[blockIdx.x + 1];
  const T alpha = (T)a.alpha;

  window_zero(wacc, win_len);
  __syncthreads();

  // batch k of this warp covers rows rb + (warp + k * nw) * G + [0, G)
  const int64_t step = (int64_t)nw * G;
  int64_t r = rb + (int64_t)warp * G + g;
  int64_t st = 0, en = 0;
  if (r < re) { st = a.row_ptr[r]; en = a.row_ptr[r + 1]; }
  // entries of the current batch (short rows), loaded one batch ahead
  T val[KG];
  int32_t col[KG];
  auto load_short = [&](int64_t rr, int64_t s, int64_t e) {
    const bool small = rr < re && e - s <= LPR * KG;
#pragma unroll
    for (int k = 0; k < KG; ++k) {
      const int64_t idx = s + q + LPR * k;
      const bool ok = small && idx < e;
      val[k] = ok ? ldg(a.vals + idx) : T(0);
      col[k] = ok ? ldg(a.col_idx + idx) : -1;
    }
  };
  load_short(r, st, en);

  for (int64_t base = rb + (int64_t)warp * G; base < re; base += step) {
    const bool has = r < re;
    const int64_t len = en - st;
    const bool small = has && len <= LPR * KG;
    T cv[KG];
    int32_t cc[KG];
#pragma unroll
    for (int k = 0; k < KG; ++k) { cv[k] = val[k]; cc[k] = col[k]; }
    const int64_t cur_r = r, cur_st = st, cur_en = en;

    // prefetch the next batch: row bounds, then its short-row entries
    r += step;
    st = en = 0;
    if (r < re) { st = a.row_ptr[r]; en = a.row_ptr[r + 1]; }
    load_short(r, st, en);

    // short rows: one lane group, entries in registers
    T d = T(0);
#pragma unroll
    for (int k = 0; k < KG; ++k)
      if (cc[k] >= 0) d = fma(cv[k], ldg(a.y + cc[k]), d);
    d = group_sum<LPR>(d);
    if (small) {
      const T vi = a.v ? ldg(a.v + cur_r) : T(1);
      const T ts = alpha * (vi * d);
#pragma unroll
      for (int k = 0; k < KG; ++k)
        if (cc[k] >= 0) win.add(cc[k], ts, cv[k]);
    }

    // medium rows: the whole warp, one row at a time
    unsigned mm = __ballot_sync(FULL_MASK, has && !small && len <= 32 * KW && q == 0);
    while (mm) {
      const int src = __ffs(mm) - 1;
      mm &= mm - 1;
      const int64_t rr = __shfl_sync(FULL_MASK, cur_r, src);
      const int64_t s2 = __shfl_sync(FULL_MASK, cur_st, src), e2 = __shfl_sync(FULL_MASK, cur_en, src);
      T mv[KW];
      int32_t mc[KW];
#pragma unroll
      for (int k = 0; k < KW; ++k) {
        const int64_t idx = s2 + lane + 32 * k;
        const bool ok = idx < e2;
        mv[k] = ok ? ldg(a.vals + idx) : T(0);
        mc[k] = ok ? ldg(a.col_idx + idx) : -1;
      }
      DotAcc<T, sizeof(T) == 4> mdot;
#pragma unroll
      for (int k = 0; k < KW; ++k)
        if (mc[k] >= 0) mdot.add(mv[k], ldg(a.y + mc[k]));
      mdot.template group_reduce<32>();
      const T vi = a.v ? ldg(a.v + rr) : T(1);
      const T ts = alpha * (vi * mdot.value());
#pragma unroll
      for (int k = 0; k < KW; ++k)
        if (mc[k] >= 0) win.add(mc[k], ts, mv[k]);
    }

    // long rows: defer to the long-row kernel
    if (has && len > 32 * KW && q == 0) {
      const unsigned long long pos = atomicAdd(&a.counters[0], 1ull);
      a.queue[pos] = cur_r;
    }
  }
  __syncthreads();
  window_flush(wacc, win_c0, win_len, a.out);
}

// Long rows: each group of LONG_GROUP threads takes queued rows one at a time.
template <typename T>
__global__ void __launch_bounds__(CSR_THREADS, 1)
    csr_long_kernel(const CsrArgs<T> a, const int64_t win_c0, const int64_t win_len) {
  constexpr int GW = LONG_GROUP / 32;  // warps per group
  constexpr int NG = CSR_THREADS / LONG_GROUP;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ long long s_row[NG];
  __shared__ double s_red[NG][GW];
  __shared__ T s_t[NG];
  T* wacc = reinterpret_cast<T*>(smem);
  const Window<T> win{wacc, win_c0, win_len, a.out};
  const int lane = threadIdx.x & 31;
  const int grp = threadIdx.x / LONG_GROUP, gt = threadIdx.x % LONG_GROUP, gw = gt >> 5;
  const int bar = 1 + grp;
  const T alpha = (T)a.alpha;

  window_zero(wacc, win_len);
  __syncthreads();
  const unsigned long long count = a.counters[0];
  for (;;) {
    if (gt == 0) {
      const unsigned long long k = atomicAdd(&a.counters[1], 1ull);
      s_row[grp] = k < count ? (long long)a.queue[k] : -1ll;
    }
    group_barrier(bar, LONG_GROUP);
    const int64_t r = s_row[grp];
    if (r < 0) break;
    const int64_t st = a.row_ptr[r], en = a.row_ptr[r + 1];

    // pass 1: the dot, LONG_UNROLL independent loads in flight per thread
    DotAcc<T, sizeof(T) == 4> d;
    for (int64_t b = st + gt; b < en; b += (int64_t)LONG_GROUP * LONG_UNROLL) {
      T xv[LONG_UNROLL];
      int32_t xc[LONG_UNROLL];
#pragma unroll
      for (int k = 0; k < LONG_UNROLL; ++k) {
        const int64_t idx = b + (int64_t)k * LONG_GROUP;
        const bool ok = idx < en;
        xv[k] = ok ? ldg(a.vals + idx) : T(0);
        xc[k] = ok ? ldg(a.col_idx + idx) : -1;
      }
      T yv[LONG_UNROLL];
#pragma unroll
      for (int k = 0; k < LONG_UNROLL; ++k) yv[k] = xc[k] >= 0 ? ldg(a.y + xc[k]) : T(0);
#pragma unroll
      for (int k = 0; k < LONG_UNROLL; ++k) d.add(xv[k], yv[k]);
    }
    d.template group_reduce<32>();
    if (lane == 0) s_red[grp][gw] = d.value_f64();
    group_barrier(bar, LONG_GROUP);
    if (gt == 0) {
      double u = 0.0;
      for (int w = 0; w < GW; ++w) u += s_red[grp][w];
      const T vi = a.v ? a.v[r] : T(1);
      s_t[grp] = alpha * (vi * (T)u);
    }
    group_barrier(bar, LONG_GROUP);
    const T ts = s_t[grp];

    // pass 2: the scatter, re-reading the row (served by L2)
    for (int64_t b = st + gt; b < en; b += (int64_t)LONG_GROUP * LONG_UNROLL) {
      T xv[LONG_UNROLL];
      int32_t xc[LONG_UNROLL];
#pragma unroll
      for (int k = 0; k < LONG_UNROLL; ++k) {
        const int64_t idx = b + (int64_t)k * LONG_GROUP;
        const bool ok = idx < en;
        xv[k] = ok ? ldg(a.vals + idx) : T(0);
        xc[k] = ok ? ldg(a.col_idx + idx) : -1;
      }
#pragma unroll
      for (int k = 0; k < LONG_UNROLL; ++k)
        if (xc[k] >= 0) win.add(xc[k], ts, xv[k]);
    }
    group_barrier(bar, LONG_GROUP);  // s_row / s_red / s_t reuse
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
