// csr.cu — fused kernels for CSR X:
//     out = alpha * X^T (v .* (X y)) + beta * z
// ("On optimizing machine learning workloads via kernel fusion", abstract: the
// fused kernel with its sparse specialisation, coarsening and hierarchical
// aggregation of partial results).
//
// Every entry is loaded once, used for the dot with y (gathered through the
// read-only cache) and reused for the scatter of t_i * vals into the output.
// Rows are binned on the fly by length:
//   short                 fp32: packed batches (consecutive short rows share a
//                         warp, 8 consecutive entries per lane, so lanes are not
//                         left idle by rows shorter than the warp); fp64: lane
//                         groups of LPR lanes x 8 entries per row, which spend
//                         fewer fp64 operations per entry
//   medium (<= WARP_LONG) one warp per row, two passes (the second from L1/L2):
//                         fp32 defers them to a queue that the long-row kernel
//                         drains after its long rows; fp64 takes them in place
//   long   (> WARP_LONG)  deferred to queues bucketed by length; in the long-row
//                         kernel a group of threads (128 by default) takes each
//                         row, longest buckets first, two passes
// The y gathers of hot columns hit a copy of y[y0, y0 + ylen) in shared memory;
// the two windows sit on the column ranges a sample of col_idx hits most.
// Row dots of a packed batch are formed lane-locally per row segment, and each
// segment's partial is added once into a per-warp fp64 buffer; t_i is then
// computed once per row. Each CTA (one per SM; 1024 threads, 768 for the fp64
// lane groups) accumulates
// scatters into a shared-memory window of columns and flushes it once with one
// atomic per column; columns outside the window go straight to out with
// atomics. fp64 window updates fold the product into the atomic itself (a CAS
// loop around one fused multiply-add).
// The prologue writes out = beta z, zeroes the counters and sets the window starts
// (from the plan's sample, or from its own sample of col_idx). Warps of the packed
// kernel take 32-row windows from one global counter; the fp64 lane-group kernel
// splits rows among CTAs by equal shares of nnz + row_cost * rows.
#include "common.cuh"
#include "kernels.h"

namespace fxtx {

namespace {

constexpr int CSR_THREADS = 1024;
// the lane-group kernel: 768 threads leave 80 registers a thread, so the 16-entry lane
// buffers of fp64 rows stay in registers (at 1024 threads, 64 registers, they spill)
constexpr int CSR_GROUP_THREADS = 768;
// consecutive entries per lane in a packed batch (fp64 keeps fewer, to fit 64 registers)
template <typename T>
struct Pack {
  static constexpr int K = sizeof(T) == 4 ? 8 : 4;
  static constexpr int CAP = 32 * K;  // entries per packed batch
};
constexpr int WARP_LONG = 2048;            // longest row a single warp takes
constexpr int WARP_UNROLL = 8;             // loads in flight per lane for warp rows
// entries per lane and batch in the long-row kernel (fp64 keeps fewer, to fit 64 registers)
template <typename T>
__host__ __device__ constexpr int long_unroll() {
  return sizeof(T) == 4 ? 8 : 4;
}
// threads that share one long row, chosen by the plan (128, 256 or 512): 128 by default, the
// fastest on the power-law workload (1,091 us per call against 1,113 at 256, 1,289 at 512 and
// 2,491 at 1,024): more rows in flight hide the latency of the gathers, which outweighs the
// pass-2 re-reads that fewer rows in flight would keep in L2
constexpr int LONG_GROUP_DEFAULT = 128;
constexpr int LONG_BUCKETS = 6;            // long-row queues: (2K, 4K], (4K, 8K], ... (32K, 64K], > 64K entries
// per-warp scratch after the window: 32 row dots (double), 32 row scales (T), 33 row starts
constexpr size_t WARP_SCRATCH = 32 * 8 + 32 * 8 + 33 * 8;

// *p += a * b in shared memory (fp64: CAS loop around one FMA, so the product folds into
// the atomic and costs one fp64 instruction per attempt; fp32: native atomic).
__device__ __forceinline__ void smem_fma_add(float* p, float a, float b) { atomicAdd(p, a * b); }
__device__ __forceinline__ void smem_fma_add(double* p, double a, double b) {
  unsigned long long* q = reinterpret_cast<unsigned long long*>(p);
  unsigned long long old = *q, assumed;
  do {
    assumed = old;
    old = atomicCAS(q, assumed, __double_as_longlong(fma(a, b, __longlong_as_double(assumed))));
  } while (old != assumed);
}

// Shared-memory windows of one CTA: scatters into columns [c0, c0 + len) are
// accumulated in `acc`, and y[y0, y0 + ylen) is held in `ys` for the gathers.
template <typename T>
struct Window {
  T* acc;
  int64_t c0;
  int64_t len;
  T* out;
  const T* ys;
  int64_t y0;
  int64_t ylen;
  const T* y;
  // out[col] += a * b, through the shared window when col falls inside it
  __device__ __forceinline__ void add(int32_t col, T a, T b) const {
    const uint64_t off = (uint64_t)((int64_t)col - c0);
    if (off < (uint64_t)len)
      smem_fma_add(acc + off, a, b);
    else
      atomicAdd(out + col, a * b);
  }
  __device__ __forceinline__ T yat(int32_t col) const {
    const uint64_t off = (uint64_t)((int64_t)col - y0);
    return off < (uint64_t)ylen ? ys[off] : ldg(y + col);
  }
};

// Workspace slots of the two window starts, written by the prologue, and of the medium-row queue.
constexpr int SLOT_WIN_C0 = 8, SLOT_Y0 = 9, SLOT_MED_COUNT = 10, SLOT_MED_CLAIM = 11;

template <typename T>
__device__ __forceinline__ Window<T> make_window(const CsrArgs<T>& a, T* acc, int64_t win_len, const T* ys,
                                                 int64_t ylen) {
  return Window<T>{acc, (int64_t)a.counters[SLOT_WIN_C0], win_len, a.out, ys, (int64_t)a.counters[SLOT_Y0], ylen,
                   a.y};
}

// Zeroes the accumulator window and copies y[y0, y0 + ylen) into shared memory.
template <typename T>
__device__ __forceinline__ void window_init(const Window<T>& w) {
  for (int64_t j = threadIdx.x; j < w.len; j += blockDim.x) w.acc[j] = T(0);
  T* ys = const_cast<T*>(w.ys);
  for (int64_t j = threadIdx.x; j < w.ylen; j += blockDim.x) ys[j] = ldg(w.y + w.y0 + j);
}

template <typename T>
__device__ __forceinline__ void window_flush(const T* acc, int64_t c0, int64_t len, T* out) {
  for (int64_t j = threadIdx.x; j < len; j += blockDim.x) {
    const T x = acc[j];
    if (x != T(0)) atomicAdd(out + c0 + j, x);
  }
}

__host__ __device__ constexpr size_t window_bytes(int64_t len, size_t elem) {
  return ((size_t)len * elem + 15) / 16 * 16;
}

// Defers row r, too long for the row kernel's batches, to the long-row kernel: rows of more
// than WARP_LONG entries to the queue of their length bucket (a group of threads each), the
// others to the medium queue (a warp each, once the long rows are done).
template <typename T>
__device__ __forceinline__ void defer_row(const CsrArgs<T>& a, int64_t r, int64_t len) {
  if (len > WARP_LONG) {
    const unsigned long long q = (unsigned long long)(len - 1) / WARP_LONG;  // >= 1
    const int b = (int)tmin<unsigned long long>(LONG_BUCKETS - 1, 63 - __clzll((long long)q));
    const unsigned long long k = atomicAdd(&a.counters[1 + b], 1ull);
    a.queue[(int64_t)b * a.queue_cap + (int64_t)k] = r;
  } else {
    const unsigned long long k = atomicAdd(&a.counters[SLOT_MED_COUNT], 1ull);
    a.med_queue[k] = r;
  }
}

}  // namespace

int take_csr_device_error() { return take_device_error(); }

size_t csr_rows_smem(int64_t win_len, int64_t ylen, int elem) {
  return window_bytes(win_len, elem) + window_bytes(ylen, elem) + 32 * WARP_SCRATCH;
}
int csr_pack_cap(int elem) { return elem == 4 ? Pack<float>::CAP : Pack<double>::CAP; }
int csr_warp_long() { return WARP_LONG; }
int csr_group_threads() { return CSR_GROUP_THREADS; }
int csr_long_buckets() { return LONG_BUCKETS; }
int csr_long_group_default() { return LONG_GROUP_DEFAULT; }

constexpr int PROLOGUE_THREADS = 1024;

// Block-wide first maximum of (count, start) keys: the largest count, the lowest start on ties.
__device__ __forceinline__ unsigned long long block_max_key(unsigned long long key, unsigned long long* red) {
  for (int o = 16; o > 0; o >>= 1) key = tmax(key, __shfl_xor_sync(FULL_MASK, key, o));
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  __syncthreads();
  if (lane == 0) red[warp] = key;
  __syncthreads();
  key = 0ull;
  for (int w = 0; w < PROLOGUE_THREADS / 32; ++w) key = tmax(key, red[w]);
  return key;
}

// The start of the len-column window holding the most sampled columns (pre: prefix sums of
// the per-bin sample counts over nb bins of wb columns): the rule of csr_place_window on the
// host, first maximum over bin-aligned starts, clamped to [0, n - len].
__device__ int64_t place_on_device(const int* pre, int nb, int64_t wb, int64_t n, int64_t len,
                                   unsigned long long* red) {
  if (len >= n) return 0;
  const int kb = (int)tmin<int64_t>(tmax<int64_t>(1, len / wb), nb);
  unsigned long long key = 0ull;
  for (int s0 = threadIdx.x; s0 + kb <= nb; s0 += PROLOGUE_THREADS) {
    const unsigned long long w = (unsigned long long)(pre[s0 + kb] - pre[s0]);
    key = tmax(key, (w << 32) | (unsigned long long)(0xffffffffu - (unsigned)s0));
  }
  key = block_max_key(key, red);
  const int64_t s0 = (int64_t)(0xffffffffu - (unsigned)(key & 0xffffffffull));
  return tmin<int64_t>(s0 * wb, n - len);
}

// Places the scatter window and the copy of y on the column ranges that a strided sample of
// kCsrSamples column indices (the positions of csr_sample_index) hits most: a histogram over
// bins of csr_bin_width(n) columns, its prefix sums, and the first maximum of each window's
// sampled count. Run by one block of PROLOGUE_THREADS threads.
template <typename T>
__device__ void place_windows(const CsrArgs<T>& a, int64_t win_len, int64_t ylen) {
  __shared__ int hist[kCsrBins + 1];
  __shared__ int part[2 * (PROLOGUE_THREADS / 32)];
  __shared__ unsigned long long red[PROLOGUE_THREADS / 32];
  const int64_t wb = csr_bin_width(a.n);
  const int nb = (int)((a.n + wb - 1) / wb);
  for (int b = threadIdx.x; b <= kCsrBins; b += PROLOGUE_THREADS) hist[b] = 0;
  __syncthreads();
  const int ns = (int)tmin<int64_t>(a.nnz, kCsrSamples);
  constexpr int U = 8;  // sampled loads in flight per thread
  for (int s0 = threadIdx.x; s0 < ns; s0 += PROLOGUE_THREADS * U) {
    int32_t c[U];
#pragma unroll
    for (int k = 0; k < U; ++k) {
      const int s1 = s0 + k * PROLOGUE_THREADS;
      c[k] = s1 < ns ? ldg(a.col_idx + csr_sample_index(s1, a.nnz)) : -1;
    }
#pragma unroll
    for (int k = 0; k < U; ++k)
      if (c[k] >= 0 && (int64_t)c[k] < a.n) atomicAdd(&hist[(int64_t)c[k] / wb], 1);
  }
  __syncthreads();
  // exclusive prefix sums in place: each thread owns kCsrBins / PROLOGUE_THREADS consecutive bins;
  // the threads' sums are scanned by warp shuffles, then the warps' totals by warp 0
  constexpr int PER = kCsrBins / PROLOGUE_THREADS;
  constexpr int NW = PROLOGUE_THREADS / 32;
  static_assert(kCsrBins % PROLOGUE_THREADS == 0 && NW <= 32, "bins per thread");
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int v[PER], sum = 0;
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    v[k] = hist[threadIdx.x * PER + k];
    sum += v[k];
  }
  int incl = sum;  // inclusive scan over the warp
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(FULL_MASK, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) part[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < NW ? part[lane] : 0, wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(FULL_MASK, wi, o);
      if (lane >= o) wi += x;
    }
    if (lane < NW) part[NW + lane] = wi - w;  // exclusive offset of each warp
    if (lane == 31) hist[kCsrBins] = wi;      // the total
  }
  __syncthreads();
  int run = part[NW + warp] + incl - sum;
#pragma unroll
  for (int k = 0; k < PER; ++k) {
    hist[threadIdx.x * PER + k] = run;
    run += v[k];
  }
  __syncthreads();
  // bins past nb are empty, so the prefix at nb is the total as well
  const int64_t c0 = place_on_device(hist, nb, wb, a.n, win_len, red);
  const int64_t y0 = place_on_device(hist, nb, wb, a.n, ylen, red);
  if (threadIdx.x == 0) {
    a.counters[SLOT_WIN_C0] = (unsigned long long)c0;
    a.counters[SLOT_Y0] = (unsigned long long)y0;
  }
}

// out = beta z (or 0); row partition; counters; the starts of the shared-memory windows
// (from the plan, or placed here from a column sample when the plan asks for it).
template <typename T>
__global__ void __launch_bounds__(PROLOGUE_THREADS)
    csr_prologue_kernel(const CsrArgs<T> a, const int nparts, const int row_cost, const int64_t win_c0,
                        const int64_t y0, const int64_t win_len, const int64_t ylen, const bool place) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int lane = threadIdx.x & 31;
  for (int64_t j = tid; j < a.n; j += stride) a.out[j] = a.use_z ? (T)(a.beta * (double)a.z[j]) : T(0);
  const int64_t total = a.nnz + (int64_t)row_cost * a.m;
  // one warp per partition point p: the first row i with key(i) = row_ptr[i] + row_cost * i >=
  // p * total / nparts, by a 32-way search (32 probes a step, so ~5 dependent loads for 4 M rows
  // instead of 22); key is non-decreasing and key(m) = total, so the answer lies in [0, m]
  auto key = [&](int64_t i) { return a.row_ptr[i] + (int64_t)row_cost * i; };
  for (int64_t p = tid >> 5; p <= nparts; p += stride >> 5) {
    int64_t r;
    if (p == 0) {
      r = 0;
    } else if (p == nparts) {
      r = a.m;
    } else {
      const int64_t target = (int64_t)((__int128)total * p / nparts);
      int64_t lo = 0, hi = a.m;  // rows below lo have key < target; key(hi) >= target
      while (hi - lo > 32) {
        const int64_t step = (hi - lo + 31) / 32;
        const int64_t q = tmin<int64_t>(lo + (int64_t)(lane + 1) * step, hi);
        const unsigned ge = __ballot_sync(FULL_MASK, key(q) >= target);  // lane 31 probes hi: never 0
        const int f = __ffs(ge) - 1;
        const int64_t qf = tmin<int64_t>(lo + (int64_t)(f + 1) * step, hi);
        lo = f == 0 ? lo : tmin<int64_t>(lo + (int64_t)f * step, hi) + 1;
        hi = qf;
      }
      const int64_t i = lo + lane;
      const unsigned ge = __ballot_sync(FULL_MASK, i < hi && key(i) >= target);
      r = ge ? lo + (__ffs(ge) - 1) : hi;
    }
    if (lane == 0) a.part[p] = r;
  }
  if (tid < LONG_BUCKETS + 2) a.counters[tid] = 0ull;
  if (tid == 0) {
    a.counters[SLOT_MED_COUNT] = 0ull;
    a.counters[SLOT_MED_CLAIM] = 0ull;
  }
  if (blockIdx.x == 0) {
    if (place) {
      place_windows(a, win_len, ylen);
    } else if (threadIdx.x == 0) {
      a.counters[SLOT_WIN_C0] = (unsigned long long)win_c0;
      a.counters[SLOT_Y0] = (unsigned long long)y0;
    }
  }
}

// One row of up to WARP_LONG entries (weight vi), taken by a whole warp: pass 1 forms the
// dot with WARP_UNROLL loads in flight per lane, pass 2 re-reads the row (from
// L1/L2) and scatters it.
template <typename T>
__device__ __forceinline__ void warp_row(const CsrArgs<T>& a, const Window<T>& win, T vi, int64_t st, int64_t en,
                                         T alpha, int lane) {
  DotAcc<T, sizeof(T) == 4> d;
  for (int64_t b = st + lane; b < en; b += 32 * WARP_UNROLL) {
    T xv[WARP_UNROLL];
    int32_t xc[WARP_UNROLL];
#pragma unroll
    for (int k = 0; k < WARP_UNROLL; ++k) {
      const int64_t idx = b + 32 * k;
      const bool ok = idx < en;
      xv[k] = ok ? ldg(a.vals + idx) : T(0);
      xc[k] = ok ? ldg(a.col_idx + idx) : -1;
    }
    T yv[WARP_UNROLL];
#pragma unroll
    for (int k = 0; k < WARP_UNROLL; ++k) yv[k] = xc[k] >= 0 ? win.yat(xc[k]) : T(0);
#pragma unroll
    for (int k = 0; k < WARP_UNROLL; ++k) d.add(xv[k], yv[k]);
  }
  d.template group_reduce<32>();
  const T ts = alpha * (vi * d.value());
  for (int64_t b = st + lane; b < en; b += 32 * WARP_UNROLL) {
    T xv[WARP_UNROLL];
    int32_t xc[WARP_UNROLL];
#pragma unroll
    for (int k = 0; k < WARP_UNROLL; ++k) {
      const int64_t idx = b + 32 * k;
      const bool ok = idx < en;
      xv[k] = ok ? ldg(a.vals + idx) : T(0);
      xc[k] = ok ? ldg(a.col_idx + idx) : -1;
    }
#pragma unroll
    for (int k = 0; k < WARP_UNROLL; ++k)
      if (xc[k] >= 0) win.add(xc[k], ts, xv[k]);
  }
}

template <typename T>
__global__ void __launch_bounds__(CSR_THREADS, 1)
    csr_rows_kernel(const CsrArgs<T> a, const int64_t win_len, const int64_t ylen) {
  constexpr int PACK_K = Pack<T>::K, PACK_CAP = Pack<T>::CAP;
  extern __shared__ __align__(128) unsigned char smem[];
  T* wacc = reinterpret_cast<T*>(smem);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  T* ys = reinterpret_cast<T*>(smem + window_bytes(win_len, sizeof(T)));
  unsigned char* scratch =
      smem + window_bytes(win_len, sizeof(T)) + window_bytes(ylen, sizeof(T)) + (size_t)warp * WARP_SCRATCH;
  double* dotb = reinterpret_cast<double*>(scratch);  // [32] row dots of the batch (fp32: [64] float-float words)
  T* tb = reinterpret_cast<T*>(scratch + 32 * 8);              // [32] row scales alpha * v_i * u_i
  int64_t* rsb = reinterpret_cast<int64_t*>(scratch + 64 * 8);  // [33] row starts of the window
  const Window<T> win = make_window(a, wacc, win_len, ys, ylen);
  const int64_t re = a.m;
  const T alpha = (T)a.alpha;

  // adds a lane's partial dot of one row segment into the warp's row-dot buffer, in fp64 (the
  // fp32 compensated pair converts exactly), with one native shared-memory atomic: segment sums
  // of one row can cancel, and fp64 keeps their sum's rounding below the fp32 bound
  auto flush = [&](int row, const DotAcc<T, sizeof(T) == 4>& part) {
    if constexpr (sizeof(T) == 4) {
      // float-float row dot: the atomic returns the old sum, so the rounding error of the
      // addition it made is recovered exactly (TwoSum) and added, with the segment's own
      // compensation, into the low word
      float* dotf = reinterpret_cast<float*>(dotb);
      const float old = atomicAdd(&dotf[row], part.s);
      float sum, err;
      two_sum(old, part.s, sum, err);
      atomicAdd(&dotf[32 + row], __fadd_rn(err, part.c));
    } else {
      atomicAdd(&dotb[row], part.value_f64());
    }
  };

  window_init(win);
  dotb[lane] = 0.0;
  __syncthreads();

  // 32-row windows from one global counter; the next window is claimed while this one runs
  // (claims of four windows were measured slower: 346 against 294 us on the power-law matrix)
  unsigned long long next = 0;
  if (lane == 0) next = atomicAdd(&a.counters[LONG_BUCKETS + 1], 32ull);
  for (;;) {
    const int64_t r0 = (int64_t)__shfl_sync(FULL_MASK, next, 0);
    if (r0 >= re) break;
    if (lane == 0) next = atomicAdd(&a.counters[LONG_BUCKETS + 1], 32ull);
    const int nr = (int)tmin<int64_t>(32, re - r0);  // rows in this window
    const bool hasrow = lane < nr;
    const int64_t rs = hasrow ? a.row_ptr[r0 + lane] : 0;
    const int64_t rend = hasrow ? a.row_ptr[r0 + lane + 1] : 0;
    const T vrow = (hasrow && a.v) ? ldg(a.v + r0 + lane) : T(1);  // this lane's row weight
    const int64_t len = rend - rs;
    const bool isshort = hasrow && len <= PACK_CAP;
    rsb[lane] = hasrow ? rs : INT64_MAX;
    if (lane == 0) rsb[32] = INT64_MAX;
    __syncwarp();
    const unsigned shortmask = __ballot_sync(FULL_MASK, isshort);

    // packed batches: maximal runs of consecutive short rows holding at most PACK_CAP entries
    int b0 = 0;
    while (b0 < nr) {
      const unsigned cand = shortmask & (0xffffffffu << b0);
      if (cand == 0) break;
      b0 = __ffs(cand) - 1;
      const int64_t s = __shfl_sync(FULL_MASK, rs, b0);
      const bool fits = lane >= b0 && isshort && rend - s <= PACK_CAP;
      const unsigned notfit = ~__ballot_sync(FULL_MASK, fits) & (0xffffffffu << b0);
      const int b1 = notfit ? __ffs(notfit) - 1 : 32;  // rows [b0, b1); b1 > b0 since row b0 fits
      const int64_t e = __shfl_sync(FULL_MASK, rend, b1 - 1);
      const int64_t base = s + (int64_t)lane * PACK_K;

      T val[PACK_K];
      int32_t col[PACK_K];
#pragma unroll
      for (int k = 0; k < PACK_K; ++k) {
        const int64_t idx = base + k;
        const bool ok = idx < e;
        val[k] = ok ? ldg(a.vals + idx) : T(0);
        col[k] = ok ? ldg(a.col_idx + idx) : -1;
      }
      T yv[PACK_K];
#pragma unroll
      for (int k = 0; k < PACK_K; ++k) yv[k] = col[k] >= 0 ? win.yat(col[k]) : T(0);

      // row of this lane's first entry: the last row of [b0, b1) starting at or before base
      int lo = b0, hi = b1 - 1;
#pragma unroll
      for (int it = 0; it < 5; ++it) {
        const int mid = (lo + hi + 1) >> 1;
        if (rsb[mid] <= base) lo = mid; else hi = mid - 1;
      }
      // lane-local segment sums, each flushed once into the warp's row-dot buffer
      int cur = lo;
      bool have = false;
      DotAcc<T, sizeof(T) == 4> acc;
#pragma unroll
      for (int k = 0; k < PACK_K; ++k) {
        if (col[k] >= 0) {
          const int64_t idx = base + k;
          while (rsb[cur + 1] <= idx) {  // rsb[b1] > idx: rows past the batch start after e
            if (have) flush(cur, acc);
            acc = DotAcc<T, sizeof(T) == 4>();
            have = false;
            ++cur;
          }
          acc.add(val[k], yv[k]);
          have = true;
        }
      }
      if (have) flush(cur, acc);
      __syncwarp();
      if (lane >= b0 && lane < b1) {
        T u;
        if constexpr (sizeof(T) == 4) {
          float* dotf = reinterpret_cast<float*>(dotb);
          u = __fadd_rn(dotf[lane], dotf[32 + lane]);
          dotf[lane] = 0.f;
          dotf[32 + lane] = 0.f;
        } else {
          u = (T)dotb[lane];
          dotb[lane] = 0.0;
        }
        tb[lane] = alpha * (vrow * u);
      }
      __syncwarp();
      // scatter, walking the same row boundaries again
      cur = lo;
#pragma unroll
      for (int k = 0; k < PACK_K; ++k) {
        if (col[k] >= 0) {
          const int64_t idx = base + k;
          while (rsb[cur + 1] <= idx) ++cur;
          win.add(col[k], tb[cur], val[k]);
        }
      }
      __syncwarp();
      b0 = b1;
    }

    // rows longer than a packed batch go to the long-row kernel's queues: the medium ones of the
    // window with one atomic for the warp (the counter is shared by every warp of the grid)
    if (hasrow && len > WARP_LONG) defer_row(a, r0 + lane, len);
    const bool med = hasrow && !isshort && len <= WARP_LONG;
    const unsigned mm = __ballot_sync(FULL_MASK, med);
    if (mm) {
      const int leader = __ffs(mm) - 1;
      unsigned long long mb = 0;
      if (lane == leader) mb = atomicAdd(&a.counters[SLOT_MED_COUNT], (unsigned long long)__popc(mm));
      mb = __shfl_sync(FULL_MASK, mb, leader);
      if (med) a.med_queue[mb + (unsigned long long)__popc(mm & ((1u << lane) - 1u))] = r0 + lane;
    }
    __syncwarp();  // rsb reuse
  }
  __syncthreads();
  window_flush(wacc, win.c0, win_len, a.out);
}

// Short rows in lane groups: LPR lanes per row, KG entries per lane held in
// registers, G = 32 / LPR rows per warp step. This costs fewer fp64 operations
// per entry than the packed batches when rows are of similar length (no
// per-segment flushes), so the fp64 path uses it. Rows longer than LPR * KG go
// to warp_row or to the long-row queue.
template <typename T, int LPR, int KG>
__global__ void __launch_bounds__(CSR_GROUP_THREADS, 1)
    csr_group_kernel(const CsrArgs<T> a, const int64_t win_len, const int64_t ylen) {
  constexpr int G = 32 / LPR;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ unsigned long long s_next;
  T* wacc = reinterpret_cast<T*>(smem);
  const T* ys = reinterpret_cast<const T*>(smem + window_bytes(win_len, sizeof(T)));
  const Window<T> win = make_window(a, wacc, win_len, ys, ylen);
  const int lane = threadIdx.x & 31;
  const int g = lane / LPR, q = lane % LPR;
  const int64_t rb = a.part[blockIdx.x], re = a.part[blockIdx.x + 1];
  const T alpha = (T)a.alpha;

  window_init(win);
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
    const bool small = has && en - st <= LPR * KG;
    const T vi = (small && a.v) ? ldg(a.v + r) : T(1);
    T val[KG];
    int32_t col[KG];
#pragma unroll
    for (int k = 0; k < KG; ++k) {
      const int64_t idx = st + q + LPR * k;
      const bool ok = small && idx < en;
      val[k] = ok ? ldg(a.vals + idx) : T(0);
      col[k] = ok ? ldg(a.col_idx + idx) : -1;
    }
    DotAcc<T, (sizeof(T) == 4 && LPR * KG > 64)> d;
#pragma unroll
    for (int k = 0; k < KG; ++k)
      if (col[k] >= 0) d.add(val[k], win.yat(col[k]));
    d.template group_reduce<LPR>();
    const T ts = alpha == T(1) ? vi * d.value() : alpha * (vi * d.value());
#pragma unroll
    for (int k = 0; k < KG; ++k)
      if (col[k] >= 0) win.add(col[k], ts, val[k]);

    // longer rows: one warp each, here (rows of similar length rarely outgrow a group, and each
    // deferral would cost an atomic on one shared counter), or the long-row queue
    unsigned lm = __ballot_sync(FULL_MASK, has && !small && q == 0);
    while (lm) {
      const int src = __ffs(lm) - 1;
      lm &= lm - 1;
      const int64_t rr = __shfl_sync(FULL_MASK, r, src);
      const int64_t s2 = __shfl_sync(FULL_MASK, st, src), e2 = __shfl_sync(FULL_MASK, en, src);
      if (e2 - s2 > WARP_LONG) {
        if (lane == 0) defer_row(a, rr, e2 - s2);
      } else {
        warp_row(a, win, a.v ? ldg(a.v + rr) : T(1), s2, e2, alpha, lane);
      }
    }
  }
  __syncthreads();
  window_flush(wacc, win.c0, win_len, a.out);
}

// Rows longer than WARP_LONG: each group of G threads takes queued rows
// one at a time, with one group barrier per row. Rows are claimed from one global
// counter that walks the length buckets from the longest down, so the longest
// rows start first and short ones fill in at the end. A group rather than a warp
// per row keeps the rows in flight few enough that a row read by pass 1 is still
// in L2 when pass 2 re-reads it. Both passes keep the next batch of entries loading
// while the current batch is used. The next row's index is claimed while the
// current one is processed, and the per-warp partial dots are double-buffered by
// row parity, so the single barrier orders both.
template <typename T, int G>
__device__ __forceinline__ void long_batch(const CsrArgs<T>& a, int64_t b, int64_t en, T* xv, int32_t* xc) {
  constexpr int U = long_unroll<T>();
#pragma unroll
  for (int k = 0; k < U; ++k) {
    const int64_t idx = b + (int64_t)k * G;
    const bool ok = idx < en;
    xv[k] = ok ? ldg(a.vals + idx) : T(0);
    xc[k] = ok ? ldg(a.col_idx + idx) : -1;
  }
}

// Named barrier over the `count` threads of one row group (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void group_barrier(int id, int count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

template <typename T, int G>
__global__ void __launch_bounds__(CSR_THREADS, 1)
    csr_long_kernel(const CsrArgs<T> a, const int64_t win_len, const int64_t ylen) {
  constexpr int U = long_unroll<T>();
  constexpr int GW = G / 32;           // warps per group
  constexpr int NG = CSR_THREADS / G;  // groups per CTA (named barriers 1 .. NG)
  static_assert(NG >= 1 && NG <= 15 && CSR_THREADS % G == 0, "named barrier ids");
  constexpr int64_t STEP = (int64_t)G * U;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ long long s_row[NG][2];
  __shared__ double s_red[NG][2][GW];
  // nothing queued (no row outgrew the row kernel): skip the windows' set-up and flush; the
  // counters are final, so every thread takes the same branch
  {
    unsigned long long queued = a.counters[SLOT_MED_COUNT];
    for (int b = 0; b < LONG_BUCKETS; ++b) queued += a.counters[1 + b];
    if (queued == 0ull) return;
  }
  T* wacc = reinterpret_cast<T*>(smem);
  const T* ys = reinterpret_cast<const T*>(smem + window_bytes(win_len, sizeof(T)));
  const Window<T> win = make_window(a, wacc, win_len, ys, ylen);
  const int lane = threadIdx.x & 31;
  const int grp = threadIdx.x / G, gt = threadIdx.x % G, gw = gt >> 5;
  const int bar = 1 + grp;
  const T alpha = (T)a.alpha;
  auto claim = [&]() -> long long {
    unsigned long long k = atomicAdd(&a.counters[0], 1ull);
    for (int b = LONG_BUCKETS - 1; b >= 0; --b) {
      const unsigned long long c = a.counters[1 + b];
      if (k < c) return (long long)a.queue[(int64_t)b * a.queue_cap + (int64_t)k];
      k -= c;
    }
    return -1ll;
  };

  window_init(win);
  if (gt == 0) s_row[grp][0] = claim();
  __syncthreads();
  for (int it = 0;; ++it) {
    const int cur = it & 1;
    const int64_t r = s_row[grp][cur];
    if (r < 0) break;
    if (gt == 0) s_row[grp][cur ^ 1] = claim();
    const int64_t st = a.row_ptr[r], en = a.row_ptr[r + 1];

    // pass 1: the dot
    DotAcc<T, sizeof(T) == 4> d;
    T xv[U];
    int32_t xc[U];
    long_batch<T, G>(a, st + gt, en, xv, xc);
    for (int64_t b = st + gt; b < en; b += STEP) {
      T nv[U];
      int32_t nc[U];
      long_batch<T, G>(a, b + STEP, en, nv, nc);
      T yv[U];
#pragma unroll
      for (int k = 0; k < U; ++k) yv[k] = xc[k] >= 0 ? win.yat(xc[k]) : T(0);
#pragma unroll
      for (int k = 0; k < U; ++k) {
        d.add(xv[k], yv[k]);
        xv[k] = nv[k];
        xc[k] = nc[k];
      }
    }
    d.template group_reduce<32>();
    if (lane == 0) s_red[grp][cur][gw] = d.value_f64();
    group_barrier(bar, G);
    double u = 0.0;
#pragma unroll
    for (int w = 0; w < GW; ++w) u += s_red[grp][cur][w];
    const T vi = a.v ? ldg(a.v + r) : T(1);
    const T ts = alpha * (vi * (T)u);

    // pass 2: the scatter, re-reading the row (served by L2)
    long_batch<T, G>(a, st + gt, en, xv, xc);
    for (int64_t b = st + gt; b < en; b += STEP) {
      T nv[U];
      int32_t nc[U];
      long_batch<T, G>(a, b + STEP, en, nv, nc);
#pragma unroll
      for (int k = 0; k < U; ++k) {
        if (xc[k] >= 0) win.add(xc[k], ts, xv[k]);
        xv[k] = nv[k];
        xc[k] = nc[k];
      }
    }
  }
  // then the medium rows (longer than the row kernel's batches, at most WARP_LONG entries):
  // one warp each, claimed one at a time, so the last rows of the call spread over every warp
  // (claims of 4 rows were measured 2 % slower on the power-law workload)
  constexpr unsigned long long MED_CLAIM = 1;
  const unsigned long long nmed = a.counters[SLOT_MED_COUNT];
  for (;;) {
    unsigned long long k0 = 0;
    if (lane == 0) k0 = atomicAdd(&a.counters[SLOT_MED_CLAIM], MED_CLAIM);
    k0 = __shfl_sync(FULL_MASK, k0, 0);
    if (k0 >= nmed) break;
    const unsigned long long k1 = tmin(nmed, k0 + MED_CLAIM);
    for (unsigned long long k = k0; k < k1; ++k) {
      const int64_t r = a.med_queue[k];
      warp_row(a, win, a.v ? ldg(a.v + r) : T(1), a.row_ptr[r], a.row_ptr[r + 1], alpha, lane);
    }
  }
  __syncthreads();
  window_flush(wacc, win.c0, win_len, a.out);
}

template <typename T, int LPR, int KG>
static cudaError_t launch_group(const CsrPlan& p, const CsrArgs<T>& a, cudaStream_t st) {
  if (p.threads != CSR_GROUP_THREADS) return cudaErrorInvalidConfiguration;
  const cudaError_t e = ensure_smem((const void*)csr_group_kernel<T, LPR, KG>, p.long_smem);
  if (e != cudaSuccess) return e;
  csr_group_kernel<T, LPR, KG><<<p.ctas, p.threads, p.long_smem, st>>>(a, p.win_len, p.ylen);
  return cudaGetLastError();
}

template <typename T, int G>
static cudaError_t launch_long(const CsrPlan& p, const CsrArgs<T>& a, cudaStream_t st) {
  const cudaError_t e = ensure_smem((const void*)csr_long_kernel<T, G>, p.long_smem);
  if (e != cudaSuccess) return e;
  csr_long_kernel<T, G><<<p.long_ctas, p.long_threads, p.long_smem, st>>>(a, p.win_len, p.ylen);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_csr(const CsrPlan& p, const CsrArgs<T>& a, cudaStream_t st) {
  {
    const int64_t work = std::max<int64_t>(a.n, ((int64_t)p.ctas + 1) * 32);  // a warp per partition point
    const int blocks = (int)std::min<int64_t>((work + PROLOGUE_THREADS - 1) / PROLOGUE_THREADS, 4096);
    csr_prologue_kernel<T><<<blocks, PROLOGUE_THREADS, 0, st>>>(a, p.ctas, p.row_cost, p.win_c0, p.y0, p.win_len,
                                                                 p.ylen, p.place_on_device && a.nnz > 0);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (a.m == 0) return cudaSuccess;
  cudaError_t e;
  if (p.group_lpr == 0) {
    e = ensure_smem((const void*)csr_rows_kernel<T>, p.smem);
    if (e != cudaSuccess) return e;
    csr_rows_kernel<T><<<p.ctas, p.threads, p.smem, st>>>(a, p.win_len, p.ylen);
  } else {
    switch (p.group_lpr * 100 + p.group_kg) {
      case 208: e = launch_group<T, 2, 8>(p, a, st); break;
      case 408: e = launch_group<T, 4, 8>(p, a, st); break;
      case 808: e = launch_group<T, 8, 8>(p, a, st); break;
      case 1608: e = launch_group<T, 16, 8>(p, a, st); break;
      case 216: e = launch_group<T, 2, 16>(p, a, st); break;
      case 416: e = launch_group<T, 4, 16>(p, a, st); break;
      case 816: e = launch_group<T, 8, 16>(p, a, st); break;
      case 1616: e = launch_group<T, 16, 16>(p, a, st); break;
      default: return cudaErrorInvalidConfiguration;
    }
    if (e != cudaSuccess) return e;
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  switch (p.long_group) {
    case 128: return launch_long<T, 128>(p, a, st);
    case 256: return launch_long<T, 256>(p, a, st);
    case 512: return launch_long<T, 512>(p, a, st);
    case 1024: return launch_long<T, 1024>(p, a, st);
    default: return cudaErrorInvalidConfiguration;
  }
}

template cudaError_t launch_csr<float>(const CsrPlan&, const CsrArgs<float>&, cudaStream_t);
template cudaError_t launch_csr<double>(const CsrPlan&, const CsrArgs<double>&, cudaStream_t);

// The strided sample the model reads: kCsrSamples row lengths and column indices at the
// positions of csr_sample_index.
__global__ void csr_sample_kernel(int64_t m, int64_t nnz, const int64_t* row_ptr, const int32_t* col_idx,
                                  int64_t* lens, int32_t* cols) {
  const int nl = (int)tmin<int64_t>(m, kCsrSamples), nc = (int)tmin<int64_t>(nnz, kCsrSamples);
  for (int s = blockIdx.x * blockDim.x + threadIdx.x; s < kCsrSamples; s += gridDim.x * blockDim.x) {
    if (s < nl) {
      const int64_t i = csr_sample_index(s, m);
      lens[s] = row_ptr[i + 1] - row_ptr[i];
    }
    if (s < nc) cols[s] = col_idx[csr_sample_index(s, nnz)];
  }
}

cudaError_t launch_csr_sample(int64_t m, int64_t nnz, const int64_t* row_ptr, const int32_t* col_idx, int64_t* lens,
                              int32_t* cols, cudaStream_t st) {
  csr_sample_kernel<<<kCsrSamples / 256, 256, 0, st>>>(m, nnz, row_ptr, col_idx, lens, cols);
  return cudaGetLastError();
}

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
