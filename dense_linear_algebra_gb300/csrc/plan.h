// plan.h — the analytical launch-parameter model (host side).
//
// "On optimizing machine learning workloads via kernel fusion" (abstract) pairs
// the fused kernel with a model that picks launch parameters from the input's
// characteristics and the GPU's resources. This is that model rebuilt for
// GB300: it reads m, n, ld, nnz, the element size, pointer alignment, the SM
// count and the shared-memory limit, and returns the kernel variant together
// with its coarsening (rows per tile, lanes per row, columns per lane), its
// pipeline depth, grid size and reduction mode. For CSR it also reads the
// matrix's data: a strided sample of row lengths (their spread sizes the fp64
// lane groups) and of column indices (which column ranges the shared-memory
// scatter window and the copy of y should cover). Without a host-side sample the
// kernels' prologue places those windows on the device from its own sample, so
// calls stay asynchronous. It costs a few microseconds at most.
#pragma once

#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <vector>

namespace fxtx {

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  int smem_optin = 0;  // max dynamic shared memory per block (bytes)
  int smem_per_sm = 0;
};

enum DenseKind { DENSE_NOOP = 0, DENSE_EMPTY_ROWS, DENSE_NARROW_TMA, DENSE_NARROW_DIRECT, DENSE_WIDE, DENSE_TILE_TMA };

struct DensePlan {
  DenseKind kind = DENSE_NOOP;
  int nb = 0;             // tile kernel: 128-byte column blocks per row, rounded up to a power of two
  int nbr = 0;            // tile kernel: column blocks actually copied, ceil(n * elem / box_bytes)
  int box_bytes = 0;      // tile kernel: width of a tensor-copy box (128, or 64 for rows of at most 64 bytes)
  int lpr = 0;            // lanes cooperating on one row (narrow)
  int vpl = 0;            // 16-byte chunks of a row held per lane (narrow)
  int rows_per_tile = 0;  // coarsening: rows a warp takes per pipeline step
  int stages = 0;         // pipeline depth per warp (narrow TMA)
  int warps = 0;          // warps per CTA
  int ctas = 0;           // grid size
  size_t smem = 0;        // dynamic shared memory per CTA
  bool smem_acc = false;  // wide: column accumulator kept in shared memory
  size_t ws_bytes = 0;    // device workspace
  double est_us = 0.0;    // the model's estimate of the launch's duration
};

// lanes-per-row / chunks-per-lane table of the narrow kernel, keyed by the
// number of 16-byte chunks in a row (1..128). Returns false when the row is
// too long for the narrow kernel.
bool narrow_shape(int64_t chunks, int* lpr, int* vpl);

// tma_ok: X 16-byte aligned and rows whole 16-byte chunks (1-D bulk copies);
// tile_ok: X 16-byte aligned and ld * elem a multiple of 16 (2-D tensor copies).
DensePlan plan_dense(const DeviceInfo& dev, int64_t m, int64_t n, int64_t ld, int elem, bool tma_ok, bool tile_ok);

// Input-data characteristics of a CSR matrix, from a strided sample of its row lengths
// and of its column indices (kCsrSamples of each, at csr_sample_index positions).
constexpr int kCsrSamples = 8192;
constexpr int kCsrBins = 1024;  // column-sample histogram bins (of csr_bin_width columns each)

struct CsrStats {
  bool valid = false;
  int row_samples = 0, col_samples = 0;
  double mean_len = 0.0, cv_len = 0.0;              // sampled row lengths: mean, coefficient of variation
  int64_t p50_len = 0, p75_len = 0, p90_len = 0, max_len = 0;
  double long_share = 0.0;                          // length-weighted share of sampled rows over the one-warp limit
  int64_t bin_width = 0;                            // columns per histogram bin
  int bins = 0;
  std::vector<int> col_hist;                        // sampled column indices per bin
};

// Position of sample s (0 <= s < kCsrSamples) among `count` items: s itself when count <=
// kCsrSamples (then only s < count are taken), else a point inside the s-th of kCsrSamples
// equal strides, offset within it by a fixed integer hash of s (so that a period in the
// matrix's structure cannot line up with the strides). The device sampler uses the same
// positions.
__host__ __device__ inline int64_t csr_sample_index(int s, int64_t count) {
  if (count <= kCsrSamples) return (int64_t)s;
  uint32_t h = (uint32_t)s * 0x9e3779b1u;  // Knuth's multiplicative hash, then an xor-shift mix
  h ^= h >> 15;
  h *= 0x85ebca6bu;
  h ^= h >> 13;
  const int64_t stride = count / kCsrSamples;  // >= 1
  return ((int64_t)s * count) / kCsrSamples + (int64_t)(h % (uint64_t)stride);
}
// Histogram bin width that spreads n columns over at most kCsrBins bins.
__host__ __device__ inline int64_t csr_bin_width(int64_t n) { return n <= 0 ? 1 : (n + kCsrBins - 1) / kCsrBins; }

// Statistics from sampled row lengths (lens[0 .. nl)) and sampled column indices
// (cols[0 .. nc)); warp_cap is the one-warp row limit of the CSR kernels.
CsrStats csr_stats_from_samples(int64_t n, const int64_t* lens, int nl, const int32_t* cols, int nc, int64_t warp_cap);
// The same statistics from host arrays row_ptr (m + 1) and col_idx (nnz).
CsrStats csr_stats_from_host(int64_t m, int64_t n, int64_t nnz, const int64_t* row_ptr, const int32_t* col_idx);

// The start of the window of `len` columns (of n) that holds the most sampled columns: the
// first maximum over bin-aligned starts of the sampled count in whole bins, clamped to
// [0, n - len]. *hits receives that count. The prologue of the CSR kernels applies the
// same rule to its own sample on the device.
int64_t csr_place_window(const CsrStats& st, int64_t n, int64_t len, int* hits);

struct CsrPlan {
  int group_lpr = 0;        // short rows in lane groups of this many lanes; 0: packed batches
  int group_kg = 0;         // entries each lane of a group holds (8 or 16)
  int pack_k = 0;           // consecutive entries per lane in a packed batch of short rows
  int pack_cap = 0;         // entries per packed batch (32 * pack_k): longer rows are not packed
  int warp_cap = 0;         // longest row one warp takes; longer rows go to the long-row kernel
  int ctas = 0, threads = 0;            // row kernel
  int long_ctas = 0, long_threads = 0;  // long-row kernel
  int long_group = 0;                   // threads sharing one long row (128, 256, 512 or 1024)
  int64_t win_c0 = 0, win_len = 0;      // columns accumulated in shared memory
  int64_t y0 = 0, ylen = 0;             // y[y0, y0 + ylen) held in shared memory for the gathers
  bool place_on_device = false;         // the prologue places both windows from its own column sample
  bool sampled = false;                 // the plan read sampled statistics (the fields below)
  double mean_len = 0.0, cv_len = 0.0, long_share = 0.0, win_hit = 0.0, y_hit = 0.0;
  int64_t p75_len = 0;
  size_t smem = 0, long_smem = 0;
  int row_cost = 0;         // nnz-equivalent cost of one row, for the partition
  size_t ws_bytes = 0;
  int64_t queue_cap = 0;    // capacity of each long-row queue
  int64_t med_cap = 0;      // capacity of the medium-row queue (rows past the short-row batches)
  double est_us = 0.0;      // the model's estimate of the call's duration
};

// Constants of the CSR kernels (csr.cu): shared memory of the row kernel for an
// accumulator window of win_len columns and a y window of ylen entries, the
// packed-batch capacity and the one-warp row limit.
size_t csr_rows_smem(int64_t win_len, int64_t ylen, int elem);
int csr_pack_cap(int elem);
int csr_warp_long();
int csr_group_threads();  // block size of the lane-group kernel
int csr_long_buckets();  // length buckets of the long-row queue
int csr_long_group_default();  // threads sharing one long row unless a candidate says otherwise

// The CSR plan from the shape alone (st == nullptr: both windows are then placed on the
// device, per call, from a column sample), or from sampled statistics of the matrix.
CsrPlan plan_csr(const DeviceInfo& dev, int64_t m, int64_t n, int64_t nnz, int elem, const CsrStats* st = nullptr);

// The cost model's roofline (in microseconds, one call): the slowest of `bytes` through
// HBM at hbm_eff of 6.8 TB/s, `fmas` at fma_eff of the device's FMA rate for elements of
// `elem` bytes, and `l2_sectors` random 32-byte L2 accesses at l2_eff of 4.9e11 per second,
// plus the fixed cost of a call.
double roofline_us(const DeviceInfo& dev, double bytes, double hbm_eff, double fmas, int elem, double fma_eff,
                   double l2_sectors, double l2_eff);

// Microseconds of `cycles` SM cycles at the clock the estimates assume.
double sm_cycles_us(double cycles);

int describe(const DensePlan& p, char* buf, size_t cap);
int describe(const CsrPlan& p, char* buf, size_t cap);

// The launches the tuner times for one call shape: the model's plan first, then the
// variants of its free parameters that fit the device (pipeline depth and warps of
// the tensor-copy kernels; the shared-memory split between the scatter window and
// the copy of y, and the fp64 lane-group width, of the CSR kernels).
std::vector<DensePlan> dense_candidates(const DeviceInfo& dev, const DensePlan& model, int64_t m, int64_t n, int elem);
std::vector<CsrPlan> csr_candidates(const DeviceInfo& dev, const CsrPlan& model, int64_t m, int64_t n, int64_t nnz,
                                    int elem, const CsrStats* st = nullptr);

}  // namespace fxtx
