// plan.h — the analytical launch-parameter model (host side).
//
// "On optimizing machine learning workloads via kernel fusion" (abstract) pairs
// the fused kernel with a model that picks launch parameters from the input's
// characteristics and the GPU's resources. This is that model rebuilt for
// GB300: it reads m, n, ld, nnz, the element size, pointer alignment, the SM
// count and the shared-memory limit, and returns the kernel variant together
// with its coarsening (rows per tile, lanes per row, columns per lane), its
// pipeline depth, grid size and reduction mode. It costs a few hundred
// nanoseconds and touches no device memory.
#pragma once

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

struct CsrPlan {
  int group_lpr = 0;        // short rows in lane groups of this many lanes; 0: packed batches
  int group_kg = 0;         // entries each lane of a group holds (8 or 16)
  int pack_k = 0;           // consecutive entries per lane in a packed batch of short rows
  int pack_cap = 0;         // entries per packed batch (32 * pack_k): longer rows are not packed
  int warp_cap = 0;         // longest row one warp takes; longer rows go to the long-row kernel
  int ctas = 0, threads = 0;            // row kernel
  int long_ctas = 0, long_threads = 0;  // long-row kernel
  int64_t win_c0 = 0, win_len = 0;      // columns accumulated in shared memory
  int64_t ylen = 0;                     // y[0, ylen) held in shared memory for the gathers
  size_t smem = 0, long_smem = 0;
  int row_cost = 0;         // nnz-equivalent cost of one row, for the partition
  size_t ws_bytes = 0;
  int64_t queue_cap = 0;    // capacity of the long-row queue
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

CsrPlan plan_csr(const DeviceInfo& dev, int64_t m, int64_t n, int64_t nnz, int elem);

// The cost model's roofline (in microseconds, one call): the slowest of `bytes` through
// HBM at hbm_eff of 6.8 TB/s, `fmas` at fma_eff of the device's FMA rate for elements of
// `elem` bytes, and `l2_sectors` random 32-byte L2 accesses at l2_eff of 4.9e11 per second,
// plus the fixed cost of a call.
double roofline_us(const DeviceInfo& dev, double bytes, double hbm_eff, double fmas, int elem, double fma_eff,
                   double l2_sectors, double l2_eff);

int describe(const DensePlan& p, char* buf, size_t cap);
int describe(const CsrPlan& p, char* buf, size_t cap);

// The launches the tuner times for one call shape: the model's plan first, then the
// variants of its free parameters that fit the device (pipeline depth and warps of
// the tensor-copy kernels; the shared-memory split between the scatter window and
// the copy of y, and the fp64 lane-group width, of the CSR kernels).
std::vector<DensePlan> dense_candidates(const DeviceInfo& dev, const DensePlan& model, int64_t m, int64_t n, int elem);
std::vector<CsrPlan> csr_candidates(const DeviceInfo& dev, const CsrPlan& model, int64_t m, int64_t n, int64_t nnz,
                                    int elem);

}  // namespace fxtx
