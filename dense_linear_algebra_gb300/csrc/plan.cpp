// plan.cpp — the analytical launch-parameter model (see plan.h).
#include "plan.h"

#include <algorithm>
#include <cmath>
#include <cstdio>

namespace fxtx {

namespace {

constexpr int64_t kTileTarget = 8 * 1024;      // bytes a warp takes per pipeline step
constexpr int64_t kSmemBudget = 200 * 1024;    // dynamic shared memory a CTA may claim
constexpr int kCsrThreads = 1024;

int64_t pow2_ceil(int64_t x) {
  int64_t p = 1;
  while (p < x) p <<= 1;
  return p;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

size_t align128(size_t x) { return (x + 127) / 128 * 128; }

// Rates of the cost model, per GB300 measurements: HBM copy bandwidth, FMA issue per
// SM and clock (fp32 124.7, fp64 2), the SM clock, and L2 random-sector throughput.
constexpr double kHbmBytesPerS = 6.8e12;
constexpr double kClockHz = 2.07e9;
constexpr double kFma32PerSmClk = 124.7;
constexpr double kFma64PerSmClk = 2.0;
constexpr double kL2SectorsPerS = 4.9e11;
constexpr double kLaunchUs = 4.0;  // launch, grid reduction and epilogue of one call
constexpr double kScatterMissWeight = 1.15;  // cost of a scatter outside the window / a gather outside y's copy
constexpr double kSplitGain = 0.02;          // least sampled gain that moves the window/y split off ¾

}  // namespace

// Roofline estimate: the slowest of HBM bytes, FMAs and random L2 sectors, each at the
// fraction of its peak the kernel kind reaches, plus the fixed cost of a call.
double roofline_us(const DeviceInfo& dev, double bytes, double hbm_eff, double fmas, int elem, double fma_eff,
                   double l2_sectors, double l2_eff) {
  const double fma_rate = (elem == 8 ? kFma64PerSmClk : kFma32PerSmClk) * std::max(dev.sm_count, 1) * kClockHz;
  double t = bytes / (kHbmBytesPerS * hbm_eff);
  t = std::max(t, fmas / (fma_rate * fma_eff));
  t = std::max(t, l2_sectors / (kL2SectorsPerS * l2_eff));
  return t * 1e6 + kLaunchUs;
}

double sm_cycles_us(double cycles) { return cycles / kClockHz * 1e6; }

namespace {

// Dense call: X once, v, y, z and out; two FMAs per element of X.
double dense_est_us(const DeviceInfo& dev, const DensePlan& p, int64_t m, int64_t n, int elem) {
  const int ce = elem == 2 ? 4 : elem;  // compute-type bytes of the vectors
  const double bytes = (double)m * n * elem + (double)m * ce + 3.0 * n * ce;
  static const double hbm_eff[] = {1.0, 1.0, 0.85, 0.5, 0.9, 0.99};  // by DenseKind
  const double fmas = 2.0 * m * n;
  return roofline_us(dev, bytes, hbm_eff[p.kind], fmas, elem == 2 ? 4 : elem, 0.7, 0.0, 1.0);
}

// CSR call: vals and col_idx once, row_ptr, v, y, z and out; two FMAs per entry; a
// random L2 sector for each gather and scatter outside the shared-memory copies, at the
// sampled hit rates of the two windows when the plan has them, else with columns taken
// as uniform over [0, n).
double csr_est_us(const DeviceInfo& dev, const CsrPlan& p, int64_t m, int64_t n, int64_t nnz, int elem) {
  const double bytes = (double)nnz * (elem + 4) + (double)(m + 1) * 8 + (double)m * elem + 3.0 * n * elem;
  const double nn = (double)std::max<int64_t>(n, 1);
  const double miss = p.sampled ? (1.0 - p.y_hit) + (1.0 - p.win_hit)
                                : (1.0 - std::min(1.0, p.ylen / nn)) + (1.0 - std::min(1.0, p.win_len / nn));
  // fp64 lane groups reach 45 % of the fp64 FMA rate (padding slots, reductions, the CAS
  // loop); fp32 packed rows are bound by memory and L2, not FMAs
  return roofline_us(dev, bytes, 0.8, 2.0 * nnz, elem, elem == 8 ? 0.45 : 0.6, miss * nnz, 0.6);
}

}  // namespace

bool narrow_shape(int64_t chunks, int* lpr, int* vpl) {
  if (chunks <= 0) return false;
  if (chunks <= 8) {
    *lpr = (int)pow2_ceil(chunks);
    *vpl = 1;
  } else if (chunks <= 16) {
    *lpr = 8; *vpl = 2;
  } else if (chunks <= 32) {
    *lpr = 8; *vpl = 4;
  } else if (chunks <= 64) {
    *lpr = 16; *vpl = 4;
  } else if (chunks <= 128) {
    *lpr = 32; *vpl = 4;
  } else {
    return false;
  }
  return true;
}

// Workspace of the wide kernels: [ctas][n] fp64 column partials (which are also the column
// sums when these do not fit shared memory); the ticket word last.
static size_t wide_ws_bytes(const DensePlan& p, int64_t n, int elem) {
  (void)elem;
  return align128((size_t)p.ctas * n * sizeof(double)) + 128;
}

static void set_wide_grid(const DeviceInfo& dev, DensePlan& p, int64_t m, int64_t n, int elem) {
  (void)n;
  (void)elem;
  p.ctas = (int)std::max<int64_t>(1, std::min<int64_t>(dev.sm_count, cdiv(m, p.rows_per_tile)));
}

static DensePlan plan_dense_model(const DeviceInfo& dev, int64_t m, int64_t n, int64_t ld, int elem, bool tma_ok,
                                  bool tile_ok) {
  DensePlan p;
  if (n == 0) return p;  // nothing to write
  if (m == 0) {
    p.kind = DENSE_EMPTY_ROWS;
    return p;
  }
  const int64_t budget = std::min<int64_t>(kSmemBudget, dev.smem_optin > 0 ? dev.smem_optin : 48 * 1024);
  // bfloat16 X (elem 2) is computed in fp32: the narrow kernel counts its chunks in fp32 elements
  const int64_t chunks = cdiv(n * (elem == 2 ? 4 : elem), 16);
  const int64_t row_bytes = n * elem;
  const int cpl = elem == 2 ? 2 : 4;  // 16-byte chunks per lane in the tile kernel
  const int64_t max_tile_row = elem == 2 ? 1024 : 2048;
  if (tile_ok && row_bytes >= 32 && row_bytes <= max_tile_row && m < (int64_t(1) << 31)) {
    // tile kernel: boxes of 128 bytes (64 for rows of at most 64 bytes); 8-KB tiles (16 KB at nb = 16)
    p.kind = DENSE_TILE_TMA;
    p.box_bytes = row_bytes <= 64 ? 64 : 128;
    p.nbr = (int)cdiv(row_bytes, p.box_bytes);
    p.nb = (int)pow2_ceil(p.nbr);
    p.lpr = (p.box_bytes / 16) * p.nb / cpl;
    p.vpl = cpl;
    p.rows_per_tile = p.box_bytes == 64 ? 128 : (p.nb >= 8 ? 8 : 64 / p.nb);
    const int64_t tile = (int64_t)p.nb * p.rows_per_tile * p.box_bytes;
    // fp32 X: 4 warps with up to 4 stages each, so that every warp streams a long run of
    // tiles (measured on 16 M x 32: 312 us against 324 us for 8 warps x 3 stages).
    // bfloat16 X (twice the widening work per byte; 5.1 TB/s with 4 warps against 6.5
    // with 8) and fp64 X (bound by the fp64 units) keep 8 warps to hide latency.
    int warps = elem == 4 ? 4 : 8, S = 0;
    const int64_t max_stages = elem == 4 ? 4 : 8;
    for (;;) {
      S = (int)std::min<int64_t>(max_stages, (budget - 1024) / (warps * (tile + 8)));
      if (S >= 3 || warps <= 2) break;
      warps >>= 1;
    }
    p.stages = std::max(S, 1);
    p.warps = warps;
    p.smem = 1024 + std::max<size_t>((size_t)warps * p.stages * (tile + 8), (size_t)warps * n * sizeof(double));
    const int64_t tiles = cdiv(m, p.rows_per_tile);
    p.ctas = (int)std::max<int64_t>(1, std::min<int64_t>((int64_t)dev.sm_count, cdiv(tiles, p.warps)));
    p.ws_bytes = align128((size_t)p.ctas * n * sizeof(double)) + 128;
    return p;
  }
  int lpr = 0, vpl = 0;
  if (narrow_shape(chunks, &lpr, &vpl)) {
    p.lpr = lpr;
    p.vpl = vpl;
    const int G = 32 / lpr;
    if (tma_ok && elem != 2) {
      // coarsening: the largest power-of-two row count (G..32) whose tile fits the target
      int R = 32;
      while (R > G && R * row_bytes > kTileTarget) R >>= 1;
      const size_t stage = align128((size_t)(R * row_bytes));
      int warps = stage <= 4096 ? 16 : 8;
      int S = 0;
      for (;;) {
        S = (int)std::min<int64_t>(8, budget / (int64_t)(warps * (stage + 8)));
        if (S >= 2 || warps <= 1) break;
        warps >>= 1;
      }
      if (S < 1) S = 1;
      p.kind = DENSE_NARROW_TMA;
      p.rows_per_tile = R;
      p.stages = S;
      p.warps = warps;
      p.smem = std::max<size_t>((size_t)warps * S * (stage + 8), (size_t)warps * n * sizeof(double));
    } else {
      p.kind = DENSE_NARROW_DIRECT;
      p.rows_per_tile = 32;
      p.stages = 1;
      p.warps = 8;
      p.smem = (size_t)p.warps * n * sizeof(double);
    }
    (void)G;
    const int64_t tiles = cdiv(m, p.rows_per_tile);
    const int per_sm = p.kind == DENSE_NARROW_DIRECT ? 4 : 1;
    p.ctas = (int)std::max<int64_t>(1, std::min<int64_t>((int64_t)dev.sm_count * per_sm, cdiv(tiles, p.warps)));
    p.ws_bytes = align128((size_t)p.ctas * n * sizeof(double)) + 128;
    return p;
  }
  // wide rows: 8 rows coarsened per step (fp64 on 20,000 x 20,000: 1,603 us per call against
  // 2,331 at 4 and 2,034 at 2 rows; the dots' independent FMA chains matter more than keeping
  // the re-read rows in L2, since the fp64 units, not HBM, bind)
  p.kind = DENSE_WIDE;
  p.warps = 16;
  p.rows_per_tile = 8;
  set_wide_grid(dev, p, m, n, elem);
  p.smem_acc = (int64_t)(n * sizeof(double)) <= budget;
  p.smem = p.smem_acc ? (size_t)n * sizeof(double) : 0;
  p.ws_bytes = wide_ws_bytes(p, n, elem);
  return p;
}

DensePlan plan_dense(const DeviceInfo& dev, int64_t m, int64_t n, int64_t ld, int elem, bool tma_ok, bool tile_ok) {
  DensePlan p = plan_dense_model(dev, m, n, ld, elem, tma_ok, tile_ok);
  if (p.kind != DENSE_NOOP) p.est_us = p.kind == DENSE_EMPTY_ROWS ? kLaunchUs : dense_est_us(dev, p, m, n, elem);
  return p;
}

std::vector<DensePlan> dense_candidates(const DeviceInfo& dev, const DensePlan& model, int64_t m, int64_t n, int elem) {
  std::vector<DensePlan> c{model};
  const int64_t budget = std::min<int64_t>(kSmemBudget, dev.smem_optin > 0 ? dev.smem_optin : 48 * 1024);
  if (model.kind == DENSE_TILE_TMA) {
    // pipeline depth and warps per CTA
    const int64_t tile = (int64_t)model.nb * model.rows_per_tile * model.box_bytes;
    const int64_t tiles = cdiv(m, model.rows_per_tile);
    for (int warps : {8, 4})
      for (int S : {2, 3, 4, 6}) {
        if (warps == model.warps && S == model.stages) continue;
        const size_t smem =
            1024 + std::max<size_t>((size_t)warps * S * (tile + 8), (size_t)warps * n * sizeof(double));
        if ((int64_t)smem > budget) continue;
        DensePlan q = model;
        q.warps = warps;
        q.stages = S;
        q.smem = smem;
        q.ctas = (int)std::max<int64_t>(1, std::min<int64_t>((int64_t)dev.sm_count, cdiv(tiles, warps)));
        q.ws_bytes = align128((size_t)q.ctas * n * sizeof(double)) + 128;
        q.est_us = dense_est_us(dev, q, m, n, elem);
        c.push_back(q);
      }
  } else if (model.kind == DENSE_WIDE) {
    // fp64: rows per step (fewer keeps more of the re-read in L2, more amortises the dot reduction)
    if (elem == 8)
      for (int r : {2, 4}) {
        DensePlan q = model;
        q.rows_per_tile = r;
        set_wide_grid(dev, q, m, n, elem);
        q.ws_bytes = wide_ws_bytes(q, n, elem);
        q.est_us = dense_est_us(dev, q, m, n, elem);
        c.push_back(q);
      }
    // the column accumulator in global memory instead of shared memory
    if (model.smem_acc) {
      DensePlan q = model;
      q.smem_acc = false;
      q.smem = 0;
      q.ws_bytes = wide_ws_bytes(q, n, elem);
      c.push_back(q);
    }
  }
  return c;
}

CsrStats csr_stats_from_samples(int64_t n, const int64_t* lens, int nl, const int32_t* cols, int nc,
                                int64_t warp_cap) {
  CsrStats st;
  st.valid = true;
  st.row_samples = nl;
  st.col_samples = nc;
  if (nl > 0) {
    std::vector<int64_t> v(lens, lens + nl);
    std::sort(v.begin(), v.end());
    double sum = 0.0, sq = 0.0, lng = 0.0;
    for (int64_t x : v) {
      sum += (double)x;
      sq += (double)x * (double)x;
      if (x > warp_cap) lng += (double)x;
    }
    st.mean_len = sum / nl;
    const double var = std::max(0.0, sq / nl - st.mean_len * st.mean_len);
    st.cv_len = st.mean_len > 0.0 ? std::sqrt(var) / st.mean_len : 0.0;
    auto pct = [&](int q) { return v[std::min<int64_t>(nl - 1, (int64_t)nl * q / 100)]; };
    st.p50_len = pct(50);
    st.p75_len = pct(75);
    st.p90_len = pct(90);
    st.max_len = v.back();
    st.long_share = sum > 0.0 ? lng / sum : 0.0;
  }
  st.bin_width = csr_bin_width(n);
  st.bins = (int)((n + st.bin_width - 1) / st.bin_width);
  st.col_hist.assign((size_t)std::max(st.bins, 1), 0);
  for (int s = 0; s < nc; ++s) {
    const int64_t c = cols[s];
    if (c >= 0 && c < n) ++st.col_hist[(size_t)(c / st.bin_width)];
  }
  return st;
}

CsrStats csr_stats_from_host(int64_t m, int64_t n, int64_t nnz, const int64_t* row_ptr, const int32_t* col_idx) {
  const int nl = (int)std::min<int64_t>(m, kCsrSamples), nc = (int)std::min<int64_t>(nnz, kCsrSamples);
  std::vector<int64_t> lens((size_t)std::max(nl, 1));
  std::vector<int32_t> cols((size_t)std::max(nc, 1));
  for (int s = 0; s < nl; ++s) {
    const int64_t i = csr_sample_index(s, m);
    lens[(size_t)s] = row_ptr[i + 1] - row_ptr[i];
  }
  for (int s = 0; s < nc; ++s) cols[(size_t)s] = col_idx[csr_sample_index(s, nnz)];
  return csr_stats_from_samples(n, lens.data(), nl, cols.data(), nc, csr_warp_long());
}

int64_t csr_place_window(const CsrStats& st, int64_t n, int64_t len, int* hits) {
  int total = 0;
  for (int c : st.col_hist) total += c;
  if (len >= n || st.bins <= 0) {
    if (hits) *hits = len >= n ? total : 0;
    return 0;
  }
  const int64_t kb = std::max<int64_t>(1, len / st.bin_width);
  std::vector<int64_t> pre((size_t)st.bins + 1, 0);
  for (int b = 0; b < st.bins; ++b) pre[(size_t)b + 1] = pre[(size_t)b] + st.col_hist[(size_t)b];
  int64_t best = -1, bs = 0;
  for (int64_t s0 = 0; s0 + kb <= st.bins; ++s0) {
    const int64_t w = pre[(size_t)(s0 + kb)] - pre[(size_t)s0];
    if (w > best) {
      best = w;
      bs = s0;
    }
  }
  if (best < 0) {  // fewer bins than the window spans
    best = pre[(size_t)st.bins];
    bs = 0;
  }
  if (hits) *hits = (int)best;
  return std::min<int64_t>(bs * st.bin_width, n - len);
}

namespace {

// Workspace of a CSR call: the row partition, the long-row queues, the medium-row queue
// (rows longer than a short-row batch or lane group, at most the one-warp limit) and the
// counters.
void csr_set_ws(CsrPlan& p, int64_t m, int64_t nnz) {
  const int64_t batch = p.group_lpr > 0 ? (int64_t)p.group_lpr * p.group_kg : (int64_t)p.pack_cap;
  p.queue_cap = std::min<int64_t>(m, nnz / (p.warp_cap + 1) + 1);
  p.med_cap = std::min<int64_t>(m, nnz / (batch + 1) + 1);
  p.ws_bytes = align128((size_t)(p.ctas + 1) * 8) +
               align128((size_t)csr_long_buckets() * std::max<int64_t>(p.queue_cap, 1) * 8) +
               align128((size_t)std::max<int64_t>(p.med_cap, 1) * 8) + 128;
}

// Fills the window placement of p from the sample (win_len and ylen already set).
void place_sampled(CsrPlan& p, const CsrStats& st, int64_t n) {
  int hw = 0, hy = 0;
  p.win_c0 = csr_place_window(st, n, p.win_len, &hw);
  p.y0 = csr_place_window(st, n, p.ylen, &hy);
  const double ns = (double)std::max(st.col_samples, 1);
  p.win_hit = st.col_samples > 0 ? hw / ns : (p.win_len >= n ? 1.0 : 0.0);
  p.y_hit = st.col_samples > 0 ? hy / ns : (p.ylen >= n ? 1.0 : 0.0);
}

}  // namespace

CsrPlan plan_csr(const DeviceInfo& dev, int64_t m, int64_t n, int64_t nnz, int elem, const CsrStats* st) {
  CsrPlan p;
  const bool sampled = st != nullptr && st->valid;
  // fp64 short rows go to lane groups sized to the rows (16 entries per lane); fp32 to packed batches
  if (elem == 8) {
    // the row length the groups are sized for: the sampled 75th percentile, which keeps a few
    // long rows from widening every group; else the mean
    const double avg = sampled && st->row_samples > 0 ? (double)st->p75_len
                                                      : (m > 0 ? (double)nnz / (double)m : 0.0);
    // 16 entries a lane and just enough lanes to cover the mean row (rows of Poisson(50)
    // entries: 4 x 16; measured 1,441 us against 1,636 for 8 x 8, one shuffle level fewer
    // per row and two rows more per warp); rows averaging 16 entries or fewer: 2 x 8
    if (avg <= 16.0) {
      p.group_lpr = 2;
      p.group_kg = 8;
    } else {
      p.group_kg = 16;
      p.group_lpr = (int)std::min<int64_t>(16, std::max<int64_t>(2, pow2_ceil((int64_t)(avg / 16.0 + 0.999))));
    }
  }
  p.pack_cap = csr_pack_cap(elem);
  p.pack_k = p.pack_cap / 32;
  p.warp_cap = csr_warp_long();
  // one CTA per SM, so that each SM's column window is as wide as possible: 1024
  // threads, or 768 for the fp64 lane groups (80 registers a thread keep their 16-entry
  // buffers from spilling; 1,399 against 1,441 us on rows of Poisson(50) entries)
  p.threads = p.group_lpr > 0 ? csr_group_threads() : kCsrThreads;
  p.long_threads = kCsrThreads;
  p.long_group = csr_long_group_default();
  const int64_t budget = std::min<int64_t>(kSmemBudget, dev.smem_optin > 0 ? dev.smem_optin : 48 * 1024);
  const int64_t fixed = (int64_t)csr_rows_smem(0, 0, elem) + 32;  // per-warp scratch of the row kernel + padding
  p.ctas = (int)std::max<int64_t>(1, std::min<int64_t>((int64_t)dev.sm_count, cdiv(std::max<int64_t>(m, 1), 1024)));
  p.long_ctas = dev.sm_count;
  // shared memory: the accumulator window takes three quarters (the unsampled default), a
  // copy of y the rest; with a column sample, the split of ½, ¾ or ⅞ whose placed windows
  // leave the fewest estimated misses, weighting a scatter miss (a global reduction, ~1.7 ns
  // on the power-law workload) kScatterMissWeight times a gather miss (~1.5 ns), and leaving
  // ¾ only for a gain of at least kSplitGain of the sampled entries (sampling noise)
  const int64_t room = std::max<int64_t>(0, budget - fixed) / elem;
  p.row_cost = 8;
  csr_set_ws(p, m, nnz);
  auto set_split = [&](CsrPlan& q, int eighths) {
    q.win_len = std::min<int64_t>(n, room * eighths / 8);
    q.ylen = std::min<int64_t>(n, room - q.win_len);
    q.smem = csr_rows_smem(q.win_len, q.ylen, elem);
    q.long_smem = q.smem - (size_t)csr_rows_smem(0, 0, elem);
  };
  set_split(p, 6);
  if (sampled) {
    p.sampled = true;
    p.mean_len = st->mean_len;
    p.cv_len = st->cv_len;
    p.long_share = st->long_share;
    p.p75_len = st->p75_len;
    place_sampled(p, *st, n);
    double best = kScatterMissWeight * (1.0 - p.win_hit) + (1.0 - p.y_hit) - kSplitGain;
    for (int eighths : {4, 7}) {
      CsrPlan q = p;
      set_split(q, eighths);
      place_sampled(q, *st, n);
      const double cost = kScatterMissWeight * (1.0 - q.win_hit) + (1.0 - q.y_hit);
      if (cost < best) {
        best = cost;
        p = q;
      }
    }
  } else {
    p.win_c0 = 0;
    p.y0 = 0;
    p.place_on_device = p.win_len < n || p.ylen < n;
  }
  p.est_us = csr_est_us(dev, p, m, n, nnz, elem);
  return p;
}

std::vector<CsrPlan> csr_candidates(const DeviceInfo& dev, const CsrPlan& model, int64_t m, int64_t n, int64_t nnz,
                                    int elem, const CsrStats* st) {
  std::vector<CsrPlan> c{model};
  const int64_t budget = std::min<int64_t>(kSmemBudget, dev.smem_optin > 0 ? dev.smem_optin : 48 * 1024);
  const int64_t fixed = (int64_t)csr_rows_smem(0, 0, elem) + 32;
  const int64_t room = std::max<int64_t>(0, budget - fixed) / elem;
  // the split of shared memory between the scatter window and the copy of y
  if (n > room / 2) {
    for (int eighths : {4, 6, 7}) {
      CsrPlan q = model;
      q.win_len = std::min<int64_t>(n, room * eighths / 8);
      q.ylen = std::min<int64_t>(n, room - q.win_len);
      if (q.win_len == model.win_len) continue;
      q.smem = csr_rows_smem(q.win_len, q.ylen, elem);
      q.long_smem = q.smem - csr_rows_smem(0, 0, elem);
      if (st != nullptr && st->valid) place_sampled(q, *st, n);
      q.est_us = csr_est_us(dev, q, m, n, nnz, elem);
      c.push_back(q);
    }
  }
  // threads sharing one long row (only when the matrix can have rows past the one-warp limit)
  if (nnz > model.warp_cap)
    for (int g : {256, 512}) {
      CsrPlan q = model;
      q.long_group = g;
      c.push_back(q);
    }
  // fp64 lane groups: the same capacity with 8 entries a lane, and one size wider
  if (model.group_lpr > 0) {
    const int cap = model.group_lpr * model.group_kg;
    for (int kg : {8, 16}) {
      for (int lpr : {cap / kg, 2 * cap / kg}) {
        if (lpr < 2 || lpr > 16 || (lpr == model.group_lpr && kg == model.group_kg)) continue;
        if (kg == 16 && lpr == cap / kg) continue;
        CsrPlan q = model;
        q.group_lpr = lpr;
        q.group_kg = kg;
        csr_set_ws(q, m, nnz);
        c.push_back(q);
      }
    }
  }
  return c;
}

int describe(const DensePlan& p, char* buf, size_t cap) {
  static const char* names[] = {"noop", "empty_rows", "narrow_tma", "narrow_direct", "wide", "tile_tma"};
  return snprintf(buf, cap,
                  "dense kind=%s lanes_per_row=%d chunks_per_lane=%d rows_per_tile=%d stages=%d warps=%d ctas=%d "
                  "smem=%zu smem_acc=%d blocks=%d box=%d ws=%zu est_us=%.1f",
                  names[p.kind], p.lpr, p.vpl, p.rows_per_tile, p.stages, p.warps, p.ctas, p.smem, (int)p.smem_acc,
                  p.nbr, p.box_bytes, p.ws_bytes, p.est_us);
}

int describe(const CsrPlan& p, char* buf, size_t cap) {
  int w = snprintf(buf, cap,
                   "csr group_lanes=%d group_entries=%d pack_k=%d pack_cap=%d warp_cap=%d ctas=%d threads=%d "
                   "long_ctas=%d long_group=%d window=[%lld,+%lld) y_window=[%lld,+%lld) placement=%s smem=%zu "
                   "queue_cap=%lld ws=%zu est_us=%.1f",
                   p.group_lpr, p.group_kg, p.pack_k, p.pack_cap, p.warp_cap, p.ctas, p.threads, p.long_ctas,
                   p.long_group,
                   (long long)p.win_c0, (long long)p.win_len, (long long)p.y0, (long long)p.ylen,
                   p.sampled ? "sampled" : (p.place_on_device ? "device" : "whole"), p.smem, (long long)p.queue_cap,
                   p.ws_bytes, p.est_us);
  if (p.sampled && w > 0 && (size_t)w < cap)
    w += snprintf(buf + w, cap - (size_t)w,
                  " mean_len=%.1f cv_len=%.2f p75_len=%lld long_share=%.3f win_hit=%.3f y_hit=%.3f", p.mean_len,
                  p.cv_len, (long long)p.p75_len, p.long_share, p.win_hit, p.y_hit);
  return w;
}

}  // namespace fxtx
