/*
 * inputgen.c — seeded synthetic inputs for the fused pattern
 *     out = alpha * X^T (v .* (X y)) + beta * z.
 *
 * This module only draws numbers and sparsity structures. It holds none of the
 * pattern's arithmetic: both the CPU oracle and the CUDA library are fed from
 * the arrays it fills, so that the two see identical bits.
 *
 * Generator: a counter-based stream built from the SplitMix64 output function
 * (Steele, Lea and Flood, "Fast splittable pseudorandom number generators",
 * OOPSLA 2014). Draw k of stream `key` is mix64(key + (k + 1) * GAMMA). Every
 * array (structure, X, y, v, z) has its own key derived from (seed, stream id),
 * and every CSR row has its own sub-key, so results do not depend on the thread
 * count that OpenMP happens to use.
 *
 *  - U[a,b]   : a + (b - a) * u with u = (r >> 11) * 2^-53 in [0, 1).
 *  - N(0,1)   : Box-Muller, z = sqrt(-2 ln u1) cos(2 pi u2), u1 in (0, 1],
 *               one normal per element (draws 2k and 2k+1).
 *  - f32      : the f64 draw rounded to nearest float.
 *  - Poisson  : inversion by sequential search (Knuth, TAOCP vol. 2, 3.4.1).
 *  - Zipf     : Walker's alias method (Vose's construction) on weights r^-s.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define GAMMA 0x9E3779B97F4A7C15ULL

static inline uint64_t mix64(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

static inline uint64_t draw(uint64_t key, uint64_t k) { return mix64(key + (k + 1) * GAMMA); }

uint64_t ig_stream_key(uint64_t seed, uint64_t stream) {
  return mix64(mix64(seed * GAMMA + 0x632BE59BD9B4E019ULL) ^ (stream + 1) * 0xD1B54A32D192ED03ULL);
}

static inline uint64_t row_key(uint64_t key, int64_t row) { return mix64(key ^ ((uint64_t)row + 1) * GAMMA); }

static inline double u01(uint64_t r) { return (double)(r >> 11) * 0x1.0p-53; }       /* [0,1) */
static inline double u01_open0(uint64_t r) { return ((double)(r >> 11) + 1.0) * 0x1.0p-53; } /* (0,1] */

static inline double normal_at(uint64_t key, int64_t k) {
  const double two_pi = 6.283185307179586476925286766559;
  double u1 = u01_open0(draw(key, 2 * (uint64_t)k));
  double u2 = u01(draw(key, 2 * (uint64_t)k + 1));
  return sqrt(-2.0 * log(u1)) * cos(two_pi * u2);
}

void ig_fill_uniform_f64(uint64_t seed, uint64_t stream, int64_t count, double a, double b, double* out) {
  uint64_t key = ig_stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < count; ++k) out[k] = a + (b - a) * u01(draw(key, (uint64_t)k));
}

void ig_fill_uniform_f32(uint64_t seed, uint64_t stream, int64_t count, double a, double b, float* out) {
  uint64_t key = ig_stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < count; ++k) out[k] = (float)(a + (b - a) * u01(draw(key, (uint64_t)k)));
}

void ig_fill_normal_f64(uint64_t seed, uint64_t stream, int64_t count, double* out) {
  uint64_t key = ig_stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < count; ++k) out[k] = normal_at(key, k);
}

void ig_fill_normal_f32(uint64_t seed, uint64_t stream, int64_t count, float* out) {
  uint64_t key = ig_stream_key(seed, stream);
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < count; ++k) out[k] = (float)normal_at(key, k);
}

/* Integers uniform in [lo, hi] (inclusive), for exact-arithmetic test inputs. */
void ig_fill_int_f64(uint64_t seed, uint64_t stream, int64_t count, int64_t lo, int64_t hi, double* out) {
  uint64_t key = ig_stream_key(seed, stream);
  uint64_t span = (uint64_t)(hi - lo + 1);
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < count; ++k) out[k] = (double)(lo + (int64_t)((draw(key, (uint64_t)k) >> 32) * span >> 32));
}

void ig_fill_int_f32(uint64_t seed, uint64_t stream, int64_t count, int64_t lo, int64_t hi, float* out) {
  uint64_t key = ig_stream_key(seed, stream);
  uint64_t span = (uint64_t)(hi - lo + 1);
#pragma omp parallel for schedule(static)
  for (int64_t k = 0; k < count; ++k) out[k] = (float)(lo + (int64_t)((draw(key, (uint64_t)k) >> 32) * span >> 32));
}

/* Row lengths ~ Poisson(lambda), clamped to [0, cap]. */
void ig_poisson_lengths(uint64_t seed, uint64_t stream, int64_t m, double lambda, int64_t cap, int64_t* len) {
  uint64_t key = ig_stream_key(seed, stream);
  double p0 = exp(-lambda);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < m; ++i) {
    double u = u01(draw(key, (uint64_t)i));
    int64_t k = 0;
    double p = p0, F = p0;
    while (u > F && k < cap) {
      ++k;
      p *= lambda / (double)k;
      F += p;
      if (p == 0.0 && F < u) break; /* far tail: numerically exhausted */
    }
    len[i] = k < cap ? k : cap;
  }
}

/* ---- Walker alias table over ranks 1..K with weights r^-s (Vose's construction) ---- */
typedef struct { int64_t K; double* prob; int32_t* alias; } alias_t;

static int alias_build(alias_t* a, int64_t K, double s) {
  a->K = K;
  a->prob = (double*)malloc((size_t)K * sizeof(double));
  a->alias = (int32_t*)malloc((size_t)K * sizeof(int32_t));
  double* w = (double*)malloc((size_t)K * sizeof(double));
  int32_t* small = (int32_t*)malloc((size_t)K * sizeof(int32_t));
  int32_t* large = (int32_t*)malloc((size_t)K * sizeof(int32_t));
  if (!a->prob || !a->alias || !w || !small || !large) {
    free(a->prob); free(a->alias); free(w); free(small); free(large);
    a->prob = NULL; a->alias = NULL;
    return -1;
  }
  double total = 0.0;
  for (int64_t r = 0; r < K; ++r) { w[r] = pow((double)(r + 1), -s); total += w[r]; }
  int64_t ns = 0, nl = 0;
  for (int64_t r = 0; r < K; ++r) {
    w[r] = w[r] * (double)K / total;
    if (w[r] < 1.0) small[ns++] = (int32_t)r; else large[nl++] = (int32_t)r;
  }
  while (ns > 0 && nl > 0) {
    int32_t sm = small[--ns], lg = large[nl - 1];
    a->prob[sm] = w[sm];
    a->alias[sm] = lg;
    w[lg] = (w[lg] + w[sm]) - 1.0;
    if (w[lg] < 1.0) { --nl; small[ns++] = lg; }
  }
  while (nl > 0) { int32_t r = large[--nl]; a->prob[r] = 1.0; a->alias[r] = r; }
  while (ns > 0) { int32_t r = small[--ns]; a->prob[r] = 1.0; a->alias[r] = r; }
  free(w); free(small); free(large);
  return 0;
}

static void alias_free(alias_t* a) { free(a->prob); free(a->alias); }

/* 0-based rank drawn from the alias table with one 64-bit draw. */
static inline int64_t alias_draw(const alias_t* a, uint64_t r) {
  int64_t idx = (int64_t)(((r >> 32) * (uint64_t)a->K) >> 32);
  double coin = (double)(r & 0xFFFFFFFFULL) * 0x1.0p-32;
  return coin < a->prob[idx] ? idx : a->alias[idx];
}

/*
 * Row lengths with a power-law tail: K_i ~ Zipf(s) on {1..kmax}, then
 * L_i = clamp(floor(c * K_i + 0.5), 1, cap) with c chosen by bisection so that
 * sum L_i is as close as possible to target_nnz. Returns the chosen c.
 */
double ig_zipf_lengths(uint64_t seed, uint64_t stream, int64_t m, double s, int64_t kmax,
                       int64_t target_nnz, int64_t cap, int64_t* len) {
  alias_t a;
  if (alias_build(&a, kmax, s) != 0) return -1.0;
  uint64_t key = ig_stream_key(seed, stream);
  int64_t* K = (int64_t*)malloc((size_t)(m > 0 ? m : 1) * sizeof(int64_t));
  if (!K) { alias_free(&a); return -1.0; }
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < m; ++i) K[i] = alias_draw(&a, draw(key, (uint64_t)i)) + 1;
  alias_free(&a);
  double lo = 0.0, hi = 1.0;
  for (;;) { /* grow hi until the sum exceeds the target */
    int64_t sum = 0;
#pragma omp parallel for reduction(+ : sum) schedule(static)
    for (int64_t i = 0; i < m; ++i) {
      int64_t L = (int64_t)floor(hi * (double)K[i] + 0.5);
      sum += L < 1 ? 1 : (L > cap ? cap : L);
    }
    if (sum >= target_nnz || hi > 1e12) break;
    lo = hi;
    hi *= 2.0;
  }
  for (int it = 0; it < 100; ++it) {
    double mid = 0.5 * (lo + hi);
    int64_t sum = 0;
#pragma omp parallel for reduction(+ : sum) schedule(static)
    for (int64_t i = 0; i < m; ++i) {
      int64_t L = (int64_t)floor(mid * (double)K[i] + 0.5);
      sum += L < 1 ? 1 : (L > cap ? cap : L);
    }
    if (sum < target_nnz) lo = mid; else hi = mid;
  }
  /* pick whichever end of the final bracket lands closer to the target */
  int64_t slo = 0, shi = 0;
  for (int64_t i = 0; i < m; ++i) {
    int64_t L1 = (int64_t)floor(lo * (double)K[i] + 0.5), L2 = (int64_t)floor(hi * (double)K[i] + 0.5);
    slo += L1 < 1 ? 1 : (L1 > cap ? cap : L1);
    shi += L2 < 1 ? 1 : (L2 > cap ? cap : L2);
  }
  double c = (llabs(target_nnz - slo) <= llabs(shi - target_nnz)) ? lo : hi;
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < m; ++i) {
    int64_t L = (int64_t)floor(c * (double)K[i] + 0.5);
    len[i] = L < 1 ? 1 : (L > cap ? cap : L);
  }
  free(K);
  return c;
}

static int cmp_i32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x > y) - (x < y);
}

static void sort_row(int32_t* c, int64_t L) {
  if (L < 32) { /* insertion sort for short rows */
    for (int64_t i = 1; i < L; ++i) {
      int32_t x = c[i];
      int64_t j = i - 1;
      while (j >= 0 && c[j] > x) { c[j + 1] = c[j]; --j; }
      c[j + 1] = x;
    }
  } else {
    qsort(c, (size_t)L, sizeof(int32_t), cmp_i32);
  }
}

/*
 * Column indices for every row of a CSR structure whose row_ptr is given:
 * distinct columns per row, drawn uniformly (zipf_s <= 0) or from Zipf(zipf_s)
 * over ranks 1..n with column = rank - 1, repeats rejected, then sorted.
 * Returns 0, or -1 when a row asks for more distinct columns than exist or
 * memory runs out.
 */
int ig_fill_csr_cols(uint64_t seed, uint64_t stream, int64_t m, int64_t n, double zipf_s,
                     const int64_t* row_ptr, int32_t* col_idx) {
  if (n <= 0) return m > 0 && row_ptr[m] > 0 ? -1 : 0;
  for (int64_t i = 0; i < m; ++i)
    if (row_ptr[i + 1] - row_ptr[i] > n) return -1;
  alias_t a = {0, NULL, NULL};
  if (zipf_s > 0.0 && alias_build(&a, n, zipf_s) != 0) return -1;
  uint64_t key = ig_stream_key(seed, stream);
  int failed = 0;
#pragma omp parallel
  {
    int32_t* mark = (int32_t*)malloc((size_t)n * sizeof(int32_t));
    if (!mark) {
#pragma omp atomic write
      failed = 1;
    } else {
      for (int64_t j = 0; j < n; ++j) mark[j] = -1;
#pragma omp for schedule(dynamic, 256)
      for (int64_t i = 0; i < m; ++i) {
        uint64_t rk = row_key(key, i);
        int64_t L = row_ptr[i + 1] - row_ptr[i];
        int32_t* c = col_idx + row_ptr[i];
        int32_t stamp = (int32_t)(i & 0x7FFFFFFF);
        uint64_t k = 0;
        for (int64_t got = 0; got < L;) {
          uint64_t r = draw(rk, k++);
          int64_t col = zipf_s > 0.0 ? alias_draw(&a, r) : (int64_t)(((r >> 32) * (uint64_t)n) >> 32);
          if (mark[col] == stamp) continue;
          mark[col] = stamp;
          c[got++] = (int32_t)col;
        }
        /* a later row with the same stamp (i + 2^31) cannot exist: m < 2^31 */
        sort_row(c, L);
      }
      free(mark);
    }
  }
  if (zipf_s > 0.0) alias_free(&a);
  return failed ? -1 : 0;
}
