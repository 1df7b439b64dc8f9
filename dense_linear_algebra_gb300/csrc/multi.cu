// multi.cu — the multi-vector instantiation OUT = alpha * X^T (V ⊙ (X Y)) + beta * Z
// (declared in multi.h): one pass over X serves kb right-hand sides at once.
//
// "On optimizing machine learning workloads via kernel fusion" (abstract): the fused
// pattern and its instantiations. Each right-hand side c is the single-vector pattern
// with y = Y[:, c], v = V[:, c] and z = Z[:, c]; reading X once for all of them raises
// the arithmetic intensity kb-fold, so small kb stays on the HBM roof and large kb
// moves to the FMA roof.
//
// Tiles of R rows of X arrive in shared memory by 2-D tensor copies (one R x 128-byte
// box per column block, a 2- to 4-deep pipeline per warp), with the tile's weights
// beside them. The warp's lanes split three ways: lane = cg + KB * (jg + NB * rs).
// Lane (rs, jg, cg) keeps in registers the eight 16-byte chunks jg, jg + NB, ... of
// Y's rows for right-hand side cg, and per row it reads the same eight chunks of X. The NB lanes of a row sum their
// partial dots with shuffles; each lane then has t = v * (x . y_cg) and adds t * x into
// its own column sums. No dot needs another right-hand side's data, so no lane holds
// more than one right-hand side.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "multi.h"
#include "tmap.h"

namespace fxtx {
namespace {

constexpr int MULTI_THREADS = 256;
constexpr size_t MULTI_SMEM_BUDGET = 220 * 1024;

template <typename T>
struct Chunk;
template <>
struct Chunk<float> {
  static constexpr CUtensorMapDataType MAP = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  __device__ static __forceinline__ void unpack(const uint4& u, float* e) {
    e[0] = __uint_as_float(u.x); e[1] = __uint_as_float(u.y); e[2] = __uint_as_float(u.z); e[3] = __uint_as_float(u.w);
  }
};
template <>
struct Chunk<double> {
  static constexpr CUtensorMapDataType MAP = CU_TENSOR_MAP_DATA_TYPE_FLOAT64;
  __device__ static __forceinline__ void unpack(const uint4& u, double* e) {
    e[0] = __hiloint2double((int)u.y, (int)u.x);
    e[1] = __hiloint2double((int)u.w, (int)u.z);
  }
};

// Rows per tile for rows of nb 128-byte blocks and kb right-hand sides of `elem` bytes:
// 8-KB tiles of X (16 KB at nb = 16), which give each lane several independent rows per
// tile; 4-KB tiles for one right-hand side (an HBM-bound pass) and where a tile's weights
// would outgrow half its X (more than 64 bytes of weights a row).
__host__ __device__ constexpr int multi_rows(int nb, int kb, int elem) {
  return nb >= 8 ? 8 : ((kb == 1 || kb * elem > 64) ? 32 : 64) / nb;
}

// Geometry for rows of NB 128-byte blocks and KB right-hand sides per pass.
template <typename T, int NB, int KB>
struct MShape {
  static constexpr int NV = 16 / (int)sizeof(T);  // elements per chunk
  static constexpr int Q = 8;                     // chunks per lane
  static constexpr int C = Q * NV;                // columns per lane
  static constexpr int RS = 32 / (NB * KB);       // row slots of a warp
  static constexpr int R = multi_rows(NB, KB, (int)sizeof(T));  // rows per tile
  static constexpr int IT = R / RS;               // rows per lane per tile
  static constexpr int BOX = R * 128;             // bytes of one 128-byte column block of a tile
  static constexpr int TILE = NB * BOX;           // bytes of X in one pipeline stage
  static constexpr int UNROLL = IT < 8 ? IT : 8;  // rows per lane between pointer updates
  static_assert(NB * KB <= 32 && RS >= 1 && R % RS == 0 && IT % UNROLL == 0, "lane split");
};

// Byte offset of chunk ch of tile row r: one R x 128-byte box per 128-byte column
// block, rows unswizzled.
template <int BOX>
__host__ __device__ __forceinline__ int chunk_offset(int r, int ch) {
  return (ch >> 3) * BOX + r * 128 + ((ch & 7) << 4);
}

// The chunk lane (rs, jg) reads at step q. The rotation by rs spreads the RS rows a
// warp reads at once over distinct 16-byte bank groups (rows are 128 bytes apart, so
// without it they would all hit the same group), and keeps every lane's offsets
// fixed from row to row.
template <int NB>
__host__ __device__ __forceinline__ int lane_chunk(int rs, int jg, int q) {
  const int rot = NB < 8 ? (rs & (8 / NB - 1)) : 0;
  return jg + ((q + rot) & 7) * NB;
}

// Element-sized asynchronous copy global -> shared (no alignment beyond the element's).
template <typename T>
__device__ __forceinline__ void cp_async_elem(T* dst, const T* src) {
  if constexpr (sizeof(T) == 4)
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
  else
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
// An arrive on `bar` once every asynchronous copy this thread issued so far has landed
// (counted in the barrier's expected arrivals).
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}
// Waits until every asynchronous copy this thread issued has landed (committed or not).
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Sums a value over the NB lanes of a row (lanes KB apart).
template <typename T, int NB, int KB>
__device__ __forceinline__ T row_sum(T s) {
#pragma unroll
  for (int o = KB; o < KB * NB; o <<= 1) s += __shfl_xor_sync(FULL_MASK, s, o);
  return s;
}

// Sums a compensated (s, c) pair over the NB lanes of a row.
template <int NB, int KB>
__device__ __forceinline__ float row_sum_comp(float s, float c) {
#pragma unroll
  for (int o = KB; o < KB * NB; o <<= 1) {
    const float s2 = __shfl_xor_sync(FULL_MASK, s, o), c2 = __shfl_xor_sync(FULL_MASK, c, o);
    float t, q;
    two_sum(s, s2, t, q);
    s = t;
    c = __fadd_rn(__fadd_rn(c, c2), q);
  }
  return __fadd_rn(s, c);
}

// A lane's per-tile column sums tacc[c] += t * x[c]. fp32 keeps them as packed pairs and
// updates two columns per instruction (fma.rn.f32x2); each element still rounds once.
template <typename T, int C>
struct ColSums {
  T v[C];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int c = 0; c < C; ++c) v[c] = T(0);
  }
  __device__ __forceinline__ void add(T t, const T* x) {
#pragma unroll
    for (int c = 0; c < C; ++c) v[c] = fma(t, x[c], v[c]);
  }
  __device__ __forceinline__ T get(int c) const { return v[c]; }
};
template <int C>
struct ColSums<float, C> {
  float2 v[C / 2];
  __device__ __forceinline__ void zero() {
#pragma unroll
    for (int c = 0; c < C / 2; ++c) v[c] = make_float2(0.f, 0.f);
  }
  __device__ __forceinline__ void add(float t, const float* x) {
    const float2 t2 = make_float2(t, t);
#pragma unroll
    for (int c = 0; c < C / 2; ++c) v[c] = __ffma2_rn(t2, make_float2(x[2 * c], x[2 * c + 1]), v[c]);
  }
  __device__ __forceinline__ float get(int c) const { return (c & 1) ? v[c >> 1].y : v[c >> 1].x; }
};

// A lane's partial dot x . y over its C columns in working precision: four independent
// chains (fp32: two chains of packed pairs).
template <typename T, int C>
__device__ __forceinline__ T lane_dot(const T* x, const T* y) {
  if constexpr (sizeof(T) == 4) {
    float2 d[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
    for (int c = 0; c < C / 2; ++c)
      d[c & 1] = __ffma2_rn(make_float2(x[2 * c], x[2 * c + 1]), make_float2(y[2 * c], y[2 * c + 1]), d[c & 1]);
    return (d[0].x + d[0].y) + (d[1].x + d[1].y);
  } else {
    T d4[4] = {T(0), T(0), T(0), T(0)};
#pragma unroll
    for (int c = 0; c < C; ++c) d4[c & 3] = fma(x[c], y[c], d4[c & 3]);
    return (d4[0] + d4[1]) + (d4[2] + d4[3]);
  }
}

// CTA partials -> workspace; the last CTA to arrive sums them in a fixed order and
// writes OUT = alpha * W + beta * Z for the pass's kb right-hand sides.
template <typename T, int KB>
__device__ __forceinline__ void multi_finish(const MultiArgs<T>& a, double* red, const int nred, const int nw) {
  __shared__ unsigned s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t N = a.n * KB;
  __syncthreads();
  for (int64_t e = threadIdx.x; e < N; e += blockDim.x) {
    double s = 0.0;
    for (int w = 0; w < nred; ++w) s += red[w * N + e];
    a.ws[blockIdx.x * N + e] = s;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(a.ticket, 1u) == gridDim.x - 1) ? 1u : 0u;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int nc = gridDim.x;
  const int cb = nc * warp / nw, ce = nc * (warp + 1) / nw;
  for (int64_t e = lane; e < N; e += 32) {
    double s = 0.0;
    for (int c = cb; c < ce; ++c) s += __ldcg(a.ws + (int64_t)c * N + e);
    red[warp * N + e] = s;
  }
  __syncthreads();
  for (int64_t e = threadIdx.x; e < N; e += blockDim.x) {
    const int64_t col = e / KB;
    const int c = (int)(e % KB);
    if (c >= a.kb) continue;
    double s = 0.0;
    for (int w = 0; w < nw; ++w) s += red[w * N + e];
    double o = a.alpha * s;
    if (a.use_z) o += a.beta * (double)a.Z[col * a.ldz + c];
    a.OUT[col * a.ldo + c] = (T)o;
  }
  if (threadIdx.x == 0) *a.ticket = 0u;
}

// vmode: 0 no weights, 1 one shared m-vector, 2 an (m x k) matrix. v16: the weights
// of a tile arrive in 16-byte copies (vmode 2, a full pass, V and ldv 16-byte aligned).
template <typename T, int NB, int KB>
__global__ void __launch_bounds__(MULTI_THREADS, 1)
    dense_multi_kernel(const __grid_constant__ CUtensorMap tmap, const MultiArgs<T> a, const int S, const int tma,
                       const int vmode, const int v16) {
  using SH = MShape<T, NB, KB>;
  constexpr int NV = SH::NV, Q = SH::Q, C = SH::C, RS = SH::RS, R = SH::R, IT = SH::IT, UNROLL = SH::UNROLL;
  constexpr int BOX = SH::BOX, TILE = SH::TILE;
  // fp32 rows longer than 64 entries (NB >= 4) take the compensated dot
  constexpr bool COMP = sizeof(T) == 4 && NB >= 4;
  // fp32: plain per-lane column sums over about 32 rows, then folded into a two-float sum
  constexpr int FOLD = IT >= 32 ? 1 : 32 / IT;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int cg = lane % KB, jg = (lane / KB) % NB, rs = lane / (KB * NB);
  const int64_t n = a.n, m = a.m;
  const int VB = vmode == 2 ? R * KB : (vmode == 1 ? R : 0);                  // weights per tile
  const int STAGE = TILE + ((VB * (int)sizeof(T) + 127) & ~127);             // X tile + weights
  unsigned char* stages = smem + (size_t)warp * S * STAGE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)nw * S * STAGE) + warp * S;

  // this lane's eight chunks (rotated order) and its slice of Y for right-hand side cg
  int off[Q];
  T yr[C];
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    const int ch = lane_chunk<NB>(rs, jg, q);
    off[q] = chunk_offset<BOX>(rs, ch);
#pragma unroll
    for (int e = 0; e < NV; ++e) {
      const int64_t col = (int64_t)ch * NV + e;
      yr[q * NV + e] = (col < n && cg < a.kb) ? ldg(a.Y + col * a.ldy + cg) : T(0);
    }
  }

  const int64_t gw = (int64_t)blockIdx.x * nw + warp, W = (int64_t)gridDim.x * nw;
  const int64_t t0 = a.tiles * gw / W, t1 = a.tiles * (gw + 1) / W, nt = t1 - t0;
  const uint64_t pol = policy_evict_first();

  // weights of one tile into vb (asynchronous copies; zeros past the last row)
  auto stage_v = [&](int64_t tile, T* vb) {
    if constexpr (KB * sizeof(T) >= 16) {
      if (v16) {
        constexpr int CPV = KB * (int)sizeof(T) / 16;  // 16-byte chunks per row of weights
        for (int e = lane; e < R * CPV; e += 32) {
          const int r = e / CPV, j = e % CPV;
          const int64_t row = tile * R + r;
          T* dst = vb + r * KB + j * NV;
          if (row < m)
            cp_async16(dst, a.V + row * a.ldv + j * NV);
          else
            *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
        return;
      }
    }
    for (int e = lane; e < VB; e += 32) {
      const int r = vmode == 2 ? e / KB : e, c = vmode == 2 ? e % KB : 0;
      const int64_t row = tile * R + r;
      if (row < m && c < a.kb)
        cp_async_elem(vb + e, a.V + (vmode == 2 ? row * a.ldv + c : row));
      else
        vb[e] = T(0);
    }
  };
  auto issue = [&](int64_t tile, int s) {
    unsigned char* st = stages + (size_t)s * STAGE;
    if (vmode) {
      stage_v(tile, reinterpret_cast<T*>(st + TILE));
      cp_async_arrive(&bars[s]);
    }
    if (lane == 0) mbar_arrive_expect_tx(&bars[s], (uint32_t)TILE);
    __syncwarp();
    if (lane < NB) tma_load_2d(st + lane * BOX, &tmap, lane * (128 / (int)sizeof(T)), (int)(tile * R), &bars[s], pol);
  };
  // X of one tile by plain loads, in the layout the tensor copy would give
  auto load_direct = [&](int64_t tile, unsigned char* stage) {
    constexpr int CPR = NB * 8;
    for (int idx = lane; idx < R * CPR; idx += 32) {
      const int r = idx / CPR, ch = idx % CPR;
      const int64_t row = tile * R + r;
      alignas(16) T e[NV];
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int64_t col = (int64_t)ch * NV + i;
        e[i] = (row < m && col < n) ? ldg(a.X + row * a.ld + col) : T(0);
      }
      *reinterpret_cast<uint4*>(stage + chunk_offset<BOX>(r, ch)) = *reinterpret_cast<const uint4*>(e);
    }
  };

  if (tma) {
    if (lane == 0) {
      // one arrival with the byte count, plus one per lane for its weight copies
      for (int s = 0; s < S; ++s) mbar_init(&bars[s], vmode ? 33u : 1u);
      fence_mbar_init();
    }
    __syncwarp();
    for (int s = 0; s < S && s < nt; ++s) issue(t0 + s, s);
  }

  typename OuterAcc<T>::type acc[C];
  ColSums<T, C> tacc;
  tacc.zero();

  for (int64_t k = 0; k < nt; ++k) {
    const int64_t tile = t0 + k;
    const int s = tma ? (int)(k % S) : 0;
    unsigned char* stage = stages + (size_t)s * STAGE;
    if (tma) {
      const bool ok = mbar_wait_bounded(&bars[s], (uint32_t)((k / S) & 1));
      if (__any_sync(FULL_MASK, !ok)) {
        if (lane == 0)
          for (int64_t j = k + 1; j < nt && j < k + S; ++j) mbar_wait_bounded(&bars[j % S], (uint32_t)((j / S) & 1));
        break;
      }
    } else {
      load_direct(tile, stage);
      if (vmode) {
        stage_v(tile, reinterpret_cast<T*>(stage + TILE));
        cp_async_wait_all();
      }
    }
    __syncwarp();  // zero fills and (direct path) plain stores are visible to the warp
    const T* vb = reinterpret_cast<const T*>(stage + TILE);

#pragma unroll 1
    for (int i0 = 0; i0 < IT; i0 += UNROLL) {
#pragma unroll
      for (int u = 0; u < UNROLL; ++u) {
        const int r = (i0 + u) * RS + rs;
        const unsigned char* rp = stage + (i0 + u) * RS * 128;
        T x[C];
#pragma unroll
        for (int q = 0; q < Q; ++q) {
          const uint4 w = *reinterpret_cast<const uint4*>(rp + off[q]);
          Chunk<T>::unpack(w, &x[q * NV]);
        }
        T d;
        if constexpr (COMP) {
          DotAcc<float, true> dacc;
#pragma unroll
          for (int c = 0; c < C; ++c) dacc.add(x[c], yr[c]);
          d = row_sum_comp<NB, KB>(dacc.s, dacc.c);
        } else {
          d = row_sum<T, NB, KB>(lane_dot<T, C>(x, yr));
        }
        const T t = vmode == 0 ? d : vb[vmode == 2 ? r * KB + cg : r] * d;
        tacc.add(t, x);
      }
    }
    if (sizeof(T) == 8 || (k + 1) % FOLD == 0 || k + 1 == nt) {
#pragma unroll
      for (int c = 0; c < C; ++c) acc[c].add(tacc.get(c));
      tacc.zero();
    }
    __syncwarp();
    if (tma && k + S < nt) {
      fence_proxy_async_smem();
      issue(tile + S, s);
    }
  }
  cp_async_wait_all();

  // per (warp, row slot) partials by column, then the CTA and grid reductions
  __syncthreads();
  double* red = reinterpret_cast<double*>(smem);  // [nw * RS][n][KB]
  const int64_t N = n * KB;
#pragma unroll
  for (int q = 0; q < Q; ++q) {
    const int ch = lane_chunk<NB>(rs, jg, q);
#pragma unroll
    for (int e = 0; e < NV; ++e) {
      const int64_t col = (int64_t)ch * NV + e;
      if (col < n) red[(warp * RS + rs) * N + col * KB + cg] = acc[q * NV + e].value();
    }
  }
  multi_finish<T, KB>(a, red, nw * RS, nw);
}

}  // namespace

// ---------------------------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------------------------
static int pow2ceil(int64_t x) {
  int p = 1;
  while (p < x) p <<= 1;
  return p;
}


MultiPlan plan_multi(const DeviceInfo& dev, int64_t m, int64_t n, int64_t k, int elem, bool tma_ok, bool full_v,
                     bool has_v) {
  MultiPlan p;
  if (n <= 0 || k <= 0 || n * elem > 2048) return p;
  p.ok = true;
  p.nb = pow2ceil((n * elem + 127) / 128);
  p.kb_max = (int)std::min<int64_t>(32 / p.nb, pow2ceil(k));
  p.passes = (int)((k + p.kb_max - 1) / p.kb_max);
  p.rows_per_tile = multi_rows(p.nb, p.kb_max, elem);
  // m == 0 runs the same kernel over no tiles (it writes beta Z); tensor maps need m > 0
  p.tma = tma_ok && m > 0 && m < (int64_t(1) << 31);
  // a stage holds a tile of X and its weights; the widest pass (all kb_max, or the
  // remainder's width) sets the stage size
  auto stage_bytes = [&](int kb) {
    const int64_t R = multi_rows(p.nb, kb, elem);
    const int64_t vb = full_v ? R * kb : (has_v ? R : 0);
    return (size_t)(p.nb * R * 128) + (size_t)((vb * elem + 127) & ~int64_t(127));
  };
  size_t tile = stage_bytes(p.kb_max);
  if (k % p.kb_max != 0) tile = std::max(tile, stage_bytes(pow2ceil(k % p.kb_max)));
  const size_t budget = std::min<size_t>(MULTI_SMEM_BUDGET, dev.smem_optin > 0 ? (size_t)dev.smem_optin : MULTI_SMEM_BUDGET);
  // eight warps with a pipeline of 2 to 8 stages each; four warps where eight do not fit
  p.warps = MULTI_THREADS / 32;
  if (p.tma) {
    for (;;) {
      const size_t room = budget - 1024;
      p.stages = (int)std::min<size_t>(8, room / (p.warps * (tile + 8)));
      if (p.stages >= 2 || p.warps == 4) break;
      p.warps = 4;
    }
  } else {
    p.stages = 1;
  }
  const size_t pipe = 1024 + p.warps * p.stages * (tile + 8);
  // partials of every (warp, row slot) by column: row slots x right-hand sides = 32 / nb
  const size_t red = 1024 + (size_t)p.warps * (32 / p.nb) * n * sizeof(double);
  p.smem = std::max(pipe, red);
  const int64_t tiles = (m + p.rows_per_tile - 1) / p.rows_per_tile;
  p.ctas = (int)std::max<int64_t>(1, std::min<int64_t>(dev.sm_count, (tiles + p.warps - 1) / p.warps));
  p.ws_bytes = (size_t)p.ctas * n * p.kb_max * sizeof(double) + 128;
  // fp32 rows of at most 32 columns with 8 or more right-hand sides: both products on the
  // tensor cores, 128-row tiles, one CTA per SM (the environment variable
  // FXTX_MULTI_TC=0 keeps such calls on the CUDA-core kernel)
  static const bool tc_on = [] {
    const char* e = getenv("FXTX_MULTI_TC");
    return !(e && e[0] == '0');
  }();
  if (tc_on && elem == 4 && n <= 32 && k >= 8 && p.tma) {
    MultiPlan q = p;
    q.tc = true;
    q.nb = 1;
    q.kb_max = k <= 8 ? 8 : (k <= 16 ? 16 : 32);
    q.passes = (int)((k + q.kb_max - 1) / q.kb_max);
    q.rows_per_tile = 128;
    q.warps = multi_tc_warps(q.kb_max);
    q.stages = multi_tc_stages(q.kb_max);
    q.smem = multi_tc_smem(q.kb_max);
    const int64_t tc_tiles = (m + 127) / 128;
    q.ctas = (int)std::max<int64_t>(1, std::min<int64_t>(dev.sm_count, tc_tiles));
    q.ws_bytes = (size_t)q.ctas * n * q.kb_max * sizeof(double) + 128;
    if (q.smem <= budget) p = q;
  }
  // the model's estimate: every pass reads X; weights, Y, Z and OUT once; two FMAs per element
  // of X and right-hand side, at the ~35 % of the FMA rate this kernel's issue rate allows
  const double vbytes = full_v ? (double)m * k * elem : (has_v ? (double)m * elem * p.passes : 0.0);
  const double bytes = (double)m * n * elem * p.passes + vbytes + 3.0 * n * k * elem;
  if (p.tc) {
    // the tensor-core form: its pipeline of roles takes a measured number of SM cycles per
    // 128-row tile (16,000,000 x 32 on GB300 at 2,070 MHz: 592, 757 and 1,144 us per call at
    // kb = 8, 16 and 32, i.e. ~1,490, ~1,910 and ~2,880 cycles a tile; the product warps'
    // issue and waits, not HBM, set it), or the HBM time if that is longer
    const double cyc = p.kb_max == 8 ? 1490.0 : (p.kb_max == 16 ? 1910.0 : 2880.0);
    const double tiles_per_cta = std::ceil((double)((m + 127) / 128) / std::max(p.ctas, 1));
    const double hbm_us = roofline_us(dev, bytes, 0.9, 0.0, elem, 1.0, 0.0, 1.0);  // includes the launch
    p.est_us = std::max(sm_cycles_us(tiles_per_cta * cyc * p.passes), hbm_us) + 4.0 * (p.passes - 1);
    return p;
  }
  const double fmas = 2.0 * m * n * k;
  p.est_us = roofline_us(dev, bytes, 0.9, fmas, elem, elem == 4 ? 0.35 : 0.8, 0.0, 1.0) + 4.0 * (p.passes - 1);
  return p;
}

int multi_pass_kb(const MultiPlan& p, int64_t k, int64_t c0) {
  return (int)std::min<int64_t>(p.kb_max, k - c0);
}

int describe_multi(const MultiPlan& p, char* buf, size_t cap) {
  return snprintf(buf, cap,
                  "multi ok=%d tma=%d tc=%d blocks=%d kb=%d passes=%d rows_per_tile=%d stages=%d warps=%d ctas=%d "
                  "smem=%zu ws=%zu est_us=%.1f",
                  (int)p.ok, (int)p.tma, (int)p.tc, p.nb, p.kb_max, p.passes, p.rows_per_tile, p.stages, p.warps,
                  p.ctas, p.smem, p.ws_bytes, p.est_us);
}

int take_multi_device_error() { return take_device_error(); }

template <typename T, int NB, int KB>
static cudaError_t launch_kb(const MultiPlan& p, const MultiArgs<T>& a0, int vmode, cudaStream_t st) {
  constexpr int R = MShape<T, NB, KB>::R;
  MultiArgs<T> a = a0;
  a.tiles = (a.m + R - 1) / R;
  CUtensorMap map;
  memset(&map, 0, sizeof map);
  // a map the driver refuses sends the pass to the plain-load staging
  MultiPlan q = p;
  q.tma = p.tma && encode_rows_map(&map, Chunk<T>::MAP, a.X, a.m, a.n, a.ld * (int64_t)sizeof(T), (int)sizeof(T), R,
                                   128, 0);
  const void* kern = (const void*)dense_multi_kernel<T, NB, KB>;
  cudaError_t e = ensure_smem(kern, q.smem);
  if (e != cudaSuccess) return e;
  // whole rows of weights in 16-byte copies: a full pass over 16-byte aligned rows
  const int v16 = vmode == 2 && a.kb == KB && KB * sizeof(T) >= 16 && (reinterpret_cast<uintptr_t>(a.V) & 15u) == 0 &&
                  (a.ldv * (int64_t)sizeof(T)) % 16 == 0;
  dense_multi_kernel<T, NB, KB><<<q.ctas, q.warps * 32, q.smem, st>>>(map, a, q.stages, q.tma ? 1 : 0, vmode, v16);
  return cudaGetLastError();
}

template <typename T, int NB>
static cudaError_t launch_nb(const MultiPlan& p, const MultiArgs<T>& a, int vmode, cudaStream_t st) {
  switch (pow2ceil(a.kb)) {
    case 1: return launch_kb<T, NB, 1>(p, a, vmode, st);
    case 2: return launch_kb<T, NB, 2>(p, a, vmode, st);
    case 4: if constexpr (NB <= 8) return launch_kb<T, NB, 4>(p, a, vmode, st); break;
    case 8: if constexpr (NB <= 4) return launch_kb<T, NB, 8>(p, a, vmode, st); break;
    case 16: if constexpr (NB <= 2) return launch_kb<T, NB, 16>(p, a, vmode, st); break;
    case 32: if constexpr (NB == 1) return launch_kb<T, NB, 32>(p, a, vmode, st); break;
    default: break;
  }
  return cudaErrorInvalidConfiguration;
}

template <typename T>
cudaError_t launch_multi(const MultiPlan& p, const MultiArgs<T>& a, cudaStream_t st) {
  if (!p.ok || a.kb < 1 || a.kb > p.kb_max) return cudaErrorInvalidConfiguration;
  if constexpr (sizeof(T) == 4) {
    if (p.tc) return launch_multi_tc(p, a, st);
  }
  const int vmode = a.V == nullptr ? 0 : (a.ldv == 0 ? 1 : 2);
  switch (p.nb) {
    case 1: return launch_nb<T, 1>(p, a, vmode, st);
    case 2: return launch_nb<T, 2>(p, a, vmode, st);
    case 4: return launch_nb<T, 4>(p, a, vmode, st);
    case 8: return launch_nb<T, 8>(p, a, vmode, st);
    case 16: return launch_nb<T, 16>(p, a, vmode, st);
    default: return cudaErrorInvalidConfiguration;
  }
}

template cudaError_t launch_multi<float>(const MultiPlan&, const MultiArgs<float>&, cudaStream_t);
template cudaError_t launch_multi<double>(const MultiPlan&, const MultiArgs<double>&, cudaStream_t);

}  // namespace fxtx
