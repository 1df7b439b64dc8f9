// dense.cu — fused kernels for dense row-major X:
//     out = alpha * X^T (v .* (X y)) + beta * z
// ("On optimizing machine learning workloads via kernel fusion", abstract: one
// fused kernel that reads X once, with coarsening and hierarchical aggregation
// of partial results).
//
// Narrow rows (at most 128 sixteen-byte chunks, i.e. n <= 512 fp32 / 256 fp64):
//   every warp owns a contiguous range of row tiles and runs its own pipeline of
//   bulk asynchronous copies (cp.async.bulk + mbarrier) into shared memory. A
//   group of LPR lanes holds one row: each lane takes VPL chunks, forms its part
//   of the dot x_i . y against y cached in registers, the group sums it with
//   shuffles, scales it by v_i, and adds t_i x_ij into register accumulators for
//   the same chunks — so each element of X is loaded from HBM once and used
//   twice. Column partials are then reduced lane -> warp (shuffles) -> CTA
//   (shared memory) -> grid (fixed-order sum by the last CTA to finish).
// Wide rows: a CTA takes rows in groups of WIDE_R, forms their dots in one pass,
//   reduces them through shared memory, and accumulates t_i x_ij into a
//   per-CTA column accumulator (shared memory when it fits); the second touch of
//   the row is served by L1/L2, not HBM. A second kernel sums the per-CTA
//   accumulators in fixed order and applies the epilogue.
#include <algorithm>
#include <mutex>
#include <tuple>
#include <vector>

#include <cuda.h>

#include "common.cuh"
#include "kernels.h"

namespace fxtx {

int take_dense_device_error() { return take_device_error(); }

__host__ __device__ constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ---------------------------------------------------------------------------------------------
// Column partials: CTA -> grid
// ---------------------------------------------------------------------------------------------
// red[w][j] holds warp w's partial of column j. Sums them into the CTA partial,
// stores it in ws[blockIdx.x], and lets the last CTA to take a ticket sum all
// CTA partials in a fixed order and write out = alpha * w + beta * z.
template <typename T, typename TX>
__device__ __forceinline__ void finish_from_red(const DenseArgs<T, TX>& a, double* red, const int nw) {
  __shared__ unsigned s_last;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t n = a.n;
  __syncthreads();
  for (int64_t j = threadIdx.x; j < n; j += blockDim.x) {
    double s = 0.0;
    for (int w = 0; w < nw; ++w) s += red[w * n + j];
    a.ws[blockIdx.x * n + j] = s;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = (atomicAdd(a.ticket, 1u) == gridDim.x - 1) ? 1u : 0u;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const int nc = gridDim.x;
  const int cb = nc * warp / nw, ce = nc * (warp + 1) / nw;
  for (int64_t j = lane; j < n; j += 32) {
    double s = 0.0;
    for (int c = cb; c < ce; ++c) s += __ldcg(a.ws + (int64_t)c * n + j);
    red[warp * n + j] = s;
  }
  __syncthreads();
  for (int64_t j = threadIdx.x; j < n; j += blockDim.x) {
    double s = 0.0;
    for (int w = 0; w < nw; ++w) s += red[w * n + j];
    double o = a.alpha * s;
    if (a.use_z) o += a.beta * (double)a.z[j];
    a.out[j] = (T)o;
  }
  if (threadIdx.x == 0) *a.ticket = 0u;
}

// One element of X in the compute type (bfloat16 widens exactly: its bits are the top
// half of the fp32 pattern).
__device__ __forceinline__ float load_x(const float* p) { return ldg(p); }
__device__ __forceinline__ double load_x(const double* p) { return ldg(p); }
__device__ __forceinline__ float load_x(const __nv_bfloat16* p) {
  return __uint_as_float((unsigned)__ldg(reinterpret_cast<const unsigned short*>(p)) << 16);
}

// ---------------------------------------------------------------------------------------------
// Narrow kernel (short rows, or X that the tensor copies cannot address)
// ---------------------------------------------------------------------------------------------
template <typename T, int LPR, int VPL, bool TMA, typename TX = T>
__global__ void __launch_bounds__(512) dense_narrow_kernel(const DenseArgs<T, TX> a, const int R, const int S) {
  static_assert(!TMA || sizeof(TX) == sizeof(T), "bulk-copied rows are read in the compute type");
  using VT = typename Vec16<T>::type;
  constexpr int NV = Vec16<T>::N;  // elements per 16-byte chunk
  constexpr int G = 32 / LPR;      // rows per warp pass
  constexpr int C = VPL * NV;      // columns per lane
  // fp32 rows longer than 64 entries take the compensated dot (cancellation grows with length)
  constexpr bool COMP = sizeof(T) == 4 && LPR * C > 64;
  extern __shared__ __align__(128) unsigned char smem[];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int g = lane / LPR, q = lane % LPR;
  const int64_t n = a.n;
  const int64_t pitch = TMA ? n : a.ld;  // elements between consecutive rows of a tile
  const size_t stage_bytes = TMA ? align_up((size_t)R * n * sizeof(T), 128) : 0;

  // y restricted to this lane's columns: chunk c = q + LPR * k covers columns c*NV .. c*NV+NV-1
  T yr[C];
#pragma unroll
  for (int k = 0; k < VPL; ++k)
#pragma unroll
    for (int e = 0; e < NV; ++e) {
      const int64_t col = (int64_t)(q + LPR * k) * NV + e;
      yr[k * NV + e] = col < n ? ldg(a.y + col) : T(0);
    }

  // this warp's tiles
  const int64_t gw = (int64_t)blockIdx.x * nw + warp, W = (int64_t)gridDim.x * nw;
  const int64_t t0 = a.tiles * gw / W, t1 = a.tiles * (gw + 1) / W, nt = t1 - t0;

  unsigned char* stages = smem + (size_t)warp * S * stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)nw * S * stage_bytes) + warp * S;
  uint64_t pol = 0;

  auto issue = [&](int64_t tile, int s) {
    const int64_t row0 = tile * R;
    const int rows = (int)tmin<int64_t>(R, a.m - row0);
    unsigned char* dst = stages + (size_t)s * stage_bytes;
    const uint32_t row_bytes = (uint32_t)(n * sizeof(T));
    if (a.ld == n) {  // the tile is one contiguous span
      if (lane == 0) {
        mbar_arrive_expect_tx(&bars[s], rows * row_bytes);
        bulk_g2s(dst, a.X + row0 * n, rows * row_bytes, &bars[s], pol);
      }
    } else {  // one copy per row, issued by as many lanes
      if (lane == 0) mbar_arrive_expect_tx(&bars[s], rows * row_bytes);
      __syncwarp();
      for (int r = lane; r < rows; r += 32)
        bulk_g2s(dst + (size_t)r * row_bytes, a.X + (row0 + r) * a.ld, row_bytes, &bars[s], pol);
    }
  };

  auto load_v = [&](int64_t tile) -> T {
    if (a.v == nullptr || tile >= t1) return T(0);
    const int64_t r = tile * R + lane;
    return (lane < R && r < a.m) ? ldg(a.v + r) : T(0);
  };

  if constexpr (TMA) {
    pol = policy_evict_first();
    if (lane == 0) {
      for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
      fence_mbar_init();
    }
    __syncwarp();
    for (int s = 0; s < S && s < nt; ++s) issue(t0 + s, s);
  }

  typename OuterAcc<T>::type acc[C];
  T vnext = load_v(t0);
  for (int64_t k = 0; k < nt; ++k) {
    const int64_t tile = t0 + k, row0 = tile * R;
    const int rows = (int)tmin<int64_t>(R, a.m - row0);
    const T vcur = vnext;
    if (k + 1 < nt) vnext = load_v(tile + 1);
    const int s = (int)(k % S);
    const T* tx = nullptr;    // the tile in shared memory (bulk-copied path)
    const TX* txg = nullptr;  // the tile in global memory (direct path)
    if constexpr (TMA) {
      const bool ok = mbar_wait_bounded(&bars[s], (uint32_t)((k / S) & 1));
      if (__any_sync(FULL_MASK, !ok)) {
        // give the copies still in flight a bounded chance to land, then stop
        if (lane == 0)
          for (int64_t j = k + 1; j < nt && j < k + S; ++j) mbar_wait_bounded(&bars[j % S], (uint32_t)((j / S) & 1));
        break;
      }
      tx = reinterpret_cast<const T*>(stages + (size_t)s * stage_bytes);
    } else {
      txg = a.X + row0 * a.ld;
    }

    T tacc[C];
#pragma unroll
    for (int c = 0; c < C; ++c) tacc[c] = T(0);
#pragma unroll 2
    for (int r0 = 0; r0 < rows; r0 += G) {
      const int r = r0 + g;
      const bool valid = r < rows;
      const T* rowp = TMA ? tx + (int64_t)r * pitch : nullptr;
      const TX* rowg = TMA ? nullptr : txg + (int64_t)r * pitch;
      T x[C];
#pragma unroll
      for (int k2 = 0; k2 < VPL; ++k2) {
        const int64_t c0 = (int64_t)(q + LPR * k2) * NV;
        if constexpr (TMA) {
          if (valid && c0 < n) {
            const VT vv = *reinterpret_cast<const VT*>(rowp + c0);
            unpack<T>(vv, &x[k2 * NV]);
          } else {
#pragma unroll
            for (int e = 0; e < NV; ++e) x[k2 * NV + e] = T(0);
          }
        } else {
#pragma unroll
          for (int e = 0; e < NV; ++e) x[k2 * NV + e] = (valid && c0 + e < n) ? load_x(rowg + c0 + e) : T(0);
        }
      }
      DotAcc<T, COMP> dacc;
#pragma unroll
      for (int c = 0; c < C; ++c) dacc.add(x[c], yr[c]);
      dacc.template group_reduce<LPR>();
      const T d = dacc.value();
      const T vi = a.v ? __shfl_sync(FULL_MASK, vcur, r & 31) : T(1);
      const T t = valid ? vi * d : T(0);
#pragma unroll
      for (int c = 0; c < C; ++c) tacc[c] = fma(t, x[c], tacc[c]);
    }
#pragma unroll
    for (int c = 0; c < C; ++c) acc[c].add(tacc[c]);
    if constexpr (TMA) {
      __syncwarp();
      if (k + S < nt) {
        fence_proxy_async_smem();
        issue(t0 + k + S, s);
      }
    }
  }

  // lane -> warp: lanes with the same q hold the same columns
  double part[C];
#pragma unroll
  for (int c = 0; c < C; ++c) part[c] = acc[c].value();
#pragma unroll
  for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
    for (int c = 0; c < C; ++c) part[c] += shfl_xor(part[c], o);

  // warp -> CTA -> grid
  __syncthreads();
  double* red = reinterpret_cast<double*>(smem);  // [nw][n]
  if (g == 0) {
#pragma unroll
    for (int k2 = 0; k2 < VPL; ++k2)
#pragma unroll
      for (int e = 0; e < NV; ++e) {
        const int64_t col = (int64_t)(q + LPR * k2) * NV + e;
        if (col < n) red[warp * n + col] = part[k2 * NV + e];
      }
  }
  finish_from_red(a, red, nw);
}

// ---------------------------------------------------------------------------------------------
// Tile kernel (rows of 64 B .. 2 KB, tensor-copied and swizzled)
// ---------------------------------------------------------------------------------------------
// A row of NB 128-byte column blocks is held by LPR = 2 * NB lanes, each taking
// four 16-byte chunks. Tiles of R rows arrive by 2-D tensor copies (one box of
// R x 128 bytes per column block) with the 128-byte swizzle, which stores chunk
// c of row r at chunk position c ^ (r mod 8). chunk_of() assigns chunks so that
// the 8 lanes of every quarter-warp read 8 distinct bank groups. Rows past m and
// columns past n arrive as zeros, so the inner loop needs no masks.
template <int LPR, int CPL, int BW>
__device__ __forceinline__ void chunk_of(int q, int j, int& b, int& c) {
  if (BW == 64) {  // one 64-byte block: LPR 1 (CPL 4) or LPR 2 (CPL 2)
    b = 0;
    c = LPR == 1 ? j : 2 * q + j;
  } else if (LPR == 2) {  // CPL 4, one block
    b = 0;
    c = 4 * q + j;
  } else if (LPR == 4 && CPL == 4) {
    b = j >> 1;
    c = 2 * q + (j & 1);
  } else if (LPR == 4) {  // CPL 2, one block
    b = 0;
    c = 2 * q + j;
  } else {
    b = (q >> 3) + j * (LPR / 8);
    c = q & 7;
  }
}

// Byte offset of chunk c of tile row r inside its box. The 128-byte swizzle stores
// chunk c of row r at chunk c ^ (r mod 8); the 64-byte swizzle (rows of 64 bytes) at
// c ^ ((r / 2) mod 4).
template <int BW>
__device__ __forceinline__ int swizzled(int r, int c) {
  return BW == 128 ? r * 128 + ((c ^ (r & 7)) << 4) : r * 64 + ((c ^ ((r >> 1) & 3)) << 4);
}

// What the tile kernel needs to know about X's storage type: elements per 16-byte
// chunk, the compute type, the tensor-map data type, and the unpacking of a chunk.
template <typename TX>
struct Store;
template <>
struct Store<float> {
  using T = float;
  static constexpr int NV = 4;
  static constexpr CUtensorMapDataType MAP = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  __device__ static __forceinline__ void unpack(const uint4& u, float* e) {
    e[0] = __uint_as_float(u.x); e[1] = __uint_as_float(u.y); e[2] = __uint_as_float(u.z); e[3] = __uint_as_float(u.w);
  }
};
template <>
struct Store<double> {
  using T = double;
  static constexpr int NV = 2;
  static constexpr CUtensorMapDataType MAP = CU_TENSOR_MAP_DATA_TYPE_FLOAT64;
  __device__ static __forceinline__ void unpack(const uint4& u, double* e) {
    e[0] = __hiloint2double((int)u.y, (int)u.x);
    e[1] = __hiloint2double((int)u.w, (int)u.z);
  }
};
template <>
struct Store<__nv_bfloat16> {
  using T = float;
  static constexpr int NV = 8;
  static constexpr CUtensorMapDataType MAP = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  // each 32-bit word holds two bfloat16, the lower-addressed one in its low half
  __device__ static __forceinline__ void unpack(const uint4& u, float* e) {
    const unsigned w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      e[2 * i] = __uint_as_float(w[i] << 16);
      e[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
  }
};

// Tile geometry for rows of NB blocks of BW bytes (BW = 128, or 64 for rows of at
// most 64 bytes) and CPL chunks per lane. A tile is 8 KB (16 KB at NB = 16).
template <int NB, int CPL, int BW = 128>
struct TileShape {
  static constexpr int CPB = BW / 16;                                      // chunks per block
  static constexpr int LPR = CPB * NB / CPL;                               // lanes per row
  static constexpr int G = 32 / LPR;                                       // rows per warp pass
  static constexpr int R = BW == 64 ? 128 : (NB >= 8 ? 8 : 64 / NB);       // rows per tile (multiple of 8)
  static constexpr int P = R / G;                                          // passes per tile
  static constexpr int BOX = R * BW;                                       // bytes of one column block of a tile
  static constexpr int TILE = NB * BOX;                                    // bytes of one pipeline stage
};

// chunks per lane: four for 4- and 8-byte elements, two for bfloat16 (16 columns either way)
template <typename TX>
__host__ __device__ constexpr int tile_cpl() {
  return sizeof(TX) == 2 ? 2 : 4;
}

template <typename TX, int NB, int BW>
__global__ void __launch_bounds__(256, 1)
    dense_tile_kernel(const __grid_constant__ CUtensorMap tmap, const DenseArgs<typename Store<TX>::T, TX> a,
                      const int nbr, const int S) {
  using T = typename Store<TX>::T;
  constexpr int CPL = tile_cpl<TX>();
  using SH = TileShape<NB, CPL, BW>;
  constexpr int NV = Store<TX>::NV;  // elements per 16-byte chunk
  constexpr int CPB = SH::CPB;
  constexpr int LPR = SH::LPR, G = SH::G, R = SH::R, P = SH::P, BOX = SH::BOX, TILE = SH::TILE;
  constexpr int C = CPL * NV;            // columns per lane
  constexpr int VR = (R + 31) / 32;      // registers holding the tile's v
  // fp32 rows longer than 64 entries take the compensated dot
  constexpr bool COMP = sizeof(T) == 4 && NB * CPB * NV > 64;
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  const int g = lane / LPR, q = lane % LPR;
  const int64_t n = a.n;

  int cb[CPL], cc[CPL];
  bool okc[CPL];
  T yr[C];
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
    chunk_of<LPR, CPL, BW>(q, j, cb[j], cc[j]);
    const int64_t col0 = ((int64_t)cb[j] * CPB + cc[j]) * NV;
    okc[j] = cb[j] < nbr && col0 < n;
#pragma unroll
    for (int e = 0; e < NV; ++e) yr[j * NV + e] = (okc[j] && col0 + e < n) ? ldg(a.y + col0 + e) : T(0);
  }

  const int64_t gw = (int64_t)blockIdx.x * nw + warp, W = (int64_t)gridDim.x * nw;
  const int64_t t0 = a.tiles * gw / W, t1 = a.tiles * (gw + 1) / W, nt = t1 - t0;
  unsigned char* stages = smem + (size_t)warp * S * TILE;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)nw * S * TILE) + warp * S;
  const uint64_t pol = policy_evict_first();

  auto issue = [&](int64_t tile, int s) {
    if (lane == 0) mbar_arrive_expect_tx(&bars[s], (uint32_t)(nbr * BOX));
    __syncwarp();
    if (lane < nbr)
      tma_load_2d(stages + (size_t)s * TILE + lane * BOX, &tmap, lane * (BW / (int)sizeof(TX)), (int)(tile * R),
                  &bars[s], pol);
  };
  auto load_v = [&](int64_t tile, T* vv) {
#pragma unroll
    for (int i = 0; i < VR; ++i) {
      const int rl = lane + 32 * i;
      const int64_t row = tile * R + rl;
      vv[i] = (a.v != nullptr && tile < t1 && rl < R && row < a.m) ? ldg(a.v + row) : T(0);
    }
  };

  if (lane == 0) {
    for (int s = 0; s < S; ++s) mbar_init(&bars[s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  for (int s = 0; s < S && s < nt; ++s) issue(t0 + s, s);

  typename OuterAcc<T>::type acc[C];
  T vnext[VR];
  load_v(t0, vnext);
  for (int64_t k = 0; k < nt; ++k) {
    T vcur[VR];
#pragma unroll
    for (int i = 0; i < VR; ++i) vcur[i] = vnext[i];
    if (k + 1 < nt) load_v(t0 + k + 1, vnext);
    const int s = (int)(k % S);
    const bool ok = mbar_wait_bounded(&bars[s], (uint32_t)((k / S) & 1));
    if (__any_sync(FULL_MASK, !ok)) {
      if (lane == 0)
        for (int64_t j = k + 1; j < nt && j < k + S; ++j) mbar_wait_bounded(&bars[j % S], (uint32_t)((j / S) & 1));
      break;
    }
    const unsigned char* stage = stages + (size_t)s * TILE;

    T tacc[C];
#pragma unroll
    for (int c = 0; c < C; ++c) tacc[c] = T(0);
#pragma unroll
    for (int p = 0; p < P; ++p) {
      const int r = p * G + g;
      T x[C];
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        if (okc[j]) {
          const uint4 u = *reinterpret_cast<const uint4*>(stage + cb[j] * BOX + swizzled<BW>(r, cc[j]));
          Store<TX>::unpack(u, &x[j * NV]);
        } else {
#pragma unroll
          for (int e = 0; e < NV; ++e) x[j * NV + e] = T(0);
        }
      }
      T dsum;
      if constexpr (COMP) {
        DotAcc<T, true> dacc;
#pragma unroll
        for (int c = 0; c < C; ++c) dacc.add(x[c], yr[c]);
        dacc.template group_reduce<LPR>();
        dsum = dacc.value();
      } else {
        // four independent partial sums: a chain of C/4 FMAs instead of C
        T d4[4] = {T(0), T(0), T(0), T(0)};
#pragma unroll
        for (int c = 0; c < C; ++c) d4[c & 3] = fma(x[c], yr[c], d4[c & 3]);
        dsum = group_sum<LPR>((d4[0] + d4[1]) + (d4[2] + d4[3]));
      }
      const T vi = a.v ? __shfl_sync(FULL_MASK, vcur[(p * G) / 32], (p * G + g) & 31) : T(1);
      const T t = vi * dsum;
#pragma unroll
      for (int c = 0; c < C; ++c) tacc[c] = fma(t, x[c], tacc[c]);
    }
#pragma unroll
    for (int c = 0; c < C; ++c) acc[c].add(tacc[c]);
    __syncwarp();
    if (k + S < nt) {
      fence_proxy_async_smem();
      issue(t0 + k + S, s);
    }
  }

  // lane -> warp: lanes with the same q hold the same columns
  double part[C];
#pragma unroll
  for (int c = 0; c < C; ++c) part[c] = acc[c].value();
#pragma unroll
  for (int o = LPR; o < 32; o <<= 1)
#pragma unroll
    for (int c = 0; c < C; ++c) part[c] += shfl_xor(part[c], o);

  __syncthreads();
  double* red = reinterpret_cast<double*>(smem);  // [nw][n]
  if (g == 0) {
#pragma unroll
    for (int j = 0; j < CPL; ++j)
#pragma unroll
      for (int e = 0; e < NV; ++e) {
        const int64_t col = ((int64_t)cb[j] * CPB + cc[j]) * NV + e;
        if (okc[j] && col < n) red[warp * n + col] = part[j * NV + e];
      }
  }
  finish_from_red(a, red, nw);
}

// ---------------------------------------------------------------------------------------------
// Wide kernel
// ---------------------------------------------------------------------------------------------
constexpr int WIDE_R = 8;        // rows coarsened per step
constexpr int WIDE_THREADS = 512;

template <typename T, bool VEC>
__global__ void __launch_bounds__(WIDE_THREADS) dense_wide_kernel(const DenseArgs<T> a, const bool smem_acc) {
  using VT = typename Vec16<T>::type;
  constexpr int NV = Vec16<T>::N;
  constexpr int NWARP = WIDE_THREADS / 32;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ double s_dot[WIDE_R][NWARP];
  __shared__ double s_t[WIDE_R];

  const int64_t n = a.n, ld = a.ld;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double* acc = smem_acc ? reinterpret_cast<double*>(smem) : a.ws + (int64_t)blockIdx.x * n;
  for (int64_t j = threadIdx.x; j < n; j += blockDim.x) acc[j] = 0.0;
  __syncthreads();

  const int64_t r_begin = a.m * blockIdx.x / gridDim.x, r_end = a.m * (blockIdx.x + 1) / gridDim.x;
  const int64_t nvec = VEC ? n / NV : 0;  // whole chunks per row (VEC: rows start 16-byte aligned)

  for (int64_t i0 = r_begin; i0 < r_end; i0 += WIDE_R) {
    const int rows = (int)tmin<int64_t>(WIDE_R, r_end - i0);
    // pass 1: WIDE_R dots at once
    DotAcc<T, sizeof(T) == 4> d[WIDE_R];
    for (int64_t c = threadIdx.x; c < nvec; c += blockDim.x) {
      T yv[NV];
      unpack<T>(*reinterpret_cast<const VT*>(a.y + c * NV), yv);
#pragma unroll
      for (int r = 0; r < WIDE_R; ++r) {
        if (r < rows) {
          T xv[NV];
          unpack<T>(*reinterpret_cast<const VT*>(a.X + (i0 + r) * ld + c * NV), xv);
#pragma unroll
          for (int e = 0; e < NV; ++e) d[r].add(xv[e], yv[e]);
        }
      }
    }
    for (int64_t j = nvec * NV + threadIdx.x; j < n; j += blockDim.x) {
      const T yj = a.y[j];
#pragma unroll
      for (int r = 0; r < WIDE_R; ++r)
        if (r < rows) d[r].add(a.X[(i0 + r) * ld + j], yj);
    }
#pragma unroll
    for (int r = 0; r < WIDE_R; ++r) {
      d[r].template group_reduce<32>();
      if (lane == 0) s_dot[r][warp] = d[r].value_f64();
    }
    __syncthreads();
    if (threadIdx.x < WIDE_R) {
      const int r = threadIdx.x;
      double u = 0.0;
      for (int w = 0; w < NWARP; ++w) u += s_dot[r][w];
      const double vi = (r < rows && a.v) ? (double)a.v[i0 + r] : 1.0;
      s_t[r] = r < rows ? (double)(T)(vi * (T)u) : 0.0;
    }
    __syncthreads();
    T t[WIDE_R];
#pragma unroll
    for (int r = 0; r < WIDE_R; ++r) t[r] = (T)s_t[r];
    // pass 2: the same rows again, scattered into the column accumulator. It walks the rows
    // in the reverse of pass 1's order, so it starts on the lines pass 1 brought into L2 last
    // and the re-read comes from L2 rather than HBM as far as L2 holds the CTAs' rows.
    for (int64_t j = nvec * NV + threadIdx.x; j < n; j += blockDim.x) {
      // fp64: the FMA chain starts from the accumulator (no separate add); fp32: a step's
      // products are summed in fp32 and added in fp64
      T s = sizeof(T) == 8 ? (T)acc[j] : T(0);
#pragma unroll
      for (int r = 0; r < WIDE_R; ++r)
        if (r < rows) s = fma(t[r], a.X[(i0 + r) * ld + j], s);
      if constexpr (sizeof(T) == 8) acc[j] = (double)s; else acc[j] += (double)s;
    }
    const int64_t nk = threadIdx.x < nvec ? (nvec - 1 - threadIdx.x) / blockDim.x + 1 : 0;
    for (int64_t kk = nk - 1; kk >= 0; --kk) {
      const int64_t c = threadIdx.x + kk * blockDim.x;
      T s[NV];
#pragma unroll
      for (int e = 0; e < NV; ++e) s[e] = sizeof(T) == 8 ? (T)acc[c * NV + e] : T(0);
#pragma unroll
      for (int r = 0; r < WIDE_R; ++r) {
        if (r < rows) {
          T xv[NV];
          unpack<T>(*reinterpret_cast<const VT*>(a.X + (i0 + r) * ld + c * NV), xv);
#pragma unroll
          for (int e = 0; e < NV; ++e) s[e] = fma(t[r], xv[e], s[e]);
        }
      }
#pragma unroll
      for (int e = 0; e < NV; ++e) {
        if constexpr (sizeof(T) == 8) acc[c * NV + e] = (double)s[e]; else acc[c * NV + e] += (double)s[e];
      }
    }
    __syncthreads();  // s_dot / s_t reuse
  }
  if (smem_acc)
    for (int64_t j = threadIdx.x; j < n; j += blockDim.x) a.ws[(int64_t)blockIdx.x * n + j] = acc[j];
}

// fp64 wide rows, software-pipelined. The fp64 units (2 FMAs per clock per SM on GB300)
// bind this kernel: every element costs two fp64 FMAs, one in the row dot and one in the
// scatter. One sweep over the columns forms the dots of step k + 1 (rows from HBM) and
// scatters step k (the same rows re-read, from L2, into the CTA's fp64 column sums in
// shared memory), so the FMAs of both passes interleave in one instruction stream and
// the memory latency of each hides behind the other's arithmetic; one CTA barrier per
// step turns the dots into the next t_i. Rows stay live for two steps: at the plan's R = 8
// (152 CTAs x 16 rows x 160 KB for n = 20,000) the re-reads exceed L2 and partly return to
// HBM, which has the bandwidth to spare while the fp64 units bind; R = 2 keeps them in L2
// but leaves too few independent FMA chains per thread.
template <int R, bool VEC>
__global__ void __launch_bounds__(WIDE_THREADS) dense_wide_f64_kernel(const DenseArgs<double> a, const bool smem_acc) {
  constexpr int NWARP = WIDE_THREADS / 32;
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ double s_dot[R][NWARP];
  __shared__ double s_t[2][R];

  const int64_t n = a.n, ld = a.ld;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  double* acc = smem_acc ? reinterpret_cast<double*>(smem) : a.ws + (int64_t)blockIdx.x * n;
  for (int64_t j = threadIdx.x; j < n; j += blockDim.x) acc[j] = 0.0;

  const int64_t r_begin = a.m * blockIdx.x / gridDim.x, r_end = a.m * (blockIdx.x + 1) / gridDim.x;
  const int64_t nvec = VEC ? n / 2 : 0;  // whole 16-byte chunks per row (VEC: rows start 16-byte aligned)

  // the dots of the R rows from i0 (rows of them real) reduced over the CTA into t = v_i u_i,
  // written to buffer b; ends with a barrier
  auto finish_dots = [&](double* d, int64_t i0, int rows, int b) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const double v = group_sum<32>(d[r]);
      if (lane == 0) s_dot[r][warp] = v;
    }
    __syncthreads();
    if (threadIdx.x < R) {
      const int r = threadIdx.x;
      double u = 0.0;
      for (int w = 0; w < NWARP; ++w) u += s_dot[r][w];
      const double vi = (r < rows && a.v) ? a.v[i0 + r] : 1.0;
      s_t[b][r] = r < rows ? vi * u : 0.0;
    }
    __syncthreads();
  };

  // step 0: its dots alone
  {
    const int rows = (int)tmax<int64_t>(0, tmin<int64_t>(R, r_end - r_begin));
    double d[R];
#pragma unroll
    for (int r = 0; r < R; ++r) d[r] = 0.0;
    for (int64_t c = threadIdx.x; c < nvec; c += blockDim.x) {
      const double2 yv = *reinterpret_cast<const double2*>(a.y + 2 * c);
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (r < rows) {
          const double2 xv = *reinterpret_cast<const double2*>(a.X + (r_begin + r) * ld + 2 * c);
          d[r] = fma(xv.y, yv.y, fma(xv.x, yv.x, d[r]));
        }
    }
    for (int64_t j = nvec * 2 + threadIdx.x; j < n; j += blockDim.x) {
      const double yj = a.y[j];
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (r < rows) d[r] = fma(a.X[(r_begin + r) * ld + j], yj, d[r]);
    }
    finish_dots(d, r_begin, rows, 0);  // its first barrier also orders the zeroing of acc
  }

  for (int k = 0;; ++k) {
    const int b = k & 1;
    const int64_t i0 = r_begin + (int64_t)k * R;
    if (i0 >= r_end) break;
    const int rows = (int)tmin<int64_t>(R, r_end - i0);
    const int64_t i1 = i0 + R;  // the next step, whose dots this sweep forms
    const int rows1 = (int)tmax<int64_t>(0, tmin<int64_t>(R, r_end - i1));
    double t[R];
#pragma unroll
    for (int r = 0; r < R; ++r) t[r] = s_t[b][r];
    double d[R];
#pragma unroll
    for (int r = 0; r < R; ++r) d[r] = 0.0;
    for (int64_t c = threadIdx.x; c < nvec; c += blockDim.x) {
      // the next step's dots (rows from HBM) ...
      if (rows1 > 0) {
        const double2 yv = *reinterpret_cast<const double2*>(a.y + 2 * c);
#pragma unroll
        for (int r = 0; r < R; ++r)
          if (r < rows1) {
            const double2 xv = *reinterpret_cast<const double2*>(a.X + (i1 + r) * ld + 2 * c);
            d[r] = fma(xv.y, yv.y, fma(xv.x, yv.x, d[r]));
          }
      }
      // ... and this step's scatter (rows from L2): the FMA chain starts from the column sum,
      // read as one 16-byte access in shared memory (half the wavefronts of two 8-byte ones)
      // and as two doubles in global memory (a CTA's sums start 8-byte aligned for odd n)
      double s0, s1;
      if (smem_acc) {
        const double2 sv = *reinterpret_cast<const double2*>(acc + 2 * c);
        s0 = sv.x;
        s1 = sv.y;
      } else {
        s0 = acc[2 * c];
        s1 = acc[2 * c + 1];
      }
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (r < rows) {
          const double2 xv = *reinterpret_cast<const double2*>(a.X + (i0 + r) * ld + 2 * c);
          s0 = fma(t[r], xv.x, s0);
          s1 = fma(t[r], xv.y, s1);
        }
      if (smem_acc) {
        *reinterpret_cast<double2*>(acc + 2 * c) = make_double2(s0, s1);
      } else {
        acc[2 * c] = s0;
        acc[2 * c + 1] = s1;
      }
    }
    for (int64_t j = nvec * 2 + threadIdx.x; j < n; j += blockDim.x) {
      if (rows1 > 0) {
        const double yj = a.y[j];
#pragma unroll
        for (int r = 0; r < R; ++r)
          if (r < rows1) d[r] = fma(a.X[(i1 + r) * ld + j], yj, d[r]);
      }
      double s = acc[j];
#pragma unroll
      for (int r = 0; r < R; ++r)
        if (r < rows) s = fma(t[r], a.X[(i0 + r) * ld + j], s);
      acc[j] = s;
    }
    if (rows1 > 0) finish_dots(d, i1, rows1, b ^ 1);  // uniform across the CTA
  }
  if (smem_acc) {
    __syncthreads();
    for (int64_t j = threadIdx.x; j < n; j += blockDim.x) a.ws[(int64_t)blockIdx.x * n + j] = acc[j];
  }
}

// Fixed-order sum of per-CTA column partials [nc][n], then out = alpha * w + beta * z.
template <typename T>
__global__ void __launch_bounds__(256) reduce_partials_kernel(const DenseArgs<T> a, const int nc) {
  __shared__ double s[8][33];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t j = (int64_t)blockIdx.x * 32 + lane;
  const int cb = nc * warp / 8, ce = nc * (warp + 1) / 8;
  double acc = 0.0;
  if (j < a.n)
    for (int c = cb; c < ce; ++c) acc += __ldcg(a.ws + (int64_t)c * a.n + j);
  s[warp][lane] = acc;
  __syncthreads();
  if (warp == 0 && j < a.n) {
    double w = 0.0;
    for (int k = 0; k < 8; ++k) w += s[k][lane];
    double o = a.alpha * w;
    if (a.use_z) o += a.beta * (double)a.z[j];
    a.out[j] = (T)o;
  }
}

// m == 0: out = beta z (or 0).
template <typename T>
__global__ void empty_rows_kernel(const DenseArgs<T> a) {
  for (int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; j < a.n; j += (int64_t)gridDim.x * blockDim.x)
    a.out[j] = a.use_z ? (T)(a.beta * (double)a.z[j]) : T(0);
}

// ---------------------------------------------------------------------------------------------
// Host launchers
// ---------------------------------------------------------------------------------------------
// The attribute is set once per (kernel, device) at the largest size asked for so
// far; later calls that fit skip the driver call.
cudaError_t ensure_smem(const void* kernel, size_t bytes) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  static std::mutex mu;
  static std::vector<std::tuple<const void*, int, size_t>> done;
  std::lock_guard<std::mutex> lock(mu);
  for (auto& d : done)
    if (std::get<0>(d) == kernel && std::get<1>(d) == dev && std::get<2>(d) >= bytes) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) {
    bool found = false;
    for (auto& d : done)
      if (std::get<0>(d) == kernel && std::get<1>(d) == dev) {
        std::get<2>(d) = bytes;
        found = true;
      }
    if (!found) done.emplace_back(kernel, dev, bytes);
  }
  return e;
}

template <typename T, int LPR, int VPL>
static cudaError_t launch_narrow(const DensePlan& p, const DenseArgs<T>& a, cudaStream_t st) {
  const void* k = p.kind == DENSE_NARROW_TMA ? (const void*)dense_narrow_kernel<T, LPR, VPL, true>
                                             : (const void*)dense_narrow_kernel<T, LPR, VPL, false>;
  cudaError_t e = ensure_smem(k, p.smem);
  if (e != cudaSuccess) return e;
  if (p.kind == DENSE_NARROW_TMA)
    dense_narrow_kernel<T, LPR, VPL, true><<<p.ctas, p.warps * 32, p.smem, st>>>(a, p.rows_per_tile, p.stages);
  else
    dense_narrow_kernel<T, LPR, VPL, false><<<p.ctas, p.warps * 32, p.smem, st>>>(a, p.rows_per_tile, 1);
  return cudaGetLastError();
}

// cuTensorMapEncodeTiled, fetched from the driver once (no link against libcuda).
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    cudaGetLastError();
  });
  return fn;
}

// Tensor map of X (n columns, m rows, row pitch ld) in boxes of rows x bw bytes, with the
// swizzle of the same width (bw = 128 or 64).
template <typename TX>
static bool encode_x_map(CUtensorMap* map, const TX* X, int64_t m, int64_t n, int64_t ld, int rows, int bw) {
  EncodeTiledFn fn = encode_tiled();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)n, (cuuint64_t)m};
  const cuuint64_t strides[1] = {(cuuint64_t)(ld * (int64_t)sizeof(TX))};
  const cuuint32_t box[2] = {(cuuint32_t)(bw / sizeof(TX)), (cuuint32_t)rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, Store<TX>::MAP, 2, const_cast<TX*>(X), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, bw == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <typename TX, int NB, int BW = 128>
static cudaError_t launch_tile_nb(const DensePlan& p, const CUtensorMap& map,
                                  const DenseArgs<typename Store<TX>::T, TX>& a, cudaStream_t st) {
  cudaError_t e = ensure_smem((const void*)dense_tile_kernel<TX, NB, BW>, p.smem);
  if (e != cudaSuccess) return e;
  dense_tile_kernel<TX, NB, BW><<<p.ctas, p.warps * 32, p.smem, st>>>(map, a, p.nbr, p.stages);
  return cudaGetLastError();
}

template <typename TX>
static cudaError_t launch_tile(const DensePlan& p, const DenseArgs<typename Store<TX>::T, TX>& a, cudaStream_t st) {
  CUtensorMap map;
  if (!encode_x_map<TX>(&map, a.X, a.m, a.n, a.ld, p.rows_per_tile, p.box_bytes)) return cudaErrorInvalidValue;
  if (p.box_bytes == 64) return launch_tile_nb<TX, 1, 64>(p, map, a, st);
  switch (p.nb) {
    case 1: return launch_tile_nb<TX, 1>(p, map, a, st);
    case 2: return launch_tile_nb<TX, 2>(p, map, a, st);
    case 4: return launch_tile_nb<TX, 4>(p, map, a, st);
    case 8: return launch_tile_nb<TX, 8>(p, map, a, st);
    case 16:
      if constexpr (tile_cpl<TX>() == 4) return launch_tile_nb<TX, 16>(p, map, a, st);
      return cudaErrorInvalidConfiguration;
    default: return cudaErrorInvalidConfiguration;
  }
}

template <int R>
static cudaError_t launch_wide_f64_r(const DensePlan& p, const DenseArgs<double>& a, bool vec, cudaStream_t st) {
  const void* k = vec ? (const void*)dense_wide_f64_kernel<R, true> : (const void*)dense_wide_f64_kernel<R, false>;
  cudaError_t e = ensure_smem(k, p.smem);
  if (e != cudaSuccess) return e;
  if (vec)
    dense_wide_f64_kernel<R, true><<<p.ctas, WIDE_THREADS, p.smem, st>>>(a, p.smem_acc);
  else
    dense_wide_f64_kernel<R, false><<<p.ctas, WIDE_THREADS, p.smem, st>>>(a, p.smem_acc);
  return cudaGetLastError();
}

template <typename T>
static cudaError_t launch_wide_f64(const DensePlan& p, const DenseArgs<T>& a, bool vec, cudaStream_t st) {
  if constexpr (sizeof(T) == 8) {
    switch (p.rows_per_tile) {
      case 2: return launch_wide_f64_r<2>(p, a, vec, st);
      case 4: return launch_wide_f64_r<4>(p, a, vec, st);
      case 8: return launch_wide_f64_r<8>(p, a, vec, st);
      default: return cudaErrorInvalidConfiguration;
    }
  }
  return cudaErrorInvalidConfiguration;
}

template <typename T>
cudaError_t launch_dense(const DensePlan& p, const DenseArgs<T>& a, cudaStream_t st) {
  switch (p.kind) {
    case DENSE_NOOP:
      return cudaSuccess;
    case DENSE_EMPTY_ROWS: {
      const int blocks = (int)std::min<int64_t>((a.n + 255) / 256, 4096);
      empty_rows_kernel<T><<<blocks, 256, 0, st>>>(a);
      return cudaGetLastError();
    }
    case DENSE_TILE_TMA:
      return launch_tile<T>(p, a, st);
    case DENSE_NARROW_TMA:
    case DENSE_NARROW_DIRECT: {
      const int key = p.lpr * 8 + p.vpl;
      switch (key) {
        case 1 * 8 + 1: return launch_narrow<T, 1, 1>(p, a, st);
        case 2 * 8 + 1: return launch_narrow<T, 2, 1>(p, a, st);
        case 4 * 8 + 1: return launch_narrow<T, 4, 1>(p, a, st);
        case 8 * 8 + 1: return launch_narrow<T, 8, 1>(p, a, st);
        case 8 * 8 + 2: return launch_narrow<T, 8, 2>(p, a, st);
        case 8 * 8 + 4: return launch_narrow<T, 8, 4>(p, a, st);
        case 16 * 8 + 4: return launch_narrow<T, 16, 4>(p, a, st);
        case 32 * 8 + 4: return launch_narrow<T, 32, 4>(p, a, st);
        default: return cudaErrorInvalidConfiguration;
      }
    }
    case DENSE_WIDE: {
      const bool vec = (reinterpret_cast<uintptr_t>(a.X) % 16 == 0) && (reinterpret_cast<uintptr_t>(a.y) % 16 == 0) &&
                       ((a.ld * (int64_t)sizeof(T)) % 16 == 0);
      if constexpr (sizeof(T) == 8) {
        cudaError_t e = launch_wide_f64(p, a, vec, st);
        if (e != cudaSuccess) return e;
        reduce_partials_kernel<T><<<(unsigned)((a.n + 31) / 32), 256, 0, st>>>(a, p.ctas);
        return cudaGetLastError();
      }
      const void* k = vec ? (const void*)dense_wide_kernel<T, true> : (const void*)dense_wide_kernel<T, false>;
      cudaError_t e = ensure_smem(k, p.smem);
      if (e != cudaSuccess) return e;
      if (vec)
        dense_wide_kernel<T, true><<<p.ctas, WIDE_THREADS, p.smem, st>>>(a, p.smem_acc);
      else
        dense_wide_kernel<T, false><<<p.ctas, WIDE_THREADS, p.smem, st>>>(a, p.smem_acc);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      reduce_partials_kernel<T><<<(unsigned)((a.n + 31) / 32), 256, 0, st>>>(a, p.ctas);
      return cudaGetLastError();
    }
  }
  return cudaErrorInvalidConfiguration;
}

cudaError_t launch_dense_bf16(const DensePlan& p, const DenseArgs<float, __nv_bfloat16>& a, cudaStream_t st) {
  switch (p.kind) {
    case DENSE_NOOP:
      return cudaSuccess;
    case DENSE_EMPTY_ROWS: {
      DenseArgs<float> e;
      e.n = a.n; e.z = a.z; e.out = a.out; e.beta = a.beta; e.use_z = a.use_z;
      const int blocks = (int)std::min<int64_t>((a.n + 255) / 256, 4096);
      empty_rows_kernel<float><<<blocks, 256, 0, st>>>(e);
      return cudaGetLastError();
    }
    case DENSE_TILE_TMA:
      return launch_tile<__nv_bfloat16>(p, a, st);
    case DENSE_NARROW_DIRECT: {
      const int key = p.lpr * 8 + p.vpl;
      auto go = [&](auto kernel) -> cudaError_t {
        cudaError_t e = ensure_smem((const void*)kernel, p.smem);
        if (e != cudaSuccess) return e;
        kernel<<<p.ctas, p.warps * 32, p.smem, st>>>(a, p.rows_per_tile, 1);
        return cudaGetLastError();
      };
      using B = __nv_bfloat16;
      switch (key) {
        case 1 * 8 + 1: return go(dense_narrow_kernel<float, 1, 1, false, B>);
        case 2 * 8 + 1: return go(dense_narrow_kernel<float, 2, 1, false, B>);
        case 4 * 8 + 1: return go(dense_narrow_kernel<float, 4, 1, false, B>);
        case 8 * 8 + 1: return go(dense_narrow_kernel<float, 8, 1, false, B>);
        case 8 * 8 + 2: return go(dense_narrow_kernel<float, 8, 2, false, B>);
        case 8 * 8 + 4: return go(dense_narrow_kernel<float, 8, 4, false, B>);
        case 16 * 8 + 4: return go(dense_narrow_kernel<float, 16, 4, false, B>);
        case 32 * 8 + 4: return go(dense_narrow_kernel<float, 32, 4, false, B>);
        default: return cudaErrorInvalidConfiguration;
      }
    }
    default:
      return cudaErrorInvalidConfiguration;  // wide rows are not offered for bfloat16 X
  }
}

template cudaError_t launch_dense<float>(const DensePlan&, const DenseArgs<float>&, cudaStream_t);
template cudaError_t launch_dense<double>(const DensePlan&, const DenseArgs<double>&, cudaStream_t);

}  // namespace fxtx
