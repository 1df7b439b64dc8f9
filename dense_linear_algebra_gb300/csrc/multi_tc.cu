// multi_tc.cu — the multi-vector instantiation OUT = alpha * X^T (V ⊙ (X Y)) + beta * Z
// with both of its products on the tensor cores (tcgen05), for fp32 X of at most 32 columns.
//
// "On optimizing machine learning workloads via kernel fusion" (abstract): the fused
// pattern and its instantiations; with k right-hand sides the pattern is two small
// matrix products per tile of 128 rows,
//     U = X_tile Y          (128 x kb: the row dots)
//     T = V_tile ⊙ U        (elementwise)
//     W += X_tile^T T       (32 x kb: the scatter),
// and X_tile is read from HBM once for both.
//
// Precision. The tensor cores take bfloat16 operands; fp32 values are split into three
// bfloat16 terms, x = x1 + x2 + x3 exactly (each rounded to nearest, every residual exact in
// fp32), and all nine products of the terms are formed, accumulated in fp32 in tensor
// memory: U per tile; W over four tiles (512 rows, 32 accumulation steps of K = 16), then
// folded into compensated two-float column sums (so the fp32 rounding of W, at most
// 32 * 2^-24 S, does not grow with the number of tiles). The error bound is the fp32 entry
// points' 2e-5 S.
//
// Throughput. An M = 128, K = 16 tensor-core product holds the tensor pipe for about 64
// cycles for any N up to 128 (measured on GB300), so the number of products per tile, not
// their width, sets the pipe's time. A tile takes 14:
//   U: the X terms stacked along K (K = 96: 6 products of K = 16) against the Y terms
//      stacked along N (N = 3 kb: column group b holds X y_b; U = the groups' sum);
//   W: K = 128 tile rows (8 products), the X terms stacked along M (M = 96 of 128), the T
//      terms along N (N = 3 kb).
//
// Roles (one CTA per SM, persistent over a contiguous range of tiles), linked by mbarriers
// only:
//   warp 0       one thread: tensor copies of X tiles (128 x 32 fp32, 128-byte swizzle);
//   warp 1       U's products, and the last warp W's: each loop run by a whole (converged)
//                warp, one elected lane issuing and committing to mbarriers;
//   warps 2..    split warps, one group of four (two at kb = 8, taking alternate tiles): one
//                row each, X into its three terms in an operand buffer;
//   next 8 warps row warps, two groups of four (tensor-memory lanes 32 (warp % 4) ..),
//                taking alternate tiles (kb = 32: every tile, half of the right-hand sides
//                each): each row's U from tensor memory, t = v u and its terms into the T
//                buffer; every four tiles, W folded into the column sums;
//   next warp    one thread: tensor copies of the tiles' rows of V (swizzled at their width).
//
// Shared-memory operand layouts (no swizzle; core matrices of 8 rows x 16 bytes):
//   X terms   128 tile rows x 96 columns (term a's column j at 32 a + j): the 16 bytes of
//             row r, columns 8 cb .. 8 cb + 7, at cb * 2048 + r * 16. For U it is the
//             K-major A operand (M = rows, K = columns); for W the MN-major A operand
//             (M = columns, K = rows) of the same bytes, M padded to 128 by reading 8 KB
//             past the buffer (those accumulator lanes are never read).
//   Y terms   96 K rows (term a's X column j at 32 a + j) x NW columns (term b's right-hand
//             side c at b * kb + c; the same y_b for every a), K-major B operand: element
//             (kk, col) at (col / 8) * 1536 + (kk / 8) * 128 + (col % 8) * 16 + (kk % 8) * 2.
//   T terms   128 rows (K) x NW columns (term b's column c at b * kb + c), MN-major B
//             operand: element (r, col) at (r / 8) * NW * 16 + (col / 8) * 128 + (r % 8) * 16
//             + (col % 8) * 2.
// A descriptor's leading byte offset is its core stride along K, the stride byte offset
// its core stride along M or N. With M = 128 the accumulator's row i sits in lane i.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "kernels.h"
#include "multi.h"
#include "tmap.h"

namespace fxtx {
namespace {

constexpr int TC_ROWS = 128;             // rows per tile
constexpr int TC_XTILE = TC_ROWS * 128;  // bytes of one X tile (32 fp32 columns)
constexpr int TC_ABUF = 12 * 2048;       // bytes of one tile's three X terms

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}

// Instruction descriptor: fp32 accumulator, bfloat16 A and B, M x N; mn = 1: both operands
// MN-major, 0: both K-major.
__host__ __device__ constexpr uint32_t tc_idesc(int M, int N, int mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)mn << 15) | ((uint32_t)mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void tc_mma(uint32_t dtmem, uint64_t ad, uint64_t bd, uint32_t idesc, int accum) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(dtmem),
      "l"(ad), "l"(bd), "r"(idesc), "r"(accum)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 fp32 columns of this warp's 32 tensor-memory lanes from column address `taddr`; the
// caller waits (tcgen05.wait::ld) before using them.
__device__ __forceinline__ void tc_load16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// x = hi + mid + lo in bfloat16, each rounded to nearest; both residuals are exact in fp32.
__device__ __forceinline__ void split3(float x0, float x1, uint32_t& a, uint32_t& b, uint32_t& c) {
  const __nv_bfloat162 p = __floats2bfloat162_rn(x0, x1);
  const float r0 = x0 - __low2float(p), r1 = x1 - __high2float(p);
  const __nv_bfloat162 q = __floats2bfloat162_rn(r0, r1);
  const __nv_bfloat162 s = __floats2bfloat162_rn(r0 - __low2float(q), r1 - __high2float(q));
  a = *reinterpret_cast<const uint32_t*>(&p);
  b = *reinterpret_cast<const uint32_t*>(&q);
  c = *reinterpret_cast<const uint32_t*>(&s);
}

// Waits for phase `parity` of `bar`; gives up when another role has given up (the CTA's
// abort word) or after WAIT_LIMIT polls (raising FXTX_ERR_TIMEOUT and setting the word).
// Polls carry no suspend-time hint: a suspended waiter wakes late, and these waits sit on the
// pipeline's critical path.
__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile int* abort_word) {
  for (uint32_t it = 0; it < WAIT_LIMIT; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u && *abort_word) return false;
  }
  raise_error(FXTX_ERR_TIMEOUT);
  *abort_word = 1;
  return false;
}

// Pulls a tensor-map box into L2 ahead of its tensor copy (no shared memory, no completion).
__device__ __forceinline__ void tma_prefetch_2d(const void* tmap, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(tmap), "r"(x), "r"(y)
               : "memory");
}

// A whole warp's wait: every lane waits, and all take the same branch after it.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_word) {
  return __all_sync(FULL_MASK, tc_wait(bar, parity, abort_word));
}

// True in one lane of the (converged) warp.
__device__ __forceinline__ bool elect_one() {
  uint32_t e;
  asm volatile("{\n.reg .b32 r;\n.reg .pred p;\nelect.sync r|p, 0xffffffff;\nselp.u32 %0, 1, 0, p;\n}" : "=r"(e));
  return e != 0;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Shape constants and the shared-memory layout of one CTA (dynamic, 1024-byte aligned base).
template <int KB>
struct TcCfg {
  static constexpr int NW = (3 * KB + 15) / 16 * 16;  // N of both products (three terms of kb)
  static constexpr int SX = KB == 8 ? 6 : (KB == 16 ? 4 : 3);  // X stages
  static constexpr int SV = KB == 8 ? 6 : (KB == 16 ? 4 : 2);  // V stages
  static constexpr int NA = 3;                        // X-terms buffers
  static constexpr int NT = KB == 8 ? 2 : (KB == 16 ? 3 : 2);  // T-terms buffers
  static constexpr int G = 4;                         // tiles summed in tensor memory per W drain
  static constexpr int RG = 2;                        // row-warp groups
  static constexpr bool CS = KB == 32;                // groups split the columns (else alternate tiles)
  static constexpr int KC = CS ? KB / 2 : KB;         // right-hand sides a row group takes
  static constexpr int TARRIVE = CS ? 8 : 4;          // row warps that form each tile's T
  static constexpr int SG = KB == 8 ? 2 : 1;          // split-warp groups (alternate tiles; registers allow 2 at kb = 8)
  static constexpr int ROW0 = 2 + 4 * SG;             // first row warp
  // U's and W's products are issued by two warps, each carrying half of the product loop's
  // waits; U may then run ahead of W, so the T buffers (released by W's products) are at
  // least two, and three at kb = 16
  static constexpr int WARPS = ROW0 + 4 * RG + 2;     // producers, U products, split, row, V copies, W products
  static constexpr int THREADS = 32 * WARPS;
  static constexpr int LBO_T = (NW / 8) * 128;        // core stride along K (rows) of the T terms
  static constexpr int TBUF = TC_ROWS * NW * 2;       // bytes of one tile's T terms
  static constexpr int YBUF = NW * 192;               // bytes of the Y terms (96 x NW bfloat16)
  static constexpr int VTILE = TC_ROWS * KB * 4;      // bytes of one tile's rows of V
  static constexpr int TMEM_USED = 4 * NW;            // U and W, two of each
  static constexpr int TMEM_COLS = TMEM_USED <= 128 ? 128 : (TMEM_USED <= 256 ? 256 : 512);
  static constexpr size_t V_OFF = (size_t)SX * TC_XTILE;
  static constexpr size_t A_OFF = V_OFF + (size_t)SV * VTILE;
  static constexpr size_t T_OFF = A_OFF + (size_t)NA * TC_ABUF;
  static constexpr size_t Y_OFF = T_OFF + (size_t)NT * TBUF;
  static constexpr size_t BYTES = Y_OFF + YBUF + 1024;
  // the W products read 8 KB past the last X-terms buffer: that must stay inside the T terms
  static_assert(NT * TBUF >= 8192, "the padded A operand of W must stay in shared memory");
  static_assert(BYTES <= 220 * 1024, "shared memory");
  static_assert(3 * 32 * KB * 8 <= SX * TC_XTILE, "the final column sums reuse the X stages");
};

template <int KB>
__global__ void __launch_bounds__(TcCfg<KB>::THREADS, 1)
    dense_multi_tc_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap vmap,
                          const MultiArgs<float> a, const int vmode, const int v_tma) {
  using C = TcCfg<KB>;
  constexpr int NW = C::NW, SX = C::SX, SV = C::SV, NA = C::NA, NT = C::NT;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ __align__(8) uint64_t xfull[SX], xfree[SX], vfull[SV], vfree[SV];
  __shared__ __align__(8) uint64_t aready[NA], opfree[NA], tready[NT], tfree[NT], uready[2], ufree[2], wready[2];
  __shared__ __align__(8) uint64_t fin_bar, fin_w_bar;
  __shared__ uint32_t s_tmem;
  __shared__ int s_abort;
  volatile int* abort_word = &s_abort;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t n = a.n;
  const int kb = a.kb;
  unsigned char* xs = smem;             // SX x 16 KB of X tiles
  unsigned char* vs = smem + C::V_OFF;  // SV x rows of V
  unsigned char* as = smem + C::A_OFF;  // NA x X terms
  unsigned char* ts = smem + C::T_OFF;  // NT x T terms
  unsigned char* ys = smem + C::Y_OFF;  // Y terms

  const int64_t tiles = (a.m + TC_ROWS - 1) / TC_ROWS;
  const int64_t t0 = tiles * blockIdx.x / gridDim.x, t1 = tiles * (blockIdx.x + 1) / gridDim.x;
  const int nt = (int)(t1 - t0);
  const uint32_t vbytes = vmode == 2 ? (uint32_t)C::VTILE : (uint32_t)(TC_ROWS * 4);
  const bool v_staged = vmode != 0 && v_tma;

  // set-up: the Y terms (zero padded); barriers; tensor memory
  if (tid == 0) s_abort = 0;
  for (int e = tid; e < 96 * NW; e += C::THREADS) {
    const int kk = e / NW, col = e % NW;
    const int j = kk & 31, b = col / KB, c = col % KB;
    float y = (b < 3 && j < n && c < kb) ? a.Y[(int64_t)j * a.ldy + c] : 0.f;
    // term b of y: y1 = bf16(y), y2 = bf16(y - y1), y3 = bf16(y - y1 - y2)
    for (int t = 0; t < b && t < 3; ++t) y -= __bfloat162float(__float2bfloat16_rn(y));
    const __nv_bfloat16 yb = __float2bfloat16_rn(b < 3 ? y : 0.f);
    const size_t off = (size_t)(col >> 3) * 1536 + (size_t)(kk >> 3) * 128 + (size_t)(col & 7) * 16 + (size_t)(kk & 7) * 2;
    *reinterpret_cast<__nv_bfloat16*>(ys + off) = yb;
  }
  if (tid == 0) {
    for (int s = 0; s < SX; ++s) { mbar_init(&xfull[s], 1); mbar_init(&xfree[s], 4); }
    for (int s = 0; s < SV; ++s) { mbar_init(&vfull[s], 1); mbar_init(&vfree[s], C::TARRIVE); }
    for (int s = 0; s < NA; ++s) { mbar_init(&aready[s], 4); mbar_init(&opfree[s], 1); }
    for (int s = 0; s < NT; ++s) { mbar_init(&tready[s], C::TARRIVE); mbar_init(&tfree[s], 1); }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&uready[s], 1);
      mbar_init(&ufree[s], C::TARRIVE);
      mbar_init(&wready[s], 1);
    }
    mbar_init(&fin_bar, 1);
    mbar_init(&fin_w_bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(&s_tmem)),
                 "r"(C::TMEM_COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem;
  const uint32_t ucol = 0, wcol = 2 * NW;  // U[2] and W[2] in tensor memory
  bool ok = true;

  // compensated column sums: a row-warp thread of quarter q < 3 holds term q of X column
  // `lane` (tensor-memory lane 32 q + lane of W), for its group's right-hand sides
  CompF32 acc[C::KC];

  if (warp == 0 || warp == C::ROW0 + 4 * C::RG) {
    // ---- tensor copies: X tiles (warp 0), rows of V (the warp after the row warps) ----
    const bool is_x = warp == 0;
    if (lane == 0 && (is_x || v_staged)) {
      const uint64_t policy = policy_evict_first();
      const int S = is_x ? SX : SV;
      uint64_t* full = is_x ? xfull : vfull;
      uint64_t* freeb = is_x ? xfree : vfree;
      int issued = 0;
      // tile i + S is pulled into L2 when tile i is copied, so twice the ring's depth is in
      // flight from HBM
      auto prefetch = [&](int j) {
        const int row = (int)((t0 + j) * TC_ROWS);
        if (is_x) tma_prefetch_2d(&xmap, 0, row);
        else if (vmode == 2) tma_prefetch_2d(&vmap, 0, row);
        else tma_prefetch_2d(&vmap, row, 0);
      };
      for (int j = S; j < 2 * S && j < nt; ++j) prefetch(j);
      for (int i = 0; i < nt; ++i) {
        const int s = i % S;
        if (i >= S && !tc_wait(&freeb[s], (uint32_t)(((i / S) - 1) & 1), abort_word)) break;
        const int row0 = (int)((t0 + i) * TC_ROWS);
        if (is_x) {
          mbar_arrive_expect_tx(&full[s], TC_XTILE);
          tma_load_2d(xs + (size_t)s * TC_XTILE, &xmap, 0, row0, &full[s], policy);
        } else {
          mbar_arrive_expect_tx(&full[s], vbytes);
          if (vmode == 2) tma_load_2d(vs + (size_t)s * C::VTILE, &vmap, 0, row0, &full[s], policy);
          else tma_load_2d(vs + (size_t)s * C::VTILE, &vmap, row0, 0, &full[s], policy);
        }
        if (i >= S && i + S < nt) prefetch(i + S);
        issued = i + 1;
      }
      // copies still in flight (only after an abort): let every stage's latest one land
      for (int j = issued > S ? issued - S : 0; j < issued; ++j)
        mbar_wait_bounded(&full[j % S], (uint32_t)((j / S) & 1));
    }
  } else if (warp == 1 || warp == C::WARPS - 1) {
    // ---- the products: warp 1 issues U's, the last warp W's; each runs its loop as a
    // converged warp (the descriptors stay warp-uniform) and one elected lane issues ----
    const bool is_u = warp == 1;
    constexpr uint32_t idesc_u = tc_idesc(128, NW, 0), idesc_w = tc_idesc(128, NW, 1);
    const uint64_t a_u0 = smem_desc(smem_addr(as), 2048, 128);      // X terms, K-major (M = rows)
    const uint64_t a_w0 = smem_desc(smem_addr(as), 128, 2048);      // X terms, MN-major (M = columns)
    const uint64_t b_u0 = smem_desc(smem_addr(ys), 128, 1536);      // Y terms, K-major
    const uint64_t b_w0 = smem_desc(smem_addr(ts), C::LBO_T, 128);  // T terms, MN-major
    const bool leader = elect_one();
    auto wait_all = [&](uint64_t* bar, uint32_t parity) -> bool { return warp_wait(bar, parity, abort_word); };
    // descriptor start addresses advance in 16-byte units (no carry: shared addresses < 256 KB)
    auto issue_u = [&](int i) {
      const uint32_t d = tmem + ucol + (uint32_t)((i & 1) * NW);
      const uint64_t ad = a_u0 + (uint64_t)((i % NA) * (TC_ABUF >> 4));
      if (leader) {
#pragma unroll
        for (int s = 0; s < 6; ++s)  // K = 16 columns of the stacked X terms (blocks 2s, 2s + 1)
          tc_mma(d, ad + (uint64_t)(s * 256), b_u0 + (uint64_t)(s * 16), idesc_u, s > 0 ? 1 : 0);
        tc_commit(&uready[i & 1]);
      }
      __syncwarp();
    };
    auto issue_w = [&](int j) {
      const uint32_t d = tmem + wcol + (uint32_t)(((j / C::G) & 1) * NW);
      const uint64_t ad = a_w0 + (uint64_t)((j % NA) * (TC_ABUF >> 4));
      const uint64_t bd = b_w0 + (uint64_t)((j % NT) * (C::TBUF >> 4));
      const int first = (j % C::G) == 0;  // the group's first tile starts the sums afresh
      if (leader) {
#pragma unroll
        for (int q = 0; q < TC_ROWS / 16; ++q)  // K = 16 rows: row blocks 2q, 2q + 1
          tc_mma(d, ad + (uint64_t)(q * 16), bd + (uint64_t)(q * 2 * (C::LBO_T >> 4)), idesc_w, (q > 0 || !first) ? 1 : 0);
        tc_commit(&opfree[j % NA]);
        tc_commit(&tfree[j % NT]);
        if (j % C::G == C::G - 1 || j == nt - 1) tc_commit(&wready[(j / C::G) & 1]);
      }
      __syncwarp();
    };
    if (is_u) {
      // U of tile i once its X terms are in place and U's accumulator i % 2 has been read
      // (by the row warps, for tile i - 2)
      for (int i = 0; i < nt; ++i) {
        if (!wait_all(&aready[i % NA], (uint32_t)((i / NA) & 1))) break;
        if (i >= 2 && !wait_all(&ufree[i & 1], (uint32_t)(((i - 2) >> 1) & 1))) break;
        tc_fence_after();
        issue_u(i);
      }
    } else {
      // W of tile j once its T terms are in place
      for (int j = 0; j < nt; ++j) {
        if (!wait_all(&tready[j % NT], (uint32_t)((j / NT) & 1))) break;
        tc_fence_after();
        issue_w(j);
      }
    }
    // every product this warp issued has completed before tensor memory is released
    uint64_t* fin = is_u ? &fin_bar : &fin_w_bar;
    if (leader) tc_commit(fin);
    __syncwarp();
    mbar_wait_bounded(fin, 0);
  } else {
    // every lane of these warps takes the same branch after a wait
    auto wait_warp = [&](uint64_t* bar, uint32_t parity) -> bool { return warp_wait(bar, parity, abort_word); };
    if (warp < C::ROW0) {
      // ---- split warps ----
      const int r = 32 * ((warp - 2) & 3) + lane;
      for (int i = (warp - 2) >> 2; i < nt; i += C::SG) {
        const int s = i % SX, ob = i % NA;
        if (!(ok = wait_warp(&xfull[s], (uint32_t)((i / SX) & 1)))) break;
        if (i >= NA && !(ok = wait_warp(&opfree[ob], (uint32_t)(((i - NA) / NA) & 1)))) break;
        // the row (128-byte swizzle: chunk c of row r at c ^ (r % 8)), then the stage is free
        float x[32];
        const unsigned char* xrow = xs + (size_t)s * TC_XTILE + (size_t)r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 f = *reinterpret_cast<const float4*>(xrow + ((c ^ (r & 7)) * 16));
          x[4 * c] = f.x; x[4 * c + 1] = f.y; x[4 * c + 2] = f.z; x[4 * c + 3] = f.w;
        }
        // the stage goes back to the tensor copies at once; the proxy fence completes the row's
        // loads first (generic-proxy reads, then an async-proxy write of the same bytes)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&xfree[s]);
        unsigned char* ab = as + (size_t)ob * TC_ABUF + (size_t)r * 16;
#pragma unroll
        for (int cb = 0; cb < 4; ++cb) {
          uint32_t w1[4], w2[4], w3[4];
#pragma unroll
          for (int p = 0; p < 4; ++p) split3(x[8 * cb + 2 * p], x[8 * cb + 2 * p + 1], w1[p], w2[p], w3[p]);
          *reinterpret_cast<uint4*>(ab + (size_t)cb * 2048) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
          *reinterpret_cast<uint4*>(ab + (size_t)(4 + cb) * 2048) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
          *reinterpret_cast<uint4*>(ab + (size_t)(8 + cb) * 2048) = make_uint4(w3[0], w3[1], w3[2], w3[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&aready[ob]);
      }
    } else {
      // ---- row warps: two groups, taking alternate tiles (group 0 also drains W) or, at
      // kb = 32, every tile with half of the right-hand sides each (columns cofs .. + KC) ----
      constexpr int KC = C::KC;
      const int h = (warp - C::ROW0) >> 2;
      const int cofs = C::CS ? KC * h : 0;
      const bool drains = C::CS || h == 0;
      const int q = warp & 3;      // quarter of the tile: tensor-memory lanes 32 q ..
      const int r = 32 * q + lane;
      const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
      // the group's KC right-hand sides of the three column groups (of KB each) from tensor
      // memory at column `col`, summed by group; `f(c, sum)` folds each, c < KC
      auto sum_groups = [&](uint32_t col, auto&& f) {
        if constexpr (KB == 8) {  // groups in columns 0..7, 8..15, 16..23
          uint32_t d0[16], d1[16];
          tc_load16(lane_base + col, d0);
          tc_load16(lane_base + col + 16u, d1);
          tc_wait_ld();
#pragma unroll
          for (int c = 0; c < 8; ++c) f(c, (__uint_as_float(d0[c]) + __uint_as_float(d0[8 + c])) + __uint_as_float(d1[c]));
        } else {
#pragma unroll
          for (int c0 = 0; c0 < KC; c0 += 16) {
            uint32_t d0[16], d1[16], d2[16];
            tc_load16(lane_base + col + (uint32_t)(cofs + c0), d0);
            tc_load16(lane_base + col + (uint32_t)(KB + cofs + c0), d1);
            tc_load16(lane_base + col + (uint32_t)(2 * KB + cofs + c0), d2);
            tc_wait_ld();
#pragma unroll
            for (int c = 0; c < 16; ++c)
              f(c0 + c, (__uint_as_float(d0[c]) + __uint_as_float(d1[c])) + __uint_as_float(d2[c]));
          }
        }
      };
      // the W rows of tile group gidx (tiles G gidx .. G gidx + G - 1) into the column sums
      auto drain = [&](int gidx) -> bool {
        if (!wait_warp(&wready[gidx & 1], (uint32_t)((gidx >> 1) & 1))) return false;
        tc_fence_after();
        if (q < 3) sum_groups(wcol + (uint32_t)((gidx & 1) * NW), [&](int c, float w) { acc[c].add(w); });
        return true;
      };
      for (int i = C::CS ? 0 : h; i < nt; i += C::CS ? 1 : C::RG) {
        const int64_t row = (t0 + i) * TC_ROWS + r;
        float v[KC];
#pragma unroll
        for (int c = 0; c < KC; ++c) v[c] = 1.f;
        if (vmode != 0 && !v_tma) {  // rows of V by plain loads, issued before the waits
#pragma unroll
          for (int c = 0; c < KC; ++c)
            v[c] = row < a.m && (vmode == 1 || cofs + c < kb)
                       ? ldg(a.V + (vmode == 1 ? row : row * a.ldv + cofs + c)) : 0.f;
        }
        if (i >= NT && !(ok = wait_warp(&tfree[i % NT], (uint32_t)(((i - NT) / NT) & 1)))) break;
        if (!(ok = wait_warp(&uready[i & 1], (uint32_t)((i >> 1) & 1)))) break;
        if (v_staged) {
          const int s = i % SV;
          if (!(ok = wait_warp(&vfull[s], (uint32_t)((i / SV) & 1)))) break;
          if (vmode == 2) {
            // the stage holds 128 rows of KB fp32 in the swizzle of their width (32, 64 or
            // 128 bytes): 16-byte chunk bits 4.. of a byte offset are XORed with its bits 7..,
            // so the eight rows a quarter-warp reads land in eight distinct chunks
            constexpr uint32_t SWZ = KB == 8 ? 1u : (KB == 16 ? 3u : 7u);
            const unsigned char* vst = vs + (size_t)s * C::VTILE;
#pragma unroll
            for (int c = 0; c < KC / 4; ++c) {
              const uint32_t o = (uint32_t)(r * KB + cofs + 4 * c) * 4u;
              const float4 w = *reinterpret_cast<const float4*>(vst + (o ^ (((o >> 7) & SWZ) << 4)));
              v[4 * c] = w.x; v[4 * c + 1] = w.y; v[4 * c + 2] = w.z; v[4 * c + 3] = w.w;
            }
          } else {
            const float w = reinterpret_cast<const float*>(vs + (size_t)s * C::VTILE)[r];
#pragma unroll
            for (int c = 0; c < KC; ++c) v[c] = w;
          }
        }
        tc_fence_after();
        float t[KC];
        sum_groups(ucol + (uint32_t)((i & 1) * NW), [&](int c, float u) { t[c] = v[c] * u; });
        unsigned char* tb = ts + (size_t)(i % NT) * C::TBUF + (size_t)(r >> 3) * C::LBO_T + (size_t)(r & 7) * 16;
#pragma unroll
        for (int c8 = 0; c8 < KC; c8 += 8) {
          uint32_t w1[4], w2[4], w3[4];
#pragma unroll
          for (int p = 0; p < 4; ++p) split3(t[c8 + 2 * p], t[c8 + 2 * p + 1], w1[p], w2[p], w3[p]);
          const int cc = cofs + c8;  // T column of term 0
          *reinterpret_cast<uint4*>(tb + (size_t)(cc >> 3) * 128) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
          *reinterpret_cast<uint4*>(tb + (size_t)((KB + cc) >> 3) * 128) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
          *reinterpret_cast<uint4*>(tb + (size_t)((2 * KB + cc) >> 3) * 128) = make_uint4(w3[0], w3[1], w3[2], w3[3]);
        }
        // one proxy fence covers the T stores (read next by the products) and the V stage's
        // loads (its bytes are rewritten next by a tensor copy)
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (v_staged) mbar_arrive(&vfree[i % SV]);
          mbar_arrive(&ufree[i & 1]);
          mbar_arrive(&tready[i % NT]);
        }
        // the previous tile group's sums, once this tile group's first tile is formed (a
        // group that drains forms every tile group's first tile, so W is read before the next
        // products overwrite it)
        if (drains && i % C::G == 0 && i >= C::G && !(ok = drain(i / C::G - 1))) break;
      }
      if (ok && drains && nt > 0) ok = drain((nt - 1) / C::G);
    }
  }

  tc_fence_before();
  const bool failed = __syncthreads_or(!ok || *abort_word);
  tc_fence_after();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS));
  if (failed) return;  // FXTX_ERR_TIMEOUT is raised; OUT is not written

  // the column sums of the three X terms through shared memory into per-CTA partials
  double* red = reinterpret_cast<double*>(smem);  // [3][32][KB], over the X stages
  if (warp >= C::ROW0 && warp < C::ROW0 + 4 * C::RG && (warp & 3) < 3 && (C::CS || warp < C::ROW0 + 4)) {
    const int q = warp & 3, cofs = C::CS ? C::KC * ((warp - C::ROW0) >> 2) : 0;
#pragma unroll
    for (int c = 0; c < C::KC; ++c) red[(q * 32 + lane) * KB + cofs + c] = acc[c].value();
  }
  __syncthreads();
  const int64_t N = n * KB;
  for (int64_t e = tid; e < N; e += C::THREADS)
    a.ws[blockIdx.x * N + e] = (red[e] + red[32 * KB + e]) + red[64 * KB + e];
  __threadfence();
  __syncthreads();
  __shared__ unsigned s_last;
  if (tid == 0) s_last = (atomicAdd(a.ticket, 1u) == gridDim.x - 1) ? 1u : 0u;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int64_t e = tid; e < N; e += C::THREADS) {
    const int64_t col = e / KB;
    const int c = (int)(e % KB);
    if (c >= kb) continue;
    double w = 0.0;
    for (unsigned k = 0; k < gridDim.x; ++k) w += __ldcg(a.ws + (int64_t)k * N + e);
    double o = a.alpha * w;
    if (a.use_z) o += a.beta * (double)a.Z[col * a.ldz + c];
    a.OUT[col * a.ldo + c] = (float)o;
  }
  if (tid == 0) *a.ticket = 0u;
}

template <int KB>
cudaError_t launch_tc_kb(const MultiPlan& p, const MultiArgs<float>& a, int vmode, cudaStream_t st) {
  CUtensorMap xmap, vmap;
  memset(&xmap, 0, sizeof xmap);
  memset(&vmap, 0, sizeof vmap);
  if (!encode_rows_map(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.X, a.m, a.n, a.ld * 4, 4, TC_ROWS, 128, 128))
    return cudaErrorInvalidValue;
  // rows of V by tensor copies where V (and its pitch) allow: an m x kb block in boxes of
  // 128 rows x KB columns (columns past kb read as zero), swizzled at the rows' width, or
  // the m-vector as one row in boxes of 128 elements
  int v_tma = 0;
  const bool v_aligned = (reinterpret_cast<uintptr_t>(a.V) & 15u) == 0;
  if (vmode == 2 && v_aligned && (a.ldv * 4) % 16 == 0)
    v_tma = encode_rows_map(&vmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.V, a.m, a.kb, a.ldv * 4, 4, TC_ROWS, KB * 4,
                            KB * 4);
  else if (vmode == 1 && v_aligned)
    v_tma = encode_rows_map(&vmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, a.V, 1, a.m, (a.m * 4 + 15) / 16 * 16, 4, 1,
                            TC_ROWS * 4, 0);
  const size_t bytes = TcCfg<KB>::BYTES;
  const void* kern = (const void*)dense_multi_tc_kernel<KB>;
  cudaError_t e = ensure_smem(kern, bytes);
  if (e != cudaSuccess) return e;
  dense_multi_tc_kernel<KB><<<p.ctas, TcCfg<KB>::THREADS, bytes, st>>>(xmap, vmap, a, vmode, v_tma);
  return cudaGetLastError();
}

}  // namespace

size_t multi_tc_smem(int kb) {
  switch (kb) {
    case 8: return TcCfg<8>::BYTES;
    case 16: return TcCfg<16>::BYTES;
    case 32: return TcCfg<32>::BYTES;
    default: return 0;
  }
}

int multi_tc_warps(int kb) {
  switch (kb) {
    case 8: return TcCfg<8>::WARPS;
    case 16: return TcCfg<16>::WARPS;
    case 32: return TcCfg<32>::WARPS;
    default: return 0;
  }
}

int multi_tc_stages(int kb) {
  switch (kb) {
    case 8: return TcCfg<8>::SX;
    case 16: return TcCfg<16>::SX;
    case 32: return TcCfg<32>::SX;
    default: return 0;
  }
}

cudaError_t launch_multi_tc(const MultiPlan& p, const MultiArgs<float>& a, cudaStream_t st) {
  if (a.m <= 0 || a.n > 32 || a.kb < 1 || a.kb > p.kb_max) return cudaErrorInvalidConfiguration;
  const int vmode = a.V == nullptr ? 0 : (a.ldv == 0 ? 1 : 2);
  switch (p.kb_max) {
    case 8: return launch_tc_kb<8>(p, a, vmode, st);
    case 16: return launch_tc_kb<16>(p, a, vmode, st);
    case 32: return launch_tc_kb<32>(p, a, vmode, st);
    default: return cudaErrorInvalidConfiguration;
  }
}

}  // namespace fxtx
