// Muon's Newton-Schulz orthogonalisation on GB300 tensor cores (sm_103a).
//
// Muon needs the whole 2-D matrix at one root rank, which runs the Newton-Schulz
// iteration (feynmanwiki walkthrough of veScale-FSDP, paper section 6.3).  Per
// matrix (a tall one is iterated as its transpose):
//   X = x / (||x||_F + eps);  repeat: A = X X^T;  B = b A + c A A;  X = a X + B X
// The products run in persistent kernels: bf16 operands staged by TMA into
// 128-byte swizzled shared memory, tcgen05.mma issued by one thread into one of
// two TMEM fp32 accumulators, an epilogue reading TMEM with tcgen05.ld and
// writing D = alpha*acc + beta*C in bf16 while the next tile's products run.
// k_gemm_p (one CTA per SM, 128 x 256 tiles) runs the two symmetric products;
// A is symmetric, so A A is computed as A A^T (both operands K-major).  They run
// and store only the tiles touching the upper triangle; a product reading A or B
// takes each k-block lying below those tiles as the transpose of its stored
// partner (MN-major TMA copies and descriptors), so no lower half is ever
// written.  k_gemm_2 runs B X on pairs of CTAs (cta_group::2, 256 x 256 tiles,
// M = 256 products reading both CTAs' shared memory), X an MN-major operand.
//
// Every wait on an mbarrier is bounded: on timeout the kernel records an error
// word in the workspace, drains its own copies, frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "bq_internal.h"
#include "tmem_ptx.h"

namespace bq {
namespace {

// ---------------------------------------------------------------- tile geometry
constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr int A_STAGE = BM * BK * 2;  // 16 KB
constexpr int B_STAGE = BN * BK * 2;  // 32 KB
constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
constexpr int EPI_WARPS = 8;       // two per TMEM lane quarter, each half of a tile's columns
constexpr int GEMM_THREADS = 64 + 32 * EPI_WARPS;  // warp 0 TMA, warp 1 MMA + TMEM, then the epilogue
constexpr int GEMM_SMEM = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
constexpr long long kWaitCycles = 1ll << 32;  // ~2 s at 2 GHz
// X X^T and (A A^T with A symmetric) have symmetric results: compute and store the
// tiles touching the upper triangle only (0: every product runs whole)
#ifndef BQ_NS_SYMMETRIC
#define BQ_NS_SYMMETRIC 1
#endif
constexpr int kSymmetric = BQ_NS_SYMMETRIC;



// ---------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// bounded wait: false (and an error word) when the phase does not complete
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, int* status, int code) {
  const long long t0 = clock64();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try(bar, parity)) return true;
    if ((it & 255) == 255 && clock64() - t0 > kWaitCycles) {
      if (status) atomicExch(status, code);
      return false;
    }
  }
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}

// c MN-major 64 x 64 chunks in one copy: a 3-D map {64 columns, rows, 64-column
// chunks} (chunk stride 128 bytes) lands them 8 KB apart, the layout of c
// separate 64 x 64 boxes
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int row, int chunk, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(chunk), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

// ---------------------------------------------------------------- UMMA descriptors
// Shared-memory matrix descriptor (tcgen05): start address >> 4 in bits 0-13,
// leading-dimension byte offset >> 4 in bits 16-29, stride-dimension byte
// offset >> 4 in bits 32-45, the fixed version value 1 in bits 46-47, base
// offset 0, swizzle mode in bits 61-63 (2 = 128-byte swizzle).
//  K-major, 128B swizzle: rows of 64 bf16 (128 B), 8-row groups 1024 B apart
//    (SBO = 1024; LBO unused for this layout).  The k-th 16-element slice of a
//    row starts 32*k bytes further.
//  MN-major, 128B swizzle: each k row holds 64 MN-contiguous elements (128 B);
//    8 k rows form a 1024 B group (SBO = 1024 between groups); 64-element MN
//    chunks sit LBO apart (one TMA box of BK rows each, LBO = BK * 128 B).
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return uint64_t((addr & 0x3FFFFu) >> 4) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
         (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16 (bits
// 7-9 = 1, 10-12 = 1), A K-major (bit 15 = 0), B major in bit 16, N >> 3 in bits
// 17-22, M >> 4 in bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n, int b_mn_major, int a_mn_major = 0) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(a_mn_major) << 15) | (uint32_t(b_mn_major) << 16) |
         (uint32_t(n >> 3) << 17) | (uint32_t(m >> 4) << 24);
}

struct GemmArgs {
  int M, N, K;
  float alpha, beta;
  const __nv_bfloat16* C;  // beta term (may be null when beta == 0), row pitch ldc
  __nv_bfloat16* D;        // output, row pitch ldd
  int64_t ldc, ldd;
  int* status;
  int sym;     // D is symmetric (M == N): only the tiles touching the upper triangle run (and are stored)
  int ntiles;  // tiles that run (symmetric: those touching the upper triangle), set by the launcher
  int a_sym;   // the A operand is such a symmetric result: its tiles below the stored ones are read transposed
  int b_sym;   // the same for a K-major B operand
};

// A symmetric result is stored as the 128 x 256 output tiles that touch its
// upper triangle, each written whole; the element (r, k) of a tile that was not
// computed equals (k, r), which lies in a stored tile.  An operand box of 128
// rows from r0 and 64 columns from k0 lies in one output tile: stored or not.
__host__ __device__ __forceinline__ bool sym_stored(int r0, int k0) { return (k0 / BN) * BN + BN > r0; }

// Epilogue of one 128 x 256 tile: TMEM accumulator columns [col_base, col_base +
// 256) -> alpha * acc + beta * C -> bf16 D, the whole tile (symmetric results
// too: their tiles touching the upper triangle are stored whole, nothing is
// mirrored).  Called by the eight epilogue warps, two per TMEM lane quarter q (the
// quarter the warp may access), each for the 32-column chunks [c_lo, c_hi).
__device__ __forceinline__ void epilogue_tile(const GemmArgs& g, uint32_t tmem, uint32_t col_base, int m0, int n0,
                                              int q, int lane, int c_lo, int c_hi) {
  const int row = m0 + 32 * q + lane;
  for (int c = c_lo; c < c_hi; ++c) {
    uint32_t r[32];
    tmem_ld32(tmem + (uint32_t(32 * q) << 16) + col_base + uint32_t(32 * c), r);
    const int col0 = n0 + 32 * c;
    if (row >= g.M || col0 >= g.N) continue;
    __nv_bfloat16* drow = g.D + int64_t(row) * g.ldd;
    const __nv_bfloat16* crow = g.C ? g.C + int64_t(row) * g.ldc : nullptr;
    const bool cterm = crow && g.beta != 0.f;
    const bool cvec = cterm && col0 + 32 <= g.N && (reinterpret_cast<uintptr_t>(crow + col0) & 15) == 0;
    __nv_bfloat162 o2[16];
#pragma unroll
    for (int v = 0; v < 4; ++v) {
      float cv[8] = {0, 0, 0, 0, 0, 0, 0, 0};
      if (cvec) {
        const uint4 cw = *reinterpret_cast<const uint4*>(crow + col0 + 8 * v);
        const __nv_bfloat162* cp = reinterpret_cast<const __nv_bfloat162*>(&cw);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 f = __bfloat1622float2(cp[j]);
          cv[2 * j] = f.x;
          cv[2 * j + 1] = f.y;
        }
      } else if (cterm) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (col0 + 8 * v + j < g.N) cv[j] = __bfloat162float(crow[col0 + 8 * v + j]);
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float lo = g.alpha * __uint_as_float(r[8 * v + 2 * j]) + g.beta * cv[2 * j];
        const float hi = g.alpha * __uint_as_float(r[8 * v + 2 * j + 1]) + g.beta * cv[2 * j + 1];
        o2[4 * v + j] = __floats2bfloat162_rn(lo, hi);
      }
    }
    if (col0 + 32 <= g.N && (reinterpret_cast<uintptr_t>(drow + col0) & 15) == 0) {
#pragma unroll
      for (int v = 0; v < 4; ++v) {
        uint4 ow;
        __nv_bfloat162* op = reinterpret_cast<__nv_bfloat162*>(&ow);
#pragma unroll
        for (int j = 0; j < 4; ++j) op[j] = o2[4 * v + j];
        *reinterpret_cast<uint4*>(drow + col0 + 8 * v) = ow;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (col0 + j < g.N) drow[col0 + j] = (j & 1) ? o2[j >> 1].y : o2[j >> 1].x;
    }
  }
}

// D[M x N] = alpha * (A[M x K] . B^T) + beta * C, A and B K-major: the two
// products with symmetric results, X X^T and A A^T (B X runs on CTA pairs, below).
// One CTA per SM walks the tiles t = blockIdx.x, + gridDim.x, ... (column blocks
// fastest; symmetric results skip the tiles wholly below the diagonal).  The
// stage ring runs on across
// tiles, and two TMEM accumulators alternate so that the epilogue of one tile
// overlaps the main loop of the next: the MMA warp waits for an accumulator's
// "empty" barrier (the eight epilogue warps' arrivals) before reusing it, and
// commits its "full" barrier when the tile's products are done.
constexpr int TMEM_COLS_P = 2 * BN;

__device__ __forceinline__ void mbar_arrive_cta(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// u-th tile that runs -> (m0, n0).  Full products: every tile, column blocks
// fastest.  Symmetric results: the tiles touching the upper triangle, listed row
// block by row block (row block bm starts at column block floor(bm BM / BN)), so
// the CTAs share out only tiles with work.
__device__ __forceinline__ void tile_at(int u, int mt, int nt, int sym, int& m0, int& n0) {
  if (sym) {
    for (int bm = 0; bm < mt; ++bm) {
      const int f = (bm * BM) / BN, cnt = nt > f ? nt - f : 0;
      if (u < cnt) {
        m0 = bm * BM;
        n0 = (f + u) * BN;
        return;
      }
      u -= cnt;
    }
    m0 = n0 = 0;  // not reached: u < the launcher's tile count
    return;
  }
  m0 = (u / nt) * BM;
  n0 = (u % nt) * BN;
}

// tmA / tmB: K-major boxes of 64 columns x BM / BN rows.  With a_sym / b_sym,
// tmAt / tmBt are 3-D maps of the same matrices ({64 columns, rows, 64-column
// chunks}, boxes of 2 / 4 chunks) for the transposed (MN-major) reads of the
// k-blocks whose tiles were not stored, one copy each: a 128-row A box or
// 256-row B box of one k-block is either stored whole or not at all.
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    k_gemm_p(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
             const __grid_constant__ CUtensorMap tmAt, const __grid_constant__ CUtensorMap tmBt, GemmArgs g) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  const uint32_t bar_base = base + STAGES * STAGE_BYTES;
  auto full_bar = [&](int s) { return bar_base + 8u * uint32_t(s); };
  auto empty_bar = [&](int s) { return bar_base + 8u * uint32_t(STAGES + s); };
  auto tfull_bar = [&](int b) { return bar_base + 8u * uint32_t(2 * STAGES + b); };
  auto tempty_bar = [&](int b) { return bar_base + 8u * uint32_t(2 * STAGES + 2 + b); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + STAGES * STAGE_BYTES + 8 * (2 * STAGES + 4));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = (g.M + BM - 1) / BM, nt = (g.N + BN - 1) / BN, ntiles = g.ntiles;
  const int nk = (g.K + BK - 1) / BK;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);   // the MMA warp's commit
      mbar_init(tempty_bar(b), EPI_WARPS);  // one arrival per epilogue warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc(smem_addr(tmem_slot), TMEM_COLS_P);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer
    uint32_t it = 0;  // k-blocks issued over all tiles
    bool ok = true;
    for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
      int m0, n0;
      tile_at(t, mt, nt, g.sym, m0, n0);
      for (int kb = 0; kb < nk; ++kb, ++it) {
        const int s = int(it % STAGES);
        if (!mbar_wait(empty_bar(s), ((it / STAGES) & 1u) ^ 1u, g.status, 1)) {
          ok = false;
          break;
        }
        const uint32_t a_dst = base + uint32_t(s) * STAGE_BYTES;
        const uint32_t b_dst = a_dst + A_STAGE;
        mbar_expect_tx(full_bar(s), STAGE_BYTES);
        if (g.a_sym && !sym_stored(m0, kb * BK)) {  // rows m0.. of the k-block, read as its transpose (MN-major)
          tma_load_3d(a_dst, &tmAt, kb * BK, m0 / 64, full_bar(s));  // two 64-row chunks
        } else {
          tma_load_2d(a_dst, &tmA, kb * BK, m0, full_bar(s));
        }
        if (g.b_sym && !sym_stored(n0, kb * BK)) {  // read transposed (MN-major): four 64-row chunks
          tma_load_3d(b_dst, &tmBt, kb * BK, n0 / 64, full_bar(s));
        } else {
          tma_load_2d(b_dst, &tmB, kb * BK, n0, full_bar(s));
        }
      }
    }
    // drain: the last load issued to each stage has landed before this CTA can exit
    for (uint32_t d = it > uint32_t(STAGES) ? it - STAGES : 0; d < it; ++d)
      mbar_wait(full_bar(int(d % STAGES)), (d / STAGES) & 1u, g.status, 2);
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer
    uint32_t it = 0, tc = 0;  // k-blocks consumed, tiles done
    bool ok = true;
    for (int t = blockIdx.x; ok && t < ntiles; t += gridDim.x) {
      int m0, n0;
      tile_at(t, mt, nt, g.sym, m0, n0);
      const int buf = int(tc & 1u);
      if (tc >= 2 && !mbar_wait(tempty_bar(buf), ((tc >> 1) & 1u) ^ 1u, g.status, 5)) break;
      tc_fence_after();
      const uint32_t acc = tmem + uint32_t(buf) * BN;
      for (int kb = 0; kb < nk; ++kb, ++it) {
        const int s = int(it % STAGES);
        if (!mbar_wait(full_bar(s), (it / STAGES) & 1u, g.status, 3)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = base + uint32_t(s) * STAGE_BYTES;
        const uint32_t b_addr = a_addr + A_STAGE;
        const bool a_t = g.a_sym && !sym_stored(m0, kb * BK);
        const bool b_t = g.b_sym && !sym_stored(n0, kb * BK);
        const uint32_t id = idesc_bf16(BM, BN, b_t ? 1 : 0, a_t ? 1 : 0);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          // K-major: 16-element k slices 32 bytes apart; MN-major: 16 k rows (2 KB)
          // apart, 64-element M / N chunks one box (8 KB) apart
          const uint64_t ad = a_t ? sdesc(a_addr + uint32_t(kk) * 16u * 128u, BK * 128, 1024)
                                  : sdesc(a_addr + 32u * kk, 16, 1024);
          const uint64_t bd = b_t ? sdesc(b_addr + uint32_t(kk) * 16u * 128u, BK * 128, 1024)
                                  : sdesc(b_addr + 32u * kk, 16, 1024);
          mma_bf16(acc, ad, bd, id, (kb | kk) != 0 ? 1u : 0u);
        }
        mma_commit(empty_bar(s));
      }
      if (!ok) break;
      mma_commit(tfull_bar(buf));
      ++tc;
    }
    // every product issued here has finished before the accumulators are freed
    if (tc > 0) mbar_wait(tfull_bar(int((tc - 1) & 1u)), ((tc - 1) >> 1) & 1u, g.status, 6);
  } else if (warp >= 2) {
    // ---------------- epilogue
    const int q = warp & 3;
    uint32_t tc = 0;
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x) {
      int m0, n0;
      tile_at(t, mt, nt, g.sym, m0, n0);
      const int buf = int(tc & 1u);
      const bool ok = mbar_wait(tfull_bar(buf), (tc >> 1) & 1u, g.status, 4);
      tc_fence_after();
      if (!ok) break;
      const int half = (warp - 2) >> 2;  // warps 2-5: columns 0-127, warps 6-9: 128-255
      epilogue_tile(g, tmem, uint32_t(buf) * BN, m0, n0, q, lane, half * (BN / 64), (half + 1) * (BN / 64));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(tempty_bar(buf));
      ++tc;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS_P);
  }
}

// ---------------------------------------------------------------- CTA pairs (cta_group::2)
// B X on pairs of CTAs (clusters of two): one 256 x 256 output tile per pair.
// Each CTA stages 128 rows of the A operand and 128 columns of X for a k-block
// (32 KB instead of the single-CTA kernel's 48 KB), the pair's first CTA (the
// leader) issues M = 256 products that read both CTAs' shared memory, and each
// CTA's tensor memory receives its own 128 accumulator rows.  Half the shared
// memory per stage leaves room for six stages: more copies in flight for the same
// tensor-core work, and a third less L2 traffic.
// Barriers: the leader's `full` (both CTAs' copies complete their bytes on it),
// each CTA's `empty` and `tfull` (the leader's commits reach both CTAs), the
// leader's `tempty` (the epilogue warps of both CTAs arrive).  Every wait is
// bounded; a cluster barrier keeps either CTA from freeing its tensor memory or
// exiting while the pair's products may still use it.
constexpr int PM = 256, STAGES2 = 6;
constexpr int HALF_STAGE = 128 * BK * 2;       // 128 rows (or columns) x 64 bf16: 16 KB
constexpr int STAGE2_BYTES = 2 * HALF_STAGE;   // one CTA's part of a k-block
constexpr int GEMM2_SMEM = STAGES2 * STAGE2_BYTES + 1024 /*align*/ + 256 /*barriers*/;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// the shared::cluster address of `addr` (a shared::cta address) in CTA `rank`
__device__ __forceinline__ uint32_t map_rank(uint32_t addr, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(addr), "r"(rank));
  return a;
}

// every thread of both CTAs
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// bounded wait on a barrier that the other CTA of the pair also arrives on
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, int* status, int code) {
  const long long t0 = clock64();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_cluster(bar, parity)) return true;
    if ((it & 255) == 255 && clock64() - t0 > kWaitCycles) {
      if (status) atomicExch(status, code);
      return false;
    }
  }
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// a box into this CTA's shared memory, its bytes completed on `cluster_bar`
// (a barrier of either CTA of the pair)
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                                 uint32_t cluster_bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(cluster_bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, int row, int chunk,
                                                 uint32_t cluster_bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
      "%3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(row), "r"(chunk), "r"(cluster_bar)
      : "memory");
}

__device__ __forceinline__ void mma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// arrive on the barrier at this shared::cta offset in both CTAs once the products
// issued so far have completed
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  const uint16_t both = 3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(both)
      : "memory");
}

// made collectively by one warp of each CTA of the pair: the same columns in both
__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D = alpha * (A B) + beta * C with B given as [K x N] N-contiguous (tmB: a 3-D
// map of 64-column chunks, two chunks a copy) and A K-major (tmA: boxes of 64
// columns x 128 rows; with a_sym, tmAt's two-chunk boxes give the transposed
// reads of A's k-blocks below its stored tiles).  Pairs walk the 256 x 256 tiles t = cluster, + clusters, ..., row
// blocks fastest.  A pair tile's rows start at a multiple of 256, so its two
// 128-row halves of a k-block are stored or transposed together and one
// instruction descriptor serves both.
__global__ void __launch_bounds__(GEMM_THREADS, 1)
    k_gemm_2(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
             const __grid_constant__ CUtensorMap tmAt, GemmArgs g) {
  extern __shared__ unsigned char smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  unsigned char* gbase = smem_raw + (base - raw);
  const uint32_t bar_base = base + STAGES2 * STAGE2_BYTES;
  auto full_bar = [&](int s) { return bar_base + 8u * uint32_t(s); };
  auto empty_bar = [&](int s) { return bar_base + 8u * uint32_t(STAGES2 + s); };
  auto tfull_bar = [&](int b) { return bar_base + 8u * uint32_t(2 * STAGES2 + b); };
  auto tempty_bar = [&](int b) { return bar_base + 8u * uint32_t(2 * STAGES2 + 2 + b); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + STAGES2 * STAGE2_BYTES + 8 * (2 * STAGES2 + 4));

  const uint32_t rank = cluster_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt = (g.M + PM - 1) / PM, ntiles = g.ntiles;
  const int nk = (g.K + BK - 1) / BK;
  const int pair = int(blockIdx.x >> 1), npairs = int(gridDim.x >> 1);
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES2; ++s) {
      mbar_init(full_bar(s), 1);   // the leader's expect_tx
      mbar_init(empty_bar(s), 1);  // the leader's commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(tfull_bar(b), 1);
      mbar_init(tempty_bar(b), 2 * EPI_WARPS);  // the epilogue warps of both CTAs
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) tmem_alloc_pair(smem_addr(tmem_slot), TMEM_COLS_P);
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers exist and the columns are held before any remote use
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    // ---------------- TMA producer (both CTAs: this CTA's halves)
    uint32_t it = 0;
    bool ok = true;
    for (int t = pair; ok && t < ntiles; t += npairs) {
      const int ma = (t % mt) * PM + 128 * int(rank), nb = (t / mt) * PM + 128 * int(rank);
      for (int kb = 0; kb < nk; ++kb, ++it) {
        const int s = int(it % STAGES2);
        if (!mbar_wait(empty_bar(s), ((it / STAGES2) & 1u) ^ 1u, g.status, 11)) {
          ok = false;
          break;
        }
        const uint32_t a_dst = base + uint32_t(s) * STAGE2_BYTES;
        const uint32_t b_dst = a_dst + HALF_STAGE;
        const uint32_t fb = map_rank(full_bar(s), 0);
        if (rank == 0) mbar_expect_tx(full_bar(s), 2 * STAGE2_BYTES);
        if (g.a_sym && !sym_stored(ma, kb * BK)) {
          tma_load_3d_pair(a_dst, &tmAt, kb * BK, ma / 64, fb);  // two 64-row chunks
        } else {
          tma_load_2d_pair(a_dst, &tmA, kb * BK, ma, fb);
        }
        tma_load_3d_pair(b_dst, &tmB, kb * BK, nb / 64, fb);  // two 64-column chunks of X
      }
    }
    // drain (leader): the pair's last copies have landed; the peer waits for this
    // at the closing cluster barrier
    if (rank == 0)
      for (uint32_t d = it > uint32_t(STAGES2) ? it - STAGES2 : 0; d < it; ++d)
        mbar_wait(full_bar(int(d % STAGES2)), (d / STAGES2) & 1u, g.status, 12);
  } else if (warp == 1 && lane == 0 && rank == 0) {
    // ---------------- MMA issuer (leader)
    uint32_t it = 0, tc = 0;
    bool ok = true;
    for (int t = pair; ok && t < ntiles; t += npairs) {
      const int m0 = (t % mt) * PM;
      const int buf = int(tc & 1u);
      if (tc >= 2 && !mbar_wait_cluster(tempty_bar(buf), ((tc >> 1) & 1u) ^ 1u, g.status, 15)) break;
      tc_fence_after();
      const uint32_t acc = tmem + uint32_t(buf) * BN;
      for (int kb = 0; kb < nk; ++kb, ++it) {
        const int s = int(it % STAGES2);
        if (!mbar_wait(full_bar(s), (it / STAGES2) & 1u, g.status, 13)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_addr = base + uint32_t(s) * STAGE2_BYTES;
        const uint32_t b_addr = a_addr + HALF_STAGE;
        const bool a_t = g.a_sym && !sym_stored(m0, kb * BK);
        const uint32_t id = idesc_bf16(PM, BN, 1, a_t ? 1 : 0);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t ad = a_t ? sdesc(a_addr + uint32_t(kk) * 16u * 128u, BK * 128, 1024)
                                  : sdesc(a_addr + 32u * kk, 16, 1024);
          const uint64_t bd = sdesc(b_addr + uint32_t(kk) * 16u * 128u, BK * 128, 1024);
          mma_bf16_pair(acc, ad, bd, id, (kb | kk) != 0 ? 1u : 0u);
        }
        mma_commit_pair(empty_bar(s));
      }
      if (!ok) break;
      mma_commit_pair(tfull_bar(buf));
      ++tc;
    }
    if (tc > 0) mbar_wait(tfull_bar(int((tc - 1) & 1u)), ((tc - 1) >> 1) & 1u, g.status, 16);
  } else if (warp >= 2) {
    // ---------------- epilogue (both CTAs: this CTA's 128 rows of the tile)
    const int q = warp & 3;
    const uint32_t te0 = map_rank(tempty_bar(0), 0), te1 = map_rank(tempty_bar(1), 0);
    uint32_t tc = 0;
    for (int t = pair; t < ntiles; t += npairs) {
      const int m0 = (t % mt) * PM + 128 * int(rank), n0 = (t / mt) * PM;
      const int buf = int(tc & 1u);
      const bool ok = mbar_wait(tfull_bar(buf), (tc >> 1) & 1u, g.status, 14);
      tc_fence_after();
      if (!ok) break;
      const int half = (warp - 2) >> 2;
      epilogue_tile(g, tmem, uint32_t(buf) * BN, m0, n0, q, lane, half * (BN / 64), (half + 1) * (BN / 64));
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_remote(buf ? te1 : te0);
      ++tc;
    }
  }
  tc_fence_before();
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, TMEM_COLS_P);
  }
}

// ---------------------------------------------------------------- normalisation and copies

constexpr int kRedThreads = 256, kRedBlocks = 1024;
constexpr size_t kStatusOffset = kRedBlocks * sizeof(float);  // device error word in every workspace

// partial sums of x^2 (fp32) per block, x: rows x cols bf16 with pitch ld;
// blocks stride over rows, threads over columns
__global__ void __launch_bounds__(kRedThreads) k_sumsq(const __nv_bfloat16* __restrict__ x, int64_t rows, int64_t cols,
                                                      int64_t ld, float* __restrict__ partial) {
  float acc = 0.f;
  for (int64_t r = blockIdx.x; r < rows; r += gridDim.x) {
    const __nv_bfloat16* row = x + r * ld;
    for (int64_t c = threadIdx.x; c < cols; c += kRedThreads) {
      const float v = __bfloat162float(row[c]);
      acc = fmaf(v, v, acc);
    }
  }
  __shared__ float red[kRedThreads / 32];
  for (int o = 16; o; o >>= 1) acc += __shfl_xor_sync(0xFFFFFFFFu, acc, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < kRedThreads / 32; ++w) t += red[w];
    partial[blockIdx.x] = t;
  }
}

// 1 / (||x||_F + eps) from the partial sums (one block, fixed summation order)
__global__ void __launch_bounds__(kRedThreads) k_inv_norm(const float* __restrict__ partial, int nparts, float eps,
                                                         float* __restrict__ inv) {
  double t = 0.0;
  for (int i = threadIdx.x; i < nparts; i += kRedThreads) t += double(partial[i]);
  __shared__ double red[kRedThreads / 32];
  for (int o = 16; o; o >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = t;
  __syncthreads();
  if (threadIdx.x == 0) {
    double tot = 0.0;
    for (int w = 0; w < kRedThreads / 32; ++w) tot += red[w];
    *inv = 1.f / (sqrtf(float(tot)) + eps);
  }
}

// out = x * (*inv) (transposed when `transpose`; inv NULL: plain copy), out row
// pitch ldo.  32 x 32
// tiles through shared memory so both sides stay coalesced.
// out = bf16(x * s) (s = *inv, or 1), optionally transposed; 64 x 64 tiles, eight
// elements per thread access (16-byte vectors where the rows allow), the
// transpose through a shared-memory tile
constexpr int kCopyTile = 64;

__device__ __forceinline__ void load8(const __nv_bfloat16* __restrict__ x, int64_t r, int64_t c, int64_t rows,
                                      int64_t cols, int64_t ldx, bool vec, float s, float* v) {
  if (r < rows && vec && c + 8 <= cols) {
    const uint4 w = *reinterpret_cast<const uint4*>(x + r * ldx + c);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      v[2 * e] = f.x * s;
      v[2 * e + 1] = f.y * s;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = (r < rows && c + e < cols) ? __bfloat162float(x[r * ldx + c + e]) * s : 0.f;
  }
}

__device__ __forceinline__ void store8(__nv_bfloat16* __restrict__ out, int64_t r, int64_t c, int64_t rows,
                                       int64_t cols, int64_t ldo, bool vec, const float* v) {
  if (r >= rows) return;
  if (vec && c + 8 <= cols) {
    uint4 w;
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(v[2 * e], v[2 * e + 1]);
    *reinterpret_cast<uint4*>(out + r * ldo + c) = w;
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (c + e < cols) out[r * ldo + c + e] = __float2bfloat16_rn(v[e]);
  }
}

__global__ void __launch_bounds__(256) k_scale_copy(const __nv_bfloat16* __restrict__ x, int64_t rows, int64_t cols,
                                                   int64_t ldx, __nv_bfloat16* __restrict__ out, int64_t ldo,
                                                   int transpose, const float* __restrict__ inv) {
  const float s = inv ? *inv : 1.f;
  __shared__ float tile[kCopyTile][kCopyTile + 1];
  const int64_t r0 = int64_t(blockIdx.y) * kCopyTile, c0 = int64_t(blockIdx.x) * kCopyTile;
  const int t = threadIdx.x;
  const bool vin = (ldx & 7) == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0;
  const bool vout = (ldo & 7) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0;
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int i = (t >> 3) + 32 * pass, j = (t & 7) << 3;  // 8 threads per 64-element row
    float v[8];
    load8(x, r0 + i, c0 + j, rows, cols, ldx, vin, s, v);
    if (!transpose) {
      store8(out, r0 + i, c0 + j, rows, cols, ldo, vout, v);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) tile[i][j + e] = v[e];
    }
  }
  if (!transpose) return;  // uniform
  __syncthreads();
  // out is cols x rows: its row c0 + i holds tile column i
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int i = (t >> 3) + 32 * pass, j = (t & 7) << 3;
    float v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) v[e] = tile[j + e][i];
    store8(out, c0 + i, r0 + j, cols, rows, ldo, vout, v);
  }
}

int check(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(BQ_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
  return BQ_OK;
}

// ---------------------------------------------------------------- tensor maps (driver entry point at run time)

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                 const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                 CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled encoder() {
  static EncodeTiled fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiled>(p);
  });
  return fn;
}

// 2-D bf16 tensor map: inner extent `inner` (contiguous), outer extent `outer`,
// row pitch `ld` elements, box inner 64 (128 bytes, the swizzle span) x box_outer
int make_map(CUtensorMap* m, const void* ptr, int64_t inner, int64_t outer, int64_t ld, int box_outer) {
  EncodeTiled enc = encoder();
  if (!enc) return set_error(BQ_EDEVICE, "bq_muon_ns: cuTensorMapEncodeTiled unavailable");
  const cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
  const cuuint64_t strides[1] = {cuuint64_t(ld) * 2};
  const cuuint32_t box[2] = {64u, cuuint32_t(box_outer)};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(BQ_EINVAL, "bq_muon_ns: tensor map encoding failed (" + std::to_string(int(r)) + ")");
  return BQ_OK;
}

// The same matrix as MN-major chunks: {64 columns, rows, ceil(cols / 64) chunks}
// with the chunk stride 128 bytes, boxes of 64 x 64 x `chunks` (a copy brings
// that many consecutive 64-column chunks of 64 rows).  Columns past `cols` inside
// the last chunk come from the row padding: they only reach output rows or
// columns past the matrix, which are never stored; rows past `rows` read as 0.
int make_map3(CUtensorMap* m, const void* ptr, int64_t cols, int64_t rows, int64_t ld, int chunks) {
  EncodeTiled enc = encoder();
  if (!enc) return set_error(BQ_EDEVICE, "bq_muon_ns: cuTensorMapEncodeTiled unavailable");
  const cuuint64_t dims[3] = {64u, cuuint64_t(rows), cuuint64_t((cols + 63) / 64)};
  const cuuint64_t strides[2] = {cuuint64_t(ld) * 2, 128u};
  const cuuint32_t box[3] = {64u, 64u, cuuint32_t(chunks)};
  const cuuint32_t estr[3] = {1u, 1u, 1u};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return set_error(BQ_EINVAL, "bq_muon_ns: tensor map encoding failed (" + std::to_string(int(r)) + ")");
  return BQ_OK;
}

int64_t pitch_of(int64_t cols) { return (cols + 63) / 64 * 64; }  // 128-byte rows

struct NsPlan {
  int64_t m, n;        // iterated shape (m <= n)
  bool tall;
  int64_t ldx, lda;    // pitches of X (m x n) and A, B (m x m)
  size_t off_part, off_status, off_x0, off_x1, off_a, off_b, bytes;
};

NsPlan ns_plan(const bq_mat& t) {
  NsPlan p;
  p.tall = t.rows > t.cols;
  p.m = p.tall ? t.cols : t.rows;
  p.n = p.tall ? t.rows : t.cols;
  p.ldx = pitch_of(p.n);
  p.lda = pitch_of(p.m);
  size_t o = 0;
  p.off_part = o;
  o += kRedBlocks * sizeof(float);
  p.off_status = o;  // == kStatusOffset for every matrix
  o += 256;
  p.off_x0 = o;
  o += size_t(p.m) * p.ldx * 2;
  o = (o + 1023) / 1024 * 1024;
  p.off_x1 = o;
  o += size_t(p.m) * p.ldx * 2;
  o = (o + 1023) / 1024 * 1024;
  p.off_a = o;
  o += size_t(p.m) * p.lda * 2;
  o = (o + 1023) / 1024 * 1024;
  p.off_b = o;
  o += size_t(p.m) * p.lda * 2;
  p.bytes = (o + 1023) / 1024 * 1024;
  return p;
}

int check_mat(const bq_mat& t) {
  if (!t.x || !t.y || t.rows < 1 || t.cols < 1 || t.ld_x < t.cols || t.ld_y < t.cols)
    return set_error(BQ_EINVAL, "bq_muon_ns: bad matrix descriptor");
  if (t.rows > (int64_t(1) << 20) || t.cols > (int64_t(1) << 20) || t.rows * t.cols > (int64_t(1) << 31))
    return set_error(BQ_EINVAL, "bq_muon_ns: matrix too large");
  if ((reinterpret_cast<uintptr_t>(t.x) | reinterpret_cast<uintptr_t>(t.y)) & 1)
    return set_error(BQ_EALIGN, "bq_muon_ns: matrices must be 2-byte aligned");
  return BQ_OK;
}

// the GEMM kernels' shared-memory attributes, set once per device (they belong
// to the current device)
int gemm_attrs() {
  if (once_per_device(kOnceGemmAttr) &&
      (cudaFuncSetAttribute(k_gemm_p, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM_SMEM) != cudaSuccess ||
       cudaFuncSetAttribute(k_gemm_2, cudaFuncAttributeMaxDynamicSharedMemorySize, GEMM2_SMEM) != cudaSuccess))
    return check("bq_muon_ns (gemm shared memory attributes)");
  return BQ_OK;
}

int gemm(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tat, const CUtensorMap& tbt,
         const GemmArgs& g, cudaStream_t s) {
  if (int rc = gemm_attrs()) return rc;
  const int mt = (g.M + BM - 1) / BM, nt = (g.N + BN - 1) / BN;
  GemmArgs a = g;
  a.ntiles = mt * nt;
  if (g.sym) {  // the same count tile_at lists
    a.ntiles = 0;
    for (int bm = 0; bm < mt; ++bm) a.ntiles += std::max(0, nt - (bm * BM) / BN);
  }
  if (a.ntiles == 0) return BQ_OK;
  const unsigned grid = unsigned(std::min(a.ntiles, sm_count()));
  k_gemm_p<<<grid, GEMM_THREADS, GEMM_SMEM, s>>>(ta, tb, tat, tbt, a);
  return check("bq_muon_ns (gemm)");
}

// Clusters of two k_gemm_2 CTAs that fit the device at once (cached per device;
// half the SMs if the occupancy query fails)
int pair_slots() {
  static std::mutex mu;
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return sm_count() / 2;
  std::lock_guard<std::mutex> lock(mu);
  if (cached[dev] == 0) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(unsigned(2 * sm_count()));
    cfg.blockDim = dim3(GEMM_THREADS);
    cfg.dynamicSmemBytes = GEMM2_SMEM;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k_gemm_2, &cfg) != cudaSuccess || n < 1) {
      cudaGetLastError();
      n = sm_count() / 2;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

// B X on CTA pairs: A K-major (ta; tat for the transposed k-blocks of a symmetric
// A), B [K x N] N-contiguous (tb)
int gemm_pair(const CUtensorMap& ta, const CUtensorMap& tb, const CUtensorMap& tat, const GemmArgs& g,
              cudaStream_t s) {
  if (int rc = gemm_attrs()) return rc;
  GemmArgs a = g;
  a.ntiles = ((g.M + PM - 1) / PM) * ((g.N + PM - 1) / PM);
  if (a.ntiles == 0) return BQ_OK;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute at[1];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(unsigned(2 * std::min(a.ntiles, pair_slots())));
  cfg.blockDim = dim3(GEMM_THREADS);
  cfg.dynamicSmemBytes = GEMM2_SMEM;
  cfg.stream = s;
  cfg.attrs = at;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, k_gemm_2, ta, tb, tat, a) != cudaSuccess) return check("bq_muon_ns (pair gemm)");
  return check("bq_muon_ns (pair gemm)");
}

// Matrix i's workspace region in the concurrent layout starts at region_off[i]
// (1024-byte multiples; region 0 at 0 holds the batch's error word).
size_t concurrent_bytes(int batch, const bq_mat* mats, std::vector<size_t>* region_off) {
  size_t o = 0;
  for (int i = 0; i < batch; ++i) {
    if (region_off) region_off->push_back(o);
    o += (ns_plan(mats[i]).bytes + 1023) / 1024 * 1024;
  }
  return std::max<size_t>(o, 256);
}

// One matrix's whole Newton-Schulz on stream s: workspace region w (its own
// scratch), error word `status` (the batch's).
int ns_one(const bq_mat& t, unsigned char* w, int* status, int steps, float a, float b, float c, float eps,
           cudaStream_t s) {
  const NsPlan p = ns_plan(t);
  float* part = reinterpret_cast<float*>(w + p.off_part);
  float* inv = reinterpret_cast<float*>(w + p.off_status + 16);  // 1 / (||x||_F + eps)
  auto* X0 = reinterpret_cast<__nv_bfloat16*>(w + p.off_x0);
  auto* X1 = reinterpret_cast<__nv_bfloat16*>(w + p.off_x1);
  auto* A = reinterpret_cast<__nv_bfloat16*>(w + p.off_a);
  auto* B = reinterpret_cast<__nv_bfloat16*>(w + p.off_b);
  const auto* x = static_cast<const __nv_bfloat16*>(t.x);
  auto* y = static_cast<__nv_bfloat16*>(t.y);

  // normalise into X0 (transposed for a tall input)
  k_sumsq<<<kRedBlocks, kRedThreads, 0, s>>>(x, t.rows, t.cols, t.ld_x, part);
  if (int rc = check("bq_muon_ns (norm)")) return rc;
  const dim3 cg(unsigned((t.cols + kCopyTile - 1) / kCopyTile), unsigned((t.rows + kCopyTile - 1) / kCopyTile));
  k_inv_norm<<<1, kRedThreads, 0, s>>>(part, kRedBlocks, eps, inv);
  if (int rc = check("bq_muon_ns (inv norm)")) return rc;
  k_scale_copy<<<cg, 256, 0, s>>>(x, t.rows, t.cols, t.ld_x, X0, p.ldx, p.tall ? 1 : 0, inv);
  if (int rc = check("bq_muon_ns (scale)")) return rc;

  // tensor maps: X as K-major A operand / K-major B operand / MN-major B operand
  // (two 64-column chunks a copy: a pair CTA's 128 columns), A and B K-major, and
  // A, B as MN-major chunks for the transposed reads (two chunks: a 128-row A
  // operand box; four: a 256-row B operand box)
  CUtensorMap mXa[2], mXb[2], mXmn[2], mAa, mAb, mAmn2, mAmn4, mBa, mBmn2;
  __nv_bfloat16* Xs[2] = {X0, X1};
  for (int j = 0; j < 2; ++j) {
    if (int rc = make_map(&mXa[j], Xs[j], p.n, p.m, p.ldx, BM)) return rc;
    if (int rc = make_map(&mXb[j], Xs[j], p.n, p.m, p.ldx, BN)) return rc;
    if (int rc = make_map3(&mXmn[j], Xs[j], p.n, p.m, p.ldx, 2)) return rc;
  }
  if (int rc = make_map(&mAa, A, p.m, p.m, p.lda, BM)) return rc;
  if (int rc = make_map(&mAb, A, p.m, p.m, p.lda, BN)) return rc;
  if (int rc = make_map3(&mAmn2, A, p.m, p.m, p.lda, 2)) return rc;
  if (int rc = make_map3(&mAmn4, A, p.m, p.m, p.lda, 4)) return rc;
  if (int rc = make_map(&mBa, B, p.m, p.m, p.lda, BM)) return rc;
  if (int rc = make_map3(&mBmn2, B, p.m, p.m, p.lda, 2)) return rc;

  int cur = 0;
  for (int it = 0; it < steps; ++it) {
    const int nxt = cur ^ 1;
    // A = X X^T (symmetric: the tiles touching the upper triangle)
    GemmArgs g1{int(p.m), int(p.m), int(p.n), 1.f, 0.f, nullptr, A, 0, p.lda, status, kSymmetric, 0, 0, 0};
    if (int rc = gemm(mXa[cur], mXb[cur], mXa[cur], mXa[cur], g1, s)) return rc;
    // B = c (A A^T) + b A   (A symmetric and stored as such: both operands read it)
    GemmArgs g2{int(p.m), int(p.m), int(p.m), c, b, A, B, p.lda, p.lda, status, kSymmetric, 0, kSymmetric, kSymmetric};
    if (int rc = gemm(mAa, mAb, mAmn2, mAmn4, g2, s)) return rc;
    // X' = B X + a X   (B symmetric and stored as such)
    GemmArgs g3{int(p.m), int(p.n), int(p.m), 1.f, a, Xs[cur], Xs[nxt], p.ldx, p.ldx, status, 0, 0, kSymmetric, 0};
    if (int rc = gemm_pair(mBa, mXmn[cur], mBmn2, g3, s)) return rc;
    cur = nxt;
  }
  // y = X (transposed back for a tall input)
  const dim3 og(unsigned((p.n + kCopyTile - 1) / kCopyTile), unsigned((p.m + kCopyTile - 1) / kCopyTile));
  k_scale_copy<<<og, 256, 0, s>>>(Xs[cur], p.m, p.n, p.ldx, y, t.ld_y, p.tall ? 1 : 0, nullptr);
  return check("bq_muon_ns (copy out)");
}

// The library's own side streams of the current device, forked from and joined
// back to the caller's stream so that independent matrices of a batch fill one
// another's idle SMs (the last wave of one matrix's product leaves SMs that the
// next matrix's products use).  Created once per device; NULL when unavailable.
constexpr int kNsStreams = 3;
struct SidePool {
  cudaStream_t st[kNsStreams];
  cudaEvent_t fork, join[kNsStreams];
  std::mutex mu;  // one batch at a time enqueues on the pool
  bool ok = false;
};

SidePool* side_pool() {
  static std::mutex mu;
  static SidePool* pools[64] = {};
  static bool tried[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!tried[dev]) {
    tried[dev] = true;
    auto* p = new SidePool();
    bool ok = cudaEventCreateWithFlags(&p->fork, cudaEventDisableTiming) == cudaSuccess;
    for (int j = 0; ok && j < kNsStreams; ++j)
      ok = cudaStreamCreateWithFlags(&p->st[j], cudaStreamNonBlocking) == cudaSuccess &&
           cudaEventCreateWithFlags(&p->join[j], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      delete p;  // the handles already made stay with the context; the batch runs in order instead
      return nullptr;
    }
    p->ok = true;
    pools[dev] = p;
  }
  return pools[dev];
}

int run_batch(int batch, const bq_mat* mats, int steps, float a, float b, float c, float eps, void* ws,
              size_t ws_bytes, void* stream, bool allow_side) {
  if (batch < 0 || (batch > 0 && !mats) || steps < 0) return set_error(BQ_EINVAL, "bq_muon_ns: bad arguments");
  if (batch > 0 && (!ws || (reinterpret_cast<uintptr_t>(ws) & 255)))
    return set_error(BQ_EALIGN, "bq_muon_ns: workspace must be 256-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // every matrix is checked before any work is queued
  for (int i = 0; i < batch; ++i) {
    if (int rc = check_mat(mats[i])) return rc;
    if (ws_bytes < ns_plan(mats[i]).bytes) return set_error(BQ_ENOSPC, "bq_muon_ns: workspace too small");
  }
  if (batch == 0) return BQ_OK;
  auto* w = static_cast<unsigned char*>(ws);
  int* status = reinterpret_cast<int*>(w + kStatusOffset);
  // the device error word is cleared once per call, so a wait that gave up on
  // any matrix of the batch stays recorded (report() keeps the first site)
  if (cudaMemsetAsync(status, 0, sizeof(int), s) != cudaSuccess) return check("bq_muon_ns (status)");
  std::vector<size_t> off;
  const size_t conc = concurrent_bytes(batch, mats, &off);
  SidePool* pool = (allow_side && batch > 1 && ws_bytes >= conc) ? side_pool() : nullptr;
  if (!pool) {  // one matrix after another on the caller's stream, one region reused
    for (int i = 0; i < batch; ++i)
      if (int rc = ns_one(mats[i], w, status, steps, a, b, c, eps, s)) return rc;
    return BQ_OK;
  }
  // matrices on the side streams, largest first to the least loaded stream
  std::lock_guard<std::mutex> lock(pool->mu);
  std::vector<int> order(static_cast<size_t>(batch));
  std::vector<double> cost(static_cast<size_t>(batch));
  for (int i = 0; i < batch; ++i) {
    const double m = double(std::min(mats[i].rows, mats[i].cols)), n = double(std::max(mats[i].rows, mats[i].cols));
    cost[size_t(i)] = 4 * m * m * n + 2 * m * m * m;
    order[size_t(i)] = i;
  }
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return cost[size_t(x)] > cost[size_t(y)]; });
  double load[kNsStreams] = {};
  if (cudaEventRecord(pool->fork, s) != cudaSuccess) return check("bq_muon_ns (fork)");
  for (int j = 0; j < kNsStreams; ++j)
    if (cudaStreamWaitEvent(pool->st[j], pool->fork, 0) != cudaSuccess) return check("bq_muon_ns (fork)");
  int rc = BQ_OK;
  for (int i : order) {
    int j = 0;
    for (int k = 1; k < kNsStreams; ++k)
      if (load[k] < load[j]) j = k;
    load[j] += cost[size_t(i)];
    rc = ns_one(mats[i], w + off[size_t(i)], status, steps, a, b, c, eps, pool->st[j]);
    if (rc != BQ_OK) break;  // what was queued is still joined below
  }
  for (int j = 0; j < kNsStreams; ++j) {  // join every stream that waited on the fork
    if (cudaEventRecord(pool->join[j], pool->st[j]) != cudaSuccess ||
        cudaStreamWaitEvent(s, pool->join[j], 0) != cudaSuccess)
      return rc != BQ_OK ? rc : check("bq_muon_ns (join)");
  }
  return rc;
}

}  // namespace

int muon_ns_workspace(int batch, const bq_mat* mats, size_t* bytes) {
  if (!bytes || batch < 0 || (batch > 0 && !mats)) return set_error(BQ_EINVAL, "bq_muon_ns_workspace: bad arguments");
  for (int i = 0; i < batch; ++i)
    if (int rc = check_mat(mats[i])) return rc;
  *bytes = concurrent_bytes(batch, mats, nullptr);
  return BQ_OK;
}

int encode_map_2d(void* map, const void* base, int elem_bytes, int64_t cols, int64_t rows, int box_cols, int box_rows) {
  EncodeTiled enc = encoder();
  if (!enc) return BQ_EDEVICE;
  const CUtensorMapDataType dt = elem_bytes == 4   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                                   : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const cuuint64_t dims[2] = {cuuint64_t(cols), cuuint64_t(rows)};
  const cuuint64_t strides[1] = {cuuint64_t(cols) * cuuint64_t(elem_bytes)};
  const cuuint32_t box[2] = {cuuint32_t(box_cols), cuuint32_t(box_rows)};
  const cuuint32_t estr[2] = {1u, 1u};
  const CUresult r = enc(static_cast<CUtensorMap*>(map), dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? BQ_OK : BQ_EINVAL;
}

int muon_ns(int batch, const bq_mat* mats, int steps, float a, float b, float c, float eps, void* ws, size_t ws_bytes,
            void* stream) {
  return run_batch(batch, mats, steps, a, b, c, eps, ws, ws_bytes, stream, true);
}

// ---------------------------------------------------------------- allocation-free variant
// Some callers cannot allocate device memory at the point where they run the
// optimizer step: runtimes that reserve every byte of the GPU up front and
// forbid later cudaMalloc calls, plug-ins inside a host framework that owns the
// allocator, or code paths that must not allocate for latency reasons.  They use
// bq_muon_ns_noalloc, whose scratch is this fixed array in the library's device
// image: every GPU that loads the library holds it until the process exits.
constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_ns_scratch[kStaticScratchBytes];

// The array's device address on the current device, looked up once per device
// with that device current (in host code the symbol is only a stand-in, not a
// device address).  The cache is never refreshed: after cudaDeviceReset the
// address may be stale.
int static_scratch(void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64)
    return set_error(BQ_EDEVICE, "bq_muon_ns_noalloc: no usable current device");
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_ns_scratch);
    if (e != cudaSuccess || !p)
      return set_error(BQ_ECUDA, std::string("bq_muon_ns_noalloc: scratch address lookup failed: ") +
                                     cudaGetErrorString(e));
    addr[dev] = p;
  }
  *out = addr[dev];
  return BQ_OK;
}

int muon_ns_noalloc(int batch, const bq_mat* mats, int steps, float a, float b, float c, float eps, void* stream) {
  void* scratch = nullptr;
  if (int rc = static_scratch(&scratch)) return rc;
  if (batch < 0 || (batch > 0 && !mats)) return set_error(BQ_EINVAL, "bq_muon_ns_noalloc: bad arguments");
  size_t need = 256;  // the matrices run one after another and reuse one region
  for (int i = 0; i < batch; ++i) {
    if (int rc = check_mat(mats[i])) return rc;
    need = std::max(need, ns_plan(mats[i]).bytes);
  }
  if (need > kStaticScratchBytes)
    return set_error(BQ_ENOSPC, "bq_muon_ns_noalloc: the batch needs " + std::to_string(need) +
                                    " bytes of scratch; the static scratch holds " +
                                    std::to_string(kStaticScratchBytes) + " (use bq_muon_ns with a workspace)");
  return run_batch(batch, mats, steps, a, b, c, eps, scratch, kStaticScratchBytes, stream, false);
}

// ws == NULL: the static scratch of the current device (bq_muon_ns_noalloc)
int muon_ns_check(const void* ws, size_t ws_bytes, void* stream) {
  if (!ws) {
    void* scratch = nullptr;
    if (int rc = static_scratch(&scratch)) return rc;
    ws = scratch;
    ws_bytes = kStaticScratchBytes;
  }
  if (ws_bytes < kStatusOffset + sizeof(int)) return set_error(BQ_EINVAL, "bq_muon_ns_check: bad workspace");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int status = 0;
  cudaError_t e = cudaStreamSynchronize(s);
  if (e == cudaSuccess)
    e = cudaMemcpy(&status, static_cast<const unsigned char*>(ws) + kStatusOffset, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return set_error(BQ_ECUDA, std::string("bq_muon_ns_check: ") + cudaGetErrorString(e));
  if (status) return set_error(BQ_ECUDA, "bq_muon_ns: a device wait timed out (site " + std::to_string(status) + ")");
  return BQ_OK;
}

}  // namespace bq
