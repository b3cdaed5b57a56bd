// Memory-bound kernels of the DBuffer step on GB300 (sm_103a):
//   k_pack         fused pre-communication copy / scale / add / zero into the
//                  bf16 gradient DBuffer (DBuffer's group-level pre-comm ops,
//                  veScale-FSDP bud-325 summary, Key claims and Method)
//   k_flat<E>      8-bit Adam over runs of flat blocks (256 or 128 elements),
//                  optionally fused with 1x128 FP8 tiles of 1-D tensors
//   k_strip<FP8>   8-bit Adam with flat 256-element blocks over a 2-D region,
//                  fused with 128x128 FP8 tiles (two phases, tile amax in smem)
//   k_tile<FP8>    8-bit Adam with 128x128 state tiles (+ FP8 of the same tile)
//   k_quant_*      standalone FP8 requantisation
// The 8-bit Adam is the pages' block-quantised optimizer state kept local to a
// shard (feynmanwiki walkthrough, paper section 6.3); FP8 is block-wise FP8 in
// the DeepSeek-V3 style (bud-325 TL;DR).
//
// Every value-producing fp32 operation uses an explicit round-to-nearest
// intrinsic (no contraction into FMA), in the order the host-side contract fixes,
// so codes, scales and master weights are reproducible bit for bit.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "bq_internal.h"

namespace bq {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
// resident CTAs per SM the Adam kernels are compiled for (register budget) and
// launched with (grid-stride kernels)
#ifndef BQ_ADAM_CTAS_PER_SM
#define BQ_ADAM_CTAS_PER_SM 3
#endif
constexpr int kAdamCtas = BQ_ADAM_CTAS_PER_SM;

// ---------------------------------------------------------------- element helpers

__device__ __forceinline__ float bf16f(uint32_t bits16) { return __uint_as_float(bits16 << 16); }

__device__ __forceinline__ uint32_t f2bf(float x) {
  return uint32_t(__bfloat16_as_ushort(__float2bfloat16_rn(x)));
}

struct Hp {
  float lr, b1, b2, eps, omb1, omb2, rbc1, rbc2;
};

__device__ __forceinline__ Hp make_hp(const bq_adam_hp& h) {
  return Hp{h.lr, h.b1, h.b2, h.eps, h.omb1, h.omb2, h.rbc1, h.rbc2};
}

// Blackwell's packed fp32 pair arithmetic: each component is rounded exactly
// like the scalar round-to-nearest operation.  A packed add takes no product as
// an operand anywhere below: ptxas contracts a packed multiply feeding a packed
// add into a fused multiply-add even when both carry an explicit .rn, so every
// multiply-then-add is written as the explicit fused operation the contract
// specifies.
__device__ __forceinline__ float2 dup(float x) { return make_float2(x, x); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }  // operands never products
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

// The Adam update of two elements; per element, each step one IEEE fp32
// operation rounded to nearest, fma(x, y, z) = x*y + z rounded once:
//   m' = fma(b1, m, omb1*g);  v' = fma(b2, v, omb2*(g*g));  mh = m'*rbc1;
//   vh = v'*rbc2;  u = mh/(sqrt(vh)+eps);  p' = fma(-lr, u, p)
__device__ __forceinline__ void adam_pair(const Hp& h, float2 g, float2 p, float2 qm, float2 qv, float2 sm, float2 sv,
                                          float2& p1, float2& m1, float2& v1) {
  const float2 m = mul2(qm, sm), v = mul2(qv, sv);
  m1 = fma2(dup(h.b1), m, mul2(dup(h.omb1), g));
  v1 = fma2(dup(h.b2), v, mul2(dup(h.omb2), mul2(g, g)));
  const float2 mh = mul2(m1, dup(h.rbc1)), vh = mul2(v1, dup(h.rbc2));
  const float2 den = add2(make_float2(__fsqrt_rn(vh.x), __fsqrt_rn(vh.y)), dup(h.eps));
  const float2 u = make_float2(__fdiv_rn(mh.x, den.x), __fdiv_rn(mh.y, den.y));
  p1 = fma2(dup(-h.lr), u, p);
}

// Block scale from an absmax (fp32 bits; all values >= 0 so bit order == value
// order): stored scale s = amax/qmax, reciprocal r = qmax/amax (one division each
// per block).  mode 0: s == 0 -> zero codes; 1: codes from x*r; 2: r overflowed
// (tiny amax) -> codes from x/s.
struct QScale {
  float s, r;
  int mode;
};

__device__ __forceinline__ QScale qscale(uint32_t amax_bits, float qmax) {
  const float a = __uint_as_float(amax_bits);
  QScale q;
  q.s = __fdiv_rn(a, qmax);
  q.r = __fdiv_rn(qmax, a);
  q.mode = q.s == 0.f ? 0 : (isinf(q.r) ? 2 : 1);
  return q;
}

// Exact small-integer conversions without I2F / F2I:
//  * a byte b placed in the low mantissa bits of 2^23 (bit pattern 0x4B0000bb)
//    is the float 2^23 + b, so subtracting 2^23 gives float(b) exactly (a signed
//    byte is first offset by 128 by flipping its top bit);
//  * for |y| < 2^22, y + 1.5*2^23 rounds y to the nearest integer, ties to even
//    (the add's own rounding; with y = x*r inside one fused multiply-add the
//    exact product is rounded), and the low byte of the sum's bit pattern is that
//    integer modulo 256 (two's complement for negative values).
__device__ __forceinline__ float2 byte_pair(uint32_t w, int i, float bias) {
  const float2 t = make_float2(__uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u | uint32_t(i))),
                               __uint_as_float(__byte_perm(w, 0x4B000000u, 0x7540u | uint32_t(i + 1))));
  return add2(t, dup(-bias));
}

// low bytes of four words -> one word
__device__ __forceinline__ uint32_t low_bytes(uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  return __byte_perm(__byte_perm(a, b, 0x0040u), __byte_perm(c, d, 0x0040u), 0x5410u);
}

// 8 int8 codes, packed little-endian into two words.  On the reciprocal path
// fma(x, r, 1.5*2^23) = 1.5*2^23 + rint(x*r) with the exact product rounded once
// to an integer; |x * r| <= 127 (1 + 2^-23) because |x| <= amax, so that integer
// already lies in [-127, 127] and needs no clamp.  The division path (tiny
// blocks, whose subnormal scale may be inexact) rounds x/s and clamps.
__device__ __forceinline__ uint2 codes_int8(const float* x, const QScale& q) {
  if (q.mode == 0) return make_uint2(0u, 0u);
  uint32_t b[8];
  if (q.mode == 1) {
    const float2 r = dup(q.r), k = dup(12582912.f);
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      const float2 y = fma2(make_float2(x[i], x[i + 1]), r, k);  // K + rint(x*r), the product unrounded
      b[i] = __float_as_uint(y.x);
      b[i + 1] = __float_as_uint(y.y);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      b[i] = __float_as_uint(__fadd_rn(fminf(fmaxf(__fdiv_rn(x[i], q.s), -127.f), 127.f), 12582912.f));
  }
  return make_uint2(low_bytes(b[0], b[1], b[2], b[3]), low_bytes(b[4], b[5], b[6], b[7]));
}

// 8 uint8 codes (v' >= 0); same reasoning, range [0, 255]
__device__ __forceinline__ uint2 codes_uint8(const float* x, const QScale& q) {
  if (q.mode == 0) return make_uint2(0u, 0u);
  uint32_t b[8];
  if (q.mode == 1) {
    const float2 r = dup(q.r), k = dup(8388608.f);
#pragma unroll
    for (int i = 0; i < 8; i += 2) {
      const float2 y = fma2(make_float2(x[i], x[i + 1]), r, k);
      b[i] = __float_as_uint(y.x);
      b[i + 1] = __float_as_uint(y.y);
    }
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      b[i] = __float_as_uint(__fadd_rn(fminf(fmaxf(__fdiv_rn(x[i], q.s), 0.f), 255.f), 8388608.f));
  }
  return make_uint2(low_bytes(b[0], b[1], b[2], b[3]), low_bytes(b[4], b[5], b[6], b[7]));
}

// 8 E4M3 codes (round to nearest even, saturating); scale 0 keeps each sign
__device__ __forceinline__ uint2 codes_e4m3(const float* x, const QScale& q) {
  uint32_t w[4];
  if (q.mode == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = ((__float_as_uint(x[2 * i]) >> 24) & 0x80u) | ((__float_as_uint(x[2 * i + 1]) >> 16) & 0x8000u);
  } else if (q.mode == 1) {
    const float2 r = dup(q.r);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = uint32_t(__nv_cvt_float2_to_fp8x2(mul2(make_float2(x[2 * i], x[2 * i + 1]), r), __NV_SATFINITE, __NV_E4M3));
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i)
      w[i] = uint32_t(__nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(x[2 * i], q.s), __fdiv_rn(x[2 * i + 1], q.s)),
                                               __NV_SATFINITE, __NV_E4M3));
  }
  return make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

__device__ __forceinline__ void store_p8(float* dst, const float* p) {
  reinterpret_cast<float4*>(dst)[0] = make_float4(p[0], p[1], p[2], p[3]);
  reinterpret_cast<float4*>(dst)[1] = make_float4(p[4], p[5], p[6], p[7]);
}

// ---------------------------------------------------------------- pack

__global__ void __launch_bounds__(kThreads) k_pack(const PackPiece* __restrict__ pieces,
                                                   const int32_t* __restrict__ chunk_first,
                                                   const uint16_t* const* __restrict__ grads,
                                                   uint16_t* __restrict__ dst, float scale, int accumulate) {
  const int64_t c = blockIdx.x;
  const int p0 = chunk_first[c], p1 = chunk_first[c + 1];
  for (int p = p0; p < p1; ++p) {
    const PackPiece pc = pieces[p];
    uint16_t* d = dst + pc.dst;
    if (pc.tensor < 0) {  // padding := +0
      if ((pc.dst & 7) == 0) {
        const int nv = pc.len >> 3;
        for (int v = threadIdx.x; v < nv; v += kThreads) reinterpret_cast<uint4*>(d)[v] = make_uint4(0, 0, 0, 0);
        for (int e = (nv << 3) + threadIdx.x; e < pc.len; e += kThreads) d[e] = 0;
      } else {
        for (int e = threadIdx.x; e < pc.len; e += kThreads) d[e] = 0;
      }
      continue;
    }
    const uint16_t* s = grads[pc.tensor] + pc.src;
    // vector path only when both sides sit on 16-byte boundaries (the source
    // pointer comes from the caller's table, so its address is checked here)
    if ((pc.dst & 7) == 0 && (reinterpret_cast<uintptr_t>(s) & 15) == 0) {
      constexpr int U = 4;
      const int nv = pc.len >> 3;
      for (int v0 = 0; v0 < nv; v0 += kThreads * U) {
        uint4 r[U], o[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + u * kThreads + threadIdx.x;
          o[u] = make_uint4(0, 0, 0, 0);
          if (v < nv) {
            r[u] = __ldg(reinterpret_cast<const uint4*>(s) + v);
            if (accumulate) o[u] = reinterpret_cast<const uint4*>(d)[v];
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + u * kThreads + threadIdx.x;
          if (v < nv) {
            const uint32_t in[4] = {r[u].x, r[u].y, r[u].z, r[u].w};
            const uint32_t old[4] = {o[u].x, o[u].y, o[u].z, o[u].w};
            uint32_t out[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              float lo = __fmul_rn(bf16f(in[i] & 0xFFFFu), scale);
              float hi = __fmul_rn(bf16f(in[i] >> 16), scale);
              if (accumulate) {
                lo = __fadd_rn(bf16f(old[i] & 0xFFFFu), lo);
                hi = __fadd_rn(bf16f(old[i] >> 16), hi);
              }
              out[i] = f2bf(lo) | (f2bf(hi) << 16);
            }
            reinterpret_cast<uint4*>(d)[v] = make_uint4(out[0], out[1], out[2], out[3]);
          }
        }
      }
      for (int e = (nv << 3) + threadIdx.x; e < pc.len; e += kThreads) {
        float y = __fmul_rn(bf16f(s[e]), scale);
        if (accumulate) y = __fadd_rn(bf16f(d[e]), y);
        d[e] = uint16_t(f2bf(y));
      }
    } else {
      for (int e = threadIdx.x; e < pc.len; e += kThreads) {
        float y = __fmul_rn(bf16f(s[e]), scale);
        if (accumulate) y = __fadd_rn(bf16f(d[e]), y);
        d[e] = uint16_t(f2bf(y));
      }
    }
  }
}

// ---------------------------------------------------------------- asynchronous staging
// A warp streams its Adam blocks through a few shared-memory stages filled with
// cp.async, so that several blocks' loads are in flight per warp with few
// registers.  Each lane reads back only the bytes it copied itself.

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async8(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

// one stage of one warp: the 8-element slices of 32 lanes, lane-contiguous
struct StageBuf {
  uint4 g[32];
  float4 p0[32], p1[32];
  uint2 m[32], v[32];
  float sc[4];  // the block's m and v scales (staged by lanes 0 and 1)
};

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// lanes 0 and 1 stage the block's two scales
__device__ __forceinline__ void stage_scales(StageBuf& sb, int lane, const AdamArgs& a, int slot) {
  if (lane == 0) cp_async4(&sb.sc[0], a.m_scale + slot);
  if (lane == 1) cp_async4(&sb.sc[1], a.v_scale + slot);
}

__device__ __forceinline__ uint32_t fastdiv(uint32_t n, uint32_t mul, uint32_t shr) {
  return mul ? (__umulhi(n, mul) >> shr) : n;
}

__device__ __forceinline__ void stage_issue(StageBuf& sb, int lane, const AdamArgs& a, int64_t pos) {
  cp_async16(&sb.g[lane], a.grad + pos);
  cp_async16(&sb.p0[lane], a.master + pos);
  cp_async16(&sb.p1[lane], a.master + pos + 4);
  cp_async8(&sb.m[lane], a.m + pos);
  cp_async8(&sb.v[lane], a.v + pos);
}

constexpr int kStages = 4;  // three blocks per warp in flight while one is computed

// ---------------------------------------------------------------- Adam over one 8-element lane slice
// The lane's inputs stay packed (bf16 pairs, fp32 quads, code bytes) and are
// unpacked element by element, which keeps the live register set small.

struct Raw8 {
  uint4 g;
  float4 p0, p1;
  uint2 m, v;
};

__device__ __forceinline__ Raw8 raw_from_stage(const StageBuf& sb, int lane) {
  Raw8 r;
  r.g = sb.g[lane];
  r.p0 = sb.p0[lane];
  r.p1 = sb.p1[lane];
  r.m = sb.m[lane];
  r.v = sb.v[lane];
  return r;
}

__device__ __forceinline__ Raw8 raw_from_global(const AdamArgs& a, int64_t pos, int n) {
  Raw8 r;
  if (n == 8) {
    r.g = *reinterpret_cast<const uint4*>(a.grad + pos);
    r.p0 = *reinterpret_cast<const float4*>(a.master + pos);
    r.p1 = *reinterpret_cast<const float4*>(a.master + pos + 4);
    r.m = *reinterpret_cast<const uint2*>(a.m + pos);
    r.v = *reinterpret_cast<const uint2*>(a.v + pos);
    return r;
  }
  uint32_t g[4] = {0, 0, 0, 0}, m[2] = {0, 0}, v[2] = {0, 0};
  float p[8] = {0, 0, 0, 0, 0, 0, 0, 0};
#pragma unroll
  for (int i = 0; i < 8; ++i)
    if (i < n) {
      g[i >> 1] |= uint32_t(a.grad[pos + i]) << (16 * (i & 1));
      p[i] = a.master[pos + i];
      m[i >> 2] |= uint32_t(uint8_t(a.m[pos + i])) << (8 * (i & 3));
      v[i >> 2] |= uint32_t(a.v[pos + i]) << (8 * (i & 3));
    }
  r.g = make_uint4(g[0], g[1], g[2], g[3]);
  r.p0 = make_float4(p[0], p[1], p[2], p[3]);
  r.p1 = make_float4(p[4], p[5], p[6], p[7]);
  r.m = make_uint2(m[0], m[1]);
  r.v = make_uint2(v[0], v[1]);
  return r;
}

// Computes p', m', v' for the lane's n valid elements (n <= 8) and the lane's
// partial maxima of |m'|, v' and |p'| (as fp32 bits).
struct Lane8 {
  float p1[8], m1[8], v1[8];
  uint32_t am, av, ap;
};

template <bool FULL>
__device__ __forceinline__ void adam_raw(const Hp& h, const Raw8& x, int n, float sm, float sv, Lane8& o) {
  o.am = o.av = o.ap = 0u;
  const uint32_t gw[4] = {x.g.x, x.g.y, x.g.z, x.g.w};
  const float pv[8] = {x.p0.x, x.p0.y, x.p0.z, x.p0.w, x.p1.x, x.p1.y, x.p1.z, x.p1.w};
  const uint32_t mw[2] = {x.m.x ^ 0x80808080u, x.m.y ^ 0x80808080u}, vw[2] = {x.v.x, x.v.y};
  const float2 sm2 = dup(sm), sv2 = dup(sv);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 g = make_float2(__uint_as_float(gw[j] << 16), __uint_as_float(gw[j] & 0xFFFF0000u));
    const float2 qm = byte_pair(mw[j >> 1], 2 * (j & 1), 8388736.f);  // 2^23 + 128 for the flipped sign bit
    const float2 qv = byte_pair(vw[j >> 1], 2 * (j & 1), 8388608.f);
    float2 p1, m1, v1;
    adam_pair(h, g, make_float2(pv[2 * j], pv[2 * j + 1]), qm, qv, sm2, sv2, p1, m1, v1);
    o.p1[2 * j] = p1.x;
    o.p1[2 * j + 1] = p1.y;
    o.m1[2 * j] = m1.x;
    o.m1[2 * j + 1] = m1.y;
    o.v1[2 * j] = v1.x;
    o.v1[2 * j + 1] = v1.y;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (FULL || i < n) {
      o.am = max(o.am, __float_as_uint(fabsf(o.m1[i])));
      o.av = max(o.av, __float_as_uint(o.v1[i]));
      o.ap = max(o.ap, __float_as_uint(fabsf(o.p1[i])));
    }
  }
}

// Block scales of m' and v' from the lanes' partial maxima: lane 0 computes the
// m scale, lane 1 the v scale (in parallel), everyone receives both.
__device__ __forceinline__ void warp_block_scales(uint32_t am, uint32_t av, int lane, QScale& qm, QScale& qv) {
  const uint32_t m_all = __reduce_max_sync(0xFFFFFFFFu, am);
  const uint32_t v_all = __reduce_max_sync(0xFFFFFFFFu, av);
  const QScale q = qscale(lane == 0 ? m_all : v_all, lane == 0 ? 127.f : 255.f);
  qm.s = __shfl_sync(0xFFFFFFFFu, q.s, 0);
  qm.r = __shfl_sync(0xFFFFFFFFu, q.r, 0);
  qm.mode = __shfl_sync(0xFFFFFFFFu, q.mode, 0);
  qv.s = __shfl_sync(0xFFFFFFFFu, q.s, 1);
  qv.r = __shfl_sync(0xFFFFFFFFu, q.r, 1);
  qv.mode = __shfl_sync(0xFFFFFFFFu, q.mode, 1);
}

__device__ __forceinline__ void store_bytes(uint8_t* dst, uint2 w, int n) {
  if (n == 8) {
    *reinterpret_cast<uint2*>(dst) = w;
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i < n) dst[i] = uint8_t(((i < 4 ? w.x : w.y) >> (8 * (i & 3))) & 0xFFu);
  }
}

__device__ __forceinline__ void store_state(const AdamArgs& a, int64_t pos, int n, const Lane8& o, const QScale& qm,
                                            const QScale& qv) {
  if (n == 8) {
    store_p8(a.master + pos, o.p1);
  } else {
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i < n) a.master[pos + i] = o.p1[i];
  }
  store_bytes(reinterpret_cast<uint8_t*>(a.m) + pos, codes_int8(o.m1, qm), n);
  store_bytes(a.v + pos, codes_uint8(o.v1, qv), n);
}

// ---------------------------------------------------------------- flat blocks (1-D / no 2-D FP8)
// Block of B = 32*E elements, one warp per block; lane l holds elements
// [l*E, l*E + E).  E = 8: 256-element blocks (FP8 1x128 tiles = half warps);
// E = 4: 128-element blocks (FP8 tile = the block).

template <int E>
__global__ void __launch_bounds__(kThreads, kAdamCtas) k_flat(const FlatGroup* __restrict__ groups, AdamArgs a) {
  constexpr int B = 32 * E;
  const FlatGroup g = groups[gridDim.x - 1 - blockIdx.x];  // back to front, see k_strip
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Hp h = make_hp(a.hp);
  const int nblk = (g.nelem + B - 1) / B;
  const bool do_fp8 = a.fp8 != nullptr && g.fslot >= 0;
  for (int b = warp; b < nblk; b += kWarps) {
    const int e0 = b * B + lane * E;             // element offset in the group
    const int n = max(0, min(E, g.nelem - e0));  // valid elements of this lane
    const int64_t pos = g.pos + e0;
    const Raw8 x = raw_from_global(a, pos, n);
    const int slot = g.mslot + b;
    const float sm = a.m_scale[slot], sv = a.v_scale[slot];
    Lane8 o;
    if (n == 8) adam_raw<true>(h, x, n, sm, sv, o);
    else adam_raw<false>(h, x, n, sm, sv, o);
    QScale qm, qv;
    warp_block_scales(o.am, o.av, lane, qm, qv);
    store_state(a, pos, n, o, qm, qv);
    if (lane == 0) {
      a.m_scale[slot] = qm.s;
      a.v_scale[slot] = qv.s;
    }
    if (do_fp8) {
      uint32_t ap = o.ap;
      // reduce over the lanes of one 128-element tile: 16 lanes (E = 8) or 32 (E = 4)
#pragma unroll
      for (int off = (E == 8 ? 8 : 16); off >= 1; off >>= 1) ap = max(ap, __shfl_xor_sync(0xFFFFFFFFu, ap, off));
      const QScale qp = qscale(ap, 448.f);
      store_bytes(a.fp8 + pos, codes_e4m3(o.p1, qp), n);
      if ((e0 & 127) == 0 && e0 < g.nelem) a.fp8_scale[g.fslot + e0 / 128] = qp.s;
    }
  }
}

// ---------------------------------------------------------------- flat 256 Adam + 2-D FP8 tiles
// One CTA per region (grid-stride, last region first: the pack that precedes
// this step writes the gradient buffer front to back, so its tail is still in
// L2 when this kernel starts).  Phase 1: warps run Adam over the region's
// 256-element blocks, write state and master, and fold |p'| into per-column-tile
// maxima in shared memory.  Phase 2: tile scales, then the updated master is
// re-read (it was written moments ago by this CTA and is served from L2) and
// converted to E4M3.  Shared memory: 2 words per column tile.

template <bool FP8>
__global__ void __launch_bounds__(kThreads, kAdamCtas) k_strip(const RegionGroup* __restrict__ groups, int ngroups, AdamArgs a) {
  // dynamic shared memory: the warps' staging pipes, then 2 words per FP8
  // column tile ([ntile] amax bits, later r; [ntile..2*ntile) s)
  extern __shared__ __align__(16) unsigned char s_dyn[];
  StageBuf* pipe = reinterpret_cast<StageBuf*>(s_dyn);
  uint32_t* s_tile = reinterpret_cast<uint32_t*>(s_dyn + sizeof(StageBuf) * kWarps * kStages);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Hp h = make_hp(a.hp);
  StageBuf* st = pipe + warp * kStages;
  for (int gi = ngroups - 1 - int(blockIdx.x); gi >= 0; gi -= int(gridDim.x)) {
    const RegionGroup g = groups[gi];
    // strip: rows x 256 columns, block = one row segment; band: rows x C,
    // flat 256-element blocks from the band start
    const bool flat = g.width == g.C;
    const int ntile = (g.width + 127) >> 7;
    if (FP8) {
      for (int t = threadIdx.x; t < ntile; t += kThreads) s_tile[t] = 0u;
      __syncthreads();
    }
    const int nel = g.rows * g.width;
    const int nblk = flat ? (nel + 255) >> 8 : g.rows;
    const int rstep = g.C >> 8;  // strip: slots per row
    // geometry of this warp's k-th block: lane position, valid count, slot
    auto geom = [&](int k, int64_t& pos, int& n, int& slot) {
      const int b = warp + k * kWarps;
      const int off = flat ? (b << 8) : b * g.C;
      slot = g.mslot + (flat ? b : b * rstep);
      n = flat ? max(0, min(8, nel - off - lane * 8)) : 8;
      pos = g.pos + off + lane * 8;
    };
    const int nb_w = warp < nblk ? (nblk - warp + kWarps - 1) / kWarps : 0;
#pragma unroll
    for (int k = 0; k < kStages - 1; ++k) {
      if (k < nb_w) {
        int64_t pos; int n, slot;
        geom(k, pos, n, slot);
        if (n == 8) stage_issue(st[k], lane, a, pos);
        stage_scales(st[k], lane, a, slot);
      }
      cp_async_commit();
    }
    for (int k = 0; k < nb_w; ++k) {
      const int kn = k + kStages - 1;
      __syncwarp();
      if (kn < nb_w) {
        int64_t pos; int n, slot;
        geom(kn, pos, n, slot);
        if (n == 8) stage_issue(st[kn % kStages], lane, a, pos);
        stage_scales(st[kn % kStages], lane, a, slot);
      }
      cp_async_commit();
      cp_async_wait<kStages - 1>();
      __syncwarp();  // lanes 0 and 1 staged the scales every lane reads
      int64_t pos; int n, slot;
      geom(k, pos, n, slot);
      const StageBuf& sb = st[k % kStages];
      const Raw8 x = n == 8 ? raw_from_stage(sb, lane) : raw_from_global(a, pos, n);
      Lane8 o;
      if (n == 8) adam_raw<true>(h, x, n, sb.sc[0], sb.sc[1], o);
      else adam_raw<false>(h, x, n, sb.sc[0], sb.sc[1], o);
      QScale qm, qv;
      warp_block_scales(o.am, o.av, lane, qm, qv);
      store_state(a, pos, n, o, qm, qv);
      if (lane == 0) {
        a.m_scale[slot] = qm.s;
        a.v_scale[slot] = qv.s;
      }
      if (FP8) {
        if (flat) {
          // column of the lane's first element; several lanes share a tile
          const int b = warp + k * kWarps;
          const uint32_t e = uint32_t((b << 8) + lane * 8);
          const int col = int(e - fastdiv(e, g.cmul, g.cshr) * uint32_t(g.C));
          const int t = col >> 7;
          const unsigned same = __match_any_sync(0xFFFFFFFFu, t);
          const uint32_t ap = __reduce_max_sync(same, o.ap);
          if (lane == __ffs(same) - 1) atomicMax(&s_tile[t], ap);
        } else {
          // strip: lanes 0-15 cover tile 0, lanes 16-31 tile 1
          uint32_t ap = o.ap;
#pragma unroll
          for (int off = 8; off >= 1; off >>= 1) ap = max(ap, __shfl_xor_sync(0xFFFFFFFFu, ap, off));
          if ((lane & 15) == 0) atomicMax(&s_tile[lane >> 4], ap);
        }
      }
    }
    cp_async_wait<0>();
    if (FP8) {
      __syncthreads();
      for (int t = threadIdx.x; t < ntile; t += kThreads) {
        const QScale q = qscale(s_tile[t], 448.f);
        a.fp8_scale[g.fslot + t] = q.s;
        s_tile[t] = __float_as_uint(q.r);
        s_tile[ntile + t] = __float_as_uint(q.s);
      }
      __syncthreads();
      const int nvec = nel >> 3;
      constexpr int U = 2;
      for (int v0 = threadIdx.x; v0 < nvec; v0 += kThreads * U) {
        float4 p0[U], p1[U];
        int64_t pos[U];
        int tile[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + u * kThreads;
          if (v < nvec) {
            if (flat) {
              const uint32_t e = uint32_t(v) << 3;
              tile[u] = int(e - fastdiv(e, g.cmul, g.cshr) * uint32_t(g.C)) >> 7;
              pos[u] = g.pos + e;
            } else {
              const int r = v >> 5, kk = v & 31;  // 32 vectors of 8 per 256-column row
              tile[u] = kk >> 4;
              pos[u] = g.pos + int64_t(r) * g.C + (kk << 3);
            }
            p0[u] = *reinterpret_cast<const float4*>(a.master + pos[u]);
            p1[u] = *reinterpret_cast<const float4*>(a.master + pos[u] + 4);
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int v = v0 + u * kThreads;
          if (v < nvec) {
            QScale q;
            q.r = __uint_as_float(s_tile[tile[u]]);
            q.s = __uint_as_float(s_tile[ntile + tile[u]]);
            q.mode = q.s == 0.f ? 0 : (isinf(q.r) ? 2 : 1);
            const float pv[8] = {p0[u].x, p0[u].y, p0[u].z, p0[u].w, p1[u].x, p1[u].y, p1[u].z, p1[u].w};
            *reinterpret_cast<uint2*>(a.fp8 + pos[u]) = codes_e4m3(pv, q);
          }
        }
      }
      __syncthreads();  // s_tile is reused by the next region
    }
  }
}

// ---------------------------------------------------------------- 128x128 Adam tiles (+ FP8 of the same tile)
// Phase 1: Adam, write master, block-reduce max|m'|, max v', max|p'|.
// Phase 2: requantise m', v' (recomputed from the untouched old codes and the
// old scales held in registers, bit-identical) and convert p' (re-read, L2).

__device__ __forceinline__ void block_max(uint32_t x, uint32_t* red, int which) {
  x = __reduce_max_sync(0xFFFFFFFFu, x);
  if ((threadIdx.x & 31) == 0) red[which * kWarps + (threadIdx.x >> 5)] = x;
}

template <bool FP8>
__global__ void __launch_bounds__(kThreads, kAdamCtas) k_tile(const RegionGroup* __restrict__ groups, int ngroups, AdamArgs a) {
  __shared__ uint32_t red[3 * kWarps];
  const Hp h = make_hp(a.hp);
  for (int gi = ngroups - 1 - int(blockIdx.x); gi >= 0; gi -= int(gridDim.x)) {
    const RegionGroup g = groups[gi];
    const bool fp8 = FP8 && g.fslot >= 0;
    const float sm = a.m_scale[g.mslot], sv = a.v_scale[g.mslot];
    const int vpr = g.width >> 3, nvec = g.rows * vpr;
    uint32_t am = 0, av = 0, ap = 0;
    for (int v = threadIdx.x; v < nvec; v += kThreads) {
      const int r = v / vpr, k = v - r * vpr;
      const int64_t pos = g.pos + int64_t(r) * g.C + (k << 3);
      const Raw8 x = raw_from_global(a, pos, 8);
      Lane8 o;
      adam_raw<true>(h, x, 8, sm, sv, o);
      store_p8(a.master + pos, o.p1);
      am = max(am, o.am);
      av = max(av, o.av);
      ap = max(ap, o.ap);
    }
    block_max(am, red, 0);
    block_max(av, red, 1);
    block_max(ap, red, 2);
    __syncthreads();
    uint32_t tm = 0, tv = 0, tp = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      tm = max(tm, red[w]);
      tv = max(tv, red[kWarps + w]);
      tp = max(tp, red[2 * kWarps + w]);
    }
    const QScale qm = qscale(tm, 127.f), qv = qscale(tv, 255.f), qp = qscale(tp, 448.f);
    if (threadIdx.x == 0) {
      a.m_scale[g.mslot] = qm.s;
      a.v_scale[g.mslot] = qv.s;
      if (fp8) a.fp8_scale[g.fslot] = qp.s;
    }
    for (int v = threadIdx.x; v < nvec; v += kThreads) {
      const int r = v / vpr, k = v - r * vpr;
      const int64_t pos = g.pos + int64_t(r) * g.C + (k << 3);
      const Raw8 x = raw_from_global(a, pos, 8);  // old codes; the master words now hold p'
      Lane8 o;
      adam_raw<true>(h, x, 8, sm, sv, o);
      *reinterpret_cast<uint2*>(a.m + pos) = codes_int8(o.m1, qm);
      *reinterpret_cast<uint2*>(a.v + pos) = codes_uint8(o.v1, qv);
      if (fp8) {
        const float pv[8] = {x.p0.x, x.p0.y, x.p0.z, x.p0.w, x.p1.x, x.p1.y, x.p1.z, x.p1.w};
        *reinterpret_cast<uint2*>(a.fp8 + pos) = codes_e4m3(pv, qp);
      }
    }
    __syncthreads();  // red is reused by the next tile
  }
}

// ---------------------------------------------------------------- standalone FP8

__global__ void __launch_bounds__(kThreads) k_quant_flat(const FlatGroup* __restrict__ groups,
                                                         const float* __restrict__ master, uint8_t* __restrict__ fp8,
                                                         float* __restrict__ fp8_scale) {
  const FlatGroup g = groups[blockIdx.x];
  if (g.fslot < 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nchunk = (g.nelem + 255) >> 8;
  for (int c = warp; c < nchunk; c += kWarps) {
    const int e0 = (c << 8) + lane * 8;
    const int n = max(0, min(8, g.nelem - e0));
    const int64_t pos = g.pos + e0;
    float p[8];
    if (n == 8) {
      const float4 p0 = *reinterpret_cast<const float4*>(master + pos);
      const float4 p1 = *reinterpret_cast<const float4*>(master + pos + 4);
      p[0] = p0.x; p[1] = p0.y; p[2] = p0.z; p[3] = p0.w; p[4] = p1.x; p[5] = p1.y; p[6] = p1.z; p[7] = p1.w;
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) p[i] = i < n ? master[pos + i] : 0.f;
    }
    uint32_t ap = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (i < n) ap = max(ap, __float_as_uint(fabsf(p[i])));
#pragma unroll
    for (int off = 8; off >= 1; off >>= 1) ap = max(ap, __shfl_xor_sync(0xFFFFFFFFu, ap, off));
    const QScale q = qscale(ap, 448.f);
    store_bytes(fp8 + pos, codes_e4m3(p, q), n);
    if ((e0 & 127) == 0 && e0 < g.nelem) fp8_scale[g.fslot + e0 / 128] = q.s;
  }
}

__global__ void __launch_bounds__(kThreads) k_quant_region(const RegionGroup* __restrict__ groups, int ngroups,
                                                           const float* __restrict__ master,
                                                           uint8_t* __restrict__ fp8, float* __restrict__ fp8_scale) {
  extern __shared__ uint32_t s_tile[];  // [ntile] amax bits, later r; [ntile..2*ntile) s
  for (int gi = blockIdx.x; gi < ngroups; gi += gridDim.x) {
    const RegionGroup g = groups[gi];
    if (g.fslot < 0) continue;  // uniform per CTA
    const bool flat = g.width == g.C;
    const int ntile = (g.width + 127) >> 7;
    for (int t = threadIdx.x; t < ntile; t += kThreads) s_tile[t] = 0u;
    __syncthreads();
    const int nvec = (g.rows * g.width) >> 3, vpr = g.width >> 3;
    for (int pass = 0; pass < 2; ++pass) {
      for (int v = threadIdx.x; v < nvec; v += kThreads) {
        int64_t pos;
        int col;
        if (flat) {
          col = (v << 3) % g.C;
          pos = g.pos + (int64_t(v) << 3);
        } else {
          const int r = v / vpr, k = v - r * vpr;
          col = k << 3;
          pos = g.pos + int64_t(r) * g.C + col;
        }
        const float4 p0 = *reinterpret_cast<const float4*>(master + pos);
        const float4 p1 = *reinterpret_cast<const float4*>(master + pos + 4);
        const float pv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
        if (pass == 0) {
          uint32_t ap = 0;
#pragma unroll
          for (int i = 0; i < 8; ++i) ap = max(ap, __float_as_uint(fabsf(pv[i])));
          atomicMax(&s_tile[col >> 7], ap);
        } else {
          QScale q;
          q.r = __uint_as_float(s_tile[col >> 7]);
          q.s = __uint_as_float(s_tile[ntile + (col >> 7)]);
          q.mode = q.s == 0.f ? 0 : (isinf(q.r) ? 2 : 1);
          *reinterpret_cast<uint2*>(fp8 + pos) = codes_e4m3(pv, q);
        }
      }
      __syncthreads();
      if (pass == 0) {
        for (int t = threadIdx.x; t < ntile; t += kThreads) {
          const QScale q = qscale(s_tile[t], 448.f);
          fp8_scale[g.fslot + t] = q.s;
          s_tile[t] = __float_as_uint(q.r);
          s_tile[ntile + t] = __float_as_uint(q.s);
        }
        __syncthreads();
      }
    }
  }
}

int check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(BQ_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
  return BQ_OK;
}

constexpr int kStripCtasPerSm = kAdamCtas;
constexpr int kTileCtasPerSm = kAdamCtas;
constexpr int kMaxStripTiles = 6144;  // 2 words per tile: 48 KB of shared memory

}  // namespace

int launch_pack(const DevTables& t, const uint16_t* const* grads, uint16_t* dst, int64_t total, float scale,
                int accumulate, void* stream) {
  (void)total;
  if (t.nchunks == 0) return BQ_OK;
  if (t.nchunks > 0x7FFFFFFF) return set_error(BQ_EINVAL, "bq_pack: too many chunks");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  k_pack<<<dim3(unsigned(t.nchunks)), kThreads, 0, s>>>(t.pieces, t.chunk_first, grads, dst, scale, accumulate);
  return check_launch("bq_pack");
}

int launch_adam8(const DevTables& t, const AdamArgs& a, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool fp8 = a.fp8 != nullptr;
  const int sms = sm_count();
  if (t.max_strip_tiles > kMaxStripTiles) return set_error(BQ_EINVAL, "bq_step_adam8: too many FP8 tiles per row");
  if (t.n_flat256) {
    k_flat<8><<<t.n_flat256, kThreads, 0, s>>>(t.flat256, a);
    if (int rc = check_launch("bq_step_adam8 (flat256)")) return rc;
  }
  if (t.n_flat128) {
    k_flat<4><<<t.n_flat128, kThreads, 0, s>>>(t.flat128, a);
    if (int rc = check_launch("bq_step_adam8 (flat128)")) return rc;
  }
  if (t.n_strips) {
    const int grid = std::min(t.n_strips, sms * kStripCtasPerSm);
    const size_t smem = sizeof(StageBuf) * kWarps * kStages + 2 * size_t(t.max_strip_tiles) * sizeof(uint32_t);
    static bool attr_done = false;
    if (!attr_done) {
      cudaFuncSetAttribute(k_strip<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
      cudaFuncSetAttribute(k_strip<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
      attr_done = true;
    }
    if (fp8)
      k_strip<true><<<grid, kThreads, smem, s>>>(t.strips, t.n_strips, a);
    else
      k_strip<false><<<grid, kThreads, smem, s>>>(t.strips, t.n_strips, a);
    if (int rc = check_launch("bq_step_adam8 (strips)")) return rc;
  }
  if (t.n_tiles) {
    const int grid = std::min(t.n_tiles, sms * kTileCtasPerSm);
    if (fp8)
      k_tile<true><<<grid, kThreads, 0, s>>>(t.tiles, t.n_tiles, a);
    else
      k_tile<false><<<grid, kThreads, 0, s>>>(t.tiles, t.n_tiles, a);
    if (int rc = check_launch("bq_step_adam8 (tiles)")) return rc;
  }
  return BQ_OK;
}

int launch_quant_fp8(const DevTables& t, const float* master, uint8_t* fp8, float* fp8_scale, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int sms = sm_count();
  if (t.max_strip_tiles > kMaxStripTiles) return set_error(BQ_EINVAL, "bq_quant_fp8: too many FP8 tiles per row");
  if (t.n_flat256) {
    k_quant_flat<<<t.n_flat256, kThreads, 0, s>>>(t.flat256, master, fp8, fp8_scale);
    if (int rc = check_launch("bq_quant_fp8 (flat256)")) return rc;
  }
  if (t.n_flat128) {
    k_quant_flat<<<t.n_flat128, kThreads, 0, s>>>(t.flat128, master, fp8, fp8_scale);
    if (int rc = check_launch("bq_quant_fp8 (flat128)")) return rc;
  }
  if (t.n_strips) {
    const size_t smem = 2 * size_t(std::max(t.max_strip_tiles, 1)) * sizeof(uint32_t);
    k_quant_region<<<std::min(t.n_strips, sms * kStripCtasPerSm), kThreads, smem, s>>>(t.strips, t.n_strips, master,
                                                                                        fp8, fp8_scale);
    if (int rc = check_launch("bq_quant_fp8 (strips)")) return rc;
  }
  if (t.n_tiles) {
    k_quant_region<<<std::min(t.n_tiles, sms * kTileCtasPerSm), kThreads, 2 * sizeof(uint32_t), s>>>(
        t.tiles, t.n_tiles, master, fp8, fp8_scale);
    if (int rc = check_launch("bq_quant_fp8 (tiles)")) return rc;
  }
  return BQ_OK;
}

}  // namespace bq
