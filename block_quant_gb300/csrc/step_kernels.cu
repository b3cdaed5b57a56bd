// Memory-bound kernels of the DBuffer step on GB300 (sm_103a):
//   k_pack         fused pre-communication copy / scale / add / zero into the
//                  bf16 gradient DBuffer (DBuffer's group-level pre-comm ops,
//                  veScale-FSDP bud-325 summary, Key claims and Method)
//   k_flat<E>      8-bit Adam over runs of flat blocks (256, 128 or 32 elements),
//                  optionally fused with 1x128 FP8 tiles of 1-D tensors
//   k_strip<FP8>   8-bit Adam with flat 256-element blocks over a 2-D region,
//                  fused with 128x128 FP8 tiles; inputs staged by a producer
//                  warp's TMA copies (tensor-map boxes or bulk copies), tile
//                  amax in shared memory, half
//                  of each region's updated master kept in tensor memory for
//                  the FP8 pass
//   k_tile<FP8>    8-bit Adam with 128x128 state tiles (+ FP8 of the same tile);
//                  the tile's inputs kept in tensor memory between its phases
//   k_tile32       8-bit Adam with the walkthrough's 32x32 state tiles (same
//                  tensor-memory scheme)
//   k_quant_*      FP8 requantisation on its own: standalone, and for the
//                  tiles of bands whose Adam ran as flat pieces
//   k_dequant_*    the bf16 view (code x tile scale) of the gathered FP8 buffer
//   k_muon_*       Muon's momentum + gather and apply around Newton-Schulz
// The 8-bit Adam is the pages' block-quantised optimizer state kept local to a
// shard (feynmanwiki walkthrough, paper section 6.3); FP8 is block-wise FP8 in
// the DeepSeek-V3 style (bud-325 TL;DR).
//
// Every value-producing fp32 operation is an explicit round-to-nearest
// intrinsic or an explicit fused multiply-add (compiled with -fmad=false, so
// nothing else is contracted), in the order the host-side contract fixes, so
// codes, scales and master weights are reproducible bit for bit.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "bq_internal.h"
#include "tmem_ptx.h"

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
// max of three floats; a NaN operand gives NaN (so a NaN in a block reaches its
// scale, as a maximum over the raw bit patterns would)
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.NaN.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

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

// ---------------------------------------------------------------- TMA staging
// The 2-D Adam kernel streams its inputs through shared memory with bulk
// asynchronous copies issued by one producer warp (the copy engine moves whole
// row segments, so many kilobytes per SM are in flight without load
// instructions or registers); completion is tracked by mbarriers.  Every wait is
// bounded: after about a second it records a status code and gives up.

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared.b64 [%0], %1;\n" ::"r"(smem_u32(b)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared.b64 _, [%0];\n" ::"r"(smem_u32(b)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared.b64 _, [%0], %1;\n" ::"r"(smem_u32(b)), "r"(bytes) : "memory");
}

// one arrival on b once every earlier cp.async of this thread has landed
__device__ __forceinline__ void mbar_arrive_cp_async(uint64_t* b) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared.b64 [%0];\n" ::"r"(smem_u32(b)) : "memory");
}

constexpr long long kWaitCycles = 1LL << 31;  // about a second at the SM clock

// wait for the completion of the phase of b with the given parity; false once
// `limit` SM clocks have passed
__device__ __forceinline__ bool mbar_wait_for(uint64_t* b, uint32_t parity, long long limit) {
  const long long t0 = clock64();
  for (;;) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(smem_u32(b)), "r"(parity)
        : "memory");
    if (done) return true;
    if (clock64() - t0 > limit) return false;
  }
}

__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity) { return mbar_wait_for(b, parity, kWaitCycles); }

// bulk copy global -> this CTA's shared memory, completion counted on bar
// (addresses 16-byte aligned, bytes a multiple of 16)
// rows [y, y + 8) x columns [x, x + 256) of a 2-D tensor map in global memory
__device__ __forceinline__ void map_load(void* dst, const void* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];\n" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ void report(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// n / d by multiply-high and shift (mul, shr from the host; mul == 0: d == 1)
__device__ __forceinline__ uint32_t fastdiv(uint32_t n, uint32_t mul, uint32_t shr) {
  return mul ? (__umulhi(n, mul) >> shr) : n;
}

// ---------------------------------------------------------------- Adam over one 8-element lane slice
// The lane's inputs stay packed (bf16 pairs, fp32 quads, code bytes) and are
// unpacked element by element, which keeps the live register set small.

struct Raw8 {
  uint4 g;
  float4 p0, p1;
  uint2 m, v;
};

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
  // lane maxima of |m'|, v' (>= 0) and |p'|, three operands per max; elements
  // past n count as 0
  float am = 0.f, av = 0.f, ap = 0.f;
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    const bool a0 = FULL || i < n, a1 = FULL || i + 1 < n;
    am = max3(am, a0 ? fabsf(o.m1[i]) : 0.f, a1 ? fabsf(o.m1[i + 1]) : 0.f);
    av = max3(av, a0 ? o.v1[i] : 0.f, a1 ? o.v1[i + 1] : 0.f);
    ap = max3(ap, a0 ? fabsf(o.p1[i]) : 0.f, a1 ? fabsf(o.p1[i + 1]) : 0.f);
  }
  o.am = __float_as_uint(am);
  o.av = __float_as_uint(av);
  o.ap = __float_as_uint(ap);
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
      // reduce over the lanes of one 128-element tile: 16 lanes (E = 8) or 32 (E = 4)
      const uint32_t ap = __reduce_max_sync(E == 4 ? 0xFFFFFFFFu : (lane < 16 ? 0x0000FFFFu : 0xFFFF0000u), o.ap);
      const QScale qp = qscale(ap, 448.f);
      store_bytes(a.fp8 + pos, codes_e4m3(o.p1, qp), n);
      if ((e0 & 127) == 0 && e0 < g.nelem) a.fp8_scale[g.fslot + e0 / 128] = qp.s;
    }
  }
}

// ---------------------------------------------------------------- flat 256 Adam + 2-D FP8 tiles
// Regions (128-row x 256-column strips, or whole 128-row bands when C % 256 != 0)
// are taken by CTAs in a grid-stride loop, last region first (the pack that
// precedes this step writes the gradient buffer front to back, so its tail is
// still in L2 when this kernel starts).  Warp kCons is the producer: it fills a
// ring of kRing shared-memory stages, each with the next kCons Adam blocks (the
// blocks' two scales by cp.async), and runs ahead across region boundaries.  A
// stage takes four copies when it can: a strip's 8 rows as one 8 x 256 box of a
// 2-D tensor map per array (maps of the caller's buffers, built on the host),
// a flat piece's 8 consecutive blocks as one bulk copy per array; otherwise
// one bulk copy per block and array (the copy engine's cost is per copy as
// much as per byte).  Warps 0..kCons-1 consume one block each per
// stage: Adam, state and master written back, |p'| folded into per-column-tile
// maxima in shared memory.  After a region's last stage they compute the tile
// scales and convert the region's updated master to E4M3: its first 64 rows
// from a copy each warp wrote to tensor memory as it went, the other rows
// re-read from global memory (this CTA wrote them moments ago, so they come
// from L2).  A block is staged only when it is whole and starts on a 16-byte
// boundary of the byte arrays; any other block (a band's ragged tail) is read
// directly from global memory.

#ifndef BQ_STRIP_CONSUMERS
#define BQ_STRIP_CONSUMERS 8
#endif
constexpr int kCons = BQ_STRIP_CONSUMERS;        // consumer warps
constexpr int kScaleLanes = 2 * kCons < 32 ? 2 * kCons : 32;  // producer lanes staging scales
constexpr int kStripThreads = 32 * (kCons + 1);  // + the producer warp
#ifndef BQ_STRIP_RING
#define BQ_STRIP_RING 4
#endif
constexpr int kRing = BQ_STRIP_RING;             // stages in the ring
#ifndef BQ_STRIP_CTAS_PER_SM
#define BQ_STRIP_CTAS_PER_SM 3
#endif
constexpr int kStripCtas = BQ_STRIP_CTAS_PER_SM;
// FP8 instantiation: the updated master of a strip's first kTmemRows rows is
// also written to tensor memory, so the FP8 pass reads it back from the SM
// instead of L2.  Row b lives in lane quarter b % 4 (the warp that updated it:
// b % kCons == warp and kCons % 4 == 0), columns (b / 4) * 8 .. + 7.
constexpr int kTmemCols = 128;
constexpr int kTmemRows = kTmemCols / 8 * 4;
static_assert(kCons % 4 == 0, "a strip row must stay in its warp's TMEM lane quarter");
static_assert(kStripCtas * kTmemCols <= 512, "the resident CTAs' TMEM columns fit one SM");

struct TmaStage {
  uint4 g[kCons][32];   // bf16 gradients, 512 B per block
  float4 p[kCons][64];  // fp32 master, 1 KB per block
  uint2 m[kCons][32];   // int8 m codes
  uint2 v[kCons][32];   // uint8 v codes
  float sc[2 * kCons];  // per block: m scale, v scale
  float pad_[32 - 2 * kCons];
};
static_assert(sizeof(TmaStage) % 128 == 0, "stages keep the 128-byte alignment of tensor copies");
static_assert(kCons == 8, "a strip stage is one 8-row box of the interval's tensor maps");
constexpr uint32_t kBlockBytes = 512 + 1024 + 256 + 256;

__device__ __forceinline__ int region_blocks(const RegionGroup& g) {
  return g.width == g.C ? (g.rows * g.width + 255) >> 8 : g.rows;
}

// first element, element count and scale slot of Adam block b of region g
// (strip: row b of the strip; band: flat 256-element block b from the band start)
__device__ __forceinline__ void region_block(const RegionGroup& g, int b, int64_t& start, int& nel, int& slot) {
  if (g.width == g.C) {
    start = g.pos + (int64_t(b) << 8);
    nel = min(256, g.rows * g.width - (b << 8));
    slot = g.mslot + b;
  } else {
    start = g.pos + int64_t(b) * g.C;
    nel = 256;
    slot = g.mslot + b * (g.C >> 8);
  }
}

__device__ __forceinline__ bool block_staged(int64_t start, int nel) { return nel == 256 && (start & 15) == 0; }

// barrier of the consumer warps only (the producer never joins it)
__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;\n" ::"n"(32 * kCons) : "memory"); }

// A consumer warp hands a ring stage back after reading it.  The reads went
// through the generic proxy and the producer's next bulk copy into the stage
// writes through the async proxy, which the mbarrier alone does not order: each
// lane fences between the two proxies before the warp arrives.
__device__ __forceinline__ void release_stage(uint64_t* empty, int lane) {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
  __syncwarp();
  if (lane == 0) mbar_arrive(empty);
}

__device__ __forceinline__ void strip_producer(const RegionGroup* __restrict__ groups, int ngroups, const AdamArgs& a,
                                               TmaStage* ring, uint64_t* full, uint64_t* empty, int lane) {
  uint32_t k = 0;  // stages issued
  bool ok = true;
  // tensor copies need 128-byte aligned destinations (the ring's start)
  const bool maps = a.tmaps != nullptr && (smem_u32(ring) & 127u) == 0;
  for (int gi = ngroups - 1 - int(blockIdx.x); ok && gi >= 0; gi -= int(gridDim.x)) {
    const RegionGroup g = groups[gi];
    const int nblk = region_blocks(g);
    for (int j = 0; j < nblk; j += kCons, ++k) {
      const int s = int(k % kRing);
      if (k >= kRing) {
        ok = __all_sync(0xFFFFFFFFu, mbar_wait(&empty[s], ((k / kRing) - 1) & 1));
        if (!ok) break;
      }
      TmaStage& S = ring[s];
      // a flat piece's blocks lie one after another in every array: a stage of
      // kCons full, aligned blocks is one bulk copy per array (4 copies instead of
      // 4 kCons; the copy engine's cost is per copy as much as per byte)
      bool merged = false;
      int64_t first = 0;
      if (g.width == g.C && j + kCons <= nblk) {
        int64_t last;
        int nf, nl, sf, sl;
        region_block(g, j, first, nf, sf);
        region_block(g, j + kCons - 1, last, nl, sl);
        merged = block_staged(first, nf) && nl == 256;
      }
      if (merged) {
        if (lane == 0) mbar_arrive_expect_tx(&full[s], kCons * kBlockBytes);
        __syncwarp();
        if (lane == 0) bulk_load(S.g[0], a.grad + first, 512 * kCons, &full[s]);
        else if (lane == 1) bulk_load(S.p[0], a.master + first, 1024 * kCons, &full[s]);
        else if (lane == 2) bulk_load(S.m[0], a.m + first, 256 * kCons, &full[s]);
        else if (lane == 3) bulk_load(S.v[0], a.v + first, 256 * kCons, &full[s]);
      } else if (maps && g.tm >= 0) {
        // a strip: rows j .. j + 7 as one 8-row box of each array's tensor map
        // (rows past the strip arrive too, zero past the interval; nobody reads them)
        if (lane == 0) mbar_arrive_expect_tx(&full[s], kCons * kBlockBytes);
        __syncwarp();
        if (lane < 4) {
          const unsigned char* mp = static_cast<const unsigned char*>(a.tmaps) + (size_t(g.tm) * 4 + lane) * kMapBytes;
          void* dst = lane == 0 ? static_cast<void*>(S.g[0])
                      : lane == 1 ? static_cast<void*>(S.p[0])
                      : lane == 2 ? static_cast<void*>(S.m[0])
                                  : static_cast<void*>(S.v[0]);
          map_load(dst, mp, g.c0, g.trow + j, &full[s]);
        }
      } else {
        // pass q, lane = 4 w + arr: array arr (g, p, m, v) of the stage's block 8 q + w
        constexpr int kPasses = (kCons + 7) / 8;
        bool staged[kPasses];
        int64_t start[kPasses];
        uint32_t nst = 0;
#pragma unroll
        for (int q = 0; q < kPasses; ++q) {
          const int w = 8 * q + (lane >> 2);
          int nel = 0, slot = 0;
          start[q] = 0;
          const bool have = w < kCons && j + w < nblk;
          if (have) region_block(g, j + w, start[q], nel, slot);
          staged[q] = have && block_staged(start[q], nel);
          nst += __popc(__ballot_sync(0xFFFFFFFFu, staged[q] && (lane & 3) == 0));
        }
        if (lane == 0) mbar_arrive_expect_tx(&full[s], nst * kBlockBytes);
        __syncwarp();
#pragma unroll
        for (int q = 0; q < kPasses; ++q) {
          const int w = 8 * q + (lane >> 2), arr = lane & 3;
          if (staged[q]) {
            if (arr == 0) bulk_load(S.g[w], a.grad + start[q], 512, &full[s]);
            else if (arr == 1) bulk_load(S.p[w], a.master + start[q], 1024, &full[s]);
            else if (arr == 2) bulk_load(S.m[w], a.m + start[q], 256, &full[s]);
            else bulk_load(S.v[w], a.v + start[q], 256, &full[s]);
          }
        }
      }
      // scale i (i & 1 ? v : m of block i >> 1) by lane i % 32
      if (lane < kScaleLanes) {
        for (int i = lane; i < 2 * kCons; i += 32) {
          const int bb = j + (i >> 1);
          if (bb < nblk) {
            int64_t st2;
            int ne2, sl2;
            region_block(g, bb, st2, ne2, sl2);
            cp_async4(&S.sc[i], ((i & 1) ? a.v_scale : a.m_scale) + sl2);
          }
        }
        mbar_arrive_cp_async(&full[s]);
      }
    }
  }
  if (!ok && lane == 0) report(a.status, 1);
  // no copy of this CTA may still be in flight when it exits
  for (uint32_t d = k > uint32_t(kRing) ? k - kRing : 0; d < k; ++d)
    if (!mbar_wait(&full[d % kRing], (d / kRing) & 1) && lane == 0) report(a.status, 2);
}

template <bool FP8>
__global__ void __launch_bounds__(kStripThreads, kStripCtas) k_strip(const RegionGroup* __restrict__ groups, int ngroups,
                                                                     AdamArgs a) {
  // dynamic shared memory: the stage ring, its full / empty mbarriers, then 2
  // words per FP8 column tile ([ntile] amax bits, later r; [ntile..2*ntile) s)
  extern __shared__ __align__(128) unsigned char s_dyn[];
  TmaStage* ring = reinterpret_cast<TmaStage*>(s_dyn);
  uint64_t* full = reinterpret_cast<uint64_t*>(s_dyn + sizeof(TmaStage) * kRing);
  uint64_t* empty = full + kRing;
  uint32_t* s_tile = reinterpret_cast<uint32_t*>(empty + kRing);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __shared__ uint32_t s_tmem;
  if (FP8 && warp == 0) tmem_alloc(smem_u32(&s_tmem), kTmemCols);
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRing; ++i) {
      mbar_init(&full[i], 1 + kScaleLanes);  // the producer's expect_tx + one per scale lane
      mbar_init(&empty[i], kCons);         // one per consumer warp
    }
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  }
  if (FP8) tc_fence_before();
  __syncthreads();
  if (FP8) tc_fence_after();
  const uint32_t tmem = FP8 ? s_tmem + (uint32_t(32 * (warp & 3)) << 16) : 0u;  // this warp's lane quarter
  if (warp == kCons) {
    strip_producer(groups, ngroups, a, ring, full, empty, lane);
    return;
  }
  constexpr int kCT = 32 * kCons;  // consumer threads
  const Hp h = make_hp(a.hp);
  uint32_t k = 0;      // stages consumed
  bool dead = false;   // a wait timed out: skip the remaining work, keep the barriers
  for (int gi = ngroups - 1 - int(blockIdx.x); gi >= 0; gi -= int(gridDim.x)) {
    const RegionGroup g = groups[gi];
    const bool fp8 = FP8 && g.fslot >= 0;  // band pieces carry no FP8 (their tiles are quantised apart)
    const int ntile = (g.width + 127) >> 7;
    const int nel = g.rows * g.width;
    const int nblk = region_blocks(g);
    if (fp8) {
      for (int t = threadIdx.x; t < ntile; t += kCT) s_tile[t] = 0u;
      consumer_sync();
    }
    for (int j = 0; j < nblk; j += kCons, ++k) {
      const int s = int(k % kRing);
      if (!dead && !__all_sync(0xFFFFFFFFu, mbar_wait(&full[s], (k / kRing) & 1))) {
        dead = true;
        if (lane == 0) report(a.status, 3);
      }
      if (dead) continue;
      const TmaStage& S = ring[s];
      const int b = j + warp;
      if (b >= nblk) {
        if (lane == 0) mbar_arrive(&empty[s]);
        continue;
      }
      int64_t start;
      int nb, slot;
      region_block(g, b, start, nb, slot);
      const bool staged = block_staged(start, nb);
      const int64_t pos = start + lane * 8;
      const int n = max(0, min(8, nb - lane * 8));
      Raw8 x;
      if (staged) {
        x.g = S.g[warp][lane];
        x.p0 = S.p[warp][2 * lane];
        x.p1 = S.p[warp][2 * lane + 1];
        x.m = S.m[warp][lane];
        x.v = S.v[warp][lane];
      } else {
        x = raw_from_global(a, pos, n);
      }
      const float sm = S.sc[2 * warp], sv = S.sc[2 * warp + 1];
      release_stage(&empty[s], lane);  // this warp no longer reads the stage
      Lane8 o;
      if (staged) adam_raw<true>(h, x, 8, sm, sv, o);
      else adam_raw<false>(h, x, n, sm, sv, o);
      QScale qm, qv;
      warp_block_scales(o.am, o.av, lane, qm, qv);
      store_state(a, pos, n, o, qm, qv);
      if (lane == 0) {
        a.m_scale[slot] = qm.s;
        a.v_scale[slot] = qv.s;
      }
      if (fp8) {
        if (b < kTmemRows && nb == 256) {
          __syncwarp();  // tcgen05 loads and stores are issued by the whole warp
          tmem_st8(tmem + uint32_t((b >> 2) * 8), o.p1);
        }
        // a strip row: lanes 0-15 cover column tile 0, lanes 16-31 tile 1
        const uint32_t ap = __reduce_max_sync(lane < 16 ? 0x0000FFFFu : 0xFFFF0000u, o.ap);
        if ((lane & 15) == 0) atomicMax(&s_tile[lane >> 4], ap);
      }
    }
    if (fp8) {
      __syncwarp();
      tmem_wait_st();
      consumer_sync();
      if (!dead) {
        for (int t = threadIdx.x; t < ntile; t += kCT) {
          const QScale q = qscale(s_tile[t], 448.f);
          a.fp8_scale[g.fslot + t] = q.s;
          s_tile[t] = __float_as_uint(q.r);
          s_tile[ntile + t] = __float_as_uint(q.s);
        }
      }
      consumer_sync();
      // rows held in TMEM: each warp converts the rows it updated (one 8-element
      // vector per lane; lanes 0-15 in column tile 0, 16-31 in tile 1)
      const int trows = dead ? 0 : min(nblk, kTmemRows);
      for (int b = warp; b < trows; b += kCons) {
        int64_t start;
        int nb, slot;
        region_block(g, b, start, nb, slot);
        const int n = max(0, min(8, nb - lane * 8));
        float pv[8];
        if (nb == 256) {
          __syncwarp();
          tmem_ld8(tmem + uint32_t((b >> 2) * 8), pv);
        } else {
#pragma unroll
          for (int i = 0; i < 8; ++i) pv[i] = i < n ? a.master[start + lane * 8 + i] : 0.f;
        }
        const int tile = lane >> 4;
        QScale qs;
        qs.r = __uint_as_float(s_tile[tile]);
        qs.s = __uint_as_float(s_tile[ntile + tile]);
        qs.mode = qs.s == 0.f ? 0 : (isinf(qs.r) ? 2 : 1);
        store_bytes(a.fp8 + start + lane * 8, codes_e4m3(pv, qs), n);
      }
      // the other rows: each thread converts two adjacent 8-element vectors of a
      // strip row (one 128-column tile) per pass, re-reading the master from L2
      const int npair = dead ? 0 : nel >> 4;
      for (int q = kTmemRows * 16 + threadIdx.x; q < npair; q += kCT) {
        const int r = q >> 4, kk = (q & 15) << 1;  // row, first of the two vectors
        const int64_t pos = g.pos + int64_t(r) * g.C + (kk << 3);
        const float4 p0 = *reinterpret_cast<const float4*>(a.master + pos);
        const float4 p1 = *reinterpret_cast<const float4*>(a.master + pos + 4);
        const float4 p2 = *reinterpret_cast<const float4*>(a.master + pos + 8);
        const float4 p3 = *reinterpret_cast<const float4*>(a.master + pos + 12);
        const int tile = kk >> 4;
        QScale qs;
        qs.r = __uint_as_float(s_tile[tile]);
        qs.s = __uint_as_float(s_tile[ntile + tile]);
        qs.mode = qs.s == 0.f ? 0 : (isinf(qs.r) ? 2 : 1);
        const float pa[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
        const float pb[8] = {p2.x, p2.y, p2.z, p2.w, p3.x, p3.y, p3.z, p3.w};
        const uint2 ca = codes_e4m3(pa, qs), cb = codes_e4m3(pb, qs);
        if ((g.pos & 15) == 0) {  // the region start fixes the alignment of every pair
          *reinterpret_cast<uint4*>(a.fp8 + pos) = make_uint4(ca.x, ca.y, cb.x, cb.y);
        } else {
          *reinterpret_cast<uint2*>(a.fp8 + pos) = ca;
          *reinterpret_cast<uint2*>(a.fp8 + pos + 8) = cb;
        }
      }
      consumer_sync();  // s_tile is reused by the next region
    }
  }
  if (FP8) {  // every consumer warp is done with TMEM before it is freed
    tc_fence_before();
    consumer_sync();
    if (warp == 0) {
      tc_fence_after();
      tmem_dealloc(s_tmem, kTmemCols);
    }
  }
}

// ---------------------------------------------------------------- 128x128 Adam tiles (+ FP8 of the same tile)
// Phase 1: Adam, write master, block-reduce max|m'|, max v', max|p'|; each
// vector's inputs (bf16 gradients, m codes, v codes: 32 bits an element) also
// go to tensor memory as loaded, and with FP8 its p' to shared memory (64 KB a
// tile).
// Its loads go in four rounds of two vectors a thread; each round first asks L2
// for the next round's lines (the last one for the next tile's first rows).
// Phase 2: requantise m', v' (recomputed bit-identically from those inputs and
// the old scales held in registers) and convert p' from shared memory.
// Thread t handles the tile's vectors t + 256 i (i < 8, a tile has at most 2048
// eight-element vectors); vector i's words live in the thread's TMEM lane (lane
// quarter warp % 4) at columns 64 (warp / 4) + 8 i .. + 7: 128 columns per CTA.

constexpr int kTileTmemCols = 128;
static_assert(kAdamCtas * kTileTmemCols <= 512, "the resident CTAs' TMEM columns fit one SM");

// row of vector v of a region with vpr vectors a row: full tile rows (vpr 16 or
// 4, a power of two, warp-uniform) take a shift instead of an integer division
__device__ __forceinline__ int vec_row(int v, int vpr) {
  return (vpr & (vpr - 1)) == 0 ? v >> (__ffs(vpr) - 1) : v / vpr;
}

// L2 prefetch of rows [r0, r0 + 32) of tile g: a row is 8 lines (master 4,
// gradient 2, m 1, v 1), one per thread.  Issued one load round ahead, it lets the
// next round's loads hit L2 without holding registers (prefetching a whole tile
// ahead instead thrashed L2: slower)
__device__ __forceinline__ void tile_prefetch(const RegionGroup& g, int r0, const AdamArgs& a) {
  const int r = r0 + (int(threadIdx.x) >> 3), kind = int(threadIdx.x) & 7;
  if (r >= g.rows) return;
  const int64_t row = g.pos + int64_t(r) * g.C;
  const void* p;
  if (kind < 4) {
    if (32 * kind >= g.width) return;
    p = a.master + row + 32 * kind;
  } else if (kind < 6) {
    if (64 * (kind - 4) >= g.width) return;
    p = a.grad + row + 64 * (kind - 4);
  } else {
    p = kind == 6 ? static_cast<const void*>(a.m + row) : static_cast<const void*>(a.v + row);
  }
  asm volatile("prefetch.global.L2 [%0];\n" ::"l"(p));
}

__device__ __forceinline__ void block_max(uint32_t x, uint32_t* red, int which) {
  x = __reduce_max_sync(0xFFFFFFFFu, x);
  if ((threadIdx.x & 31) == 0) red[which * kWarps + (threadIdx.x >> 5)] = x;
}

// A vector's inputs as they were loaded, in 8 tensor-memory words: the four
// words of bf16 gradient pairs, the two of m codes, the two of v codes (the
// same 32 bits an element as any packed form, with no repacking either way)
__device__ __forceinline__ void pack_inputs(const Raw8& x, uint32_t* w) {
  w[0] = x.g.x;
  w[1] = x.g.y;
  w[2] = x.g.z;
  w[3] = x.g.w;
  w[4] = x.m.x;
  w[5] = x.m.y;
  w[6] = x.v.x;
  w[7] = x.v.y;
}

__device__ __forceinline__ void unpack_inputs(const uint32_t* w, Raw8& x) {
  x.g = make_uint4(w[0], w[1], w[2], w[3]);
  x.m = make_uint2(w[4], w[5]);
  x.v = make_uint2(w[6], w[7]);
}

template <bool FP8>
__global__ void __launch_bounds__(kThreads, kAdamCtas) k_tile(const RegionGroup* __restrict__ groups, int ngroups, AdamArgs a) {
  __shared__ uint32_t red[3 * kWarps];
  __shared__ uint32_t s_tmem;
  // FP8: the tile's p', vector v (= 256 i + t) as float4s v and 2048 + v (a warp's
  // 16-byte accesses are contiguous, free of bank conflicts): the second phase
  // converts it from here instead of re-reading the master
  extern __shared__ float4 s_p[];
  const int warp = threadIdx.x >> 5;
  if (warp == 0) tmem_alloc(smem_u32(&s_tmem), kTileTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tcell = s_tmem + (uint32_t(32 * (warp & 3)) << 16) + uint32_t(64 * (warp >> 2));
  const Hp h = make_hp(a.hp);
  for (int gi = ngroups - 1 - int(blockIdx.x); gi >= 0; gi -= int(gridDim.x)) {
    const RegionGroup g = groups[gi];
    const bool fp8 = FP8 && g.fslot >= 0;
    const float sm = a.m_scale[g.mslot], sv = a.v_scale[g.mslot];
    const int vpr = g.width >> 3, nvec = g.rows * vpr;
    if (nvec > 8 * kThreads && threadIdx.x == 0) report(a.status, 8);  // not a 128x128 tile: the planner never emits one
    uint32_t am = 0, av = 0, ap = 0;
    // i advances by two (two vectors' loads in flight per thread); the loop test
    // is warp-uniform so the whole warp issues the TMEM stores
    for (int i = 0; i < 8 && kThreads * i + 32 * warp < nvec; i += 2) {
      const int v0 = threadIdx.x + kThreads * i, v1 = v0 + kThreads;
      const bool ok0 = v0 < nvec, ok1 = v1 < nvec;
      const int r0 = vec_row(v0, vpr), k0 = v0 - r0 * vpr;
      const int64_t pos0 = g.pos + int64_t(r0) * g.C + (k0 << 3);
      int64_t pos1 = pos0;
      if (ok1) {
        const int r1 = vec_row(v1, vpr), k1 = v1 - r1 * vpr;
        pos1 = g.pos + int64_t(r1) * g.C + (k1 << 3);
      }
      const Raw8 x0 = raw_from_global(a, pos0, ok0 ? 8 : 0);
      const Raw8 x1 = raw_from_global(a, pos1, ok1 ? 8 : 0);
      // the next 32 rows (or the next tile's first 32) into L2 while these are used
      if (i < 6) tile_prefetch(g, 16 * (i + 2), a);
      else if (gi >= int(gridDim.x)) tile_prefetch(groups[gi - int(gridDim.x)], 0, a);
      uint32_t w[8];
      pack_inputs(x0, w);
      __syncwarp();
      tmem_st8(tcell + uint32_t(8 * i), w);
      if (kThreads * (i + 1) + 32 * warp < nvec) {
        pack_inputs(x1, w);
        tmem_st8(tcell + uint32_t(8 * (i + 1)), w);
      }
      Lane8 o;
      if (ok0) {
        adam_raw<true>(h, x0, 8, sm, sv, o);
        store_p8(a.master + pos0, o.p1);
        if (fp8) {
          const int vi = kThreads * i + int(threadIdx.x);
          s_p[vi] = make_float4(o.p1[0], o.p1[1], o.p1[2], o.p1[3]);
          s_p[8 * kThreads + vi] = make_float4(o.p1[4], o.p1[5], o.p1[6], o.p1[7]);
        }
        am = max(am, o.am);
        av = max(av, o.av);
        ap = max(ap, o.ap);
      }
      if (ok1) {
        adam_raw<true>(h, x1, 8, sm, sv, o);
        store_p8(a.master + pos1, o.p1);
        if (fp8) {
          const int vi = kThreads * (i + 1) + int(threadIdx.x);
          s_p[vi] = make_float4(o.p1[0], o.p1[1], o.p1[2], o.p1[3]);
          s_p[8 * kThreads + vi] = make_float4(o.p1[4], o.p1[5], o.p1[6], o.p1[7]);
        }
        am = max(am, o.am);
        av = max(av, o.av);
        ap = max(ap, o.ap);
      }
    }
    block_max(am, red, 0);
    block_max(av, red, 1);
    block_max(ap, red, 2);
    __syncwarp();
    tmem_wait_st();
    __syncthreads();
    // each warp combines the 3 x kWarps maxima with one word a lane; lanes 0, 1
    // and 2 derive the m, v and p' scales side by side and the warp shares them
    static_assert(3 * kWarps <= 32, "one maximum word per lane");
    const int lane = threadIdx.x & 31;
    const uint32_t word = lane < 3 * kWarps ? red[lane] : 0u;
    const uint32_t tm = __reduce_max_sync(0xFFFFFFFFu, lane < kWarps ? word : 0u);
    const uint32_t tv = __reduce_max_sync(0xFFFFFFFFu, lane >= kWarps && lane < 2 * kWarps ? word : 0u);
    const uint32_t tp = __reduce_max_sync(0xFFFFFFFFu, lane >= 2 * kWarps ? word : 0u);
    const QScale q3 = qscale(lane == 0 ? tm : lane == 1 ? tv : tp, lane == 0 ? 127.f : lane == 1 ? 255.f : 448.f);
    auto take = [&](int from) {
      QScale q;
      q.s = __shfl_sync(0xFFFFFFFFu, q3.s, from);
      q.r = __shfl_sync(0xFFFFFFFFu, q3.r, from);
      q.mode = __shfl_sync(0xFFFFFFFFu, q3.mode, from);
      return q;
    };
    const QScale qm = take(0), qv = take(1), qp = take(2);
    if (threadIdx.x == 0) {
      a.m_scale[g.mslot] = qm.s;
      a.v_scale[g.mslot] = qv.s;
      if (fp8) a.fp8_scale[g.fslot] = qp.s;
    }
    for (int i = 0; i < 8 && kThreads * i + 32 * warp < nvec; ++i) {
      uint32_t w[8];
      __syncwarp();
      tmem_ld8(tcell + uint32_t(8 * i), w);
      const int v = threadIdx.x + kThreads * i;
      if (v < nvec) {
        const int r = vec_row(v, vpr), k = v - r * vpr;
        const int64_t pos = g.pos + int64_t(r) * g.C + (k << 3);
        Raw8 x;
        unpack_inputs(w, x);
        x.p0 = x.p1 = make_float4(0.f, 0.f, 0.f, 0.f);
        Lane8 o;
        adam_raw<true>(h, x, 8, sm, sv, o);
        *reinterpret_cast<uint2*>(a.m + pos) = codes_int8(o.m1, qm);
        *reinterpret_cast<uint2*>(a.v + pos) = codes_uint8(o.v1, qv);
        if (fp8) {  // this thread's p' of vector v, kept in shared memory by the first phase
          const float4 p0 = s_p[v], p1 = s_p[8 * kThreads + v];
          const float pv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
          *reinterpret_cast<uint2*>(a.fp8 + pos) = codes_e4m3(pv, qp);
        }
      }
    }
    __syncthreads();  // red and s_p are reused by the next tile
  }
  tc_fence_before();
  __syncthreads();  // every warp is done with TMEM before it is freed
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(s_tmem, kTileTmemCols);
  }
}

// ---------------------------------------------------------------- 32x32 Adam tiles
// The pages' own 8-bit Adam geometry (walkthrough of veScale-FSDP, paper section
// 6.3): 32x32 blocks of the 2-D view, kept whole on one device by a 32-row
// granularity.  A group is a 32-row band x <= 256 columns; warp w takes the
// group's tile w (1..4 eight-element vectors per row).  Phase 1: Adam over the
// tile, p' written, max|m'| and max v' reduced over the warp; each vector's
// inputs (bf16 gradients, m and v codes) also go to tensor memory as loaded.
// Phase 2: m' and v' recomputed bit-identically from those words and
// requantised.  Lane l handles the tile's vectors l + 32 i (i < 4); vector i's
// words live in the lane's TMEM row (lane quarter warp % 4) at columns
// 32 (warp / 4) + 8 i .. + 7: 64 columns per CTA.

constexpr int kTile32TmemCols = 64;
static_assert(kAdamCtas * kTile32TmemCols <= 512, "the resident CTAs' TMEM columns fit one SM");

__global__ void __launch_bounds__(kThreads, kAdamCtas) k_tile32(const RegionGroup* __restrict__ groups, int ngroups,
                                                              AdamArgs a) {
  __shared__ uint32_t s_tmem;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (warp == 0) tmem_alloc(smem_u32(&s_tmem), kTile32TmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tcell = s_tmem + (uint32_t(32 * (warp & 3)) << 16) + uint32_t(32 * (warp >> 2));
  const Hp h = make_hp(a.hp);
  for (int gi = ngroups - 1 - int(blockIdx.x); gi >= 0; gi -= int(gridDim.x)) {
    const RegionGroup g = groups[gi];
    const int c = warp << 5;
    if (c >= g.width) continue;  // warp-uniform
    const int vpr = min(32, g.width - c) >> 3;
    const int nvec = g.rows * vpr;
    if (nvec > 128 && lane == 0) report(a.status, 8);  // not a 32x32 tile: the planner never emits one
    const int slot = g.mslot + warp;
    const float sm = a.m_scale[slot], sv = a.v_scale[slot];
    auto vpos = [&](int v) {
      const int r = vec_row(v, vpr), k = v - r * vpr;
      return g.pos + int64_t(r) * g.C + c + (k << 3);
    };
    uint32_t am = 0, av = 0;
    for (int i = 0; i < 4 && 32 * i < nvec; i += 2) {  // two vectors' loads in flight per lane
      const int v0 = lane + 32 * i, v1 = v0 + 32;
      const bool ok0 = v0 < nvec, ok1 = v1 < nvec;
      const int64_t p0 = ok0 ? vpos(v0) : g.pos, p1 = ok1 ? vpos(v1) : g.pos;
      const Raw8 x0 = raw_from_global(a, p0, ok0 ? 8 : 0);
      const Raw8 x1 = raw_from_global(a, p1, ok1 ? 8 : 0);
      {  // this warp's next 16 rows (or the next group's first 16) into L2: lane -> row, two lines each
        const RegionGroup* ng = i == 0 ? &g : (gi >= int(gridDim.x) ? &groups[gi - int(gridDim.x)] : nullptr);
        const int r = (i == 0 ? 16 : 0) + (lane & 15);
        if (ng && c < ng->width && r < ng->rows) {
          const int64_t row = ng->pos + int64_t(r) * ng->C + c;
          if (lane < 16) {
            asm volatile("prefetch.global.L2 [%0];\n" ::"l"(a.master + row));
            asm volatile("prefetch.global.L2 [%0];\n" ::"l"(a.grad + row));
          } else {
            asm volatile("prefetch.global.L2 [%0];\n" ::"l"(a.m + row));
            asm volatile("prefetch.global.L2 [%0];\n" ::"l"(a.v + row));
          }
        }
      }
      uint32_t w[8];
      pack_inputs(x0, w);
      __syncwarp();  // tcgen05 loads and stores are issued by the whole warp
      tmem_st8(tcell + uint32_t(8 * i), w);
      if (32 * (i + 1) < nvec) {
        pack_inputs(x1, w);
        tmem_st8(tcell + uint32_t(8 * (i + 1)), w);
      }
      Lane8 o;
      if (ok0) {
        adam_raw<true>(h, x0, 8, sm, sv, o);
        store_p8(a.master + p0, o.p1);
        am = max(am, o.am);
        av = max(av, o.av);
      }
      if (ok1) {
        adam_raw<true>(h, x1, 8, sm, sv, o);
        store_p8(a.master + p1, o.p1);
        am = max(am, o.am);
        av = max(av, o.av);
      }
    }
    QScale qm, qv;
    warp_block_scales(am, av, lane, qm, qv);
    if (lane == 0) {
      a.m_scale[slot] = qm.s;
      a.v_scale[slot] = qv.s;
    }
    __syncwarp();
    tmem_wait_st();
    for (int i = 0; i < 4 && 32 * i < nvec; ++i) {
      uint32_t w[8];
      __syncwarp();
      tmem_ld8(tcell + uint32_t(8 * i), w);
      const int v = lane + 32 * i;
      if (v < nvec) {
        const int64_t pos = vpos(v);
        Raw8 x;
        unpack_inputs(w, x);
        x.p0 = x.p1 = make_float4(0.f, 0.f, 0.f, 0.f);
        Lane8 o;
        adam_raw<true>(h, x, 8, sm, sv, o);
        *reinterpret_cast<uint2*>(a.m + pos) = codes_int8(o.m1, qm);
        *reinterpret_cast<uint2*>(a.v + pos) = codes_uint8(o.v1, qv);
      }
    }
  }
  tc_fence_before();
  __syncthreads();  // every warp is done with TMEM before it is freed
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(s_tmem, kTile32TmemCols);
  }
}

// ---------------------------------------------------------------- Muon momentum and apply
// Muon around Newton-Schulz (walkthrough of veScale-FSDP, paper section 6.3): the
// momentum update runs on the local shards, the full momentum matrix is
// materialised for the root, and the root's result is applied back to the owned
// ranges.  One CTA per Muon piece (<= 8192 elements of one tensor interval).
//   k_muon_momentum: M = fma(mu, M, G) in fp32, stored; bf16(M) (nearest even)
//                    written to the tensor's row-major matrix at its offset
//   k_muon_apply:    W = fma(-lr_i, O_i, W), O_i the bf16 Newton-Schulz output

__global__ void __launch_bounds__(kThreads) k_muon_momentum(const PackPiece* __restrict__ pieces,
                                                            const uint16_t* __restrict__ grad, float* __restrict__ mom,
                                                            float mu, uint16_t* const* __restrict__ gather) {
  const PackPiece pc = pieces[blockIdx.x];
  uint16_t* out = gather[pc.tensor];
  if (!out) return;
  out += pc.src;
  const uint16_t* g = grad + pc.dst;
  float* m = mom + pc.dst;
  int e0 = 0;
  if ((pc.dst & 7) == 0 && (reinterpret_cast<uintptr_t>(out) & 15) == 0) {
    const int nv = pc.len >> 3;
    const float2 mu2 = dup(mu);
    for (int v = threadIdx.x; v < nv; v += kThreads) {
      const uint4 gw = reinterpret_cast<const uint4*>(g)[v];
      const float4 a = reinterpret_cast<const float4*>(m)[2 * v], b = reinterpret_cast<const float4*>(m)[2 * v + 1];
      const uint32_t w[4] = {gw.x, gw.y, gw.z, gw.w};
      const float mv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      float r[8];
      uint32_t o[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 gg = make_float2(bf16f(w[j] & 0xFFFFu), bf16f(w[j] >> 16));
        const float2 y = fma2(mu2, make_float2(mv[2 * j], mv[2 * j + 1]), gg);
        r[2 * j] = y.x;
        r[2 * j + 1] = y.y;
        o[j] = f2bf(y.x) | (f2bf(y.y) << 16);
      }
      reinterpret_cast<float4*>(m)[2 * v] = make_float4(r[0], r[1], r[2], r[3]);
      reinterpret_cast<float4*>(m)[2 * v + 1] = make_float4(r[4], r[5], r[6], r[7]);
      reinterpret_cast<uint4*>(out)[v] = make_uint4(o[0], o[1], o[2], o[3]);
    }
    e0 = nv << 3;
  }
  for (int e = e0 + threadIdx.x; e < pc.len; e += kThreads) {
    const float y = __fmaf_rn(mu, m[e], bf16f(g[e]));
    m[e] = y;
    out[e] = uint16_t(f2bf(y));
  }
}

__global__ void __launch_bounds__(kThreads) k_muon_apply(const PackPiece* __restrict__ pieces, float* __restrict__ master,
                                                         const uint16_t* const* __restrict__ upd,
                                                         const float* __restrict__ lr) {
  const PackPiece pc = pieces[blockIdx.x];
  const uint16_t* o = upd[pc.tensor];
  if (!o) return;
  o += pc.src;
  float* w = master + pc.dst;
  const float nlr = -lr[pc.tensor];
  int e0 = 0;
  if ((pc.dst & 7) == 0 && (reinterpret_cast<uintptr_t>(o) & 15) == 0) {
    const int nv = pc.len >> 3;
    const float2 n2 = dup(nlr);
    for (int v = threadIdx.x; v < nv; v += kThreads) {
      const uint4 ow = reinterpret_cast<const uint4*>(o)[v];
      const float4 a = reinterpret_cast<const float4*>(w)[2 * v], b = reinterpret_cast<const float4*>(w)[2 * v + 1];
      const uint32_t q[4] = {ow.x, ow.y, ow.z, ow.w};
      const float wv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
      float r[8];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 y = fma2(n2, make_float2(bf16f(q[j] & 0xFFFFu), bf16f(q[j] >> 16)),
                              make_float2(wv[2 * j], wv[2 * j + 1]));
        r[2 * j] = y.x;
        r[2 * j + 1] = y.y;
      }
      reinterpret_cast<float4*>(w)[2 * v] = make_float4(r[0], r[1], r[2], r[3]);
      reinterpret_cast<float4*>(w)[2 * v + 1] = make_float4(r[4], r[5], r[6], r[7]);
    }
    e0 = nv << 3;
  }
  for (int e = e0 + threadIdx.x; e < pc.len; e += kThreads) w[e] = __fmaf_rn(nlr, bf16f(o[e]), w[e]);
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
          const int r = vec_row(v, vpr), k = v - r * vpr;
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

// FP8 tiles (<= 128 x 128: the band-tile and tile lists) in two passes: the
// first reads the tile, reduces max|p'| and keeps rows 0-63 in shared memory
// (32 KB); the second converts those from shared memory and re-reads only rows
// 64-127 (from L2), so half as many lines must stay in L2 between the passes.
constexpr int kHalfVecs = 64 * 16;  // 8-element vectors in rows 0-63 of a 128-column tile
constexpr int kQuantTileCtas = 6;   // 197 KB of shared memory per SM (32 rows: 8 CTAs, 96 rows: 4 were slower)

__global__ void __launch_bounds__(kThreads) k_quant_tile(const RegionGroup* __restrict__ groups, int ngroups,
                                                         const float* __restrict__ master, uint8_t* __restrict__ fp8,
                                                         float* __restrict__ fp8_scale) {
  __shared__ float4 s_half[2 * kHalfVecs];  // vector v's halves at v and kHalfVecs + v
  __shared__ uint32_t red[kWarps];
  __shared__ QScale s_q;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int gi = blockIdx.x; gi < ngroups; gi += gridDim.x) {
    const RegionGroup g = groups[gi];
    if (g.fslot < 0) continue;  // uniform per CTA
    const int vpr = g.width >> 3, nvec = g.rows * vpr, nlow = min(nvec, 64 * vpr);
    uint32_t ap = 0;
    for (int v = threadIdx.x; v < nvec; v += kThreads) {
      const int r = vec_row(v, vpr), k = v - r * vpr;
      const int64_t pos = g.pos + int64_t(r) * g.C + (k << 3);
      const float4 p0 = *reinterpret_cast<const float4*>(master + pos);
      const float4 p1 = *reinterpret_cast<const float4*>(master + pos + 4);
      if (v < nlow) {
        s_half[v] = p0;
        s_half[kHalfVecs + v] = p1;
      }
      ap = max(ap, max(max(__float_as_uint(fabsf(p0.x)), __float_as_uint(fabsf(p0.y))),
                       max(__float_as_uint(fabsf(p0.z)), __float_as_uint(fabsf(p0.w)))));
      ap = max(ap, max(max(__float_as_uint(fabsf(p1.x)), __float_as_uint(fabsf(p1.y))),
                       max(__float_as_uint(fabsf(p1.z)), __float_as_uint(fabsf(p1.w)))));
    }
    ap = __reduce_max_sync(0xFFFFFFFFu, ap);
    if (lane == 0) red[warp] = ap;
    __syncthreads();
    if (warp == 0) {
      const uint32_t t = __reduce_max_sync(0xFFFFFFFFu, lane < kWarps ? red[lane] : 0u);
      if (lane == 0) {
        s_q = qscale(t, 448.f);
        fp8_scale[g.fslot] = s_q.s;
      }
    }
    __syncthreads();
    const QScale q = s_q;
    for (int v = threadIdx.x; v < nvec; v += kThreads) {
      const int r = vec_row(v, vpr), k = v - r * vpr;
      const int64_t pos = g.pos + int64_t(r) * g.C + (k << 3);
      float4 p0, p1;
      if (v < nlow) {
        p0 = s_half[v];
        p1 = s_half[kHalfVecs + v];
      } else {
        p0 = *reinterpret_cast<const float4*>(master + pos);
        p1 = *reinterpret_cast<const float4*>(master + pos + 4);
      }
      const float pv[8] = {p0.x, p0.y, p0.z, p0.w, p1.x, p1.y, p1.z, p1.w};
      *reinterpret_cast<uint2*>(fp8 + pos) = codes_e4m3(pv, q);
    }
    __syncthreads();  // s_half, red and s_q are reused by the next tile
  }
}

// ---------------------------------------------------------------- the bf16 view after the AllGather
// Compute reads each gathered FP8 parameter as code x tile scale: the E4M3 code
// decoded exactly (every E4M3 value is a half), times the fp32 scale (one fp32
// rounding), rounded to bf16 (nearest even).  Only FP8 tiles are written.

__device__ __forceinline__ uint4 dequant8(uint2 w, float s) {
  const uint32_t b[2] = {w.x, w.y};
  uint32_t o[4];
  const float2 s2 = dup(s);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const __nv_fp8x2_storage_t pair = __nv_fp8x2_storage_t((b[j >> 1] >> (16 * (j & 1))) & 0xFFFFu);
    const __half2 h = __half2(__nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3));
    const float2 x = mul2(__half22float2(h), s2);
    o[j] = f2bf(x.x) | (f2bf(x.y) << 16);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

__device__ __forceinline__ uint16_t dequant1(uint8_t c, float s) {
  const __half h = __half(__nv_cvt_fp8_to_halfraw(__nv_fp8_storage_t(c), __NV_E4M3));
  return uint16_t(f2bf(__fmul_rn(__half2float(h), s)));
}

__global__ void __launch_bounds__(kThreads) k_dequant_flat(const FlatGroup* __restrict__ groups,
                                                           const uint8_t* __restrict__ fp8,
                                                           const float* __restrict__ fp8_scale,
                                                           uint16_t* __restrict__ out) {
  const FlatGroup g = groups[blockIdx.x];
  if (g.fslot < 0) return;
  const int nv = g.nelem >> 3;
  for (int v = threadIdx.x; v < nv; v += kThreads) {
    const int e = v << 3;  // 8 elements never cross a 128-element tile
    const int64_t pos = g.pos + e;
    *reinterpret_cast<uint4*>(out + pos) =
        dequant8(*reinterpret_cast<const uint2*>(fp8 + pos), fp8_scale[g.fslot + (e >> 7)]);
  }
  for (int e = (nv << 3) + threadIdx.x; e < g.nelem; e += kThreads)
    out[g.pos + e] = dequant1(fp8[g.pos + e], fp8_scale[g.fslot + (e >> 7)]);
}

__global__ void __launch_bounds__(kThreads) k_dequant_region(const RegionGroup* __restrict__ groups, int ngroups,
                                                             const uint8_t* __restrict__ fp8,
                                                             const float* __restrict__ fp8_scale,
                                                             uint16_t* __restrict__ out) {
  for (int gi = blockIdx.x; gi < ngroups; gi += gridDim.x) {
    const RegionGroup g = groups[gi];
    if (g.fslot < 0) continue;
    const bool flat = g.width == g.C;
    const int nvec = (g.rows * g.width) >> 3, vpr = g.width >> 3;
    for (int v = threadIdx.x; v < nvec; v += kThreads) {
      int64_t pos;
      int col;
      if (flat) {
        const uint32_t e = uint32_t(v) << 3;
        col = int(e - fastdiv(e, g.cmul, g.cshr) * uint32_t(g.C));
        pos = g.pos + e;
      } else {
        const int r = vec_row(v, vpr), k = v - r * vpr;
        col = k << 3;
        pos = g.pos + int64_t(r) * g.C + col;
      }
      *reinterpret_cast<uint4*>(out + pos) =
          dequant8(*reinterpret_cast<const uint2*>(fp8 + pos), fp8_scale[g.fslot + (col >> 7)]);
    }
  }
}

// ---------------------------------------------------------------- bounded-wait self-test
// One thread waits on an mbarrier that nothing arrives at, through the same wait
// loop as the step kernels but with a short limit, and records code 7 when the
// wait gives up (1 if it ever completed, which cannot happen).
__global__ void k_wait_selftest(int* status, long long limit) {
  __shared__ __align__(8) uint64_t bar;
  mbar_init(&bar, 1);
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
  const bool done = mbar_wait_for(&bar, 0, limit);
  *status = done ? 1 : 7;
}

int check_launch(const char* what) {
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(BQ_ECUDA, std::string(what) + ": " + cudaGetErrorString(e));
  return BQ_OK;
}

constexpr int kQuantCtasPerSm = kAdamCtas;
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
  if (t.n_flat32) {
    k_flat<1><<<t.n_flat32, kThreads, 0, s>>>(t.flat32, a);
    if (int rc = check_launch("bq_step_adam8 (flat32)")) return rc;
  }
  if (t.n_tiles32) {
    k_tile32<<<std::min(t.n_tiles32, sms * kAdamCtas), kThreads, 0, s>>>(t.tiles32, t.n_tiles32, a);
    if (int rc = check_launch("bq_step_adam8 (tiles32)")) return rc;
  }
  if (t.n_strips) {
    const int grid = std::min(t.n_strips, sms * kStripCtas);
    const size_t smem = sizeof(TmaStage) * kRing + 2 * kRing * sizeof(uint64_t) +
                        2 * size_t(t.max_strip_tiles) * sizeof(uint32_t);
    if (once_per_device(kOnceStripAttr)) {  // the attribute belongs to the current device
      // the 227 KB opt-in limit covers static and dynamic shared memory; 1 KB is
      // left for the static part (k_strip<true> keeps its TMEM address there)
      constexpr int kDyn = 227 * 1024 - 1024;
      if (cudaFuncSetAttribute(k_strip<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDyn) != cudaSuccess ||
          cudaFuncSetAttribute(k_strip<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kDyn) != cudaSuccess)
        return check_launch("bq_step_adam8 (strip shared memory attribute)");
    }
    if (fp8)
      k_strip<true><<<grid, kStripThreads, smem, s>>>(t.strips, t.n_strips, a);
    else
      k_strip<false><<<grid, kStripThreads, smem, s>>>(t.strips, t.n_strips, a);
    if (int rc = check_launch("bq_step_adam8 (strips)")) return rc;
  }
  if (fp8 && t.n_band_tiles) {
    // FP8 of tensors whose Adam ran as band pieces: two passes per tile over the
    // just-written master, half the tile held on chip between them
    k_quant_tile<<<std::min(t.n_band_tiles, sms * kQuantTileCtas), kThreads, 0, s>>>(
        t.band_tiles, t.n_band_tiles, a.master, a.fp8, a.fp8_scale);
    if (int rc = check_launch("bq_step_adam8 (band FP8 tiles)")) return rc;
  }
  if (t.n_tiles) {
    const int grid = std::min(t.n_tiles, sms * kTileCtasPerSm);
    constexpr int kTileP = 8 * kThreads * 2 * int(sizeof(float4));  // a 128x128 tile's p' (64 KB)
    if (once_per_device(kOnceTileAttr) &&
        cudaFuncSetAttribute(k_tile<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTileP) != cudaSuccess)
      return check_launch("bq_step_adam8 (tile shared memory attribute)");
    if (fp8)
      k_tile<true><<<grid, kThreads, kTileP, s>>>(t.tiles, t.n_tiles, a);
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
    k_quant_region<<<std::min(t.n_strips, sms * kQuantCtasPerSm), kThreads, smem, s>>>(t.strips, t.n_strips, master,
                                                                                        fp8, fp8_scale);
    if (int rc = check_launch("bq_quant_fp8 (strips)")) return rc;
  }
  if (t.n_band_tiles) {
    k_quant_tile<<<std::min(t.n_band_tiles, sms * kQuantTileCtas), kThreads, 0, s>>>(t.band_tiles, t.n_band_tiles,
                                                                                     master, fp8, fp8_scale);
    if (int rc = check_launch("bq_quant_fp8 (band tiles)")) return rc;
  }
  if (t.n_tiles) {
    k_quant_tile<<<std::min(t.n_tiles, sms * kQuantTileCtas), kThreads, 0, s>>>(t.tiles, t.n_tiles, master, fp8,
                                                                                fp8_scale);
    if (int rc = check_launch("bq_quant_fp8 (tiles)")) return rc;
  }
  return BQ_OK;
}

int launch_dequant_fp8(const DevTables& t, const uint8_t* fp8, const float* fp8_scale, uint16_t* out, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int sms = sm_count();
  if (t.n_flat256) {
    k_dequant_flat<<<t.n_flat256, kThreads, 0, s>>>(t.flat256, fp8, fp8_scale, out);
    if (int rc = check_launch("bq_dequant_fp8 (flat256)")) return rc;
  }
  if (t.n_flat128) {
    k_dequant_flat<<<t.n_flat128, kThreads, 0, s>>>(t.flat128, fp8, fp8_scale, out);
    if (int rc = check_launch("bq_dequant_fp8 (flat128)")) return rc;
  }
  if (t.n_strips) {
    k_dequant_region<<<std::min(t.n_strips, sms * 8), kThreads, 0, s>>>(t.strips, t.n_strips, fp8, fp8_scale, out);
    if (int rc = check_launch("bq_dequant_fp8 (strips)")) return rc;
  }
  if (t.n_tiles) {
    k_dequant_region<<<std::min(t.n_tiles, sms * 8), kThreads, 0, s>>>(t.tiles, t.n_tiles, fp8, fp8_scale, out);
    if (int rc = check_launch("bq_dequant_fp8 (tiles)")) return rc;
  }
  if (t.n_band_tiles) {
    k_dequant_region<<<std::min(t.n_band_tiles, sms * 8), kThreads, 0, s>>>(t.band_tiles, t.n_band_tiles, fp8,
                                                                           fp8_scale, out);
    if (int rc = check_launch("bq_dequant_fp8 (band tiles)")) return rc;
  }
  return BQ_OK;
}

int launch_wait_selftest(int* status, void* stream) {
  k_wait_selftest<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(status, 1LL << 21);  // about a millisecond
  return check_launch("bq_wait_selftest");
}

int launch_muon_momentum(const DevTables& t, const uint16_t* grad, float* mom, float mu, uint16_t* const* gather,
                         void* stream) {
  if (!t.n_muon) return BQ_OK;
  k_muon_momentum<<<t.n_muon, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(t.muon, grad, mom, mu, gather);
  return check_launch("bq_muon_momentum");
}

int launch_muon_apply(const DevTables& t, float* master, const uint16_t* const* upd, const float* lr, void* stream) {
  if (!t.n_muon) return BQ_OK;
  k_muon_apply<<<t.n_muon, kThreads, 0, static_cast<cudaStream_t>(stream)>>>(t.muon, master, upd, lr);
  return check_launch("bq_muon_apply");
}

}  // namespace bq
