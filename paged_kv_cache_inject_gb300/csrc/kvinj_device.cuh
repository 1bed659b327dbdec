// kvinj_device.cuh -- device helpers shared by the sm_103a kernels: 16-bit
// element conversions, the RoPE pair rotation, status reporting, and inline
// PTX for mbarriers, 1-D/2-D TMA bulk copies and named barriers.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kvinj.h"

namespace kvinj {

// ---------------------------------------------------------------------------
// status
// ---------------------------------------------------------------------------
__device__ __forceinline__ void report(int32_t *status, int bits) {
  if (status) atomicOr(status, bits);
}

// ---------------------------------------------------------------------------
// 16-bit <-> fp32. DT 0 = bf16, 1 = fp16. A 32-bit word holds two elements,
// the lower address in the low half.
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
  if constexpr (DT == 0) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  } else {
    __half2 h = *reinterpret_cast<__half2 *>(&w);
    return __half22float2(h);
  }
}

template <int DT>
__device__ __forceinline__ uint32_t pack2(float a, float b) {  // round to nearest even
  if constexpr (DT == 0) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
  } else {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
  }
}

// 2^x by the special-function unit's approximation (ex2.approx.ftz: relative error near
// 2^-22; 2^-inf = +0). The softmax kernels call it with x <= their lazy-maximum threshold;
// it is several times cheaper per element here than exp2f.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// RoPE rotation of one pair (a = x_i, b = x_{i+D/2}) by the angle whose cos
// and sin are c = t.x + t.z and s = t.y + t.w (hi + lo parts of the fp64
// values). Rotate-half convention: y_i = a c - b s, y_{i+D/2} = b c + a s.
//
// The products with the hi parts are split with fma (t = b*s_hi is exact up
// to et = fma(b, s_hi, -t)), so the result carries an error of a few fp32
// ulps of |y| plus ~2^-46 |x|, rather than 2^-24 |x|. That keeps the value
// rounded to bf16/fp16 within one ulp of the exactly rounded rotation even
// where a c and b s nearly cancel.
// ---------------------------------------------------------------------------
__device__ __forceinline__ float2 rope_pair(float a, float b, float4 t) {
  const float ch = t.x, sh = t.y, cl = t.z, sl = t.w;
  // first: a*c - b*s
  float t1 = b * sh;
  float e1 = __fmaf_rn(b, sh, -t1);
  float u1 = __fmaf_rn(a, ch, -t1);
  float r1 = __fmaf_rn(a, cl, -(b * sl)) - e1;
  // second: b*c + a*s
  float t2 = a * sh;
  float e2 = __fmaf_rn(a, sh, -t2);
  float u2 = __fmaf_rn(b, ch, t2);
  float r2 = __fmaf_rn(b, cl, a * sl) + e2;
  return make_float2(u1 + r1, u2 + r2);
}

// ---------------------------------------------------------------------------
// Exactly rounded rotation (the int8 paths). The stored 16-bit key must be the
// rounding of the fp64 rotation a*c - b*s, b*c + a*s (products and sum each
// rounded in fp64) with c, s the fp64 table values: the int8 code of a row
// depends on every bit of it. rope_pair's fp32 result y differs from the exact
// a*C - b*S (C, S = the hi + lo table values) by less than 2^-23|y| +
// 2^-44(|a| + |b|), and C, S differ from the fp64 values by less than 2^-48,
// so with E = 2^-22|y| + 2^-43(|a| + |b|) the fp64 result lies in
// [y - E, y + E]. When both ends of that interval round to the same 16-bit
// value, so does the fp64 result; otherwise (a rounding boundary inside the
// interval, about 2^-14 of the elements for bf16) the rotation is recomputed
// in fp64 from the fp64 table, with the fp64 operations in the same order.
// ---------------------------------------------------------------------------
template <int DT>
__device__ __forceinline__ uint16_t f32_to16(float x) {
  if constexpr (DT == 0) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  else return __half_as_ushort(__float2half_rn(x));
}

// round-to-nearest-even of an fp64 value to the 16-bit type: round to odd into
// fp32 (truncate; set the last bit when inexact), then to nearest even -- the
// same result as a single rounding, fp32 carrying more than two extra bits
// (Boldo and Melquiond, "Emulation of FMA and correctly rounded sums: proved
// algorithms using rounding to odd", IEEE Trans. Computers 57(4), 2008)
template <int DT>
__device__ __forceinline__ uint16_t f64_to16(double x) {
  float f = __double2float_rz(x);
  if ((double)f != x) f = __uint_as_float(__float_as_uint(f) | 1u);
  return f32_to16<DT>(f);
}

template <int DT>
__device__ __forceinline__ bool rounds_alike(float y, float e) {
  return f32_to16<DT>(__fsub_rd(y, e)) == f32_to16<DT>(__fadd_ru(y, e));
}

// bf16: whether every value within 2^-22|y| + 2^-43(|a| + |b|) of y rounds as y does, from
// y's bits alone in the common case: a bf16 rounding boundary is an fp32 whose low 16 bits
// are 0x8000, so |low16 - 0x8000| is y's distance to the nearest one in fp32 ulps of y;
// 2^-22|y| is under 4 of those ulps, and 2^-43(|a| + |b|) under one while |y| >= 2^-18
// (|a| + |b|). Anything else (near a boundary, heavy cancellation, zero) reports false and
// takes the exact path.
__device__ __forceinline__ bool bf16_rounding_safe(float y, float ab) {
  const uint32_t t = __float_as_uint(y);
  const int d = abs((int)(t & 0xFFFFu) - 0x8000);
  return d > 6 && fabsf(y) > 0x1p-18f * ab;
}

// rotated pair (a, b) at the position whose table entries are t (float hi/lo)
// and *t64 (fp64 {cos, sin}), each output rounded once to the 16-bit type
template <int DT>
__device__ __forceinline__ ushort2 rope_pair_exact(float a, float b, float4 t,
                                                   const double2 *t64) {
  const float2 y = rope_pair(a, b, t);
  const float ab = fabsf(a) + fabsf(b);
  bool safe;
  if constexpr (DT == 0) {
    safe = bf16_rounding_safe(y.x, ab) && bf16_rounding_safe(y.y, ab);
  } else {
    const float base = 0x1p-43f * ab;
    safe = rounds_alike<DT>(y.x, __fmaf_ru(0x1p-22f, fabsf(y.x), base)) &&
           rounds_alike<DT>(y.y, __fmaf_ru(0x1p-22f, fabsf(y.y), base));
  }
  if (safe) return make_ushort2(f32_to16<DT>(y.x), f32_to16<DT>(y.y));
  const double2 cs = *t64;
  const double da = a, db = b;
  const double r0 = __dsub_rn(__dmul_rn(da, cs.x), __dmul_rn(db, cs.y));
  const double r1 = __dadd_rn(__dmul_rn(db, cs.x), __dmul_rn(da, cs.y));
  return make_ushort2(f64_to16<DT>(r0), f64_to16<DT>(r1));
}

// ---------------------------------------------------------------------------
// int8 row quantization ("Latency Optimization > KV Cache Management", KV cache
// quantization): s = max|x| / 127 rounded to fp32 (one correctly rounded fp32
// division gives the fp64 quotient's fp32 rounding here: the quotient of a
// 16-bit value by 127 never lies within the fp64 rounding error of an fp32
// rounding boundary), code = x / s rounded to nearest even, clamped to
// [-127, 127]. The code is decided exactly: c0 = rint(x * (1/s)) is within one
// of it (the product is within 2^-16 of the quotient, which is below 128), and
// the signs of x - (c0 +- 1/2) s, each computed with one fma (rounding keeps the
// sign and keeps zero as zero), say whether the exact quotient lies past a
// half-way point or on it. inv = the row's 1/s (any nearby value will do).
// ---------------------------------------------------------------------------
__device__ __forceinline__ float quant_scale(float amax) { return __fdiv_rn(amax, 127.f); }
__device__ __forceinline__ float quant_inv(float s) { return s > 0.f ? __frcp_rn(s) : 0.f; }

__device__ __forceinline__ int quant_code(float x, float s, float inv) {
  if (!(s > 0.f)) return 0;
  const float q = x * inv, c0 = rintf(q);
  // the product is within 2^-16 of the quotient: away from a half-way point c0 is the code
  if (fabsf(q - c0) < 0.4995f) return min(max((int)c0, -127), 127);
  const float hi = __fmaf_rn(-(c0 + 0.5f), s, x);  // x - (c0 + 1/2) s
  const float lo = __fmaf_rn(-(c0 - 0.5f), s, x);  // x - (c0 - 1/2) s
  const int ci = (int)c0, odd = ci & 1;
  int c = ci;
  if (hi > 0.f || (hi == 0.f && odd)) c = ci + 1;        // past c0 + 1/2, or a tie: the even one
  else if (lo < 0.f || (lo == 0.f && odd)) c = ci - 1;
  return min(max(c, -127), 127);
}

// ---------------------------------------------------------------------------
// cache-hinted global memory access
// ---------------------------------------------------------------------------
template <int BYTES>
struct Vec;
template <>
struct Vec<4> {
  using T = uint32_t;
};
template <>
struct Vec<8> {
  using T = uint2;
};
template <>
struct Vec<16> {
  using T = uint4;
};

// streaming read (read once: do not keep in L1)
__device__ __forceinline__ uint32_t ld_stream(const uint32_t *p) {
  uint32_t v;
  asm volatile("ld.global.nc.L1::no_allocate.b32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ld_stream(const uint2 *p) {
  uint2 v;
  asm volatile("ld.global.nc.L1::no_allocate.v2.b32 {%0, %1}, [%2];"
               : "=r"(v.x), "=r"(v.y)
               : "l"(p));
  return v;
}
__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ void st_global(uint32_t *p, uint32_t v) {
  asm volatile("st.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_global(uint2 *p, uint2 v) {
  asm volatile("st.global.v2.b32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}
__device__ __forceinline__ void st_global(uint4 *p, uint4 v) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// ---------------------------------------------------------------------------
// shared memory, mbarriers, TMA
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar_addr, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar_addr), "r"(parity)
      : "memory");
  return ok != 0;
}

// non-blocking test of the phase with `parity`
__device__ __forceinline__ bool mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// A wait that gives up: true when the phase with `parity` completed, false
// after ~`limit_ns` of wall time or 2^26 polls, whichever comes first. A
// legitimate wait in these kernels lasts microseconds.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity,
                                                  uint64_t limit_ns = 1000000000ull) {
  uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0; i < (1u << 26); ++i) {
    if (mbar_try_wait(a, parity)) return true;
    if ((i & 255u) == 255u && globaltimer_ns() - t0 > limit_ns) return false;
  }
  return false;
}

// 2-D tiled TMA load of one box into shared memory, completion counted on `bar`
__device__ __forceinline__ void tma_load_2d(void *smem_dst, const CUtensorMap *map, int32_t x,
                                            int32_t y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

// 1-D bulk copy global -> shared (both 16-byte aligned, bytes % 16 == 0),
// completion counted on `bar`
__device__ __forceinline__ void bulk_load(void *smem_dst, const void *gsrc, uint32_t bytes,
                                          uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// hint: bring the line holding p into L2 (and its address translation)
__device__ __forceinline__ void prefetch_l2(const void *p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// programmatic dependent launch: let the next kernel on the stream (launched
// with the programmatic serialization attribute) start; it waits with
// griddep_wait until this grid has completed and its writes are visible
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// named barrier over `nthreads` threads (a multiple of 32)
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint32_t lds32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr));
  return v;
}

}  // namespace kvinj
