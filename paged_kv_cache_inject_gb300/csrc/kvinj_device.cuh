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
