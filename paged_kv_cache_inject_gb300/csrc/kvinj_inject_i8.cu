// kvinj_inject_i8.cu -- inject and append into an int8 paged cache.
//
// "Latency Optimization > KV Cache Management", KV cache quantization: storing
// the cache as int8 halves its bytes. Each stored row (one token of one kv
// head, D = 128 values) is quantized on its own, symmetrically, with one fp32
// scale (quant_scale / quant_code in kvinj_device.cuh). Keys are rotated at
// their absolute position first ("InferScale" §3.3: RoPE applied to the
// stored pre-RoPE keys at the assigned positions) and rounded once to the
// 16-bit type exactly as the fp64 rotation would be (rope_pair_exact), so that
// the codes are those of the 16-bit rotated key the unquantized cache holds.
//
// Layout: codes [L][num_blocks][Hkv][16][D] int8 (one 128-byte row per token
// and head), scales [L][num_blocks][Hkv][16] fp32. The work split is the one
// of the 16-bit inject: a warp takes one (chunk, layer, token) -- or one
// appended token -- and each 16-lane half-warp one row, lane k owning elements
// [4k, 4k + 4) and [64 + 4k, 64 + 4k + 4), so a rotate-half pair sits in one
// lane and a row's maximum is a reduction over the 16 lanes of its half.
#include "kvinj_device.cuh"
#include "kvinj_internal.h"

namespace kvinj {

namespace {

constexpr int D8 = 128, E8 = 4, HALF8 = 64, RB8 = 4;

// quantize a row held as x[0..3] = elements [4k, 4k + 4), x[4..7] = [64 + 4k, ..) by the
// 16 lanes of a half-warp; store its codes and (lane k == 0) its scale. Every lane of the
// warp takes part in the reduction; `live` = false (a head past Hkv) stores nothing.
__device__ __forceinline__ void quant_store(const float (&x)[8], int k, int8_t *codes,
                                            float *scale, bool live) {
  float m = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(x[i]));
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float s = quant_scale(m), inv = quant_inv(s);
  uint32_t w[2];
#pragma unroll
  for (int hh = 0; hh < 2; ++hh) {
    uint32_t v = 0;
#pragma unroll
    for (int e = 0; e < E8; ++e)
      v |= (uint32_t)(quant_code(x[hh * 4 + e], s, inv) & 0xFF) << (8 * e);
    w[hh] = v;
  }
  if (!live) return;
  st_global(reinterpret_cast<uint32_t *>(codes + E8 * k), w[0]);
  st_global(reinterpret_cast<uint32_t *>(codes + HALF8 + E8 * k), w[1]);
  if (k == 0) *scale = s;
}

template <int DT>
__device__ __forceinline__ float from16(uint16_t b) {
  if constexpr (DT == 0) return __uint_as_float((uint32_t)b << 16);
  else return __half2float(__ushort_as_half(b));
}

// the Hkv K rows (rotated at the position whose table rows are rot / rot64, or taken as
// given when rot == nullptr) and Hkv V rows of one token: source row of head h at
// sk / sv + h * D, destination row (codes) at dk / dv + h * 16 * D, scale at ks / vs + h * 16
template <int DT>
__device__ __forceinline__ void token_i8(const uint16_t *sk, const uint16_t *sv, int8_t *dk,
                                         int8_t *dv, float *ks, float *vs, int Hkv,
                                         const float4 *rot, const double2 *rot64, int lane) {
  const int half = lane >> 4, k = lane & 15;
  float4 tab[E8];
  if (rot) {
#pragma unroll
    for (int e = 0; e < E8; ++e) tab[e] = __ldg(rot + k * E8 + e);
  }
  for (int h0 = 0; h0 < Hkv; h0 += 2 * RB8) {
    uint2 klo[RB8], khi[RB8], vlo[RB8], vhi[RB8];
#pragma unroll
    for (int i = 0; i < RB8; ++i) {
      const int h = h0 + 2 * i + half;
      klo[i] = khi[i] = vlo[i] = vhi[i] = make_uint2(0, 0);
      if (h < Hkv) {
        const uint16_t *a = sk + (int64_t)h * D8 + k * E8;
        const uint16_t *b = sv + (int64_t)h * D8 + k * E8;
        klo[i] = ld_stream(reinterpret_cast<const uint2 *>(a));
        khi[i] = ld_stream(reinterpret_cast<const uint2 *>(a + HALF8));
        vlo[i] = ld_stream(reinterpret_cast<const uint2 *>(b));
        vhi[i] = ld_stream(reinterpret_cast<const uint2 *>(b + HALF8));
      }
    }
#pragma unroll
    for (int i = 0; i < RB8; ++i) {
      const int h = h0 + 2 * i + half;
      const bool live = h < Hkv;
      const uint16_t ka[4] = {(uint16_t)klo[i].x, (uint16_t)(klo[i].x >> 16), (uint16_t)klo[i].y,
                              (uint16_t)(klo[i].y >> 16)};
      const uint16_t kb[4] = {(uint16_t)khi[i].x, (uint16_t)(khi[i].x >> 16), (uint16_t)khi[i].y,
                              (uint16_t)(khi[i].y >> 16)};
      float x[8];
#pragma unroll
      for (int e = 0; e < E8; ++e) {
        if (rot && live) {
          const ushort2 y = rope_pair_exact<DT>(from16<DT>(ka[e]), from16<DT>(kb[e]), tab[e],
                                                rot64 + k * E8 + e);
          x[e] = from16<DT>(y.x);
          x[4 + e] = from16<DT>(y.y);
        } else {
          x[e] = from16<DT>(ka[e]);
          x[4 + e] = from16<DT>(kb[e]);
        }
      }
      quant_store(x, k, dk + (int64_t)h * 16 * D8, ks + h * 16, live);
      const uint16_t va[4] = {(uint16_t)vlo[i].x, (uint16_t)(vlo[i].x >> 16), (uint16_t)vlo[i].y,
                              (uint16_t)(vlo[i].y >> 16)};
      const uint16_t vb[4] = {(uint16_t)vhi[i].x, (uint16_t)(vhi[i].x >> 16), (uint16_t)vhi[i].y,
                              (uint16_t)(vhi[i].y >> 16)};
#pragma unroll
      for (int e = 0; e < E8; ++e) {
        x[e] = from16<DT>(va[e]);
        x[4 + e] = from16<DT>(vb[e]);
      }
      quant_store(x, k, dv + (int64_t)h * 16 * D8, vs + h * 16, live);
    }
  }
}

template <int DT>
__global__ void __launch_bounds__(256) inject_i8_kernel(I8Args a) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t c = a.chunk_len;
  const int64_t n_units = a.n * a.n_layers * c;
  const int64_t row = (int64_t)a.Hkv * D8;
  const int64_t nslots = a.num_blocks * a.B;
  for (int64_t u = warp; u < n_units; u += nwarps) {
    const int t = (int)(u % c);
    const int64_t jl = u / c;
    const int l = a.layer_begin + (int)(jl % a.n_layers);
    const int64_t j = jl / a.n_layers;
    const int id = a.chunk_ids[j];
    const int64_t slot = a.slot_mapping[j * c + t];
    const int pos = a.start_pos[j] + t;
    int bad = 0;
    if (id < 0 || id >= a.num_chunks) bad |= KVINJ_ST_BAD_CHUNK;
    if (slot < 0 || slot >= nslots) bad |= KVINJ_ST_BAD_SLOT;
    if (pos < 0 || pos >= a.max_pos) bad |= KVINJ_ST_BAD_POS;
    if (bad) {
      if (lane == 0) report(a.status, bad);
      continue;
    }
    const uint16_t *sk = a.src_k + (((int64_t)id * a.L + l) * 2 * c + t) * row;
    const int64_t r0 = ((int64_t)l * a.num_blocks + slot / a.B) * a.Hkv * a.B + slot % a.B;
    token_i8<DT>(sk, sk + c * row, a.k + r0 * D8, a.v + r0 * D8, a.ks + r0, a.vs + r0, a.Hkv,
                 a.rope + (int64_t)pos * (D8 / 2), a.rope64 + (int64_t)pos * (D8 / 2), lane);
  }
}

template <int DT>
__global__ void __launch_bounds__(256) append_i8_kernel(I8Args a) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t row = (int64_t)a.Hkv * D8;
  const int64_t nslots = a.num_blocks * a.B;
  for (int64_t i = warp; i < a.n; i += nwarps) {
    const int pos = a.positions[i];
    const int64_t slot = a.slot_mapping[i];
    int bad = 0;
    if (pos < 0 || (a.rope && pos >= a.max_pos)) bad |= KVINJ_ST_BAD_POS;
    if (slot < 0 || slot >= nslots) bad |= KVINJ_ST_BAD_SLOT;
    if (bad) {
      if (lane == 0) report(a.status, bad);
      continue;
    }
    const int64_t r0 = ((int64_t)a.layer * a.num_blocks + slot / a.B) * a.Hkv * a.B + slot % a.B;
    token_i8<DT>(a.src_k + i * row, a.src_v + i * row, a.k + r0 * D8, a.v + r0 * D8, a.ks + r0,
                 a.vs + r0, a.Hkv, a.rope ? a.rope + (int64_t)pos * (D8 / 2) : nullptr,
                 a.rope ? a.rope64 + (int64_t)pos * (D8 / 2) : nullptr, lane);
  }
}

int grid_for(int64_t warps_of_work) {
  int64_t ctas = (warps_of_work + 7) / 8;
  const int64_t cap = (int64_t)num_sms() * 8;
  if (ctas > cap) ctas = cap;
  return (int)(ctas < 1 ? 1 : ctas);
}

}  // namespace

cudaError_t launch_inject_i8(const I8Args &a, int dtype, cudaStream_t s) {
  const int grid = grid_for(a.n * a.n_layers * a.chunk_len);
  if (dtype == 0) inject_i8_kernel<0><<<grid, 256, 0, s>>>(a);
  else inject_i8_kernel<1><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_append_i8(const I8Args &a, int dtype, cudaStream_t s) {
  const int grid = grid_for(a.n);
  if (dtype == 0) append_i8_kernel<0><<<grid, 256, 0, s>>>(a);
  else append_i8_kernel<1><<<grid, 256, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace kvinj
