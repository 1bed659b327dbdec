// kvinj_decode.cu -- split-K paged GQA decode attention, CUDA-core consumer.
//
// Computes, per request r and query head qh (kv head h = qh / G):
//   out = sum_p softmax_p(scale * (R_{q_pos} q) . K_p) V_p
// over the request's context, read block by block through its block table
// ("LLM Inference: KV Caching": attention softmax(QK^T/sqrt d)V and "Paged
// attention"; "Latency Optimization > KV Cache Management": 16-token pages
// gathered through a page table; "Inside LLM Inference Engines ...":
// PagedAttention). Decode is bound by memory bandwidth (InferScale, the
// decode phase; "Inside LLM Inference Engines ...", Decode Phase).
//
// Work split, TMA producer and end-of-piece protocol:
// kvinj_decode_common.cuh. This consumer does the arithmetic on the CUDA
// cores, one warp per kv head: for QK, 8 lanes per token split the head
// dimension and the G per-head partial dot products are combined with a
// reduce-scatter across those 8 lanes (G = 8: 7 shuffles for 8 sums); for PV
// each lane owns D/32 dimensions of all G heads. It needs ~2*G*D FMAs per
// token and is kept beside the tensor-core consumer (kvinj_decode_mma.cu) as
// the measured alternative.
#include <math.h>

#include "kvinj_decode_common.cuh"

namespace kvinj {

// reduce-scatter of N per-lane values across the 8 lanes of a token group
// (xor masks M, M/2, ..., 1): returns the sum over the group of value index
// hs(dg), where hs = dg >> log2(8/N); then a plain butterfly for the rest.
template <int N, int M>
struct RedScatter {
  static __device__ __forceinline__ float run(const float *v, int dg) {
    float a[N / 2];
    const bool up = (dg & M) != 0;
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      float send = up ? v[i] : v[i + N / 2];
      float keep = up ? v[i + N / 2] : v[i];
      a[i] = keep + __shfl_xor_sync(0xffffffffu, send, M);
    }
    return RedScatter<N / 2, M / 2>::run(a, dg);
  }
};
template <int M>
struct RedScatter<1, M> {
  static __device__ __forceinline__ float run(const float *v, int) {
    float x = v[0];
#pragma unroll
    for (int m = M; m >= 1; m >>= 1) x += __shfl_xor_sync(0xffffffffu, x, m);
    return x;
  }
};
template <>
struct RedScatter<1, 0> {
  static __device__ __forceinline__ float run(const float *v, int) { return v[0]; }
};

// q of the G heads of kv head h, rotated at q_pos[r], times scale*log2(e).
// The lane keeps, for every 64-element box b, the 8 elements of chunk dg:
// dims [64b + 8dg, 64b + 8dg + 8).
template <int D, int G, int DT, int NBOX>
__device__ __forceinline__ void load_q_rows(const DecodeArgs &a, int r, int h, int dg,
                                            float (&qr)[G][NBOX][8]) {
  constexpr int HALF = D / 2;
  const int qp = a.q_pos[r];
  const bool rotate = a.rope != nullptr;
  const bool pos_ok = !rotate || (qp >= 0 && qp < a.max_pos);
  if (!pos_ok && (threadIdx.x & 31) == 0) report(a.status, KVINJ_ST_BAD_POS);
  const float4 *trow = rotate && pos_ok ? a.rope + (int64_t)qp * HALF : nullptr;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const uint16_t *qrow = a.q + ((int64_t)r * a.Hq + (int64_t)h * G + g) * D;
#pragma unroll
    for (int b = 0; b < NBOX; ++b) {
      const int d0 = 64 * b + 8 * dg;
      const uint4 own = *reinterpret_cast<const uint4 *>(qrow + d0);
      float x[8];
      float2 f;
      f = unpack2<DT>(own.x); x[0] = f.x; x[1] = f.y;
      f = unpack2<DT>(own.y); x[2] = f.x; x[3] = f.y;
      f = unpack2<DT>(own.z); x[4] = f.x; x[5] = f.y;
      f = unpack2<DT>(own.w); x[6] = f.x; x[7] = f.y;
      if (trow) {
        const int dp = (d0 + HALF) % D;  // the rotate-half partners
        const uint4 par = *reinterpret_cast<const uint4 *>(qrow + dp);
        float y[8];
        f = unpack2<DT>(par.x); y[0] = f.x; y[1] = f.y;
        f = unpack2<DT>(par.y); y[2] = f.x; y[3] = f.y;
        f = unpack2<DT>(par.z); y[4] = f.x; y[5] = f.y;
        f = unpack2<DT>(par.w); y[6] = f.x; y[7] = f.y;
        const bool first = d0 < HALF;
        const int f0 = d0 % HALF;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float4 t = __ldg(trow + f0 + e);
          x[e] = first ? rope_pair(x[e], y[e], t).x : rope_pair(y[e], x[e], t).y;
        }
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) qr[g][b][e] = x[e] * a.scale_log2;
    }
  }
}

template <int D, int G, int HG, int S, int DT>
__global__ void __launch_bounds__((HG + 1) * 32, 1)
    decode_ffma_kernel(const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, DecodeArgs a) {
  using Lay = DecodeLayout<D, G, HG, S>;
  constexpr int NBOX = D / 64;
  constexpr int DPL = D / 32;  // dims per lane in the PV product
  constexpr int HSHIFT = (G == 8) ? 0 : (G == 4) ? 1 : (G == 2) ? 2 : 3;
  constexpr int PF = partial_floats(G, D), SLOT = HG * PF;
  static_assert(G == 1 || G == 2 || G == 4 || G == 8, "FMA decode: G in {1,2,4,8}");

  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = align_smem(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  CtaRange rg;
  if (!decode_prologue<Lay, (HG + 1) * 32>(a, sm, rg)) return;

  uint64_t *full = reinterpret_cast<uint64_t *>(sm + Lay::off_bar);
  uint64_t *empty = full + S;
  volatile int *flags = reinterpret_cast<volatile int *>(sm + Lay::off_flags);
  const int *valid = reinterpret_cast<const int *>(sm + Lay::off_valid);

  if (warp == HG) {
    decode_producer<Lay>(a, tmK, tmV, sm, rg, lane);
    return;
  }

  // ------------------------------ consumers ------------------------------
  const int tp = lane >> 3, dg = lane & 7;
  const int hs = dg >> HSHIFT;  // head whose score this lane ends up holding
  const bool head_owner = (dg & ((1 << HSHIFT) - 1)) == 0;  // lowest lane of its head
  float *p_sm = reinterpret_cast<float *>(sm + Lay::off_scratch) + warp * Lay::SCRATCH_FLOATS;
  float *alpha_sm = p_sm + 16 * G;
  const int *pre = reinterpret_cast<const int *>(sm + Lay::off_pre);
  const uint32_t stage0 = smem_u32(sm + Lay::off_stage);
  const int ngrp = a.Hkv / HG;
  const int e0 = lane * DPL;  // first PV dimension of this lane

  int P = rg.b0, g = 0;
  while (P < rg.b1) {
    const Piece pc = find_piece(a, pre, ngrp, P, rg.b1);
    const int h = pc.hg * HG + warp;

    float qr[G][NBOX][8];
    load_q_rows<D, G, DT, NBOX>(a, pc.r, h, dg, qr);

    float m_run = -INFINITY, l_run = 0.f;
    float acc[G][DPL];
#pragma unroll
    for (int gg = 0; gg < G; ++gg)
#pragma unroll
      for (int e = 0; e < DPL; ++e) acc[gg][e] = 0.f;

    const int np = pc.end - P;
    for (int i = 0; i < np; ++i) {
      const int gi = g + i, st = gi % S;
      const bool ok = consumer_wait(a, full, flags, gi, S);
      int nv = 0;
      if (ok && valid[st]) nv = min(16, pc.ctx - (pc.pg0 + i) * 16);
      const uint32_t kb = stage0 + st * Lay::STAGE_BYTES;
      const uint32_t vb = kb + Lay::UNIT_BYTES;

      // ---- scores of the block's 16 tokens: 4 passes of 4 tokens ----
      float sc[4];
#pragma unroll
      for (int pass = 0; pass < 4; ++pass) {
        const int t = pass * 4 + tp;
        float part[G];
#pragma unroll
        for (int gg = 0; gg < G; ++gg) part[gg] = 0.f;
        if (nv > 0) {
#pragma unroll
          for (int b = 0; b < NBOX; ++b) {
            const uint4 kw = lds128(kb + unit_off<Lay::BOXB>(warp, 8 * b + dg, t));
            float k8[8];
            float2 f;
            f = unpack2<DT>(kw.x); k8[0] = f.x; k8[1] = f.y;
            f = unpack2<DT>(kw.y); k8[2] = f.x; k8[3] = f.y;
            f = unpack2<DT>(kw.z); k8[4] = f.x; k8[5] = f.y;
            f = unpack2<DT>(kw.w); k8[6] = f.x; k8[7] = f.y;
#pragma unroll
            for (int gg = 0; gg < G; ++gg)
#pragma unroll
              for (int e = 0; e < 8; ++e) part[gg] = __fmaf_rn(qr[gg][b][e], k8[e], part[gg]);
          }
        }
        const float s = RedScatter<G, 4>::run(part, dg);
        sc[pass] = (t < nv) ? s : -INFINITY;
      }

      // ---- online softmax for head hs ----
      float pm = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
      pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 8));
      pm = fmaxf(pm, __shfl_xor_sync(0xffffffffu, pm, 16));
      const float m_new = fmaxf(m_run, pm);
      const float alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);
      float pr[4], ps = 0.f;
#pragma unroll
      for (int pass = 0; pass < 4; ++pass) {
        pr[pass] = (sc[pass] == -INFINITY) ? 0.f : exp2f(sc[pass] - m_new);
        ps += pr[pass];
      }
      ps += __shfl_xor_sync(0xffffffffu, ps, 8);
      ps += __shfl_xor_sync(0xffffffffu, ps, 16);
      l_run = l_run * alpha + ps;
      m_run = m_new;
      if (head_owner) {
#pragma unroll
        for (int pass = 0; pass < 4; ++pass) p_sm[(pass * 4 + tp) * G + hs] = pr[pass];
        if (tp == 0) alpha_sm[hs] = alpha;
      }
      __syncwarp();

      // ---- acc = alpha * acc + sum_t p_t V_t over the lane's DPL dims ----
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        const float al = alpha_sm[gg];
#pragma unroll
        for (int e = 0; e < DPL; ++e) acc[gg][e] *= al;
      }
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        if (t < nv) {
          const uint32_t addr = vb + unit_off<Lay::BOXB>(warp, e0 / 8, t) + (e0 % 8) * 2;
          float v[DPL];
          if constexpr (DPL == 4) {
            const uint2 w = lds64(addr);
            float2 f = unpack2<DT>(w.x);
            v[0] = f.x; v[1] = f.y;
            f = unpack2<DT>(w.y);
            v[2] = f.x; v[3] = f.y;
          } else {
            const float2 f = unpack2<DT>(lds32(addr));
            v[0] = f.x; v[1] = f.y;
          }
#pragma unroll
          for (int gg = 0; gg < G; ++gg) {
            const float pt = p_sm[t * G + gg];
#pragma unroll
            for (int e = 0; e < DPL; ++e) acc[gg][e] = __fmaf_rn(pt, v[e], acc[gg][e]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + st);
    }

    // ---- this warp's head: final output or partial state ----
    const bool complete = (P == pc.seg_start) && (pc.end == pc.seg_end);
    float* slot = a.partials + (size_t)(2 * blockIdx.x + (pc.seg_start <= rg.b0 ? 0 : 1)) * SLOT +
                  warp * PF;
#pragma unroll
    for (int gg = 0; gg < G; ++gg) {
      const float mg = __shfl_sync(0xffffffffu, m_run, gg << HSHIFT);
      const float lg = __shfl_sync(0xffffffffu, l_run, gg << HSHIFT);
      if (complete) {
        uint16_t *orow = a.out + ((int64_t)pc.r * a.Hq + (int64_t)h * G + gg) * D;
        const float inv = lg > 0.f ? 1.f / lg : 0.f;
#pragma unroll
        for (int e = 0; e < DPL; e += 2)
          *reinterpret_cast<uint32_t *>(orow + e0 + e) =
              pack2<DT>(acc[gg][e] * inv, acc[gg][e + 1] * inv);
      } else {
        if (lane == 0) {
          slot[gg] = mg;
          slot[G + gg] = lg;
        }
#pragma unroll
        for (int e = 0; e < DPL; e += 2)
          *reinterpret_cast<float2 *>(slot + 2 * G + gg * D + e0 + e) =
              make_float2(acc[gg][e], acc[gg][e + 1]);
      }
    }

    g += np;
    P = pc.end;
  }
}

template <int D, int G, int HG, int DT>
static cudaError_t launch_ffma(const DecodeArgs &a, const CUtensorMap &tmK,
                               const CUtensorMap &tmV, int ctas, cudaStream_t s) {
  constexpr int STAGE = 2 * (D / 64) * HG * BLK * 128;
  constexpr int S = (192 * 1024 / STAGE) < 2 ? 2 : (192 * 1024 / STAGE) > 24 ? 24
                                                                            : (192 * 1024 / STAGE);
  using Lay = DecodeLayout<D, G, HG, S>;
  auto kern = decode_ffma_kernel<D, G, HG, S, DT>;
  const size_t smem = Lay::bytes(a.batch);
  if (smem > (size_t)DECODE_MAX_SMEM) return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DECODE_MAX_SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaError_t e = launch_pdl(kern, dim3(ctas), dim3((HG + 1) * 32), smem, s, tmK, tmV, a);
  if (e != cudaSuccess) return e;
  return launch_combine<D, G, HG, DT>(a, ctas, s);
}

cudaError_t launch_decode_ffma(const DecodeArgs &a, const CUtensorMap &tmK,
                               const CUtensorMap &tmV, int D, int G, int HG, int dtype, int ctas,
                               cudaStream_t s) {
#define KVINJ_FFMA_CASE(DD, GG, HH, TT)                    \
  if (D == DD && G == GG && HG == HH && dtype == TT) \
    return launch_ffma<DD, GG, HH, TT>(a, tmK, tmV, ctas, s);
#define KVINJ_FFMA_G(DD, HH, TT)                                                         \
  KVINJ_FFMA_CASE(DD, 1, HH, TT) KVINJ_FFMA_CASE(DD, 2, HH, TT) KVINJ_FFMA_CASE(DD, 4, HH, TT) \
  KVINJ_FFMA_CASE(DD, 8, HH, TT)
#define KVINJ_FFMA_H(DD, TT) \
  KVINJ_FFMA_G(DD, 1, TT) KVINJ_FFMA_G(DD, 2, TT) KVINJ_FFMA_G(DD, 4, TT) KVINJ_FFMA_G(DD, 8, TT)
  KVINJ_FFMA_H(64, 0)
  KVINJ_FFMA_H(64, 1)
  KVINJ_FFMA_H(128, 0)
  KVINJ_FFMA_H(128, 1)
#undef KVINJ_FFMA_H
#undef KVINJ_FFMA_G
#undef KVINJ_FFMA_CASE
  return cudaErrorInvalidValue;
}

}  // namespace kvinj
