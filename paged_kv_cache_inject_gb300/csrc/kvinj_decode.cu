// kvinj_decode.cu -- split-K paged GQA decode attention, sm_103a.
//
// Computes, per request r and query head qh (kv head h = qh / G):
//   out = sum_p softmax_p(scale * (R_{q_pos} q) . K_p) V_p
// over the request's context, read page by page through its block table
// ("LLM Inference: KV Caching": attention softmax(QK^T/sqrt d)V and "Paged
// attention"; "Latency Optimization > KV Cache Management": 16-token pages
// gathered through a page table; "Inside LLM Inference Engines ...":
// PagedAttention). Decode is bound by memory bandwidth (InferScale, the
// decode phase; "Inside LLM Inference Engines ...", Decode Phase).
//
// Work split. The (request, kv head) pairs are "segments" of ceil(C_r/16)
// pages; their pages, flattened request-major, are cut into gridDim.x equal
// contiguous ranges, one per CTA (one CTA per SM), so every CTA streams the
// same number of bytes whatever the mix of context lengths. A segment that
// lies inside one CTA is finished there; a segment cut by range boundaries
// leaves one partial softmax state (m, l, acc) per CTA piece in the
// workspace, and the CTA that finishes last (an atomic counter per segment,
// no waiting) merges them and writes the output. Every CTA therefore needs
// only its own data; nothing spins on another CTA.
//
// Inside a CTA, one producer warp streams pages into a ring of S stages with
// 2-D TMA (two 16 x 64-element boxes per K or V page at D = 128, 128-byte
// swizzle, so the consumers' 16-byte shared loads are bank-conflict free);
// block-table entries are fetched 32 at a time, one per lane, a batch ahead.
// NW consumer warps take the pages round-robin, each keeping its own online
// softmax state for the current segment, merged through shared memory at the
// end of each piece. All mbarrier waits are bounded; a wait that gives up
// raises KVINJ_ST_TIMEOUT and the CTA winds down instead of hanging.
//
// This file holds the CUDA-core (FMA) consumer: 8 lanes per token split the
// head dimension; the G per-head partial dot products are combined with a
// reduce-scatter across those 8 lanes (G = 8: 7 shuffles for 8 sums).
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

template <int D, int G, int NW, int S, int DT>
__global__ void __launch_bounds__((NW + 1) * 32, 1)
    decode_ffma_kernel(const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, DecodeArgs a) {
  using Lay = DecodeLayout<D, G, NW, S>;
  constexpr int NBOX = D / 64;
  constexpr int DPL = D / 32;  // dims per lane in the PV product
  constexpr int HSHIFT = (G == 8) ? 0 : (G == 4) ? 1 : (G == 2) ? 2 : 3;
  static_assert(G == 1 || G == 2 || G == 4 || G == 8, "FMA decode: G in {1,2,4,8}");
  // every use of a stage goes to the same consumer warp, which therefore sees
  // the stage's phases in order (the mbarrier parity waits rely on it)
  static_assert(S % NW == 0, "stages must be a multiple of the consumer warps");

  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = align_smem(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  CtaRange rg;
  if (!decode_prologue<Lay, (NW + 1) * 32>(a, sm, rg)) return;

  uint64_t *full = reinterpret_cast<uint64_t *>(sm + Lay::off_bar);
  uint64_t *empty = full + S;
  volatile int *flags = reinterpret_cast<volatile int *>(sm + Lay::off_flags);
  int *valid = reinterpret_cast<int *>(sm + Lay::off_valid);

  if (warp == NW) {
    decode_producer<Lay>(a, tmK, tmV, sm, rg, lane);
    return;
  }

  // ------------------------------ consumers ------------------------------
  const int tp = lane >> 3, dg = lane & 7;
  const int hs = dg >> HSHIFT;  // head whose score this lane ends up holding
  const bool head_owner = (dg & ((1 << HSHIFT) - 1)) == 0;  // lowest lane of its head
  float *p_sm = reinterpret_cast<float *>(sm + Lay::off_p) + warp * 16 * G;
  float *alpha_sm = reinterpret_cast<float *>(sm + Lay::off_alpha) + warp * G;
  float *mm = reinterpret_cast<float *>(sm + Lay::off_mm);
  float *ml = reinterpret_cast<float *>(sm + Lay::off_ml);
  float *macc = reinterpret_cast<float *>(sm + Lay::off_macc);
  const int *pre = reinterpret_cast<const int *>(sm + Lay::off_pre);
  const uint32_t stage0 = smem_u32(sm + Lay::off_stage);

  int P = rg.b0, g = 0;
  while (P < rg.b1) {
    Piece pc = find_piece(a, pre, P, rg.b1);

    // q of the G heads of this group, rotated, in log2 units: lane keeps the
    // dims of chunk dg (8 elements) of every 64-element box
    float qr[G][NBOX][8];
    load_q_rows<D, G, DT, NBOX>(a, pc.r, pc.h, dg, qr);

    float m_run = -INFINITY, l_run = 0.f;
    float acc[G][DPL];
#pragma unroll
    for (int gg = 0; gg < G; ++gg)
#pragma unroll
      for (int e = 0; e < DPL; ++e) acc[gg][e] = 0.f;

    const int np = pc.end - P;
    for (int i = ((warp - g) % NW + NW) % NW; i < np; i += NW) {
      const int gi = g + i, st = gi % S;
      bool ok = !flags[0] && mbar_wait_bounded(full + st, (uint32_t)(gi / S) & 1u);
      if (!ok) {
        if (!flags[0]) report(a.status, KVINJ_ST_TIMEOUT);
        flags[0] = 1;
      }
      int nv = 0;
      if (ok && valid[st]) nv = min(16, pc.ctx - (pc.pg0 + i) * 16);
      const uint32_t kbase = stage0 + st * Lay::STAGE_BYTES;
      const uint32_t vbase = kbase + Lay::PAGE_BYTES;

      // ---- scores of the page's 16 tokens: 4 passes of 4 tokens ----
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
            uint4 kw = lds128(kbase + b * BOX_BYTES + t * 128 + ((dg ^ (t & 7)) << 4));
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
        float s = RedScatter<G, 4>::run(part, dg);
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
      const int e0 = lane * DPL;
      const uint32_t voff = (e0 / 64) * BOX_BYTES + (e0 % 8) * 2;
      const int vch = (e0 % 64) / 8;
#pragma unroll
      for (int t = 0; t < 16; ++t) {
        if (t < nv) {
          const uint32_t addr = vbase + voff + t * 128 + ((vch ^ (t & 7)) << 4);
          float v[DPL];
          if constexpr (DPL == 4) {
            uint2 w = lds64(addr);
            float2 f = unpack2<DT>(w.x);
            v[0] = f.x; v[1] = f.y;
            f = unpack2<DT>(w.y);
            v[2] = f.x; v[3] = f.y;
          } else {
            uint32_t w = lds32(addr);
            float2 f = unpack2<DT>(w);
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

    // ---- merge the NW warp states of this piece ----
    if (head_owner && tp == 0) {
      mm[warp * G + hs] = m_run;
      ml[warp * G + hs] = l_run;
    }
#pragma unroll
    for (int gg = 0; gg < G; ++gg)
#pragma unroll
      for (int e = 0; e < DPL; ++e) macc[(warp * G + gg) * D + lane * DPL + e] = acc[gg][e];
    finish_piece<Lay, DT>(a, sm, rg, pc, P, tid);

    g += np;
    P = pc.end;
  }
}

template <int D, int G, int DT>
static cudaError_t launch_ffma(const DecodeArgs &a, const CUtensorMap &tmK,
                               const CUtensorMap &tmV, int ctas, cudaStream_t s) {
  constexpr int NW = 8, S = 16;
  using Lay = DecodeLayout<D, G, NW, S>;
  auto kern = decode_ffma_kernel<D, G, NW, S, DT>;
  const size_t smem = Lay::bytes(a.batch);
  if (smem > (size_t)DECODE_MAX_SMEM) return cudaErrorInvalidValue;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DECODE_MAX_SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  kern<<<ctas, (NW + 1) * 32, smem, s>>>(tmK, tmV, a);
  return cudaGetLastError();
}

cudaError_t launch_decode_ffma(const DecodeArgs &a, const CUtensorMap &tmK,
                               const CUtensorMap &tmV, int D, int G, int dtype, int ctas,
                               cudaStream_t s) {
#define KVINJ_FFMA_CASE(DD, GG, TT)                                  \
  if (D == DD && G == GG && dtype == TT) return launch_ffma<DD, GG, TT>(a, tmK, tmV, ctas, s);
#define KVINJ_FFMA_D(DD, TT) \
  KVINJ_FFMA_CASE(DD, 1, TT) KVINJ_FFMA_CASE(DD, 2, TT) KVINJ_FFMA_CASE(DD, 4, TT) KVINJ_FFMA_CASE(DD, 8, TT)
  KVINJ_FFMA_D(64, 0)
  KVINJ_FFMA_D(64, 1)
  KVINJ_FFMA_D(128, 0)
  KVINJ_FFMA_D(128, 1)
#undef KVINJ_FFMA_D
#undef KVINJ_FFMA_CASE
  return cudaErrorInvalidValue;
}

}  // namespace kvinj
