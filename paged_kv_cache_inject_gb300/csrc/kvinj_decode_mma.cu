// kvinj_decode_mma.cu -- split-K paged GQA decode, tensor-core consumer.
//
// Work split, producer (which also stages each piece's query rows and RoPE
// row with 1-D bulk copies) and end-of-piece protocol:
// kvinj_decode_common.cuh. Each consumer warp owns one kv head of the unit's
// head group. For its G query heads and the unit's 16 tokens it runs the two
// small contractions on the tensor cores with mma.sync m16n8k16 (fp32
// accumulation), with the tokens on the M side:
//   QK: S^T[16 tokens x N] = K[16 x D] Q^T[D x N]. A = the head's 16 K rows
//       (ldmatrix from the swizzled stage); B = the rotated, scaled queries,
//       built in registers once per piece from the staged rows.
//   softmax over the 16 tokens of each column: two rows per lane, then
//       xor-shuffles across the 8 row groups.
//   PV: O^T[D x N] += V^T[D x 16] P^T[16 x N]. A = V rows via
//       ldmatrix.trans; B = P^T, the exponentiated scores moved across the
//       warp with movmatrix (transpose of an 8x8 16-bit tile in registers).
// Columns (N). The tensor cores take 16-bit operands while Q (rotated,
// scaled) and P are fp32; each is split x = hi + lo, hi = round16(x),
// lo = round16(x - hi) (~16 significant bits together). The hi and lo parts
// of every query head are separate columns and their results are summed:
// for G <= 4 one 8-column tile holds them all (hi of head j in column j, lo
// in column j + 4), so a 16-token unit costs D/16 mmas for QK and D/16 for
// PV; for G = 8 (16) the hi heads fill 1 (2) tiles and the lo heads as many.
// K and V are used as stored.
#include <math.h>

#include "kvinj_decode_common.cuh"

namespace kvinj {

template <int DT>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (DT == 0) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// transpose of an 8x8 16-bit tile held one row pair per lane (row lane/4,
// columns 2*(lane%4), +1) into the same layout of the transposed tile
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// (x, y) -> hi = round16 of both, lo = round16 of what hi missed
template <int DT>
__device__ __forceinline__ uint32_t split_hi_lo(float x, float y, uint32_t &lo) {
  const uint32_t hi = pack2<DT>(x, y);
  const float2 h = unpack2<DT>(hi);
  lo = pack2<DT>(x - h.x, y - h.y);
  return hi;
}

// B fragments of one query row for every k-step (elements at dims
// ks*16 + j*8 + 2*c4 + {0,1}, j in {0,1}) from the staged row in shared
// memory: rotated with the staged table row (tab == nullptr: as given),
// times scale*log2(e), split hi/lo. With rotate-half the partner of dim
// d < D/2 is d + D/2: the same offsets of k-step ks + D/32, held by the lane.
template <int D, int DT>
__device__ __forceinline__ void q_row_frags(const uint16_t *qrow, const float4 *tab, float sc,
                                            int c4, uint32_t (&hi)[D / 16][2],
                                            uint32_t (&lo)[D / 16][2]) {
  constexpr int KS = D / 16, HALF = D / 2;
#pragma unroll
  for (int ks = 0; ks < KS / 2; ++ks)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int d = ks * 16 + j * 8 + 2 * c4;
      const float2 x = unpack2<DT>(*reinterpret_cast<const uint32_t *>(qrow + d));
      const float2 y = unpack2<DT>(*reinterpret_cast<const uint32_t *>(qrow + d + HALF));
      float x0 = x.x, x1 = x.y, y0 = y.x, y1 = y.y;
      if (tab) {
        const float2 r0 = rope_pair(x.x, y.x, tab[d]);
        const float2 r1 = rope_pair(x.y, y.y, tab[d + 1]);
        x0 = r0.x;
        y0 = r0.y;
        x1 = r1.x;
        y1 = r1.y;
      }
      hi[ks][j] = split_hi_lo<DT>(x0 * sc, x1 * sc, lo[ks][j]);
      hi[ks + KS / 2][j] = split_hi_lo<DT>(y0 * sc, y1 * sc, lo[ks + KS / 2][j]);
    }
}

template <int G>
struct Cols {
  static constexpr bool SMALL = G <= 4;             // hi and lo of all heads in one tile
  static constexpr int NTN = SMALL ? 1 : 2 * G / 8;  // n-tiles (8 columns each)
  static constexpr int HT = SMALL ? 1 : NTN / 2;     // tiles of hi columns
  static constexpr int HC = 2 * HT;                  // head columns a lane holds after hi+lo
};

template <int D, int G, int HG, int S, int QB, int DT>
__global__ void __launch_bounds__((HG + 1) * 32, 1)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, DecodeArgs a) {
  using Lay = DecodeLayout<D, G, HG, S, QB>;
  using C = Cols<G>;
  constexpr int KS = D / 16;  // k-steps of QK = m-tiles of PV
  constexpr int NTN = C::NTN, HT = C::HT;
  constexpr int PF = partial_floats(G, D), SLOT = HG * PF;
  static_assert(G == 1 || G == 2 || G == 4 || G == 8 || G == 16, "tensor-core decode: G");
  static_assert(QB >= 1, "the tensor-core consumer reads staged query rows");

  extern __shared__ uint8_t smem_raw[];
  uint8_t *sm = align_smem(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  CtaRange rg;
  if (!decode_prologue<Lay, (HG + 1) * 32>(a, sm, rg)) return;

  uint64_t *full = reinterpret_cast<uint64_t *>(sm + Lay::off_bar);
  uint64_t *empty = full + S;
  uint64_t *qfull = full + 2 * S, *qempty = qfull + QB;
  volatile int *flags = reinterpret_cast<volatile int *>(sm + Lay::off_flags);
  const int *valid = reinterpret_cast<const int *>(sm + Lay::off_valid);
  const int *qinfo = reinterpret_cast<const int *>(sm + Lay::off_qinfo);

  if (warp == HG) {
    decode_producer<Lay>(a, tmK, tmV, sm, rg, lane);
    return;
  }

  // ------------------------------ consumers ------------------------------
  const int g4 = lane >> 2, c4 = lane & 3;
  const int lm = lane >> 3, lr = lane & 7;  // ldmatrix roles: matrix, row
  const int *pre = reinterpret_cast<const int *>(sm + Lay::off_pre);
  const uint32_t stage0 = smem_u32(sm + Lay::off_stage);
  const int ngrp = a.Hkv / HG;
  // the head of each column slot this lane holds after summing hi and lo:
  // slot k = 2*t + j -> head (SMALL) 2*(c4 & 1) + j, else t*8 + 2*c4 + j
  auto head_of = [&](int t, int j) { return C::SMALL ? 2 * (c4 & 1) + j : t * 8 + 2 * c4 + j; };

  int P = rg.b0, g = 0, piece = 0;
  while (P < rg.b1) {
    const Piece pc = find_piece(a, pre, ngrp, P, rg.b1);
    const int h = pc.hg * HG + warp;  // this warp's kv head

    // ---- query B fragments from the staged rows ----
    uint32_t qb[NTN][KS][2];
    {
      const int qbuf = piece % QB;
      bool ok = !flags[0] && mbar_wait_bounded(qfull + qbuf, (uint32_t)(piece / QB) & 1u);
      if (!ok) {
        if (!flags[0]) report(a.status, KVINJ_ST_TIMEOUT);
        flags[0] = 1;
      }
      const uint16_t *qs = reinterpret_cast<const uint16_t *>(sm + Lay::off_q +
                                                              qbuf * Lay::Q_BYTES) +
                           warp * G * D;
      const float4 *tab = qinfo[qbuf] >= 0
                              ? reinterpret_cast<const float4 *>(sm + Lay::off_t + qbuf * Lay::T_BYTES)
                              : nullptr;
#pragma unroll
      for (int t = 0; t < NTN; ++t)
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) qb[t][ks][0] = qb[t][ks][1] = 0u;
      if (ok) {
        if constexpr (C::SMALL) {
          // column g4: hi (g4 < 4) or lo (g4 >= 4) of head g4 & 3
          const int hd = g4 & 3;
          if (hd < G) {
            uint32_t hi[KS][2], lo[KS][2];
            q_row_frags<D, DT>(qs + hd * D, tab, a.scale_log2, c4, hi, lo);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
              qb[0][ks][0] = g4 < 4 ? hi[ks][0] : lo[ks][0];
              qb[0][ks][1] = g4 < 4 ? hi[ks][1] : lo[ks][1];
            }
          }
        } else {
#pragma unroll
          for (int t = 0; t < HT; ++t) {  // column g4 of hi tile t: head t*8 + g4
            uint32_t hi[KS][2], lo[KS][2];
            q_row_frags<D, DT>(qs + (t * 8 + g4) * D, tab, a.scale_log2, c4, hi, lo);
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
              qb[t][ks][0] = hi[ks][0];
              qb[t][ks][1] = hi[ks][1];
              qb[HT + t][ks][0] = lo[ks][0];
              qb[HT + t][ks][1] = lo[ks][1];
            }
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(qempty + qbuf);
    }

    float m_run[2 * HT], l_run[2 * HT];
#pragma unroll
    for (int k = 0; k < 2 * HT; ++k) {
      m_run[k] = -INFINITY;
      l_run[k] = 0.f;
    }
    float o[KS][NTN][4];
#pragma unroll
    for (int mt = 0; mt < KS; ++mt)
#pragma unroll
      for (int t = 0; t < NTN; ++t) o[mt][t][0] = o[mt][t][1] = o[mt][t][2] = o[mt][t][3] = 0.f;

    const int np = pc.end - P;
    for (int i = 0; i < np; ++i) {
      const int gi = g + i, st = gi % S;
      const bool ok = consumer_wait(a, full, flags, gi, S);
      int nv = 0;
      if (ok && valid[st]) nv = min(16, pc.ctx - (pc.pg0 + i) * 16);
      const uint32_t kb = stage0 + st * Lay::STAGE_BYTES;
      const uint32_t vb = kb + Lay::UNIT_BYTES;

      if (nv > 0) {
        // ---- S^T = K Q^T: rows = tokens (g4, g4 + 8), cols = hi/lo heads ----
        float s[NTN][4];
#pragma unroll
        for (int t = 0; t < NTN; ++t) s[t][0] = s[t][1] = s[t][2] = s[t][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t ka[4];
          ldsm_x4(kb + unit_off<Lay::BOXB>(warp, 2 * ks + (lm >> 1), (lm & 1) * 8 + lr), ka);
#pragma unroll
          for (int t = 0; t < NTN; ++t) mma16816<DT>(s[t], ka, qb[t][ks][0], qb[t][ks][1]);
        }
        // hi + lo -> one score per (token row, head column slot)
        float sc[HT][4];
#pragma unroll
        for (int t = 0; t < HT; ++t)
#pragma unroll
          for (int c = 0; c < 4; ++c)
            sc[t][c] = C::SMALL ? s[0][c] + __shfl_xor_sync(0xffffffffu, s[0][c], 2)
                                : s[t][c] + s[HT + t][c];
        if (nv < 16) {  // tokens past the context (ragged last block)
#pragma unroll
          for (int t = 0; t < HT; ++t) {
            if (g4 >= nv) sc[t][0] = sc[t][1] = -INFINITY;
            if (g4 + 8 >= nv) sc[t][2] = sc[t][3] = -INFINITY;
          }
        }
        // ---- online softmax per head column (over the 16 tokens) ----
        float alpha[HT][2];
#pragma unroll
        for (int t = 0; t < HT; ++t)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            float mx = fmaxf(sc[t][j], sc[t][j + 2]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            const int k = 2 * t + j;
            const float m_new = fmaxf(m_run[k], mx);
            alpha[t][j] = (m_new == -INFINITY) ? 1.f : exp2f(m_run[k] - m_new);
            const float p0 = (sc[t][j] == -INFINITY) ? 0.f : exp2f(sc[t][j] - m_new);
            const float p1 = (sc[t][j + 2] == -INFINITY) ? 0.f : exp2f(sc[t][j + 2] - m_new);
            sc[t][j] = p0;
            sc[t][j + 2] = p1;
            float sum = p0 + p1;
            sum += __shfl_xor_sync(0xffffffffu, sum, 4);
            sum += __shfl_xor_sync(0xffffffffu, sum, 8);
            sum += __shfl_xor_sync(0xffffffffu, sum, 16);
            l_run[k] = l_run[k] * alpha[t][j] + sum;
            m_run[k] = m_new;
          }
        // ---- P^T as the B operand: hi / lo columns, transposed with movmatrix ----
        uint32_t pb[NTN][2];
#pragma unroll
        for (int t = 0; t < HT; ++t) {
          uint32_t lo0, lo1;
          const uint32_t hi0 = split_hi_lo<DT>(sc[t][0], sc[t][1], lo0);  // token g4
          const uint32_t hi1 = split_hi_lo<DT>(sc[t][2], sc[t][3], lo1);  // token g4 + 8
          if constexpr (C::SMALL) {  // lanes c4 < 2 hold the hi columns, c4 >= 2 the lo ones
            pb[0][0] = movmatrix_t(c4 < 2 ? hi0 : lo0);
            pb[0][1] = movmatrix_t(c4 < 2 ? hi1 : lo1);
          } else {
            pb[t][0] = movmatrix_t(hi0);
            pb[t][1] = movmatrix_t(hi1);
            pb[HT + t][0] = movmatrix_t(lo0);
            pb[HT + t][1] = movmatrix_t(lo1);
          }
        }
        // ---- rescale O^T columns, then O^T += V^T P^T ----
#pragma unroll
        for (int mt = 0; mt < KS; ++mt)
#pragma unroll
          for (int t = 0; t < NTN; ++t) {
            const int th = C::SMALL ? 0 : t % HT;
            o[mt][t][0] *= alpha[th][0];
            o[mt][t][1] *= alpha[th][1];
            o[mt][t][2] *= alpha[th][0];
            o[mt][t][3] *= alpha[th][1];
          }
        // V rows of a ragged block past the context may hold anything (even
        // NaN bit patterns): zero this head's rows so that 0 * V stays 0
        if (nv < 16) {
          for (int idx = lane; idx < (16 - nv) * (D / 8); idx += 32) {
            const int tok = nv + idx / (D / 8), chunk = idx % (D / 8);
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(
                             vb + unit_off<Lay::BOXB>(warp, chunk, tok)),
                         "r"(0)
                         : "memory");
          }
          __syncwarp();
        }
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          uint32_t va[4];
          ldsm_x4_t(vb + unit_off<Lay::BOXB>(warp, 2 * mt + (lm & 1), (lm >> 1) * 8 + lr), va);
#pragma unroll
          for (int t = 0; t < NTN; ++t) mma16816<DT>(o[mt][t], va, pb[t][0], pb[t][1]);
        }
        if (nv < 16) fence_proxy_async_smem();  // generic writes before the next TMA fill
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + st);
    }

    // ---- this warp's head: final output or partial state ----
    // O[head][dim] = O^T[dim][hi col] + O^T[dim][lo col]
    const bool complete = (P == pc.seg_start) && (pc.end == pc.seg_end);
    float *slot = a.partials +
                  (size_t)(2 * blockIdx.x + (pc.seg_start <= rg.b0 ? 0 : 1)) * SLOT + warp * PF;
    uint16_t *obase = a.out + ((int64_t)pc.r * a.Hq + (int64_t)h * G) * D;
    const bool writer = C::SMALL ? c4 < 2 : true;
#pragma unroll
    for (int t = 0; t < HT; ++t)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int hd = head_of(t, j);
        const int k = 2 * t + j;
        const float inv = l_run[k] > 0.f ? 1.f / l_run[k] : 0.f;
        if (!complete && writer && hd < G && g4 == 0) {
          slot[hd] = m_run[k];
          slot[G + hd] = l_run[k];
        }
#pragma unroll
        for (int mt = 0; mt < KS; ++mt)
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const int c = 2 * half + j;
            float v = C::SMALL ? o[mt][0][c] + __shfl_xor_sync(0xffffffffu, o[mt][0][c], 2)
                               : o[mt][t][c] + o[mt][HT + t][c];
            const int dim = mt * 16 + half * 8 + g4;
            if (writer && hd < G) {
              if (complete)
                obase[hd * D + dim] = to16<DT>(v * inv);
              else
                slot[2 * G + hd * D + dim] = v;
            }
          }
      }

    g += np;
    P = pc.end;
    ++piece;
  }
}

template <int D, int G, int HG, int DT>
static cudaError_t launch_mma(const DecodeArgs &a, const CUtensorMap &tmK, const CUtensorMap &tmV,
                              int ctas, cudaStream_t s) {
  // stages and q buffers within ~210 KiB: prefer 3+ stages and double q buffers
  constexpr int STAGE = 2 * (D / 64) * HG * BLK * 128;
  constexpr int QBYTES = HG * G * D * 2 + (D / 2) * 16;
  constexpr int BUDGET = 210 * 1024;
  constexpr int S2 = (BUDGET - 2 * QBYTES) / STAGE;
  constexpr int QB = S2 >= 3 ? 2 : 1;
  constexpr int SRAW = (BUDGET - QB * QBYTES) / STAGE;
  constexpr int S = SRAW < 2 ? 2 : (SRAW > 24 ? 24 : SRAW);
  using Lay = DecodeLayout<D, G, HG, S, QB>;
  auto kern = decode_mma_kernel<D, G, HG, S, QB, DT>;
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

cudaError_t launch_decode_mma(const DecodeArgs &a, const CUtensorMap &tmK, const CUtensorMap &tmV,
                              int D, int G, int HG, int dtype, int ctas, cudaStream_t s) {
#define KVINJ_MMA_CASE(DD, GG, HH, TT)                     \
  if (D == DD && G == GG && HG == HH && dtype == TT) \
    return launch_mma<DD, GG, HH, TT>(a, tmK, tmV, ctas, s);
#define KVINJ_MMA_G(DD, HH, TT)                                                        \
  KVINJ_MMA_CASE(DD, 1, HH, TT) KVINJ_MMA_CASE(DD, 2, HH, TT) KVINJ_MMA_CASE(DD, 4, HH, TT) \
  KVINJ_MMA_CASE(DD, 8, HH, TT) KVINJ_MMA_CASE(DD, 16, HH, TT)
#define KVINJ_MMA_H(DD, TT) \
  KVINJ_MMA_G(DD, 1, TT) KVINJ_MMA_G(DD, 2, TT) KVINJ_MMA_G(DD, 4, TT) KVINJ_MMA_G(DD, 8, TT)
  KVINJ_MMA_H(64, 0)
  KVINJ_MMA_H(64, 1)
  KVINJ_MMA_H(128, 0)
  KVINJ_MMA_H(128, 1)
#undef KVINJ_MMA_H
#undef KVINJ_MMA_G
#undef KVINJ_MMA_CASE
  return cudaErrorInvalidValue;
}

}  // namespace kvinj
