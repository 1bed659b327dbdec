// kvinj_decode_i8.cu -- split-K paged GQA decode over an int8 KV cache on the
// tcgen05 tensor cores.
//
// "Latency Optimization > KV Cache Management", KV cache quantization: int8
// halves the cache's bytes, and decode reads the whole cache every step ("Inside
// LLM Inference Engines ...", the memory-bound Decode Phase). Each stored row
// (token, kv head) holds D = 128 int8 codes and one fp32 scale; its value is
// code * scale. Per request r and query head qh (kv head h = qh / G):
//   out = sum_p softmax_p((R_{q_pos} q * scale) . (c^K_p s^K_p)) c^V_p s^V_p
//       = sum_p w_p s^V_p c^V_p,  w_p = softmax_p(s^K_p * (q' . c^K_p)).
//
// Work split, producer, partial states and combine pass are those of the
// 16-bit kernels (kvinj_decode_common.cuh); the unit is the tcgen05 kernel's
// (128 rows: one block of 8 kv heads, or at G = 8 two blocks of 4), staged by
// TMA as int8 code tiles plus the rows' scales (34 KiB a stage, three stages).
// There is no int8 tensor-core path here (its rate on this part is low), so
// the codes become 16-bit operands on the chip -- exactly, an int8 value being
// a 16-bit float too:
//   K: each converter thread turns its row's 128 codes into 16-bit values and
//      stores them in tensor memory, where they are the A operand of the QK
//      MMA (lane = unit row, two values per column); the row's K scale, V
//      scale and block valid bit go to tensor memory beside them.
//   V: each converter thread writes its row's 128 values into a 16-bit V tile
//      in shared memory (two of them, by unit parity), in the 128-byte swizzled
//      layout the PV MMA reads as its MN-major A operand.
// The stage is released as soon as the converters have read it, so the stages
// stay in flight instead of waiting for their unit's softmax, and with two V
// tiles and two K operands the converters run a unit ahead of the MMAs.
//   QK: S[128 x N] = codes^K[128 x 128] Q^T[128 x N] (N = 2*HG*G: hi and lo
//       parts of each rotated, scaled query, as in the 16-bit kernel). The MMA
//       operands are fp16 whatever the query type.
//   softmax: the row's score is (S_hi + S_lo) * s^K; the probability written
//       to the P tile is p * s^V (p itself goes into the running sum l).
//   PV: O^T[128 x N] += V^T[128 x 128] P^T[128 x N].
// The fused append writes the new token's codes and scales (rotated exactly,
// then quantized, as the int8 inject does) before its block is streamed.
//
// Warp roles (384 threads, 512 with two softmax sets at G >= 2):
//   warp 0      TMA producer (int8 stages)
//   warp 1      TMEM owner; lane 0 issues every MMA and commit
//   warps 2-3   query preparation and the fused append
//   warps 4-7   softmax, P tile, rescaling of O, end-of-piece output (set 0)
//   warps 8-11  converters (warp 8 + i owns unit rows 32i .. 32i + 31)
//   warps 12-15 softmax set 1 at G >= 2: the same rows as set 0, the other half of each kv
//               head's query heads (and of O's columns)
// Every wait is bounded; a wait that gives up sets the abort flag and
// KVINJ_ST_TIMEOUT, and all roles still reach the final barrier.
#include <math.h>

#include "kvinj_decode_common.cuh"
#include "kvinj_umma.cuh"

namespace kvinj {

namespace {

constexpr float I8_TAU = 8.f;  // lazy-maximum threshold, log2 units
// threads: 0 producer, 1 MMA, 2-3 queries, 4-7 softmax set 0, 8-11 converters, and with
// two softmax sets (G >= 2) 12-15 set 1 (the same tensor-memory lanes as set 0; each set owns
// half of the query heads of every kv head)
template <int SW>
constexpr int i8_threads() { return 256 + 128 * SW; }
template <int G>
constexpr int I8_SOFTMAX_SETS = G >= 2 ? 2 : 1;

template <int G_, int S_, int QBUF_, int HG_, int BPU_>
struct I8Layout {
  static constexpr int D = 128, G = G_, HG = HG_, S = S_, BPU = BPU_;
  static constexpr int QB = 0;               // the producer stages no query rows
  static constexpr int QBUF = QBUF_;         // Q tiles, written by the query warps
  static constexpr int EMPTY_ARRIVALS = 4;   // the four converter warps free a stage
  static constexpr bool SPLIT_KV = false;
  static constexpr int VR = S;
  static constexpr bool I8 = true;
  static constexpr bool QPOS_SM = true;      // the query warps read q positions there
  static constexpr bool APPEND_WAIT = true;  // the producer waits for a fused append
  static constexpr int N = HG * 2 * G;       // MMA N
  static constexpr int ROWS = HG * BPU * BLK;           // 128 unit rows
  static constexpr int CODE_BYTES = ROWS * D;           // 16 KiB of K (or V) codes
  static constexpr int SC_BYTES = ROWS * 4;             // the rows' K (or V) scales
  static constexpr int STAGE_TX = 2 * CODE_BYTES + 2 * SC_BYTES;
  static constexpr int STAGE_BYTES = (STAGE_TX + 1023) / 1024 * 1024;
  static constexpr int NBOX = 1, BOXB = CODE_BYTES;
  static constexpr int TILE_BYTES = N * 2 * D;          // Q / P tiles: N rows x 128 16-bit
  static constexpr int VT_BYTES = ROWS * D * 2;         // V as 16-bit values: 32 KiB
  static constexpr int VT_BLOCK = ROWS * 128;           // one 64-column block of it
  static constexpr int Q_BYTES = 0, T_BYTES = 0;
  static constexpr int off_stage = 0;
  static constexpr int off_vt = S * STAGE_BYTES;        // [2] V tiles
  static constexpr int off_q = off_vt + 2 * VT_BYTES;   // [QBUF] Q tiles
  static constexpr int off_t = off_q;                   // unused
  static constexpr int off_p = off_q + QBUF * TILE_BYTES;
  static constexpr int off_bar = off_p + TILE_BYTES;    // full[S] empty[S]
  // sfull[2] sfree[2] pfull pvdone qfull[QBUF] qempty[QBUF] ofree done kfull[2] vfull[2]
  // vfree[2]
  static constexpr int NXBAR = 14 + 2 * QBUF;
  static constexpr int off_xbar = off_bar + 2 * S * 8;
  static constexpr int off_qfull = off_xbar + 6 * 8;
  static constexpr int off_valid = off_xbar + NXBAR * 8;   // [VR] valid bits
  static constexpr int off_qinfo = off_valid + VR * 4;     // unused (no bytes)
  static constexpr int off_flags = off_qinfo;              // [0] abort [8..24) scan
  static constexpr int off_alpha = off_flags + 96;         // [2][N] factors, [2][8] flags
  static constexpr int off_ml = off_alpha + 2 * N * 4 + 64;
  static constexpr int off_tmem = off_ml + 2 * HG * G * 4;
  static constexpr int off_pre = off_tmem + 16;            // pre[batch + 1], then qpos[batch]
  // tensor memory: S[2] at columns 0 and N, O at 2N, the K operands [2] at KT and KT + 64,
  // the rows' {K scale, V scale, valid} [2] at SC and SC + 4
  static constexpr int KT = (3 * N + 63) / 64 * 64;
  static constexpr int SC = KT + 128;
  static constexpr uint32_t TMEM_COLS = SC + 8 <= 256 ? 256 : 512;
  static size_t bytes(int batch) { return (size_t)off_pre + (size_t)(2 * batch + 1) * 4; }
  static_assert(ROWS == 128, "a unit is 128 rows: the MMA's M");
  static_assert(STAGE_BYTES % 1024 == 0 && off_vt % 1024 == 0 && off_q % 1024 == 0 &&
                    off_p % 1024 == 0,
                "swizzle atoms are 1024-byte aligned");
};

template <int NR>
__device__ __forceinline__ uint32_t i8_tile_off(int n, int c) {
  return (c >> 6) * (NR * 128) + n * 128 + ((((c & 63) >> 3) ^ (n & 7)) << 4) + (c & 7) * 2;
}

__device__ __forceinline__ void sts16_(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ void sts32_(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void sts128_(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                        uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ void sts128z_(uint32_t addr) { sts128_(addr, 0, 0, 0, 0); }

// D[tmem] (+)= A[tmem] * B[smem], issued by one thread; acc = 0 overwrites D
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                            uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc)
      : "memory");
}

// four int8 codes (lowest byte first) -> two words of two 16-bit values each, exactly.
// bf16: a code's byte b in the 7 mantissa bits under the exponent of 128 is 128 + (b & 127);
// subtracting 128, or 256 when b's top bit is set (the byte of a negative code), leaves
// the code. fp16: 1024 + u - 1152 with u = code + 128.
template <int DT>
__device__ __forceinline__ void codes_to16(uint32_t x, uint32_t &w01, uint32_t &w23) {
  if constexpr (DT == 0) {
    const uint32_t p01 = __byte_perm(x, 0u, 0x4140), p23 = __byte_perm(x, 0u, 0x4342);
    const uint32_t a01 = (p01 & 0x007F007Fu) | 0x43004300u, s01 = (p01 & 0x00800080u) | 0x43004300u;
    const uint32_t a23 = (p23 & 0x007F007Fu) | 0x43004300u, s23 = (p23 & 0x00800080u) | 0x43004300u;
    const __nv_bfloat162 r01 = __hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&a01),
                                       *reinterpret_cast<const __nv_bfloat162 *>(&s01));
    const __nv_bfloat162 r23 = __hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&a23),
                                       *reinterpret_cast<const __nv_bfloat162 *>(&s23));
    w01 = *reinterpret_cast<const uint32_t *>(&r01);
    w23 = *reinterpret_cast<const uint32_t *>(&r23);
  } else {
    const uint32_t u = x ^ 0x80808080u;
    const uint32_t h01 = __byte_perm(u, 0x64646464u, 0x5140);
    const uint32_t h23 = __byte_perm(u, 0x64646464u, 0x5342);
    const __half2 off = __floats2half2_rn(1152.f, 1152.f);
    const __half2 a = __hsub2(*reinterpret_cast<const __half2 *>(&h01), off);
    const __half2 b = __hsub2(*reinterpret_cast<const __half2 *>(&h23), off);
    w01 = *reinterpret_cast<const uint32_t *>(&a);
    w23 = *reinterpret_cast<const uint32_t *>(&b);
  }
}

// a row of D = 128 values held by one warp (lane l: x = dims 2l, 2l+1, y = 64+2l, 64+2l+1)
// quantized and stored: codes at codes[d], scale at *scale (lane 0)
__device__ __forceinline__ void quant_row_warp(float x0, float x1, float y0, float y1,
                                               int lane, int8_t *codes, float *scale) {
  float m = fmaxf(fmaxf(fabsf(x0), fabsf(x1)), fmaxf(fabsf(y0), fabsf(y1)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  const float s = quant_scale(m), inv = quant_inv(s);
  const uint16_t cx =
      (uint16_t)((quant_code(x0, s, inv) & 0xFF) | ((quant_code(x1, s, inv) & 0xFF) << 8));
  const uint16_t cy =
      (uint16_t)((quant_code(y0, s, inv) & 0xFF) | ((quant_code(y1, s, inv) & 0xFF) << 8));
  *reinterpret_cast<uint16_t *>(codes + 2 * lane) = cx;
  *reinterpret_cast<uint16_t *>(codes + 64 + 2 * lane) = cy;
  if (lane == 0) *scale = s;
}

template <int DT>
__device__ __forceinline__ float val16(uint16_t b) {
  if constexpr (DT == 0) return __uint_as_float((uint32_t)b << 16);
  else return __half2float(__ushort_as_half(b));
}

template <int G, int S, int QBUF, int DT, int HG, int BPU, int SW>
__global__ void __launch_bounds__(i8_threads<SW>(), 1)
    decode_i8_kernel(const __grid_constant__ CUtensorMap tmK,
                     const __grid_constant__ CUtensorMap tmV, DecodeArgs a) {
  using Lay = I8Layout<G, S, QBUF, HG, BPU>;
  constexpr int D = 128, N = Lay::N, PF = partial_floats(G, D), SLOT = HG * PF;
  // MMA operands are fp16 whatever the query type: codes are exact in it, its conversion
  // is the cheaper one, and its hi/lo parts carry more of q and p than bf16's would
  constexpr int OT = 1;
  constexpr int TPH = BLK * BPU;   // tokens of a head in a unit (its rows are consecutive)
  constexpr int HPW = 32 / TPH;    // heads per softmax warp
  static_assert(G == 1 || G == 2 || G == 4 || G == 8, "int8 decode: G");
  constexpr int NT = i8_threads<SW>();
  constexpr int GS = G / SW;       // query heads per kv head of one softmax set
  static_assert(SW == 1 || (SW == 2 && G >= 2 && HG % 2 == 0), "softmax sets");

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *sm = smem_raw;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (smem_u32(sm) & 1023u) {  // the swizzled tiles need 1024-byte alignment
    if (tid == 0) report(a.status, KVINJ_ST_INTERNAL);
    return;
  }
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + Lay::off_bar);
  uint64_t *empty = full + S;
  uint64_t *sfull = reinterpret_cast<uint64_t *>(sm + Lay::off_xbar);
  uint64_t *sfree = sfull + 2, *pfull = sfull + 4, *pvdone = sfull + 5;
  uint64_t *qfull = sfull + 6, *qempty = qfull + QBUF, *ofree = qempty + QBUF, *done = ofree + 1;
  uint64_t *kfull = done + 1, *vfull = kfull + 2, *vfree = vfull + 2;
  volatile int *flags = reinterpret_cast<volatile int *>(sm + Lay::off_flags);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + Lay::off_tmem);
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(sfull + b, 1);
      mbar_init(sfree + b, 4 * SW);
      mbar_init(kfull + b, 4);
    }
    mbar_init(pfull, 4 * SW);
    mbar_init(pvdone, 1);
    for (int b = 0; b < QBUF; ++b) {
      mbar_init(qfull + b, 2);
      mbar_init(qempty + b, 1);
    }
    mbar_init(ofree, 4 * SW);
    mbar_init(done, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(vfull + b, 4);
      mbar_init(vfree + b, 1);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tslot, Lay::TMEM_COLS);
    tmem_relinquish();
  }
  CtaRange rg;
  const bool has_units = decode_prologue<Lay, NT>(a, sm, rg);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (!has_units) {
    if (warp == 1) tmem_dealloc(*tslot, Lay::TMEM_COLS);
    return;
  }
  const uint32_t tbase = *tslot;
  const int *pre = reinterpret_cast<const int *>(sm + Lay::off_pre);
  const int ngrp = a.Hkv / HG;
  const uint32_t stage0 = smem_u32(sm + Lay::off_stage);
  const uint32_t q0 = smem_u32(sm + Lay::off_q), p0 = smem_u32(sm + Lay::off_p);
  const uint32_t vt0 = smem_u32(sm + Lay::off_vt);

  auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
    if (flags[0]) return false;
    if (mbar_wait_bounded(bar, parity)) return true;
    report(a.status, KVINJ_ST_TIMEOUT);
    flags[0] = 1;
    return false;
  };

  if (warp == 0) {
    decode_producer<Lay>(a, tmK, tmV, sm, rg, lane);
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      constexpr uint32_t ID_QK = umma_idesc_f16<OT>(128, N, 0, 0);  // A (codes) from TMEM
      constexpr uint32_t ID_PV = umma_idesc_f16<OT>(128, N, 1, 0);  // A = V^T, MN-major smem
      auto issue_qk = [&](int gi, int qbuf) {
        const int par = gi & 1;
        if (!wait(kfull + par, (uint32_t)(gi >> 1) & 1u)) return;
        if (gi >= 2 && !wait(sfree + par, (uint32_t)((gi >> 1) - 1) & 1u)) return;
        tc_fence_after();
        const uint32_t qb = q0 + qbuf * Lay::TILE_BYTES;
        const uint32_t d = tbase + par * N, ka = tbase + Lay::KT + par * 64;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_f16_ta(d, ka + kk * 8,
                      umma_desc_sw128(qb + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024),
                      ID_QK, kk > 0);
        umma_commit(sfull + par);
      };
      int P = rg.b0, gi0 = 0, piece = 0;
      while (P < rg.b1) {
        const Piece pc = find_piece<BPU>(a, pre, ngrp, P, rg.b1);
        const int np = pc.end - P, qbuf = piece % QBUF;
        if (wait(qfull + qbuf, (uint32_t)(piece / QBUF) & 1u)) issue_qk(gi0, qbuf);
        if (piece > 0) wait(ofree, (uint32_t)(piece - 1) & 1u);  // O read out
        for (int j = 0; j < np; ++j) {
          const int gi = gi0 + j;
          // QK of the next unit of the piece goes out before this unit's PV: its K operand
          // comes from the converters (which run a unit ahead), never from this unit's P,
          // so the next S is computed while this unit's softmax runs
          if (j + 1 >= np) umma_commit(qempty + qbuf);  // the Q tile is free once its QKs are
          if (j + 1 < np) issue_qk(gi + 1, qbuf);
          if (!wait(pfull, (uint32_t)gi & 1u)) continue;
          if (!wait(vfull + (gi & 1), (uint32_t)(gi >> 1) & 1u)) continue;
          tc_fence_after();
          const uint32_t vt = vt0 + (gi & 1) * Lay::VT_BYTES;
#pragma unroll
          for (int kk = 0; kk < Lay::ROWS / 16; ++kk)
            umma_f16(tbase + 2 * N, umma_desc_sw128(vt + kk * 2048, Lay::VT_BLOCK, 1024),
                     umma_desc_sw128(p0 + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024),
                     ID_PV, (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit(vfree + (gi & 1));
          umma_commit(pvdone);
        }
        gi0 += np;
        P = pc.end;
        ++piece;
      }
      umma_commit(done);
      if (!mbar_wait_bounded(done, 0, 100000000ull)) {
        report(a.status, KVINJ_ST_TIMEOUT);
        flags[0] = 1;
      }
    }
    __syncwarp();
  } else if (warp < 4) {
    // --------------------------- query preparation ---------------------------
    const int qw = warp - 2;
    constexpr int RPW = HG * G / 2;  // rows per warp
    const int *qpos_sm = pre + a.batch + 1;
    int P = rg.b0, piece = 0;
    while (P < rg.b1) {
      const Piece pc = find_piece<BPU>(a, pre, ngrp, P, rg.b1);
      const int qbuf = piece % QBUF;
      int qp = a.rope ? qpos_sm[pc.r] : -1;
      if (a.rope && (qp < 0 || qp >= a.max_pos)) {
        if (qw == 0 && lane == 0) report(a.status, KVINJ_ST_BAD_POS);
        qp = -1;
      }
      float4 t0 = make_float4(1.f, 0.f, 0.f, 0.f), t1 = t0;
      if (qp >= 0) {
        const float4 *tab = a.rope + (int64_t)qp * (D / 2);
        t0 = __ldg(tab + 2 * lane);
        t1 = __ldg(tab + 2 * lane + 1);
      }
      uint32_t xw[RPW], yw[RPW];
      const uint16_t *qg = a.q + ((int64_t)pc.r * a.Hq + (int64_t)pc.hg * HG * G) * D;
#pragma unroll
      for (int k = 0; k < RPW; ++k) {
        const uint16_t *row = qg + (int64_t)(2 * k + qw) * D;
        xw[k] = __ldg(reinterpret_cast<const unsigned int *>(row + 2 * lane));
        yw[k] = __ldg(reinterpret_cast<const unsigned int *>(row + 64 + 2 * lane));
      }
      // fused append: the token at q_pos, if its block is one of this piece's units
      const int qa = qpos_sm[pc.r];
      const int pg_a = qa >= 0 ? qa / BLK : -1;
      const bool app = a.k_new && qa >= 0 && (!a.rope || qa < a.max_pos) &&
                       pg_a / BPU >= pc.pg0 && pg_a / BPU < pc.pg0 + (pc.end - P);
      uint32_t akx[HG / 2], aky[HG / 2], avx[HG / 2], avy[HG / 2];
      int64_t abl = -1;
      if (app) {
        abl = a.block_tables[(int64_t)pc.r * a.max_blocks + pg_a];
#pragma unroll
        for (int k = 0; k < HG / 2; ++k) {
          const int64_t src = ((int64_t)pc.r * a.Hkv + pc.hg * HG + qw * (HG / 2) + k) * D;
          akx[k] = __ldg(reinterpret_cast<const unsigned int *>(a.k_new + src + 2 * lane));
          aky[k] = __ldg(reinterpret_cast<const unsigned int *>(a.k_new + src + 64 + 2 * lane));
          avx[k] = __ldg(reinterpret_cast<const unsigned int *>(a.v_new + src + 2 * lane));
          avy[k] = __ldg(reinterpret_cast<const unsigned int *>(a.v_new + src + 64 + 2 * lane));
        }
      }
      bool ok = true;
      if (piece >= QBUF) ok = wait(qempty + qbuf, (uint32_t)(piece / QBUF - 1) & 1u);
      if (ok) {
        const uint32_t qt = q0 + qbuf * Lay::TILE_BYTES;
        const float sc = a.scale_log2;
#pragma unroll
        for (int k = 0; k < RPW; ++k) {
          const int row = 2 * k + qw, h = row / G, g = row % G;
          const float2 x = unpack2<DT>(xw[k]), y = unpack2<DT>(yw[k]);
          float x0 = x.x, x1 = x.y, y0 = y.x, y1 = y.y;
          if (qp >= 0) {
            const float2 r0 = rope_pair(x.x, y.x, t0);
            const float2 r1 = rope_pair(x.y, y.y, t1);
            x0 = r0.x;
            y0 = r0.y;
            x1 = r1.x;
            y1 = r1.y;
          }
          x0 *= sc, x1 *= sc, y0 *= sc, y1 *= sc;
          // fp16 hi and lo parts (the MMA operand type of this kernel)
          const uint32_t xh = pack2<OT>(x0, x1), yh = pack2<OT>(y0, y1);
          const float2 xf = unpack2<OT>(xh), yf = unpack2<OT>(yh);
          const uint32_t xl = pack2<OT>(x0 - xf.x, x1 - xf.y), yl = pack2<OT>(y0 - yf.x, y1 - yf.y);
          const int nh = h * 2 * G + g, nl = nh + G;
          sts32_(qt + i8_tile_off<N>(nh, 2 * lane), xh);
          sts32_(qt + i8_tile_off<N>(nh, 64 + 2 * lane), yh);
          sts32_(qt + i8_tile_off<N>(nl, 2 * lane), xl);
          sts32_(qt + i8_tile_off<N>(nl, 64 + 2 * lane), yl);
        }
        if (app) {
          if (abl < 0 || abl >= a.num_blocks) {
            if (lane == 0) report(a.status, KVINJ_ST_BAD_BLOCK);
          } else {
            int8_t *kc = reinterpret_cast<int8_t *>(a.k_cache);
            int8_t *vc = reinterpret_cast<int8_t *>(a.v_cache);
            const double2 *t64 = a.rope ? a.rope64 + (int64_t)qa * (D / 2) : nullptr;
#pragma unroll
            for (int k = 0; k < HG / 2; ++k) {
              const int h = pc.hg * HG + qw * (HG / 2) + k;
              const int64_t r = ((int64_t)a.layer * a.num_blocks + abl) * a.Hkv * BLK +
                                (int64_t)h * BLK + qa % BLK;
              float2 kx = unpack2<DT>(akx[k]), ky = unpack2<DT>(aky[k]);
              if (a.rope) {
                const ushort2 e0 = rope_pair_exact<DT>(kx.x, ky.x, t0, t64 + 2 * lane);
                const ushort2 e1 = rope_pair_exact<DT>(kx.y, ky.y, t1, t64 + 2 * lane + 1);
                kx = make_float2(val16<DT>(e0.x), val16<DT>(e1.x));
                ky = make_float2(val16<DT>(e0.y), val16<DT>(e1.y));
              }
              quant_row_warp(kx.x, kx.y, ky.x, ky.y, lane, kc + r * D, a.k_scale + r);
              const float2 vx = unpack2<DT>(avx[k]), vy = unpack2<DT>(avy[k]);
              quant_row_warp(vx.x, vx.y, vy.x, vy.y, lane, vc + r * D, a.v_scale + r);
            }
            // these generic stores precede the producer's tensor copy of the block
            asm volatile("fence.proxy.async.global;" ::: "memory");
          }
        }
        fence_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(qfull + qbuf);
      P = pc.end;
      ++piece;
    }
  } else if (warp < 8 || warp >= 12) {
    // -------------------------------- softmax --------------------------------
    const int qd = warp & 3;
    const int set = SW == 1 ? 0 : (warp >= 12 ? 1 : 0);  // query heads g0 .. g0 + GS - 1
    const int g0 = set * GS, hh0 = set * (HG / SW);     // ... and this set's O columns
    const int row = 32 * qd + lane;  // unit row = head * TPH + token; O row = dimension
    const int hs = lane / TPH, h = HPW * qd + hs, t = lane % TPH;
    float *alpha_sm = reinterpret_cast<float *>(sm + Lay::off_alpha);
    volatile int *rflag = reinterpret_cast<volatile int *>(alpha_sm + 2 * N);
    float *m_sm = reinterpret_cast<float *>(sm + Lay::off_ml), *l_sm = m_sm + HG * G;
    // the P tile's off-diagonal blocks stay zero
    for (int i = 128 * set + 32 * qd + lane; i < Lay::TILE_BYTES / 16; i += 128 * SW)
      sts128z_(p0 + 16 * i);
    fence_async_smem();

    int P = rg.b0, gi0 = 0;
    while (P < rg.b1) {
      const Piece pc = find_piece<BPU>(a, pre, ngrp, P, rg.b1);
      const int np = pc.end - P;
      float m_run[GS], l_part[GS];
#pragma unroll
      for (int g = 0; g < GS; ++g) {
        m_run[g] = -INFINITY;
        l_part[g] = 0.f;
      }
      for (int j = 0; j < np; ++j) {
        const int gi = gi0 + j, par = gi & 1;
        const bool ok = wait(sfull + par, (uint32_t)(gi >> 1) & 1u);
        const int tok = (pc.pg0 + j) * TPH + t;
        float s[GS], sk = 0.f, sv = 0.f;
        uint32_t vflag = 0;
        if (ok) {
          tc_fence_after();
          uint32_t r[HPW * 2 * G];
          tmem_ld<HPW * 2 * G>(tmem_addr(tbase + par * N, 32 * qd, HPW * 2 * G * qd), r);
          uint32_t q4[4];
          tmem_ld<4>(tmem_addr(tbase + Lay::SC + par * 4, 32 * qd, 0), q4);
          sk = __uint_as_float(q4[0]);
          sv = __uint_as_float(q4[1]);
          vflag = q4[2];
          // (register indices stay compile-time: a set picks its half by a select)
          auto score = [&](int g) {
            return (HPW == 2 && hs) ? __uint_as_float(r[(2 * G + g) % (HPW * 2 * G)]) +
                                          __uint_as_float(r[(3 * G + g) % (HPW * 2 * G)])
                                    : __uint_as_float(r[g]) + __uint_as_float(r[G + g]);
          };
#pragma unroll
          for (int gl = 0; gl < GS; ++gl) s[gl] = (SW == 2 && set) ? score(GS + gl) : score(gl);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sfree + par);
        const bool live = ok && vflag && tok < pc.ctx && tok >= pc.lo;
#pragma unroll
        for (int g = 0; g < GS; ++g) s[g] = live ? s[g] * sk : -INFINITY;
        float alpha[GS], p[GS];
        bool resc = false;
#pragma unroll
        for (int g = 0; g < GS; ++g) {
          float mu = s[g];
#pragma unroll
          for (int o = 1; o < TPH; o <<= 1) mu = fmaxf(mu, __shfl_xor_sync(0xffffffffu, mu, o));
          alpha[g] = 1.f;
          if (mu > m_run[g] + I8_TAU) {
            alpha[g] = exp2f(m_run[g] - mu);
            m_run[g] = mu;
            resc = true;
          }
          p[g] = (s[g] == -INFINITY) ? 0.f : ex2_approx(s[g] - m_run[g]);
          l_part[g] = __fmaf_rn(l_part[g], alpha[g], p[g]);
        }
        if (t == 0) {
#pragma unroll
          for (int g = 0; g < GS; ++g) {
            alpha_sm[par * N + h * 2 * G + g0 + g] = alpha[g];
            alpha_sm[par * N + h * 2 * G + G + g0 + g] = alpha[g];
          }
        }
        const int any = __any_sync(0xffffffffu, resc);
        if (lane == 0) rflag[par * 8 + set * 4 + qd] = any;
        named_bar_sync(1, 128 * SW);
        int anyr = 0;
#pragma unroll
        for (int f = 0; f < 4 * SW; ++f) anyr |= rflag[par * 8 + f];
        const bool need = j > 0 && anyr;
        // PV of the previous unit done: the P tile is free and O is current
        bool okpv = true;
        if (j > 0) {
          okpv = wait(pvdone, (uint32_t)(gi - 1) & 1u);
          if (okpv) tc_fence_after();
        }
        if (need && okpv) {
#pragma unroll
          for (int k = 0; k < HG / SW; ++k) {
            const int hh = hh0 + k;
            uint32_t o[2 * G];
            const uint32_t ta = tmem_addr(tbase + 2 * N, 32 * qd, hh * 2 * G);
            tmem_ld<2 * G>(ta, o);
#pragma unroll
            for (int c = 0; c < 2 * G; ++c)
              o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha_sm[par * N + hh * 2 * G + c]);
            tmem_st<2 * G>(ta, o);
          }
        }
        // P^T: column k = row of this thread; each probability times its row's V scale
#pragma unroll
        for (int gl = 0; gl < GS; ++gl) {
          const int g = g0 + gl;
          const float pv = live ? p[gl] * sv : 0.f;
          const uint16_t hi = f32_to16<OT>(pv);
          const uint16_t lo = f32_to16<OT>(pv - val16<OT>(hi));
          sts16_(p0 + i8_tile_off<N>(h * 2 * G + g, row), hi);
          sts16_(p0 + i8_tile_off<N>(h * 2 * G + G + g, row), lo);
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(pfull);
      }

      // ---- end of piece: outputs or the partial state ----
      float l_tot[GS];
#pragma unroll
      for (int g = 0; g < GS; ++g) {
        float x = l_part[g];
#pragma unroll
        for (int o = 1; o < TPH; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        l_tot[g] = x;
      }
      if (t == 0) {
#pragma unroll
        for (int g = 0; g < GS; ++g) {
          m_sm[h * G + g0 + g] = m_run[g];
          l_sm[h * G + g0 + g] = l_tot[g];
        }
      }
      named_bar_sync(1, 128 * SW);
      const bool complete = (P == pc.seg_start) && (pc.end == pc.seg_end);
      float *slot = a.partials + (size_t)(2 * blockIdx.x + (pc.seg_start <= rg.b0 ? 0 : 1)) * SLOT;
      if (wait(pvdone, (uint32_t)(gi0 + np - 1) & 1u)) {
        tc_fence_after();
        const int d = row;
        uint16_t *obase = a.out + ((int64_t)pc.r * a.Hq + (int64_t)pc.hg * HG * G) * D + d;
#pragma unroll
        for (int k = 0; k < HG / SW; ++k) {
          const int hh = hh0 + k;
          uint32_t o[2 * G];
          tmem_ld<2 * G>(tmem_addr(tbase + 2 * N, 32 * qd, hh * 2 * G), o);
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const float v = __uint_as_float(o[g]) + __uint_as_float(o[G + g]);
            if (complete) {
              const float l = l_sm[hh * G + g];
              obase[(hh * G + g) * D] = f32_to16<DT>(l > 0.f ? v * (1.f / l) : 0.f);
            } else {
              slot[hh * PF + 2 * G + g * D + d] = v;
            }
          }
        }
        if (!complete && set == 0 && row < HG * G) {
          slot[(row / G) * PF + row % G] = m_sm[row];
          slot[(row / G) * PF + G + row % G] = l_sm[row];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(ofree);
      gi0 += np;
      P = pc.end;
    }
  } else {
    // ------------------------------- converters -------------------------------
    // thread = unit row r (warp 8 + i: rows 32i .. 32i + 31, its tensor-memory lanes)
    const int cw = warp - 8, r = 32 * cw + lane;
    const int *valid = reinterpret_cast<const int *>(sm + Lay::off_valid);
    // the row's scale index in the stage: rows (head, token) with one block per unit,
    // (head, block, token) with two, whose scales were copied as [block][head][token]
    const int sidx = BPU == 1 ? r : ((r >> 4) & 1) * (HG * BLK) + (r >> 5) * BLK + (r & 15);
    const int vbit = BPU == 1 ? 0 : ((r >> 4) & 1);
    const int n = rg.b1 - rg.b0;
    for (int gi = 0; gi < n; ++gi) {
      const int st = gi % S, par = gi & 1;
      if (!wait(full + st, (uint32_t)(gi / S) & 1u)) break;
      // the K operand and scale columns of this parity were read by QK(gi - 2) and the
      // softmax of unit gi - 2
      if (gi >= 2 && !wait(sfree + par, (uint32_t)((gi >> 1) - 1) & 1u)) break;
      tc_fence_after();
      const uint32_t sb = stage0 + st * Lay::STAGE_BYTES;
      const uint8_t *sp = sm + Lay::off_stage + (size_t)st * Lay::STAGE_BYTES;
      const uint32_t rk = sb + r * 128, rv = sb + Lay::CODE_BYTES + r * 128;
      // K codes of the row -> 16-bit values in tensor memory (both halves issued, then one
      // wait), with the row's scales and valid bit beside them
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t w[32];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint4 v = lds128(rk + (((hh * 4 + c) ^ (r & 7)) << 4));
          codes_to16<OT>(v.x, w[8 * c + 0], w[8 * c + 1]);
          codes_to16<OT>(v.y, w[8 * c + 2], w[8 * c + 3]);
          codes_to16<OT>(v.z, w[8 * c + 4], w[8 * c + 5]);
          codes_to16<OT>(v.w, w[8 * c + 6], w[8 * c + 7]);
        }
        tmem_st32_nw(tmem_addr(tbase + Lay::KT + par * 64 + hh * 32, 32 * cw, 0), w);
      }
      {
        const float *scs = reinterpret_cast<const float *>(sp + 2 * Lay::CODE_BYTES);
        uint32_t q4[4];
        q4[0] = __float_as_uint(scs[sidx]);
        q4[1] = __float_as_uint(scs[Lay::ROWS + sidx]);
        q4[2] = (uint32_t)((valid[st] >> vbit) & 1);
        q4[3] = 0;
        tmem_st4_nw(tmem_addr(tbase + Lay::SC + par * 4, 32 * cw, 0), q4);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(kfull + par);
      // V codes of the row, read before the stage is released
      uint4 vr[8];
#pragma unroll
      for (int c = 0; c < 8; ++c) vr[c] = lds128(rv + ((c ^ (r & 7)) << 4));
      __syncwarp();
      if (lane == 0) mbar_arrive(empty + st);
      // V tile `par` is free once PV(gi - 2) is done
      if (gi >= 2 && !wait(vfree + par, (uint32_t)((gi >> 1) - 1) & 1u)) break;
      const uint32_t vt = vt0 + par * Lay::VT_BYTES;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t w[8];
        codes_to16<OT>(vr[c].x, w[0], w[1]);
        codes_to16<OT>(vr[c].y, w[2], w[3]);
        codes_to16<OT>(vr[c].z, w[4], w[5]);
        codes_to16<OT>(vr[c].w, w[6], w[7]);
        // 16 values = two 16-byte chunks of the 64-column block c / 4 of row r
        const int col = c * 16;
        const uint32_t base = vt + (col >> 6) * Lay::VT_BLOCK + r * 128;
        const int ch = (col & 63) >> 3;
        sts128_(base + ((ch ^ (r & 7)) << 4), w[0], w[1], w[2], w[3]);
        sts128_(base + (((ch + 1) ^ (r & 7)) << 4), w[4], w[5], w[6], w[7]);
      }
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(vfull + par);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, Lay::TMEM_COLS);
  }
}

template <int G, int S, int QBUF, int DT, int HG, int BPU>
cudaError_t launch_i8_cfg(const DecodeArgs &a, const CUtensorMap &tmK, const CUtensorMap &tmV,
                          int ctas, cudaStream_t s) {
  constexpr int SW = I8_SOFTMAX_SETS<G>;
  auto kern = decode_i8_kernel<G, S, QBUF, DT, HG, BPU, SW>;
  const size_t smem = I8Layout<G, S, QBUF, HG, BPU>::bytes(a.batch);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DECODE_MAX_SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaError_t e = launch_pdl(kern, dim3(ctas), dim3(i8_threads<SW>()), smem, s, tmK, tmV, a);
  if (e != cudaSuccess) return e;
  return launch_combine<128, G, HG, DT, BPU, false, BPU == 2 ? 12 : 4>(a, ctas, s);
}

// three stages beside two V tiles and two Q tiles when they fit, else two stages and one Q
// tile (a large batch's prefix sums need the room); G = 8 takes units of two blocks of 4 kv
// heads (N = 64), as the 16-bit kernel does. (Measured on one GB300, 8B- and 70B-shaped
// batches: two stages with two P tiles were slower than this.)
template <int G, int DT>
cudaError_t launch_i8(const DecodeArgs &a, const CUtensorMap &tmK, const CUtensorMap &tmV,
                      int ctas, cudaStream_t s) {
  constexpr int HG = G == 8 ? 4 : 8, BPU = G == 8 ? 2 : 1;
  if (I8Layout<G, 3, 2, HG, BPU>::bytes(a.batch) <= (size_t)DECODE_MAX_SMEM)
    return launch_i8_cfg<G, 3, 2, DT, HG, BPU>(a, tmK, tmV, ctas, s);
  if (I8Layout<G, 2, 1, HG, BPU>::bytes(a.batch) <= (size_t)DECODE_MAX_SMEM)
    return launch_i8_cfg<G, 2, 1, DT, HG, BPU>(a, tmK, tmV, ctas, s);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode_i8(const DecodeArgs &a, const CUtensorMap &tmK, const CUtensorMap &tmV,
                             int G, int dtype, int ctas, cudaStream_t s) {
#define KVINJ_I8_CASE(GG, TT) \
  if (G == GG && dtype == TT) return launch_i8<GG, TT>(a, tmK, tmV, ctas, s);
  KVINJ_I8_CASE(1, 0)
  KVINJ_I8_CASE(2, 0)
  KVINJ_I8_CASE(4, 0)
  KVINJ_I8_CASE(8, 0)
  KVINJ_I8_CASE(1, 1)
  KVINJ_I8_CASE(2, 1)
  KVINJ_I8_CASE(4, 1)
  KVINJ_I8_CASE(8, 1)
#undef KVINJ_I8_CASE
  return cudaErrorInvalidValue;
}

}  // namespace kvinj
