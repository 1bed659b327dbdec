// kvinj_decode_umma.cuh -- split-K paged GQA decode attention on the 5th-
// generation tensor cores (tcgen05, accumulators in tensor memory). The kernel
// template; kvinj_decode_umma.cu instantiates it for calls that wait for the
// kernel ahead before any read, kvinj_decode_umma_early.cu for calls that
// stream their first pages before that wait (KVINJ_DECODE_KV_READY).
//
// Computes, per request r and query head qh (kv head h = qh / G):
//   out = sum_p softmax_p(scale * (R_{q_pos} q) . K_p) V_p
// over the request's context, read block by block through its block table
// ("LLM Inference: KV Caching": attention softmax(QK^T/sqrt d)V and "Paged
// attention"; "Latency Optimization > KV Cache Management": 16-token pages
// gathered through a page table; "Inside LLM Inference Engines ...":
// PagedAttention and the memory-bound Decode Phase).
//
// Work split, TMA producer and partial-state protocol are those of
// kvinj_decode_common.cuh (D = 128). A unit is 128 rows of K and 128 rows of
// V: for G <= 4 one block of a head group of HG = 8 kv heads, for G = 8 two
// consecutive blocks of a group of HG = 4 kv heads (BPU = 2 blocks per unit),
// which keeps N = 2*HG*G at 64 so that three stages fit beside the Q and P
// tiles. What differs from the other kernels is the consumer: one MMA per
// k-step over the whole unit instead of one small contraction per kv head.
//
//   QK: S[128 x N] = K_unit[128 x 128] Q^T[128 x N]. Row i of the unit is
//       (head i / TPH, token i % TPH of the unit), TPH = 16*BPU; the N columns
//       are, per kv head h of the group, the hi and the lo 16-bit parts of its
//       G rotated, scaled queries (columns h*2G + g and h*2G + G + g). Row i
//       only uses the 2G columns of its own head; the other products are
//       computed and ignored (the tensor cores have ample slack in this
//       memory-bound loop).
//   softmax: warps 4..7 each own 32 rows of S (two heads, or one at G = 8),
//       one row per thread; a head's tokens are TPH lanes, reduced with
//       shuffles. At G >= 2 warps 8..11 are a second set on the same rows:
//       each set takes half of the query heads of every kv head (its own
//       exponentials, P columns, O rescale and readout), and the two sets
//       meet at one named barrier per unit.
//   PV: O^T[128 x N] += V_unit^T[128 x 128] P^T[128 x N], where P^T is block
//       diagonal: the column of query head (h, g) holds that head's 16
//       probabilities in the rows of head h and zeros elsewhere, so each
//       head's output only sees its own V rows. V is the A operand as stored
//       (MN-major: the head dimension is contiguous).
//
// Both products accumulate in fp32 in TMEM (S double buffered, O per piece).
// Q and P are fp32 values split x = hi + lo into two 16-bit numbers, so the
// products carry ~16 significant bits of them; K and V are used as stored.
//
// Online softmax with a lazy maximum: per query head the running maximum m
// only moves when a unit's maximum exceeds it by more than TAU (in log2
// units); exponentials are taken against the current m (so are at most
// 2^TAU), and O and l are rescaled only when m moves. The final
// O / l is the same quotient as with an always-current maximum.
//
// At G = 8 the K and V halves of a stage have their own barrier pairs: K is released by a
// commit after its QK, V after its PV, so the next units' K can land while this unit's
// softmax runs; the softmax waits on the V half (the K half's barrier may already be phases
// ahead), and the block valid bits sit in a ring deep enough for that lead.
//
// Sliding window (a.window > 0): a request's units start at the one holding its first
// attended token (context length minus the window); the softmax masks tokens before it as
// it masks those past the context.
//
// Warp roles (256 threads, 384 with two softmax sets):
//   warp 0     TMA producer (stages of K and V rows)
//   warp 1     TMEM owner; lane 0 issues every MMA and commit
//   warps 2-3  query preparation: rotate (RoPE at the request's position),
//              scale, split hi/lo, write the swizzled Q tile of each piece
//   warps 4-7  softmax, P tile, rescaling of O, end-of-piece output
//   warps 8-11 (G >= 2) the second softmax set
// Every wait is bounded; a wait that gives up sets the abort flag and
// KVINJ_ST_TIMEOUT, later waits return at once, and all roles still reach
// the final barrier, after which TMEM is released.
//
// EARLY (a call with KVINJ_DECODE_KV_READY): the prologue and the producer's
// first stages run before the dependency wait on the kernel ahead; every other
// role waits for it first. A separate instantiation, so that the waiting
// kernel carries none of this code.
#pragma once

#include <math.h>

#include "kvinj_decode_common.cuh"
#include "kvinj_umma.cuh"

namespace kvinj {

constexpr float UMMA_TAU = 8.f;  // lazy-maximum threshold, log2 units

// where the combine pass releases the kernel after it (see decode_combine_kernel): at its
// start when this call read its pages early (the next call of a decode step normally does
// too, and its CTAs then take SMs as this call's CTAs leave them), else after its wait
template <bool EARLY, int BPU>
constexpr bool UMMA_COMBINE_RELEASE_EARLY = EARLY;

// softmax warp sets of the kernel at a given G (two halve each softmax thread's query heads)
template <int G>
constexpr int UMMA_SOFTMAX_SETS = G >= 2 ? 2 : 1;

template <int G_, int S_, int QBUF_, int HG_ = 8, int BPU_ = 1>
struct UmmaLayout {
  static constexpr int D = 128, G = G_, HG = HG_, S = S_;
  static constexpr int BPU = BPU_;           // 16-token blocks per unit (HG*BPU*16 = 128 rows)
  static constexpr int QB = 0;               // the producer stages no query rows
  static constexpr int QBUF = QBUF_;         // Q tiles, written by the query warps
  static constexpr int EMPTY_ARRIVALS = 1;   // one MMA commit frees a stage half
  // two-block units (G = 8): K and V halves of a stage have their own barriers, K is freed
  // after its QK and V after its PV (measured faster there; one-block units keep one pair)
  static constexpr bool SPLIT_KV = BPU == 2;
  // valid bits of each unit's blocks: one entry per stage; split stages keep them in a
  // ring, as unit gi's entry is written when its K is issued (after QK(gi - S)), when the
  // softmax has read the entries of units up to gi - S - 2
  static constexpr int VR = SPLIT_KV ? 8 : S;
  static constexpr bool I8 = false;          // 16-bit cache
  static constexpr int CODE_BYTES = 0, SC_BYTES = 0, STAGE_TX = 0;
  static constexpr bool QPOS_SM = true;      // the query warps read q positions there
  static constexpr bool APPEND_WAIT = true;  // the producer waits for a fused append
  static constexpr int N = HG * 2 * G;       // MMA N
  static constexpr int NBOX = D / 64;
  static constexpr int BOXB = HG * BPU * BLK * 128;    // 16 KiB: 128 rows of 128 bytes
  static constexpr int UNIT_BYTES = NBOX * BOXB;       // 32 KiB of K (or V)
  static constexpr int STAGE_BYTES = 2 * UNIT_BYTES;
  static constexpr int TILE_BYTES = N * 2 * D;         // N rows x 128 elements
  static constexpr int Q_BYTES = 0, T_BYTES = 0;       // producer q staging: unused
  static constexpr int off_stage = 0;
  static constexpr int off_q = S * STAGE_BYTES;        // [QBUF] Q tiles
  static constexpr int off_t = off_q;                  // unused
  static constexpr int off_p = off_q + QBUF * TILE_BYTES;
  static constexpr int off_bar = off_p + TILE_BYTES;   // full[S] empty[S] (K), fullV[S] emptyV[S]
                                                       // (split stages; else full/empty cover both)
  // sfull[2] sfree[2] pfull pvdone qfull[QBUF] qempty[QBUF] ofree done
  static constexpr int NXBAR = 8 + 2 * QBUF;
  static constexpr int off_xbar = off_bar + (SPLIT_KV ? 4 : 2) * S * 8;
  static constexpr int off_qfull = off_xbar + 6 * 8;  // qfull[QBUF] (see below)
  static constexpr int off_valid = off_xbar + NXBAR * 8;  // [VR] valid bits
  static constexpr int off_qinfo = off_valid + VR * 4;  // unused (no bytes)
  static constexpr int off_flags = off_qinfo;          // [0] abort [1] unused [8..20) scan
  static constexpr int off_alpha = off_flags + 96;     // [2][N] factors, [2][8] flags
  static constexpr int off_ml = off_alpha + 2 * N * 4 + 64;
  static constexpr int off_tmem = off_ml + 2 * HG * G * 4;
  static constexpr int off_pre = off_tmem + 16;        // pre[batch + 1], then qpos[batch]
  // S[2] at columns 0 and N, O at 2N
  static constexpr uint32_t TMEM_COLS =
      3 * N <= 32 ? 32 : 3 * N <= 64 ? 64 : 3 * N <= 128 ? 128 : 3 * N <= 256 ? 256 : 512;
  // the dynamic shared array is declared 1024-byte aligned: no slack for alignment (the
  // bytes saved let a combine CTA stay resident beside this one)
  static size_t bytes(int batch) { return (size_t)off_pre + (size_t)(2 * batch + 1) * 4; }
  static_assert(3 * N <= 512, "tensor memory: S[2] and O");
  static_assert(HG * BPU * BLK == 128, "a unit is 128 rows: the MMA's M");
  static_assert(off_q % 1024 == 0 && off_p % 1024 == 0, "swizzle atoms are 1024-byte aligned");
};

// byte offset of element (row n, column c) of a K-major tile of NR rows x 128
// columns in the 128-byte swizzle: two blocks of 64 columns, NR*128 bytes each
template <int NR>
__device__ __forceinline__ uint32_t tile_off(int n, int c) {
  return (c >> 6) * (NR * 128) + n * 128 + ((((c & 63) >> 3) ^ (n & 7)) << 4) + (c & 7) * 2;
}

__device__ __forceinline__ void sts16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
__device__ __forceinline__ void sts32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ void sts128_zero(uint32_t addr) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0) : "memory");
}

// warps: 0 producer, 1 MMA issuer and TMEM owner, 2-3 queries, then SW sets of four softmax
// warps (set k: warps 4 + 4k .. 7 + 4k, query heads g in [k G/SW, (k + 1) G/SW) of each kv
// head, the same TMEM lanes as the other sets)
template <int SW>
constexpr int umma_threads() { return 128 + 128 * SW; }

template <int G, int S, int QBUF, int DT, int HG = 8, int BPU = 1, bool EARLY = false,
          int SW = 1>
__global__ void __launch_bounds__(umma_threads<SW>(), 1)
    decode_umma_kernel(const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, DecodeArgs a) {
  using Lay = UmmaLayout<G, S, QBUF, HG, BPU>;
  constexpr int D = 128, N = Lay::N, PF = partial_floats(G, D), SLOT = HG * PF;
  constexpr int NT = umma_threads<SW>();
  constexpr int GS = G / SW;       // query heads per kv head of one softmax set
  static_assert(SW == 1 || (SW == 2 && G >= 2 && HG % 2 == 0), "softmax sets");
  constexpr int TPH = BLK * BPU;   // tokens of a head in a unit (its rows are consecutive)
  constexpr int HPW = 32 / TPH;    // heads per softmax warp
  static_assert(G == 1 || G == 2 || G == 4 || G == 8, "tcgen05 decode: G");

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t *sm = smem_raw;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (smem_u32(sm) & 1023u) {  // the swizzled tiles need 1024-byte alignment
    if (tid == 0) report(a.status, KVINJ_ST_INTERNAL);
    return;
  }

  uint64_t *full = reinterpret_cast<uint64_t *>(sm + Lay::off_bar);  // K halves of the stages
  uint64_t *empty = full + S;
  uint64_t *fullV = full + 2 * S, *emptyV = full + 3 * S;             // V halves
  uint64_t *sfull = reinterpret_cast<uint64_t *>(sm + Lay::off_xbar);
  uint64_t *sfree = sfull + 2, *pfull = sfull + 4, *pvdone = sfull + 5;
  uint64_t *qfull = sfull + 6, *qempty = qfull + QBUF, *ofree = qempty + QBUF, *done = ofree + 1;
  volatile int *flags = reinterpret_cast<volatile int *>(sm + Lay::off_flags);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + Lay::off_tmem);
  // set-up that reads no input runs before the dependency wait (in the prologue)
  if (tid == 0) {
    for (int b = 0; b < 2; ++b) {
      mbar_init(sfull + b, 1);
      mbar_init(sfree + b, 4 * SW);
    }
    mbar_init(pfull, 4 * SW);
    mbar_init(pvdone, 1);
    for (int b = 0; b < QBUF; ++b) {
      mbar_init(qfull + b, 2);
      mbar_init(qempty + b, 1);
    }
    mbar_init(ofree, 4 * SW);
    mbar_init(done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tslot, Lay::TMEM_COLS);
    tmem_relinquish();
  }
  CtaRange rg;
  const bool has_units = decode_prologue<Lay, NT, EARLY>(a, sm, rg);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (!has_units) {
    if constexpr (EARLY) {
      decode_dependency_wait();
      zero_invalid_outputs<128>(a, reinterpret_cast<const int *>(sm + Lay::off_pre), tid, NT);
    }
    if (warp == 1) tmem_dealloc(*tslot, Lay::TMEM_COLS);
    return;
  }
  if constexpr (EARLY) {
    // every role but the producer (which first issues its first stages) waits for the
    // kernel ahead here, before it reads q, the new token or the RoPE table, or writes
    // an output or a partial state (the combine pass of the previous call may still be
    // reading the workspace)
    if (warp != 0) {
      decode_dependency_wait();
      if (warp >= 4)
        zero_invalid_outputs<128>(a, reinterpret_cast<const int *>(sm + Lay::off_pre), tid - 128,
                                  NT - 128);
    }
  }
  const uint32_t tbase = *tslot;
  const int *pre = reinterpret_cast<const int *>(sm + Lay::off_pre);
  const int ngrp = a.Hkv / HG;
  const uint32_t stage0 = smem_u32(sm + Lay::off_stage);
  const uint32_t q0 = smem_u32(sm + Lay::off_q), p0 = smem_u32(sm + Lay::off_p);

  // bounded wait; false once the CTA is aborting
  auto wait = [&](uint64_t *bar, uint32_t parity) -> bool {
    if (flags[0]) return false;
    if (mbar_wait_bounded(bar, parity)) return true;
    report(a.status, KVINJ_ST_TIMEOUT);
    flags[0] = 1;
    return false;
  };

  if (warp == 0) {
    decode_producer<Lay, EARLY>(a, tmK, tmV, sm, rg, lane);
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      constexpr uint32_t ID_QK = umma_idesc_f16<DT>(128, N, 0, 0);
      constexpr uint32_t ID_PV = umma_idesc_f16<DT>(128, N, 1, 0);
      auto issue_qk = [&](int gi, int qbuf) {
        const int st = gi % S;
        if (!wait(full + st, (uint32_t)(gi / S) & 1u)) return;
        if (gi >= 2 && !wait(sfree + (gi & 1), (uint32_t)((gi >> 1) - 1) & 1u)) return;
        tc_fence_after();
        const uint32_t kb = stage0 + st * Lay::STAGE_BYTES, qb = q0 + qbuf * Lay::TILE_BYTES;
        const uint32_t d = tbase + (gi & 1) * N;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_f16(d, umma_desc_sw128(kb + (kk >> 2) * Lay::BOXB + (kk & 3) * 32, 16, 1024),
                   umma_desc_sw128(qb + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024), ID_QK,
                   kk > 0);
        umma_commit(sfull + (gi & 1));
        if constexpr (Lay::SPLIT_KV) umma_commit(empty + st);  // the K half is free
      };
      int P = rg.b0, gi0 = 0, piece = 0;
      while (P < rg.b1) {
        const Piece pc = find_piece<BPU>(a, pre, ngrp, P, rg.b1);
        const int np = pc.end - P, qbuf = piece % QBUF;
        if (wait(qfull + qbuf, (uint32_t)(piece / QBUF) & 1u)) issue_qk(gi0, qbuf);
        if (piece > 0) wait(ofree, (uint32_t)(piece - 1) & 1u);  // O read out
        for (int j = 0; j < np; ++j) {
          const int gi = gi0 + j, st = gi % S;
          // QK of the next unit goes first only if its rows have landed:
          // blocking on them here would hold this unit's stage meanwhile
          bool qk_next = j + 1 >= np;
          if (!qk_next && mbar_test(full + (gi + 1) % S, (uint32_t)((gi + 1) / S) & 1u) &&
              (gi + 1 < 2 || mbar_test(sfree + ((gi + 1) & 1), (uint32_t)(((gi + 1) >> 1) - 1) & 1u))) {
            issue_qk(gi + 1, qbuf);
            qk_next = true;
          }
          if (j + 1 >= np) umma_commit(qempty + qbuf);  // the Q tile is free once its QKs are done
          if (!wait(pfull, (uint32_t)gi & 1u)) continue;
          if (Lay::SPLIT_KV && !wait(fullV + st, (uint32_t)(gi / S) & 1u)) continue;
          tc_fence_after();
          const uint32_t vb = stage0 + st * Lay::STAGE_BYTES + Lay::UNIT_BYTES;
#pragma unroll
          for (int kk = 0; kk < HG * BPU * BLK / 16; ++kk)
            umma_f16(tbase + 2 * N, umma_desc_sw128(vb + kk * 2048, Lay::BOXB, 1024),
                     umma_desc_sw128(p0 + (kk >> 2) * (N * 128) + (kk & 3) * 32, 16, 1024),
                     ID_PV, (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit(Lay::SPLIT_KV ? emptyV + st : empty + st);
          umma_commit(pvdone);
          if (!qk_next) issue_qk(gi + 1, qbuf);
        }
        gi0 += np;
        P = pc.end;
        ++piece;
      }
      // every MMA complete before TMEM and shared memory are released; a wait that
      // gives up leaves this call's output invalid, which the status word says
      umma_commit(done);
      if (!mbar_wait_bounded(done, 0, 100000000ull)) {
        report(a.status, KVINJ_ST_TIMEOUT);
        flags[0] = 1;
      }
    }
    __syncwarp();
  } else if (warp < 4) {
    // --------------------------- query preparation ---------------------------
    // warp qw handles rows qw, qw + 2, ... of the group's HG*G query heads;
    // lane l the dimension pairs (2l, 2l + 64) and (2l + 1, 2l + 65)
    const int qw = warp - 2;
    constexpr int RPW = HG * G / 2;  // rows per warp
    const int *qpos_sm = pre + a.batch + 1;  // copied by the prologue (-1 without RoPE)
    int P = rg.b0, piece = 0;
    while (P < rg.b1) {
      const Piece pc = find_piece<BPU>(a, pre, ngrp, P, rg.b1);
      const int qbuf = piece % QBUF;
      // the loads (query rows, RoPE row) go out before the wait for the tile
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
      // fused append: the token at q_pos, if its block is one of this piece's
      // units, is written here (K rotated at q_pos with the same table row)
      const int qa = qpos_sm[pc.r];
      const int pg_a = qa >= 0 ? qa / BLK : -1;  // the block of the new token
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
          const uint32_t xh = pack2<DT>(x0, x1), yh = pack2<DT>(y0, y1);
          const float2 xf = unpack2<DT>(xh), yf = unpack2<DT>(yh);
          const uint32_t xl = pack2<DT>(x0 - xf.x, x1 - xf.y), yl = pack2<DT>(y0 - yf.x, y1 - yf.y);
          const int nh = h * 2 * G + g, nl = nh + G;
          sts32(qt + tile_off<N>(nh, 2 * lane), xh);
          sts32(qt + tile_off<N>(nh, 64 + 2 * lane), yh);
          sts32(qt + tile_off<N>(nl, 2 * lane), xl);
          sts32(qt + tile_off<N>(nl, 64 + 2 * lane), yl);
        }
        if (app) {
          if (abl < 0 || abl >= a.num_blocks) {
            if (lane == 0) report(a.status, KVINJ_ST_BAD_BLOCK);
          } else {
#pragma unroll
            for (int k = 0; k < HG / 2; ++k) {
              const int h = pc.hg * HG + qw * (HG / 2) + k;
              const int64_t dst =
                  ((((int64_t)a.layer * a.num_blocks + abl) * a.Hkv + h) * BLK + qa % BLK) * D;
              uint32_t kx = akx[k], ky = aky[k];
              if (a.rope) {
                const float2 x = unpack2<DT>(kx), y = unpack2<DT>(ky);
                const float2 r0 = rope_pair(x.x, y.x, t0);
                const float2 r1 = rope_pair(x.y, y.y, t1);
                kx = pack2<DT>(r0.x, r1.x);
                ky = pack2<DT>(r0.y, r1.y);
              }
              st_global(reinterpret_cast<uint32_t *>(a.k_cache + dst + 2 * lane), kx);
              st_global(reinterpret_cast<uint32_t *>(a.k_cache + dst + 64 + 2 * lane), ky);
              st_global(reinterpret_cast<uint32_t *>(a.v_cache + dst + 2 * lane), avx[k]);
              st_global(reinterpret_cast<uint32_t *>(a.v_cache + dst + 64 + 2 * lane), avy[k]);
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
  } else if (warp < 4 + 4 * SW) {
    // -------------------------------- softmax --------------------------------
    const int qd = warp & 3;            // TMEM lane quadrant
    const int set = SW == 1 ? 0 : (warp - 4) >> 2;  // softmax set: heads g0 .. g0 + GS - 1
    const int g0 = set * GS;
    const int hh0 = set * (HG / SW);    // kv heads whose O columns this set rescales and reads
    const int row = 32 * qd + lane;     // unit row = head * 16 + token; O row = dimension
    // unit row = (head, token of the unit): head h owns rows TPH*h .. TPH*h + TPH-1
    const int hs = lane / TPH, h = HPW * qd + hs, t = lane % TPH;
    float *alpha_sm = reinterpret_cast<float *>(sm + Lay::off_alpha);
    volatile int *rflag = reinterpret_cast<volatile int *>(alpha_sm + 2 * N);
    float *m_sm = reinterpret_cast<float *>(sm + Lay::off_ml), *l_sm = m_sm + HG * G;
    const int *valid = reinterpret_cast<const int *>(sm + Lay::off_valid);
    // the P tile's off-diagonal blocks stay zero
    for (int i = tid - 128; i < Lay::TILE_BYTES / 16; i += 128 * SW) sts128_zero(p0 + 16 * i);
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
        const int gi = gi0 + j, st = gi % S, par = gi & 1;
        // the stage's V rows and S. With split stages the wait is on the V half: the K
        // half is released after its QK and its barrier may already be phases ahead, while
        // V is held until this unit's PV (the producer writes the valid bits before it
        // issues the V half).
        const bool ok = wait((Lay::SPLIT_KV ? fullV : full) + st, (uint32_t)(gi / S) & 1u) &&
                        wait(sfull + par, (uint32_t)(gi >> 1) & 1u);
        // this thread's token: in the context and in a block the cache holds
        const int tok = (pc.pg0 + j) * TPH + t;
        const bool live = ok && ((valid[Lay::SPLIT_KV ? gi % Lay::VR : st] >> (t / BLK)) & 1) &&
                          tok < pc.ctx && tok >= pc.lo;
        float s[GS];
        if (ok) {
          tc_fence_after();
          uint32_t r[HPW * 2 * G];
          tmem_ld<HPW * 2 * G>(tmem_addr(tbase + par * N, 32 * qd, HPW * 2 * G * qd), r);
          // (register indices stay compile-time: a set picks its half by a select)
          auto score = [&](int g) {
            return (HPW == 2 && hs) ? __uint_as_float(r[(2 * G + g) % (HPW * 2 * G)]) +
                                          __uint_as_float(r[(3 * G + g) % (HPW * 2 * G)])
                                    : __uint_as_float(r[g]) + __uint_as_float(r[G + g]);
          };
#pragma unroll
          for (int gl = 0; gl < GS; ++gl)
            s[gl] = (SW == 2 && set) ? score(GS + gl) : score(gl);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sfree + par);
        if (!live) {
#pragma unroll
          for (int g = 0; g < GS; ++g) s[g] = -INFINITY;
        }
        // unit maximum per query head; move m only past the threshold
        float alpha[GS], p[GS];
        bool resc = false;
#pragma unroll
        for (int g = 0; g < GS; ++g) {
          float mu = s[g];
#pragma unroll
          for (int o = 1; o < TPH; o <<= 1) mu = fmaxf(mu, __shfl_xor_sync(0xffffffffu, mu, o));
          alpha[g] = 1.f;
          if (mu > m_run[g] + UMMA_TAU) {  // also the first finite maximum
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
          // O row `row` (dimension), every column of this set's kv heads times its factor
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
        // P^T: column k = row of this thread, rows n = (h, g, hi | lo)
#pragma unroll
        for (int gl = 0; gl < GS; ++gl) {
          const int g = g0 + gl;
          const uint16_t hi = to16<DT>(p[gl]);
          const float hf = DT == 0 ? __bfloat162float(__ushort_as_bfloat16(hi))
                                   : __half2float(__ushort_as_half(hi));
          const uint16_t lo = to16<DT>(p[gl] - hf);
          sts16(p0 + tile_off<N>(h * 2 * G + g, row), hi);
          sts16(p0 + tile_off<N>(h * 2 * G + G + g, row), lo);
        }
        // V rows past the context may hold anything (even NaN bit patterns):
        // zero them so that 0 * V stays 0 (each set its column boxes)
        if (!live) {
          const uint32_t vr = stage0 + st * Lay::STAGE_BYTES + Lay::UNIT_BYTES + row * 128;
#pragma unroll
          for (int b = 0; b < Lay::NBOX; ++b)
            if (b % SW == set) {
#pragma unroll
              for (int c = 0; c < 8; ++c) sts128_zero(vr + b * Lay::BOXB + 16 * c);
            }
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
              obase[(hh * G + g) * D] = to16<DT>(l > 0.f ? v * (1.f / l) : 0.f);
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
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, Lay::TMEM_COLS);
  }
}

template <int G, int S, int QBUF, int DT, int HG, int BPU, bool EARLY>
static cudaError_t launch_umma_cfg(const DecodeArgs &a, const CUtensorMap &tmK,
                                   const CUtensorMap &tmV, int ctas, cudaStream_t s) {
  constexpr int SW = UMMA_SOFTMAX_SETS<G>;
  auto kern = decode_umma_kernel<G, S, QBUF, DT, HG, BPU, EARLY, SW>;
  const size_t smem = UmmaLayout<G, S, QBUF, HG, BPU>::bytes(a.batch);
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         DECODE_MAX_SMEM);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaError_t e = launch_pdl(kern, dim3(ctas), dim3(umma_threads<SW>()), smem, s, tmK, tmV, a);
  if (e != cudaSuccess) return e;
  // two-block units (G = 8): twelve pieces per round, in CTAs of four warps (small enough to
  // stay resident beside the split pass at that round size)
  constexpr int CR = BPU == 2 ? 12 : 4, CWN = BPU == 2 ? 4 : COMBINE_WARPS;
  return launch_combine<128, G, HG, DT, BPU, UMMA_COMBINE_RELEASE_EARLY<EARLY, BPU>, CR, CWN>(
      a, ctas, s);
}

// three stages when they fit beside the Q and P tiles, else two. G = 8 takes units of two
// blocks of 4 kv heads (N = 64: the tiles of G = 4, three stages) instead of one block of 8
// (N = 128: two stages).
template <int G, int DT, bool EARLY>
static cudaError_t launch_umma(const DecodeArgs &a, const CUtensorMap &tmK,
                               const CUtensorMap &tmV, int ctas, cudaStream_t s) {
  constexpr int HG = G == 8 ? 4 : 8, BPU = G == 8 ? 2 : 1;
  if (UmmaLayout<G, 3, 2, HG, BPU>::bytes(a.batch) <= (size_t)DECODE_MAX_SMEM)
    return launch_umma_cfg<G, 3, 2, DT, HG, BPU, EARLY>(a, tmK, tmV, ctas, s);
  if (UmmaLayout<G, 3, 1, HG, BPU>::bytes(a.batch) <= (size_t)DECODE_MAX_SMEM)
    return launch_umma_cfg<G, 3, 1, DT, HG, BPU, EARLY>(a, tmK, tmV, ctas, s);
  if (UmmaLayout<G, 2, 1, HG, BPU>::bytes(a.batch) <= (size_t)DECODE_MAX_SMEM)
    return launch_umma_cfg<G, 2, 1, DT, HG, BPU, EARLY>(a, tmK, tmV, ctas, s);
  return cudaErrorInvalidValue;
}

// every (G, dtype) the tcgen05 kernel takes, for one value of EARLY
template <bool EARLY>
cudaError_t launch_decode_umma_t(const DecodeArgs &a, const CUtensorMap &tmK,
                                 const CUtensorMap &tmV, int G, int dtype, int ctas,
                                 cudaStream_t s) {
#define KVINJ_UMMA_CASE(GG, TT) \
  if (G == GG && dtype == TT) return launch_umma<GG, TT, EARLY>(a, tmK, tmV, ctas, s);
  KVINJ_UMMA_CASE(1, 0)
  KVINJ_UMMA_CASE(2, 0)
  KVINJ_UMMA_CASE(4, 0)
  KVINJ_UMMA_CASE(8, 0)
  KVINJ_UMMA_CASE(1, 1)
  KVINJ_UMMA_CASE(2, 1)
  KVINJ_UMMA_CASE(4, 1)
  KVINJ_UMMA_CASE(8, 1)
#undef KVINJ_UMMA_CASE
  return cudaErrorInvalidValue;
}

}  // namespace kvinj
