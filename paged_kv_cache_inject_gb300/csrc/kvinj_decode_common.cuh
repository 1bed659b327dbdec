// kvinj_decode_common.cuh -- the parts of the split-K paged decode shared by
// the CUDA-core and tensor-core consumers: shared-memory layout, prologue
// (units per request, prefix sums, this CTA's range), the TMA producer warp,
// piece lookup, and the end-of-piece protocol (final outputs, or partial
// softmax states combined in-kernel by the CTA that finishes a segment last).
//
// Work unit. A physical block of the cache holds, per layer, the 16 tokens
// of every kv head contiguously ([Hkv][16][D] for K, the same for V). The
// unit of work is one block of one group of HG consecutive kv heads: HG*16
// rows of K and of V, contiguous, fetched with two TMA boxes each (16 KiB
// boxes for HG = 8, D = 128). Streaming units of 16-32 KiB reaches the HBM
// rate where 4 KiB pages of a single head do not. Consumer warp w owns kv
// head hg*HG + w of the group and every unit passes through all HG warps.
//
// Segments and pieces. The units of (request r, head group hg) form a
// segment of ceil(C_r/16) units. Units are flattened request-major and cut
// into gridDim.x equal contiguous ranges, one per CTA. A segment inside one
// CTA range is finished there; a segment cut by range boundaries leaves one
// partial softmax state per piece in the workspace, and a second, small
// kernel launched after this one on the same stream combines the pieces
// (stream order makes every partial visible to it; which pieces make up a
// segment follows from the context lengths alone). The streaming kernel thus
// needs no fence, atomic or counter, and nothing waits on another CTA.
#pragma once

#include <math.h>

#include "kvinj_device.cuh"
#include "kvinj_internal.h"

namespace kvinj {

constexpr int BLK = 16;                      // tokens per block
constexpr int DECODE_MAX_SMEM = 227 * 1024;  // opt-in dynamic shared memory per CTA

template <int D_, int G_, int HG_, int S_, int QB_ = 0>
struct DecodeLayout {
  static constexpr int D = D_, G = G_, HG = HG_, S = S_;
  static constexpr int QB = QB_;                        // q staging buffers (0 = none)
  static constexpr int EMPTY_ARRIVALS = HG;             // consumer warps free a stage
  static constexpr bool QPOS_SM = false;  // q positions copied to shared memory after pre[]
  static constexpr bool APPEND_WAIT = false;  // the producer waits for a fused append
  static constexpr int BPU = 1;               // 16-token blocks per unit
  static constexpr bool SPLIT_KV = false;     // K and V of a stage share one barrier pair
  static constexpr int VR = S;                // valid bits: one entry per stage
  static constexpr bool I8 = false;           // 16-bit cache
  static constexpr int CODE_BYTES = 0, SC_BYTES = 0, STAGE_TX = 0;
  static constexpr int off_qfull = 0, QBUF = 1;
  static constexpr int NBOX = D / 64;                   // 64-element (128-byte) column boxes
  static constexpr int BOXB = HG * BLK * 128;           // bytes of one box: HG*16 rows
  static constexpr int UNIT_BYTES = NBOX * BOXB;        // K (or V) of one unit
  static constexpr int STAGE_BYTES = 2 * UNIT_BYTES;    // K then V
  static constexpr int Q_BYTES = HG * G * D * 2;        // q rows of one head group
  static constexpr int T_BYTES = (D / 2) * 16;          // one RoPE table row
  static constexpr int off_stage = 0;                   // 1024-byte aligned
  static constexpr int off_q = S * STAGE_BYTES;         // [QB][Q_BYTES]
  static constexpr int off_t = off_q + QB * Q_BYTES;    // [QB][T_BYTES]
  static constexpr int off_bar = off_t + QB * T_BYTES;  // full[S], empty[S], qfull[QB], qempty[QB]
  static constexpr int off_valid = off_bar + (2 * S + 2 * QB) * 8;
  static constexpr int off_qinfo = off_valid + S * 4;   // [QB] q position (-1: no rotation)
  static constexpr int off_flags = off_qinfo + 16;      // [0] abort [1] last [8..40) scan
  static constexpr int off_scratch = off_flags + 256;   // per warp: p[16][G], alpha[G]
  static constexpr int SCRATCH_FLOATS = 17 * G;
  static constexpr int off_pre = off_scratch + HG * SCRATCH_FLOATS * 4;
  static size_t bytes(int batch) { return (size_t)off_pre + (size_t)(batch + 1) * 4 + 1024; }
};

__device__ __forceinline__ uint8_t *align_smem(uint8_t *p) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return reinterpret_cast<uint8_t *>((a + 1023) & ~uintptr_t(1023));
}

// byte offset, inside a unit's K (or V) half, of 16-byte chunk `chunk`
// (0 .. D/8-1) of token `tok` of the warp's head `w`: the 128-byte swizzle
// of the TMA boxes XORs the chunk index with the row index mod 8
template <int BOXB>
__device__ __forceinline__ uint32_t unit_off(int w, int chunk, int tok) {
  return (chunk >> 3) * BOXB + (w * BLK + tok) * 128 + (((chunk & 7) ^ (tok & 7)) << 4);
}

struct CtaRange {
  int b0, b1;  // this CTA's units [b0, b1) of the flattened unit sequence
  int n_eff;   // CTAs that received units
  int Ptot;    // total units
};

__device__ __forceinline__ int range_begin(int c, const CtaRange &rg) {
  return (int)((int64_t)c * rg.Ptot / rg.n_eff);
}
// the CTA whose range holds unit P
__device__ __forceinline__ int cta_of(int P, const CtaRange &rg) {
  return (int)(((int64_t)(P + 1) * rg.n_eff - 1) / rg.Ptot);
}

struct Piece {
  int r, hg;      // request, head group
  int pg0;        // first block (within the request) of this piece
  int ctx;        // context length of the request
  int lo;         // first token attended to (sliding window; 0 without one)
  int seg_start;  // flattened index of the segment's first unit
  int seg_end;    // one past its last unit
  int end;        // one past this piece's last unit (<= seg_end)
};

// largest r with pre[r] <= P (requests without units have pre[r] == pre[r+1])
__device__ __forceinline__ int find_request(const int *pre, int batch, int P) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= P) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// sliding window ("LLM Inference: KV Caching", sliding window attention): a query attends
// to the last a.window tokens of its context only (a.window == 0: to all of them); the
// first token attended to
__device__ __forceinline__ int window_lo(const DecodeArgs &a, int c) {
  return (a.window > 0 && c > a.window) ? c - a.window : 0;
}

// the piece of unit P: units of a head group are 16*BPU-token spans of the request's
// context from the one holding its first attended token
template <int BPU = 1>
__device__ __forceinline__ Piece find_piece(const DecodeArgs &a, const int *pre, int ngrp, int P,
                                            int b1) {
  Piece pc;
  pc.r = find_request(pre, a.batch, P);
  const int pages = (pre[pc.r + 1] - pre[pc.r]) / ngrp;
  const int off = P - pre[pc.r];
  pc.ctx = a.context_lens[pc.r];
  pc.lo = window_lo(a, pc.ctx);
  pc.hg = off / pages;
  pc.pg0 = off - pc.hg * pages + pc.lo / (BLK * BPU);
  pc.seg_start = pre[pc.r] + pc.hg * pages;
  pc.seg_end = pc.seg_start + pages;
  pc.end = min(b1, pc.seg_end);
  return pc;
}

// Units per request -> pre[0..batch] (exclusive prefix sums, in shared
// memory), by all NT threads of the CTA. `units(r, c)` gives request r's units
// from its context length c (and may act on it); `scratch` holds NT/32 ints.
template <int NT, class F>
__device__ void unit_prefix(const DecodeArgs &a, int *pre, int *scratch, F units) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NWARP = NT / 32;
  int carry = 0;
  for (int base = 0; base < a.batch; base += NT) {
    const int r = base + tid;
    const int v = r < a.batch ? units(r, __ldg(a.context_lens + r)) : 0;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = lane < NWARP ? scratch[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < NWARP) scratch[lane] = w;
    }
    __syncthreads();
    const int incl = x + (warp > 0 ? scratch[warp - 1] : 0);
    if (r < a.batch) pre[r + 1] = carry + incl;
    carry += scratch[NWARP - 1];
    __syncthreads();
  }
  if (tid == 0) pre[0] = 0;
  __syncthreads();
}

// 16-token blocks of a valid context (0 for an invalid one)
__device__ __forceinline__ int context_pages(const DecodeArgs &a, int c) {
  return (c > 0 && c <= a.max_blocks * BLK) ? (c + BLK - 1) / BLK : 0;
}
// work units of one head group of a request whose context is c tokens long
template <int BPU>
__device__ __forceinline__ int context_units(const DecodeArgs &a, int c) {
  const int u = (context_pages(a, c) + BPU - 1) / BPU;
  return u > 0 ? u - window_lo(a, c) / (BLK * BPU) : 0;  // from the first attended token's
}

// The wait for the kernel ahead of this one on the stream (launched as its
// programmatic dependent), then the release of this kernel's own dependent
// (the combine pass, which waits for this grid's completion). Every thread
// that reads an input another kernel may produce, or writes anything, runs
// this first. Releasing only after the wait keeps the chain that early reads
// rely on: once a kernel after this one starts, everything enqueued before
// this kernel has completed.
__device__ __forceinline__ void decode_dependency_wait() {
  griddep_wait();
  griddep_launch_dependents();
}

// CTA 0, after the dependency wait: a zero output and KVINJ_ST_BAD_CTX for
// every request whose context length is invalid (pre[r + 1] == pre[r]);
// threads t0, t0 + nt, ... of the CTA take the requests in turn.
template <int D>
__device__ void zero_invalid_outputs(const DecodeArgs &a, const int *pre, int t0, int nt) {
  if (blockIdx.x != 0) return;
  for (int r = t0; r < a.batch; r += nt) {
    if (pre[r + 1] != pre[r]) continue;
    uint4 *o = reinterpret_cast<uint4 *>(a.out + (int64_t)r * a.Hq * D);
    for (int i = 0; i < a.Hq * D / 8; ++i) o[i] = make_uint4(0, 0, 0, 0);
    report(a.status, KVINJ_ST_BAD_CTX);
  }
}

// Units per request -> prefix sums pre[0..batch], this CTA's range, barrier
// set-up. Returns false when this CTA has no units.
//
// EARLY = false (every input may come from the kernel before this one): all
// threads wait for that kernel first, and CTA 0 zeroes the output of requests
// whose context length is invalid. EARLY = true (a call with
// KVINJ_DECODE_KV_READY): the context lengths, q positions and block tables
// were written before the previous decode call on the stream, so they are read
// here before the wait; the caller then runs decode_dependency_wait() in each
// thread before any other read or write (the producer after it has issued the
// first stages) and zero_invalid_outputs() from CTA 0. The two are separate
// instantiations: the waiting one carries none of the early code.
template <class Lay, int NT, bool EARLY = false>
__device__ bool decode_prologue(const DecodeArgs &a, uint8_t *sm, CtaRange &rg) {
  if constexpr (!EARLY) decode_dependency_wait();
  int *pre = reinterpret_cast<int *>(sm + Lay::off_pre);
  int *flags = reinterpret_cast<int *>(sm + Lay::off_flags);
  const int tid = threadIdx.x;
  const int ngrp = a.Hkv / Lay::HG;
  unit_prefix<NT>(a, pre, flags + 8, [&](int r, int c) {
    if constexpr (Lay::QPOS_SM) pre[a.batch + 1 + r] = a.q_pos ? __ldg(a.q_pos + r) : -1;
    const int v = context_units<Lay::BPU>(a, c) * ngrp;
    if (!EARLY && v == 0 && blockIdx.x == 0) {
      uint4 *o = reinterpret_cast<uint4 *>(a.out + (int64_t)r * a.Hq * Lay::D);
      for (int i = 0; i < a.Hq * Lay::D / 8; ++i) o[i] = make_uint4(0, 0, 0, 0);
      report(a.status, KVINJ_ST_BAD_CTX);
    }
    return v;
  });
  rg.Ptot = pre[a.batch];
  rg.n_eff = min((int)gridDim.x, rg.Ptot);
  if ((int)blockIdx.x >= rg.n_eff) return false;
  rg.b0 = range_begin(blockIdx.x, rg);
  rg.b1 = range_begin(blockIdx.x + 1, rg);
  if (tid == 0) {
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + Lay::off_bar);
    for (int s = 0; s < Lay::S; ++s) {
      mbar_init(full + s, 1);                 // the producer's arrive + the TMA bytes
      mbar_init(full + Lay::S + s, Lay::EMPTY_ARRIVALS);  // the consumers' releases
    }
    for (int b = 0; b < Lay::QB; ++b) {
      mbar_init(full + 2 * Lay::S + b, 1);
      mbar_init(full + 2 * Lay::S + Lay::QB + b, Lay::HG);
    }
    if constexpr (Lay::SPLIT_KV) {
      static_assert(Lay::QB == 0, "split stages: the producer stages no query rows");
      for (int s = 0; s < Lay::S; ++s) {
        mbar_init(full + 2 * Lay::S + s, 1);                    // V landed
        mbar_init(full + 3 * Lay::S + s, Lay::EMPTY_ARRIVALS);  // V released
      }
    }
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
  }
  __syncthreads();
  return true;
}

// Producer warp: stream this CTA's units into the stage ring. Block-table
// entries are fetched one per lane, a batch of 32 ahead of their use; lane 0
// issues the copies (NBOX boxes of K and NBOX boxes of V per unit). With
// EARLY, the first stages are issued before the dependency wait (see
// decode_prologue).
template <class Lay, bool EARLY = false>
__device__ void decode_producer(const DecodeArgs &a, const CUtensorMap &tmK,
                                const CUtensorMap &tmV, uint8_t *sm, const CtaRange &rg,
                                int lane) {
  constexpr int S = Lay::S, NBOX = Lay::NBOX, HG = Lay::HG;
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + Lay::off_bar);
  uint64_t *empty = full + S;
  // split stages: full/empty cover the K half, fullV/emptyV the V half
  uint64_t *fullV = full + 2 * S, *emptyV = full + 3 * S;
  volatile int *flags = reinterpret_cast<volatile int *>(sm + Lay::off_flags);
  int *valid = reinterpret_cast<int *>(sm + Lay::off_valid);
  const int *pre = reinterpret_cast<const int *>(sm + Lay::off_pre);
  uint8_t *stages = sm + Lay::off_stage;
  const int ngrp = a.Hkv / HG;
  if (lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  const int n = rg.b1 - rg.b0;
  // lookup of unit g0 + lane: block-table entry (and, when q is staged, the
  // request's q position); the loads are consumed one batch later
  // with two blocks per unit, blk2 is the second one (-2: the context ends before it)
  auto start_lookup = [&](int gi, int &blk, int &blk2, int &hg, int &rq, int &first, int &qp,
                          int &ap) {
    blk = -1;
    blk2 = -2;
    hg = 0;
    rq = 0;
    first = 0;
    qp = -1;
    ap = 0;
    if (gi < n) {
      const int P = rg.b0 + gi;
      const int r = find_request(pre, a.batch, P);
      const int pages = (pre[r + 1] - pre[r]) / ngrp;
      const int off = P - pre[r];
      hg = off / pages;
      const int c = __ldg(a.context_lens + r);
      const int fp = window_lo(a, c) / BLK;  // first page holding an attended token
      const int pgr = off - hg * pages;
      const int pg = pgr + fp / Lay::BPU;    // unit index within the request
      rq = r;
      first = (gi == 0 || pgr == 0) ? 1 : 0;  // first unit of a piece
      // (a two-block unit that starts one page before the window loads the window's first
      // block in both halves: the page before holds no attended token and is not read)
      blk = a.block_tables[(int64_t)r * a.max_blocks + max(pg * Lay::BPU, fp)];
      if constexpr (Lay::BPU == 2) {
        if (pg * 2 + 1 < context_pages(a, c))
          blk2 = a.block_tables[(int64_t)r * a.max_blocks + pg * 2 + 1];
      }
      if (Lay::QB && first && a.rope) qp = a.q_pos[r];
      if constexpr (Lay::APPEND_WAIT) {
        // this unit holds the token appended by this call (written by the query warps)
        const int qa = pre[a.batch + 1 + r];
        ap = (a.k_new && qa >= 0 && (!a.rope || qa < a.max_pos) && qa / BLK / Lay::BPU == pg)
                 ? 1 : 0;
      }
    }
  };
  int blk, blk2, hg, rq, first, qp, ap;
  start_lookup(lane, blk, blk2, hg, rq, first, qp, ap);
  int pieces = 0, cur_piece = -1;
  int kiss = 0, viss = 0;  // (lane 0) units whose K (V) copies were issued
  bool aborted = false;
  // early: the first stages are issued before the dependency wait, up to the first
  // unit that holds a fused append (its rows are written after the wait); status
  // bits found before the wait are reported after it
  bool waited = !EARLY;
  int pending = 0;
  for (int g0 = 0; g0 < n && !aborted; g0 += 32) {
    // valid bits: block 0 (and, with two blocks per unit, block 1) in the cache
    const int ok0 = (blk >= 0 && blk < a.num_blocks) ? 1 : 0;
    const int ok1 = (Lay::BPU == 2 && blk2 >= 0 && blk2 < a.num_blocks) ? 2 : 0;
    if (g0 + lane < n && (!ok0 || (blk2 != -2 && Lay::BPU == 2 && !ok1))) {
      if constexpr (EARLY) pending |= KVINJ_ST_BAD_BLOCK;
      else report(a.status, KVINJ_ST_BAD_BLOCK);
    }
    if constexpr (EARLY) {
      if (waited && pending) {
        report(a.status, pending);
        pending = 0;
      }
    }
    const int ok = ok0 | ok1;
    const int row0 = (int)((((int64_t)a.layer * a.num_blocks + (ok0 ? blk : 0)) * a.Hkv +
                            (int64_t)hg * HG) * BLK);
    const int row1 = (int)((((int64_t)a.layer * a.num_blocks + (ok1 ? blk2 : (ok0 ? blk : 0))) *
                                a.Hkv + (int64_t)hg * HG) * BLK);
    const int qpos_ok = (qp >= 0 && qp < a.max_pos) ? qp : -1;
    // (the kernels that stage q in the producer run without EARLY)
    if (Lay::QB && first && a.rope && qpos_ok < 0 && g0 + lane < n) report(a.status, KVINJ_ST_BAD_POS);
    const int qrow0 = rq * a.Hq + hg * HG * Lay::G;  // first q row of the head group
    int nblk, nblk2, nhg, nrq, nfirst, nqp, nap;
    start_lookup(g0 + 32 + lane, nblk, nblk2, nhg, nrq, nfirst, nqp, nap);
    const int cnt = min(32, n - g0);
    for (int i = 0; i < cnt; ++i) {
      const int r0 = __shfl_sync(0xffffffffu, row0, i);
      const int r1 = __shfl_sync(0xffffffffu, row1, i);
      const int oki = __shfl_sync(0xffffffffu, ok, i);
      const int fi = __shfl_sync(0xffffffffu, first, i);
      const int qri = __shfl_sync(0xffffffffu, qrow0, i);
      const int qpi = __shfl_sync(0xffffffffu, qpos_ok, i);
      const int api = __shfl_sync(0xffffffffu, ap, i);
      const int gi = g0 + i, st = gi % S;
      int go = 1;
      if (fi) ++cur_piece;
      if constexpr (EARLY) {
        if (!waited && (gi >= S || api)) {
          // the stages are all issued (the next needs a consumer), or this unit holds
          // the fused append: wait for the kernel ahead, then report what was found
          decode_dependency_wait();
          waited = true;
          if (pending) report(a.status, pending);
          pending = 0;
        }
      }
      if (lane == 0) {
        if constexpr (Lay::APPEND_WAIT) {
          // the piece's query warps write the appended token before its block is read
          uint64_t *qf = reinterpret_cast<uint64_t *>(sm + Lay::off_qfull) + cur_piece % Lay::QBUF;
          if (api && !flags[0] &&
              !mbar_wait_bounded(qf, (uint32_t)(cur_piece / Lay::QBUF) & 1u)) {
            report(a.status, KVINJ_ST_TIMEOUT);
            flags[0] = 1;
          }
        }
        if (Lay::QB && fi && !flags[0]) {
          // q rows (and RoPE row) of the piece starting here
          constexpr int QBD = Lay::QB ? Lay::QB : 1;
          const int qb = pieces % QBD;
          uint64_t *qfull = full + 2 * S + qb, *qempty = full + 2 * S + Lay::QB + qb;
          if (pieces >= Lay::QB &&
              !mbar_wait_bounded(qempty, (uint32_t)(pieces / QBD - 1) & 1u)) {
            report(a.status, KVINJ_ST_TIMEOUT);
            flags[0] = 1;
          } else {
            int *qinfo = reinterpret_cast<int *>(sm + Lay::off_qinfo);
            qinfo[qb] = a.rope ? qpi : -2;
            const bool trow = a.rope && qpi >= 0;
            mbar_arrive_expect_tx(qfull, Lay::Q_BYTES + (trow ? Lay::T_BYTES : 0));
            bulk_load(sm + Lay::off_q + qb * Lay::Q_BYTES, a.q + (int64_t)qri * Lay::D,
                      Lay::Q_BYTES, qfull);
            if (trow)
              bulk_load(sm + Lay::off_t + qb * Lay::T_BYTES, a.rope + (int64_t)qpi * (Lay::D / 2),
                        Lay::T_BYTES, qfull);
          }
          ++pieces;
        }
        if (flags[0]) {
          go = 0;
        } else if (gi >= S && !mbar_wait_bounded(empty + st, (uint32_t)(gi / S - 1) & 1u)) {
          report(a.status, KVINJ_ST_TIMEOUT);
          flags[0] = 1;
          go = 0;
        }
        if (go) {
          valid[Lay::SPLIT_KV ? gi % Lay::VR : st] = oki;
          uint8_t *kd = stages + st * Lay::STAGE_BYTES;
          // the boxes of one tensor (K or V) of this unit into dst, counted on bar
          auto load_half = [&](uint8_t *dst, const CUtensorMap *tm, uint64_t *bar) {
            if constexpr (Lay::BPU == 1) {
#pragma unroll
              for (int b = 0; b < NBOX; ++b) tma_load_2d(dst + b * Lay::BOXB, tm, 64 * b, r0, bar);
            } else {
              // 16-row boxes (one head of one block) placed in (head, block, token) order
#pragma unroll
              for (int b = 0; b < NBOX; ++b)
#pragma unroll
                for (int h = 0; h < HG; ++h)
#pragma unroll
                  for (int j = 0; j < 2; ++j)
                    tma_load_2d(dst + b * Lay::BOXB + (h * 2 + j) * BLK * 128, tm, 64 * b,
                                (j ? r1 : r0) + h * BLK, bar);
            }
          };
          if constexpr (Lay::I8) {
            // int8 cache: the K and V code tiles (the 128-byte swizzle, like the 16-bit
            // tiles' column blocks) and the rows' K and V scales, all on one barrier
            uint8_t *sc = kd + 2 * Lay::CODE_BYTES;
            mbar_arrive_expect_tx(full + st, Lay::STAGE_TX);
            if constexpr (Lay::BPU == 1) {
              tma_load_2d(kd, &tmK, 0, r0, full + st);
              tma_load_2d(kd + Lay::CODE_BYTES, &tmV, 0, r0, full + st);
              bulk_load(sc, a.k_scale + r0, Lay::SC_BYTES, full + st);
              bulk_load(sc + Lay::SC_BYTES, a.v_scale + r0, Lay::SC_BYTES, full + st);
            } else {
              // rows in (head, block, token) order, one 16-row box per (head, block); the
              // scales of block j are copied as [j][head][token]
#pragma unroll
              for (int h = 0; h < HG; ++h)
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                  tma_load_2d(kd + (h * 2 + j) * BLK * 128, &tmK, 0, (j ? r1 : r0) + h * BLK,
                              full + st);
                  tma_load_2d(kd + Lay::CODE_BYTES + (h * 2 + j) * BLK * 128, &tmV, 0,
                              (j ? r1 : r0) + h * BLK, full + st);
                }
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                bulk_load(sc + j * (Lay::SC_BYTES / 2), a.k_scale + (j ? r1 : r0),
                          Lay::SC_BYTES / 2, full + st);
                bulk_load(sc + Lay::SC_BYTES + j * (Lay::SC_BYTES / 2), a.v_scale + (j ? r1 : r0),
                          Lay::SC_BYTES / 2, full + st);
              }
            }
            kiss = viss = gi + 1;
          } else if constexpr (Lay::SPLIT_KV) {
            // K is released once its QK is done, V once its PV is: K runs ahead of V
            mbar_arrive_expect_tx(full + st, Lay::UNIT_BYTES);
            load_half(kd, &tmK, full + st);
            kiss = gi + 1;
            if (gi >= S && !mbar_wait_bounded(emptyV + st, (uint32_t)(gi / S - 1) & 1u)) {
              report(a.status, KVINJ_ST_TIMEOUT);
              flags[0] = 1;
              go = 0;
            } else {
              mbar_arrive_expect_tx(fullV + st, Lay::UNIT_BYTES);
              load_half(kd + Lay::UNIT_BYTES, &tmV, fullV + st);
              viss = gi + 1;
            }
          } else {
            mbar_arrive_expect_tx(full + st, Lay::STAGE_BYTES);
            load_half(kd, &tmK, full + st);
            load_half(kd + Lay::UNIT_BYTES, &tmV, full + st);
            kiss = viss = gi + 1;
          }
        }
      }
      go = __shfl_sync(0xffffffffu, go, 0);
      if (!go) {
        aborted = true;
        break;
      }
    }
    blk = nblk;
    blk2 = nblk2;
    hg = nhg;
    rq = nrq;
    first = nfirst;
    qp = nqp;
    ap = nap;
  }
  if constexpr (EARLY) {
    if (!waited) {
      // fewer units than stages, none with an append: the wait still precedes the exit
      decode_dependency_wait();
      if (pending) report(a.status, pending);
    }
  }
  if (aborted && lane == 0) {
    // let the copies already in flight land before the CTA can exit
    for (int gi = max(0, kiss - S); gi < kiss; ++gi)
      mbar_wait_bounded(full + gi % S, (uint32_t)(gi / S) & 1u, 100000000ull);
    if constexpr (Lay::SPLIT_KV)
      for (int gi = max(0, viss - S); gi < viss; ++gi)
        mbar_wait_bounded(fullV + gi % S, (uint32_t)(gi / S) & 1u, 100000000ull);
    for (int k = max(0, pieces - Lay::QB); k < pieces; ++k)
      mbar_wait_bounded(full + 2 * S + k % (Lay::QB ? Lay::QB : 1), (uint32_t)(k / (Lay::QB ? Lay::QB : 1)) & 1u,
                        100000000ull);
  }
}

// wait for unit gi's stage; false (and the abort flag) when the wait gave up
__device__ __forceinline__ bool consumer_wait(const DecodeArgs &a, uint64_t *full,
                                              volatile int *flags, int gi, int S) {
  const bool ok = !flags[0] && mbar_wait_bounded(full + gi % S, (uint32_t)(gi / S) & 1u);
  if (!ok) {
    if (!flags[0]) report(a.status, KVINJ_ST_TIMEOUT);
    flags[0] = 1;
  }
  return ok;
}

template <int DT>
__device__ __forceinline__ uint16_t to16(float x) {
  if constexpr (DT == 0) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  else return __half_as_ushort(__float2half_rn(x));
}

// floats of one head's partial state in a workspace slot: m[G], l[G], acc[G][D]
__host__ __device__ constexpr int partial_floats(int G, int D) { return G * (D + 2); }

// The partial slot of CTA c for the segment starting at unit seg_start:
// 2c for the first segment in c's range, 2c + 1 for its last one.
__device__ __forceinline__ float *partial_slot(const DecodeArgs &a, int c, int seg_start,
                                               const CtaRange &rg, int slot_floats) {
  return a.partials + (size_t)(2 * c + (seg_start <= range_begin(c, rg) ? 0 : 1)) * slot_floats;
}

// Combine the partial states of all pieces of a segment into output rows
// (row = query head g of kv head w of the group), one warp per NR rows, lane l
// owning dimensions [l*D/32, (l+1)*D/32) of each. Pieces go in rounds of R
// (a segment over a few CTAs takes one or two); a round issues every load it needs -- each
// row's and piece's m and l (the same address in all lanes) and the lane's
// slice of the accumulator -- before using any of them, so a segment costs
// one dependent round trip after the descriptor.
template <int D, int G, int HG, int DT, int NR, int R = 4>
__device__ void combine_rows(const DecodeArgs &a, const CtaRange &rg, const Piece &pc,
                             const int (&rows)[NR], int lane) {
  constexpr int PF = partial_floats(G, D), SLOT = HG * PF, DPL = D / 32;
  const int cf = cta_of(pc.seg_start, rg), cl = cta_of(pc.seg_end - 1, rg);
  const int npc = cl - cf + 1;
  float A[NR][DPL], M[NR], Ls[NR];
#pragma unroll
  for (int k = 0; k < NR; ++k) {
    M[k] = -INFINITY;
    Ls[k] = 0.f;
#pragma unroll
    for (int e = 0; e < DPL; ++e) A[k][e] = 0.f;
  }
  for (int c0 = 0; c0 < npc; c0 += R) {
    const int cnt = min(R, npc - c0);
    float m[NR][R], l[NR][R], v[NR][R][DPL];
#pragma unroll
    for (int u = 0; u < R; ++u) {
      const float *slot = partial_slot(a, cf + c0 + min(u, cnt - 1), pc.seg_start, rg, SLOT);
#pragma unroll
      for (int k = 0; k < NR; ++k) {
        const int w = rows[k] / G, g = rows[k] % G;
        const float *p = slot + w * PF;
        m[k][u] = __ldcg(p + g);
        l[k][u] = __ldcg(p + G + g);
#pragma unroll
        for (int e = 0; e < DPL; ++e) v[k][u][e] = __ldcg(p + 2 * G + g * D + lane * DPL + e);
      }
    }
#pragma unroll
    for (int k = 0; k < NR; ++k) {
      float Mr = -INFINITY;
#pragma unroll
      for (int u = 0; u < R; ++u)
        if (u < cnt) Mr = fmaxf(Mr, m[k][u]);
      const float Mn = fmaxf(M[k], Mr);
      if (Mn == -INFINITY) continue;  // nothing but empty pieces so far
      const float rescale = (M[k] == -INFINITY) ? 0.f : exp2f(M[k] - Mn);
#pragma unroll
      for (int e = 0; e < DPL; ++e) A[k][e] *= rescale;
      Ls[k] *= rescale;
      M[k] = Mn;
#pragma unroll
      for (int u = 0; u < R; ++u) {
        const float f = (u < cnt && m[k][u] != -INFINITY) ? exp2f(m[k][u] - Mn) : 0.f;
        Ls[k] = __fmaf_rn(l[k][u], f, Ls[k]);
#pragma unroll
        for (int e = 0; e < DPL; ++e) A[k][e] = __fmaf_rn(v[k][u][e], f, A[k][e]);
      }
    }
  }
#pragma unroll
  for (int k = 0; k < NR; ++k) {
    const int w = rows[k] / G, g = rows[k] % G;
    const float inv = Ls[k] > 0.f ? 1.f / Ls[k] : 0.f;
    const int h = pc.hg * HG + w;
    uint16_t *orow = a.out + ((int64_t)pc.r * a.Hq + (int64_t)h * G + g) * D + lane * DPL;
#pragma unroll
    for (int e = 0; e < DPL; e += 2)
      *reinterpret_cast<uint32_t *>(orow + e) = pack2<DT>(A[k][e] * inv, A[k][e + 1] * inv);
  }
}

// The combine pass: grid (segments, ceil(HG*G / CW)), CW warps per CTA, one warp
// per output row: CTA (s, y) takes segment s = (request, head group) and, if the
// split-K ranges cut it, combines its rows CW*y .. CW*y + CW - 1, R pieces' loads
// in flight per round. By default R = 4 and CW = 8; with two-block units (G = 8),
// whose segments span about twice as many ranges, R = 12 -- in CTAs of four warps
// after the 16-bit split pass (so that they stay resident beside it), of eight
// after the int8 decode (whose 512-thread CTAs leave no room beside them anyway).
// Whether and where a segment was cut follows from the context lengths alone,
// which the split-K pass read after its own dependency wait (before it let this
// grid start): that is worked out, and the segment's partial-state lines are
// prefetched, before this grid waits for the split-K pass. A grid of segments (a
// few per SM at serving batch sizes) leaves its CTAs resident beside the decode
// CTAs, so only the loads of the partial states follow the wait. (Measured at
// batch 32, split-K pass + combine per layer: one CTA per segment with two rows
// per warp 50.5 us; one warp per row over a grid of decode CTAs 42.9 us; one warp
// per row over this grid of segments 41.2 us.)
//
// RELEASE_EARLY: the kernel after this one is released at this pass's start
// instead of after its dependency wait. That kernel still waits for this grid's
// completion before it reads anything this pass writes; what it gains is that
// its CTAs may be scheduled (and a decode call with early page reads may start
// streaming) as soon as the split-K pass's CTAs leave their SMs. Everything
// enqueued before the split-K pass has completed by then (the split-K pass
// released this grid only after its own dependency wait).
constexpr int COMBINE_WARPS = 8;
template <int D, int G, int HG, int DT, int BPU, bool RELEASE_EARLY = false, int R = 4,
          int CW = COMBINE_WARPS>
__global__ void __launch_bounds__(CW * 32) decode_combine_kernel(DecodeArgs a) {
  extern __shared__ int comb_sm[];  // scratch[CW], pre[batch + 1]
  if constexpr (RELEASE_EARLY) griddep_launch_dependents();
  int *pre = comb_sm + CW;
  const int ngrp = a.Hkv / HG;
  unit_prefix<CW * 32>(a, pre, comb_sm,
                                  [&](int, int c) { return context_units<BPU>(a, c) * ngrp; });
  CtaRange rg;
  rg.Ptot = pre[a.batch];
  rg.n_eff = min(a.ctas, rg.Ptot);
  Piece pc;
  pc.r = blockIdx.x / ngrp;
  pc.hg = blockIdx.x % ngrp;
  const int pages = (pre[pc.r + 1] - pre[pc.r]) / ngrp;
  pc.seg_start = pre[pc.r] + pc.hg * pages;
  pc.seg_end = pc.seg_start + pages;
  constexpr int ROWS = HG * G, PF = partial_floats(G, D), SLOT = HG * PF;
  const int row = blockIdx.y * CW + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int cf = pages > 0 ? cta_of(pc.seg_start, rg) : 0;
  const int cl = pages > 0 ? cta_of(pc.seg_end - 1, rg) : 0;
  if (cf == cl) return;  // finished inside one split-K range (or empty)
  if (row < ROWS) {
    // warm L2 and the address translations for this row's partial states while the
    // split-K pass still runs (a hint: the lines it writes later are current in L2)
    const int w = row / G, g = row % G;
    const int j = lane & 7;  // per piece: m/l, then the D-float slice (up to 5 lines)
    if (j <= 5) {
      for (int c = cf + (lane >> 3); c <= cl; c += 4) {
        const float *p = partial_slot(a, c, pc.seg_start, rg, SLOT) + w * PF;
        prefetch_l2(j == 0 ? p + g : p + 2 * G + g * D + min((j - 1) * 32, D - 1));
      }
    }
  }
  griddep_wait();  // the split-K pass complete, its partial states visible
  if constexpr (!RELEASE_EARLY) griddep_launch_dependents();
  if (row >= ROWS) return;
  const int rows[1] = {row};
  combine_rows<D, G, HG, DT, 1, R>(a, rg, pc, rows, lane);
}

// Launch `kern` on stream s as a programmatic dependent of the kernel launched
// just before it: its CTAs may be scheduled while that kernel still runs
// (once that kernel's CTAs have all called griddep_launch_dependents), and
// they wait for its completion in griddep_wait before reading anything.
template <class... P, class... A>
cudaError_t launch_pdl(void (*kern)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       A &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<A &&>(args)...);
}

// the combine pass for a split-K grid of `ctas` CTAs
template <int D, int G, int HG, int DT, int BPU = 1, bool RELEASE_EARLY = false, int R = 4,
          int CW = COMBINE_WARPS>
cudaError_t launch_combine(const DecodeArgs &a, int ctas, cudaStream_t s) {
  DecodeArgs c = a;
  c.ctas = ctas;
  return launch_pdl(decode_combine_kernel<D, G, HG, DT, BPU, RELEASE_EARLY, R, CW>,
                    dim3(a.batch * (a.Hkv / HG), (HG * G + CW - 1) / CW),
                    dim3(CW * 32), (size_t)(CW + a.batch + 1) * sizeof(int),
                    s, c);
}

}  // namespace kvinj
