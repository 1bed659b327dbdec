// kvinj_decode_common.cuh -- parts of the split-K paged decode shared by the
// CUDA-core and tensor-core consumers: shared-memory layout, the prologue
// (pages per request, prefix sums, this CTA's range), the TMA producer warp,
// the query load/rotation, and the end-of-piece merge with the in-kernel
// combine of pieces that several CTAs produced.
#pragma once

#include <math.h>

#include "kvinj_device.cuh"
#include "kvinj_internal.h"

namespace kvinj {

constexpr int BLK = 16;                  // tokens per page (block size)
constexpr int DECODE_MAX_SMEM = 227 * 1024;  // opt-in dynamic shared memory per CTA
constexpr int BOX_BYTES = BLK * 64 * 2;  // one TMA box: 16 rows x 64 elements

template <int D_, int G_, int NW_, int S_>
struct DecodeLayout {
  static constexpr int D = D_, G = G_, NW = NW_, S = S_;
  static constexpr int NBOX = D / 64;
  static constexpr int PAGE_BYTES = NBOX * BOX_BYTES;  // K (or V) page of one head
  static constexpr int STAGE_BYTES = 2 * PAGE_BYTES;   // K page then V page
  static constexpr int off_stage = 0;                  // 1024-byte aligned
  static constexpr int off_bar = S * STAGE_BYTES;      // full[S], empty[S]
  static constexpr int off_valid = off_bar + 2 * S * 8;
  static constexpr int off_flags = off_valid + S * 4;  // [0] abort [1] last [8..40) scan
  static constexpr int off_p = off_flags + 256;        // float [NW][16][G]
  static constexpr int off_alpha = off_p + NW * 16 * G * 4;
  static constexpr int off_mm = off_alpha + NW * G * 4;  // float [NW][G]
  static constexpr int off_ml = off_mm + NW * G * 4;     // float [NW][G]
  static constexpr int off_macc = off_ml + NW * G * 4;   // float [NW][G][D]
  static constexpr int off_pre = off_macc + NW * G * D * 4;
  static size_t bytes(int batch) { return (size_t)off_pre + (size_t)(batch + 1) * 4 + 1024; }
};

__device__ __forceinline__ uint8_t *align_smem(uint8_t *p) {
  uintptr_t a = reinterpret_cast<uintptr_t>(p);
  return reinterpret_cast<uint8_t *>((a + 1023) & ~uintptr_t(1023));
}

struct CtaRange {
  int b0, b1;   // this CTA's pages [b0, b1) of the flattened page sequence
  int n_eff;    // CTAs that received pages
  int Ptot;     // total pages
};

__device__ __forceinline__ int range_begin(int c, const CtaRange &rg) {
  return (int)((int64_t)c * rg.Ptot / rg.n_eff);
}
// the CTA whose range holds page P
__device__ __forceinline__ int cta_of(int P, const CtaRange &rg) {
  return (int)(((int64_t)(P + 1) * rg.n_eff - 1) / rg.Ptot);
}

struct Piece {
  int r, h;        // request, kv head
  int pg0;         // first page (within the request) of this piece
  int ctx;         // context length of the request
  int seg_start;   // flattened index of the segment's first page
  int seg_end;     // one past its last page
  int end;         // one past this piece's last page (<= seg_end)
};

// largest r with pre[r] <= P (requests without pages have pre[r] == pre[r+1])
__device__ __forceinline__ int find_request(const int *pre, int batch, int P) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= P) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ Piece find_piece(const DecodeArgs &a, const int *pre, int P, int b1) {
  Piece pc;
  pc.r = find_request(pre, a.batch, P);
  const int pages = (pre[pc.r + 1] - pre[pc.r]) / a.Hkv;
  const int off = P - pre[pc.r];
  pc.h = off / pages;
  pc.pg0 = off - pc.h * pages;
  pc.seg_start = pre[pc.r] + pc.h * pages;
  pc.seg_end = pc.seg_start + pages;
  pc.end = min(b1, pc.seg_end);
  pc.ctx = a.context_lens[pc.r];
  return pc;
}

__device__ __forceinline__ int valid_pages(const DecodeArgs &a, int r) {
  const int c = a.context_lens[r];
  return (c > 0 && c <= a.max_blocks * BLK) ? (c + BLK - 1) / BLK : 0;
}

// Pages per request -> prefix sums pre[0..batch] (in pages x Hkv), this CTA's
// range, barrier set-up. CTA 0 also zeroes the output of requests whose
// context length is invalid. Returns false when this CTA has no pages.
template <class Lay, int NT>
__device__ bool decode_prologue(const DecodeArgs &a, uint8_t *sm, CtaRange &rg) {
  int *pre = reinterpret_cast<int *>(sm + Lay::off_pre);
  int *flags = reinterpret_cast<int *>(sm + Lay::off_flags);
  int *ws = flags + 8;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NWARP = NT / 32;
  int carry = 0;
  for (int base = 0; base < a.batch; base += NT) {
    const int r = base + tid;
    int v = 0;
    if (r < a.batch) {
      v = valid_pages(a, r) * a.Hkv;
      if (v == 0 && blockIdx.x == 0) {
        uint4 *o = reinterpret_cast<uint4 *>(a.out + (int64_t)r * a.Hq * Lay::D);
        for (int i = 0; i < a.Hq * Lay::D / 8; ++i) o[i] = make_uint4(0, 0, 0, 0);
        report(a.status, KVINJ_ST_BAD_CTX);
      }
    }
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) ws[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = lane < NWARP ? ws[lane] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      if (lane < NWARP) ws[lane] = w;
    }
    __syncthreads();
    const int incl = x + (warp > 0 ? ws[warp - 1] : 0);
    if (r < a.batch) pre[r + 1] = carry + incl;
    carry += ws[NWARP - 1];
    __syncthreads();
  }
  if (tid == 0) pre[0] = 0;
  __syncthreads();
  rg.Ptot = pre[a.batch];
  rg.n_eff = min((int)gridDim.x, rg.Ptot);
  if ((int)blockIdx.x >= rg.n_eff) return false;
  rg.b0 = range_begin(blockIdx.x, rg);
  rg.b1 = range_begin(blockIdx.x + 1, rg);
  if (tid == 0) {
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + Lay::off_bar);
    for (int s = 0; s < Lay::S; ++s) {
      mbar_init(full + s, 1);
      mbar_init(full + Lay::S + s, 1);
    }
    flags[0] = 0;
    flags[1] = 0;
    fence_mbar_init();
  }
  __syncthreads();
  return true;
}

// Producer warp: stream this CTA's pages (K page then V page of one head)
// into the stage ring. Block-table entries are fetched one per lane, a batch
// of 32 ahead of their use. Lane 0 issues the TMA copies.
template <class Lay>
__device__ void decode_producer(const DecodeArgs &a, const CUtensorMap &tmK,
                                const CUtensorMap &tmV, uint8_t *sm, const CtaRange &rg,
                                int lane) {
  constexpr int S = Lay::S, NBOX = Lay::NBOX;
  uint64_t *full = reinterpret_cast<uint64_t *>(sm + Lay::off_bar);
  uint64_t *empty = full + S;
  volatile int *flags = reinterpret_cast<volatile int *>(sm + Lay::off_flags);
  int *valid = reinterpret_cast<int *>(sm + Lay::off_valid);
  const int *pre = reinterpret_cast<const int *>(sm + Lay::off_pre);
  uint8_t *stages = sm + Lay::off_stage;
  if (lane == 0) {
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  const int n = rg.b1 - rg.b0;
  // lookup of page g0 + lane: the block-table load is issued here and
  // consumed one batch later
  auto start_lookup = [&](int gi, int &blk, int &h) {
    blk = -1;
    h = 0;
    if (gi < n) {
      const int P = rg.b0 + gi;
      const int r = find_request(pre, a.batch, P);
      const int pages = (pre[r + 1] - pre[r]) / a.Hkv;
      const int off = P - pre[r];
      h = off / pages;
      const int pg = off - h * pages;
      blk = a.block_tables[(int64_t)r * a.max_blocks + pg];
    }
  };
  int blk, h;
  start_lookup(lane, blk, h);
  int issued = 0;
  bool aborted = false;
  for (int g0 = 0; g0 < n && !aborted; g0 += 32) {
    int ok = (blk >= 0 && blk < a.num_blocks) ? 1 : 0;
    if (!ok && g0 + lane < n) report(a.status, KVINJ_ST_BAD_BLOCK);
    const int row0 =
        (int)((((int64_t)a.layer * a.num_blocks + (ok ? blk : 0)) * a.Hkv + h) * BLK);
    int nblk, nh;
    start_lookup(g0 + 32 + lane, nblk, nh);
    const int cnt = min(32, n - g0);
    for (int i = 0; i < cnt; ++i) {
      const int r0 = __shfl_sync(0xffffffffu, row0, i);
      const int oki = __shfl_sync(0xffffffffu, ok, i);
      const int gi = g0 + i, st = gi % S;
      int go = 1;
      if (lane == 0) {
        if (flags[0]) {
          go = 0;
        } else if (gi >= S && !mbar_wait_bounded(empty + st, (uint32_t)(gi / S - 1) & 1u)) {
          report(a.status, KVINJ_ST_TIMEOUT);
          flags[0] = 1;
          go = 0;
        }
        if (go) {
          valid[st] = oki;
          uint64_t *fb = full + st;
          mbar_arrive_expect_tx(fb, Lay::STAGE_BYTES);
          uint8_t *kd = stages + st * Lay::STAGE_BYTES;
#pragma unroll
          for (int b = 0; b < NBOX; ++b) {
            tma_load_2d(kd + b * BOX_BYTES, &tmK, 64 * b, r0, fb);
            tma_load_2d(kd + Lay::PAGE_BYTES + b * BOX_BYTES, &tmV, 64 * b, r0, fb);
          }
        }
      }
      go = __shfl_sync(0xffffffffu, go, 0);
      if (!go) {
        aborted = true;
        break;
      }
      issued = gi + 1;
    }
    blk = nblk;
    h = nh;
  }
  if (aborted && lane == 0) {
    // let the copies already in flight land before the CTA can exit
    for (int gi = max(0, issued - S); gi < issued; ++gi)
      mbar_wait_bounded(full + gi % S, (uint32_t)(gi / S) & 1u, 100000000ull);
  }
}

// q rows of the G heads of kv group h of request r, rotated at q_pos[r],
// times scale*log2(e). The lane keeps, for every 64-element box b, the 8
// elements of chunk `dg`: dims [64b + 8dg, 64b + 8dg + 8).
template <int D, int G, int DT, int NBOX>
__device__ __forceinline__ void load_q_rows(const DecodeArgs &a, int r, int h, int dg,
                                            float (&qr)[G][NBOX][8]) {
  constexpr int HALF = D / 2;
  const int qp = a.q_pos[r];
  const bool rotate = a.rope != nullptr;
  const bool pos_ok = !rotate || (qp >= 0 && qp < a.max_pos);
  if (!pos_ok && dg == 0 && (threadIdx.x & 31) == 0) report(a.status, KVINJ_ST_BAD_POS);
  const float4 *trow = rotate && pos_ok ? a.rope + (int64_t)qp * HALF : nullptr;
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const uint16_t *qrow = a.q + ((int64_t)r * a.Hq + h * G + g) * D;
#pragma unroll
    for (int b = 0; b < NBOX; ++b) {
      const int d0 = 64 * b + 8 * dg;
      uint4 own = *reinterpret_cast<const uint4 *>(qrow + d0);
      float x[8];
      float2 f;
      f = unpack2<DT>(own.x); x[0] = f.x; x[1] = f.y;
      f = unpack2<DT>(own.y); x[2] = f.x; x[3] = f.y;
      f = unpack2<DT>(own.z); x[4] = f.x; x[5] = f.y;
      f = unpack2<DT>(own.w); x[6] = f.x; x[7] = f.y;
      if (trow) {
        const int dp = (d0 + HALF) % D;  // the rotate-half partners
        uint4 par = *reinterpret_cast<const uint4 *>(qrow + dp);
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

template <int DT>
__device__ __forceinline__ uint16_t to16(float x) {
  if constexpr (DT == 0) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  else return __half_as_ushort(__float2half_rn(x));
}

// End of a piece: merge the NW per-warp states (already in mm/ml/macc), then
// either write the output (piece == whole segment) or store this CTA's
// partial and, if it is the last piece of its segment to arrive, combine all
// pieces. Called by the NW consumer warps only (named barrier 1).
template <class Lay, int DT>
__device__ void finish_piece(const DecodeArgs &a, uint8_t *sm, const CtaRange &rg,
                             const Piece &pc, int P, int tid) {
  constexpr int G = Lay::G, D = Lay::D, NW = Lay::NW, NT = NW * 32;
  volatile int *flags = reinterpret_cast<volatile int *>(sm + Lay::off_flags);
  const float *mm = reinterpret_cast<const float *>(sm + Lay::off_mm);
  const float *ml = reinterpret_cast<const float *>(sm + Lay::off_ml);
  const float *macc = reinterpret_cast<const float *>(sm + Lay::off_macc);
  named_bar_sync(1, NT);
  const bool complete = (P == pc.seg_start) && (pc.end == pc.seg_end);
  uint16_t *orow = a.out + ((int64_t)pc.r * a.Hq + pc.h * G) * D;
  constexpr int PF = G * (D + 2);  // floats per partial slot: m[G], l[G], acc[G][D]
  float *mine = a.partials +
                (size_t)(2 * blockIdx.x + (pc.seg_start <= rg.b0 ? 0 : 1)) * PF;
  for (int idx = tid; idx < G * D; idx += NT) {
    const int g = idx / D, d = idx - g * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, mm[w * G + g]);
    float Ls = 0.f, A = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const float mw = mm[w * G + g];
      const float f = (mw == -INFINITY) ? 0.f : exp2f(mw - M);
      Ls = __fmaf_rn(ml[w * G + g], f, Ls);
      A = __fmaf_rn(macc[(w * G + g) * D + d], f, A);
    }
    if (complete) {
      orow[idx] = to16<DT>(Ls > 0.f ? A / Ls : 0.f);
    } else {
      mine[2 * G + idx] = A;
      if (d == 0) {
        mine[g] = M;
        mine[G + g] = Ls;
      }
    }
  }
  if (!complete) {
    __threadfence();
    named_bar_sync(1, NT);
    const int cf = cta_of(pc.seg_start, rg), cl = cta_of(pc.seg_end - 1, rg);
    if (tid == 0) {
      const int old = atomicAdd(a.counters + pc.r * a.Hkv + pc.h, 1);
      flags[1] = (old == cl - cf) ? 1 : 0;
    }
    named_bar_sync(1, NT);
    if (flags[1]) {
      __threadfence();
      for (int idx = tid; idx < G * D; idx += NT) {
        const int g = idx / D;
        float M = -INFINITY;
        for (int c = cf; c <= cl; ++c) {
          const float *pp = a.partials +
                            (size_t)(2 * c + (pc.seg_start <= range_begin(c, rg) ? 0 : 1)) * PF;
          M = fmaxf(M, __ldcg(pp + g));
        }
        float Ls = 0.f, A = 0.f;
        for (int c = cf; c <= cl; ++c) {
          const float *pp = a.partials +
                            (size_t)(2 * c + (pc.seg_start <= range_begin(c, rg) ? 0 : 1)) * PF;
          const float mc = __ldcg(pp + g);
          const float f = (mc == -INFINITY) ? 0.f : exp2f(mc - M);
          Ls = __fmaf_rn(__ldcg(pp + G + g), f, Ls);
          A = __fmaf_rn(__ldcg(pp + 2 * G + idx), f, A);
        }
        orow[idx] = to16<DT>(Ls > 0.f ? A / Ls : 0.f);
      }
      if (tid == 0) atomicExch(a.counters + pc.r * a.Hkv + pc.h, 0);
    }
  }
  named_bar_sync(1, NT);
}

}  // namespace kvinj
