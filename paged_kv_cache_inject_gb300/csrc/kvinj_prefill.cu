// kvinj_prefill.cu -- paged prefill of query tokens on the tensor cores.
//
// "InferScale: GPU-Native KV Injection for Personalized LLM Serving", §3.4 step
// 4: once the memory chunks are injected, only the query tokens are prefilled,
// each attending to the injected memory (and to the earlier query tokens)
// through the request's block table as if the memory had been prefilled. Query
// token i of request seq[i] sits at position pos[i], its own K/V already in the
// cache, and attends to the request's tokens 0 .. pos[i]:
//   out[i][qh] = sum_j softmax_j(scale * (R_{pos[i]} q[i][qh]) . K_j) V_j,  j <= pos[i]
// over kv head qh / G ("LLM Inference: KV Caching": softmax(QK^T / sqrt d) V).
//
// Tiles. The query rows of one request that share a kv head are the MMA's M
// dimension: a tile is up to T = 128 / G consecutive tokens of the token list
// that belong to one request, its 128 rows the (token, query head of the
// group) pairs, row = t * G + g. A unit of work is (tile, kv head, chunk of 128
// keys = 8 pages): K and V of the chunk are read once for all rows of the tile.
// prefill_setup_kernel finds the tiles in its first CTA (zeroing the rows of
// invalid tokens and laying the units out (tile, head, chunk) with prefix
// sums) while its other CTAs prepare every query row as the MMA reads it
// (rotated, scaled, split into hi + lo 16-bit parts). The units are split into
// equal contiguous ranges, one per CTA of prefill_umma_kernel. A segment (tile,
// head) cut by a range boundary leaves one partial softmax state per piece,
// which prefill_combine_kernel merges.
//
// prefill_umma_kernel, per CTA (12 warps; warps 2-3 only lend their registers):
//   warp 0     producer: the chunk's 8 pages of K and V (16-row TMA boxes of
//              64 columns, 128-byte swizzle) into a 3-stage ring, the pages'
//              valid bits beside them
//   warp 1     tensor-memory owner and MMA issuer, per unit
//                S  = Q K^T  (A = Q hi, lo from tensor memory, B = K, K-major)
//                O += P V    (A = P hi, lo from tensor memory, B = V, MN-major)
//   warps 4-11 softmax in two sets on the same rows, one row per thread
//              (tensor-memory lanes 32 (warp % 4) onward): set 0 (warps 4-7)
//              keys 0-63 of each chunk and O columns 0-63, set 1 (warps 8-11)
//              keys 64-127 and O columns 64-127. Per unit: this set's part of
//              the row of S masked (keys after the row's position, or in a page
//              outside the cache), the rows' maxima exchanged, a lazy running
//              maximum, P = 2^(S - m) split into hi + lo 16-bit parts written
//              over the set's own columns of S, O rescaled when the maximum
//              moved; at the end
//              of a piece O / l to the output, or (m, l, O) to the workspace,
//              and the next piece's prepared query rows into tensor memory
//              (set 0 the hi parts, set 1 the lo parts)
// Tensor memory (512 columns): S[2] at 0 and 128 (P over them: keys 64k ..
// 64k + 63 as hi words at 64k + j, lo words at 64k + 32 + j), O at 256,
// Q hi at 384, Q lo at 448. Every wait is bounded and reports
// KVINJ_ST_TIMEOUT when it gives up.
#include "kvinj_device.cuh"
#include "kvinj_internal.h"
#include "kvinj_umma.cuh"

namespace kvinj {

namespace {

constexpr int PF_D = 128;
constexpr int BLK = 16;                   // tokens per page
constexpr int PF_S = 3;                   // stages
constexpr int PF_THREADS = 384;           // 12 warps = 3 warpgroups
// registers per thread of each warpgroup after setmaxnreg (warps 0-3: 168 -> 120, each
// softmax set: 168 -> 192): the launch provides 384 x 168 = 64512, and 128 x (120 + 2 x 192)
// = 64512 -- the softmax sets' increase is exactly what the first warpgroup frees
constexpr int PF_REG_LAUNCH = 168, PF_REG_CTRL = 120, PF_REG_SOFTMAX = 192;
static_assert(128 * (PF_REG_CTRL + 2 * PF_REG_SOFTMAX) <= PF_THREADS * PF_REG_LAUNCH,
              "prefill: register split");
constexpr int PF_TB = 1024;               // threads of the tile builder
constexpr int PF_SLOT = 128 * (PF_D + 2); // floats of a partial state: m[128] l[128] O[D][128]
constexpr int PF_COMBINE_THREADS = 512;  // four per row

// tensor-memory columns
constexpr uint32_t TM_S = 0, TM_O = 256, TM_QHI = 384, TM_QLO = 448;

struct PfLayout {
  static constexpr int BOX = 128 * 128;           // one 64-column block of 128 rows
  static constexpr int KV = 2 * BOX;              // K (or V) of a chunk
  static constexpr int STAGE = 2 * KV;            // K then V
  static constexpr int off_bar = PF_S * STAGE;
  // full[S] empty[S] tq qfree sfull[2] pfull[2] pvdone done
  static constexpr int NBAR = 2 * PF_S + 2 + 4 + 2;
  static constexpr int off_valid = off_bar + NBAR * 8;  // [S] page bits of each stage
  static constexpr int off_flags = off_valid + PF_S * 4;  // [0] abort
  static constexpr int off_tmem = off_flags + 16;
  // the softmax sets' exchange: rows' maxima [2 parities][2 sets][128], sums [2 sets][128]
  static constexpr int off_mx = (off_tmem + 16 + 15) / 16 * 16;
  static constexpr int bytes = off_mx + (4 * 128 + 2 * 128) * 4;
};
static_assert(PfLayout::bytes <= 227 * 1024, "prefill: shared memory");

// register budget of the executing warpgroup (all its threads execute it)
template <int N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

__device__ __forceinline__ void sts128_zero(uint32_t addr) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0) : "memory");
}

// 32x32b.x16 store that does not wait for its completion (tmem_wait_st does)
__device__ __forceinline__ void tmem_st16_nw(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
               :
               : "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
               : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], issued by one thread; acc = 0 overwrites D
__device__ __forceinline__ void umma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(acc)
      : "memory");
}

// inclusive scan over the builder's PF_TB threads with operator op; *total = all of them
template <class Op>
__device__ int cta_scan(int v, int *sh, int &total, Op op) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int x = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v = op(v, x);
  }
  if (lane == 31) sh[w] = v;
  __syncthreads();
  if (w == 0) {
    int s = sh[lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xffffffffu, s, o);
      if (lane >= o) s = op(s, x);
    }
    sh[lane] = s;
  }
  __syncthreads();
  const int r = w ? op(v, sh[w - 1]) : v;
  total = sh[31];
  __syncthreads();
  return r;
}

__device__ __forceinline__ bool token_ok(const PrefillArgs &a, int i, int &r, int &p) {
  r = a.seq[i];
  p = a.pos[i];
  return r >= 0 && r < a.batch && p >= 0 && (int64_t)p < (int64_t)a.max_blocks * BLK;
}

// CTAs with a range: no more than units, so that every range holds one at least
__device__ __forceinline__ int ranges(int total, int grid) { return total < grid ? total : grid; }

// first unit of CTA c's range (c < ranges(total, grid)): c * total / ranges
__device__ __forceinline__ int range_start(int c, int total, int ng) {
  return (int)((int64_t)c * total / ng);
}

// The tiles: runs of consecutive valid tokens of one request, cut every T tokens.
// tiles[k] = {request, first token, tokens, largest position}; the units of tile k
// (Hkv heads x its chunks) start at tile_pre[k]; cta_tile[c] = the tile of CTA c's
// first unit; hdr = {tiles, units}.
__device__ void prefill_tiles(const PrefillArgs &a, int T) {
  __shared__ int sh[32];
  const int tid = threadIdx.x;
  auto add = [](int x, int y) { return x + y; };
  auto mx = [](int x, int y) { return x > y ? x : y; };
  int bad = 0, carry_rs = -1, carry_k = 0;
  for (int i0 = 0; i0 < a.n; i0 += PF_TB) {
    const int i = i0 + tid;
    int r = 0, p = 0;
    const bool ok = i < a.n && token_ok(a, i, r, p);
    if (i < a.n && !ok) {
      // a request id outside the batch or a position outside the table: zero row
      bad |= (r < 0 || r >= a.batch) ? (KVINJ_ST_BAD_SEQ | KVINJ_ST_BAD_CTX)
                                     : (KVINJ_ST_BAD_POS | KVINJ_ST_BAD_CTX);
      uint4 *o = reinterpret_cast<uint4 *>(a.out + (int64_t)i * a.Hq * PF_D);
      for (int e = 0; e < a.Hq * PF_D / 8; ++e) o[e] = make_uint4(0, 0, 0, 0);
    }
    int rp = 0, pp = 0;
    const bool run0 = ok && (i == 0 || !token_ok(a, i - 1, rp, pp) || rp != r);
    int tot;
    const int rs = mx(cta_scan(run0 ? i : -1, sh, tot, mx), carry_rs);
    carry_rs = mx(carry_rs, tot);
    const bool t0 = ok && (i - rs) % T == 0;
    const int k = carry_k + cta_scan(t0 ? 1 : 0, sh, tot, add) - (t0 ? 1 : 0);
    carry_k += tot;
    if (t0) {
      // the tile: this token and the next ones of the same run, T at most (the loads do
      // not wait on one another: no early exit)
      int nt = 1, mp = p;
      bool run = true;
      for (int j = i + 1; j < i + T; ++j) {
        int rj = -1, pj = 0;
        const bool okj = j < a.n && token_ok(a, j, rj, pj);
        run = run && okj && rj == r;
        if (run) {
          mp = max(mp, pj);
          ++nt;
        }
      }
      a.tiles[k] = make_int4(r, i, nt, mp);
    }
  }
  if (bad) report(a.status, bad);
  const int n_tiles = carry_k;
  __syncthreads();
  int carry_u = 0;
  for (int k0 = 0; k0 < n_tiles; k0 += PF_TB) {
    const int k = k0 + tid;
    const int units = k < n_tiles ? a.Hkv * (a.tiles[k].w / PF_D + 1) : 0;
    int tot;
    const int inc = cta_scan(units, sh, tot, add);
    if (k < n_tiles) a.tile_pre[k] = carry_u + inc - units;
    carry_u += tot;
  }
  if (tid == 0) {
    a.tile_pre[n_tiles] = carry_u;
    a.hdr[0] = n_tiles;
    a.hdr[1] = carry_u;
  }
  __syncthreads();
  const int64_t total = carry_u;
  if (total == 0) return;
  const int64_t ng = ranges(carry_u, a.grid);
  for (int k = tid; k < n_tiles; k += PF_TB) {
    // the CTAs whose range starts inside this tile's units [lo, hi)
    const int64_t lo = a.tile_pre[k], hi = a.tile_pre[k + 1];
    const int64_t c0 = (lo * ng + total - 1) / total, c1 = (hi * ng + total - 1) / total;
    for (int64_t c = c0; c < c1 && c < ng; ++c) a.cta_tile[c] = k;
  }
}

// Query rows as the MMA reads them: row (token i, query head qh) rotated at pos[i] (as
// given without a RoPE table; a position outside the table leaves it unrotated and is
// flagged), times scale * log2(e), as 16-bit hi parts (words 0-63, word j = elements 2j,
// 2j + 1) and lo parts (words 64-127). One warp per row: lane l the pairs (2l, 2l + 64) and
// (2l + 1, 2l + 65). Rows of invalid tokens are not written (no tile holds them).
template <int DT>
__device__ void prefill_q_rows(const PrefillArgs &a, int cta, int ctas) {
  const int lane = threadIdx.x & 31;
  const int64_t rows = (int64_t)a.n * a.Hq;
  for (int64_t row = ((int64_t)cta * blockDim.x + threadIdx.x) >> 5; row < rows;
       row += ((int64_t)ctas * blockDim.x) >> 5) {
    const int i = (int)(row / a.Hq);
    int r, p;
    if (!token_ok(a, i, r, p)) continue;
    const bool rot = a.rope && p < a.max_pos;
    if (a.rope && !rot && lane == 0 && row % a.Hq == 0) report(a.status, KVINJ_ST_BAD_POS);
    const uint32_t *src = reinterpret_cast<const uint32_t *>(a.q + row * PF_D);
    const float2 x = unpack2<DT>(__ldg(src + lane)), y = unpack2<DT>(__ldg(src + 32 + lane));
    float a0 = x.x, a1 = x.y, b0 = y.x, b1 = y.y;
    if (rot) {
      const float4 *tab = a.rope + (int64_t)p * (PF_D / 2) + 2 * lane;
      const float2 r0 = rope_pair(a0, b0, __ldg(tab)), r1 = rope_pair(a1, b1, __ldg(tab + 1));
      a0 = r0.x;
      b0 = r0.y;
      a1 = r1.x;
      b1 = r1.y;
    }
    const float sc = a.scale_log2;
    a0 *= sc;
    a1 *= sc;
    b0 *= sc;
    b1 *= sc;
    uint32_t *dst = a.qhl + row * PF_D;
    const uint32_t h1 = pack2<DT>(a0, a1), h2 = pack2<DT>(b0, b1);
    const float2 f1 = unpack2<DT>(h1), f2 = unpack2<DT>(h2);
    dst[lane] = h1;
    dst[32 + lane] = h2;
    dst[64 + lane] = pack2<DT>(a0 - f1.x, a1 - f1.y);
    dst[96 + lane] = pack2<DT>(b0 - f2.x, b1 - f2.y);
  }
}

// CTA 0 lays out the tiles and units, the other CTAs prepare the query rows
template <int DT>
__global__ void __launch_bounds__(PF_TB) prefill_setup_kernel(PrefillArgs a, int T) {
  if (blockIdx.x == 0) prefill_tiles(a, T);
  else prefill_q_rows<DT>(a, blockIdx.x - 1, gridDim.x - 1);
}

// sequential walk over the tiles of a CTA's units
struct PfWalk {
  int k = 0, kb = 0, ke = 0, nch = 1;
  int4 t = make_int4(0, 0, 0, 0);
  __device__ void set(const PrefillArgs &a, int kk) {
    k = kk;
    t = a.tiles[k];
    kb = a.tile_pre[k];
    ke = a.tile_pre[k + 1];
    nch = t.w / PF_D + 1;
  }
  __device__ void seek(const PrefillArgs &a, int u) {
    while (u >= ke) set(a, k + 1);
  }
};

// the piece of a segment (tile, head) that starts at unit u of a range ending at b1
struct PfPiece {
  int u1, h, c0, seg0, seg1;
};
__device__ __forceinline__ PfPiece pf_piece(const PfWalk &w, int u, int b1) {
  PfPiece p;
  const int off = u - w.kb;
  p.h = off / w.nch;
  p.c0 = off - p.h * w.nch;
  p.seg0 = w.kb + p.h * w.nch;
  p.seg1 = p.seg0 + w.nch;
  p.u1 = min(p.seg1, b1);
  return p;
}

template <int G, int DT>
__global__ void __launch_bounds__(PF_THREADS, 1)
    prefill_umma_kernel(const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, PrefillArgs a) {
  using Lay = PfLayout;
  extern __shared__ __align__(1024) uint8_t sm[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (smem_u32(sm) & 1023u) {  // the swizzled tiles need 1024-byte alignment
    if (tid == 0) report(a.status, KVINJ_ST_INTERNAL);
    return;
  }
  const int total = a.hdr[1], ng = ranges(total, a.grid);
  if ((int)blockIdx.x >= ng) return;
  const int b0 = range_start(blockIdx.x, total, ng);
  const int b1 = range_start(blockIdx.x + 1, total, ng);

  uint64_t *bar = reinterpret_cast<uint64_t *>(sm + Lay::off_bar);
  uint64_t *full = bar, *empty = bar + PF_S, *tq = bar + 2 * PF_S, *qfree = tq + 1;
  uint64_t *sfull = tq + 2, *pfull = sfull + 2, *pvdone = pfull + 2, *done = pvdone + 1;
  int *valid = reinterpret_cast<int *>(sm + Lay::off_valid);
  volatile int *flags = reinterpret_cast<volatile int *>(sm + Lay::off_flags);
  uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + Lay::off_tmem);
  if (tid == 0) {
    for (int s = 0; s < PF_S; ++s) {
      mbar_init(full + s, 1);   // the producer's arrive + the copies' bytes
      mbar_init(empty + s, 1);  // the MMA's commit after the unit's PV
    }
    mbar_init(tq, 8);     // the softmax warps: Q of a piece in tensor memory
    mbar_init(qfree, 1);  // the MMA's commit after a piece's last QK
    for (int b = 0; b < 2; ++b) {
      mbar_init(sfull + b, 1);
      mbar_init(pfull + b, 8);  // the softmax warps: P in tensor memory, O rescaled
    }
    mbar_init(pvdone, 1);
    mbar_init(done, 1);
    flags[0] = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tslot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = *tslot;
  auto wait = [&](uint64_t *b, uint32_t parity) -> bool {
    if (flags[0]) return false;
    if (mbar_wait_bounded(b, parity)) return true;
    report(a.status, KVINJ_ST_TIMEOUT);
    flags[0] = 1;
    return false;
  };
  PfWalk w;
  w.set(a, a.cta_tile[blockIdx.x]);
  if (warp < 4) regs_dec<PF_REG_CTRL>();  // the whole first warpgroup
  if (warp == 0) {
    // -------------------------------- producer --------------------------------
    if (lane == 0) {
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
    }
    // unit u's kv head and (lanes 0-7) the table entries of its chunk's 8 pages, looked up
    // one unit ahead of its copies; a page past the tile's last position is not needed (its
    // copy re-reads the chunk's first page, masked)
    struct Look {
      int blk, h;
      bool need;
    };
    auto look = [&](int u) {
      Look l{-1, 0, false};
      if (u < b1) {
        w.seek(a, u);
        const int off = u - w.kb;
        l.h = off / w.nch;
        const int pg = (off - l.h * w.nch) * 8 + (lane & 7);
        l.need = lane < 8 && pg * BLK <= w.t.w;
        if (l.need) l.blk = __ldg(a.block_tables + (int64_t)w.t.x * a.max_blocks + pg);
      }
      return l;
    };
    int issued = 0;
    Look cur = look(b0);
    for (int u = b0, gi = 0; u < b1; ++u, ++gi) {
      const Look nxt = look(u + 1);  // in flight while this unit waits for its stage
      const int st = gi % PF_S;
      const bool okb = cur.need && cur.blk >= 0 && cur.blk < a.num_blocks;
      if (cur.need && !okb) report(a.status, KVINJ_ST_BAD_BLOCK);
      const int vbits = (int)(__ballot_sync(0xffffffffu, okb) & 0xFFu);
      const int first = __shfl_sync(0xffffffffu, okb ? cur.blk : 0, 0);
      const int use = okb ? cur.blk : first;
      bool go = true;
      if (lane == 0) go = gi < PF_S || wait(empty + st, (uint32_t)(gi / PF_S - 1) & 1u);
      if (!__shfl_sync(0xffffffffu, go, 0)) break;
      if (lane == 0) {
        valid[st] = vbits;
        mbar_arrive_expect_tx(full + st, Lay::STAGE);
      }
      __syncwarp();
      if (lane < 8) {
        const int row = (int)((((int64_t)a.layer * a.num_blocks + use) * a.Hkv + cur.h) * BLK);
        uint8_t *kd = sm + st * Lay::STAGE + lane * BLK * 128;
#pragma unroll
        for (int cb = 0; cb < 2; ++cb) {
          tma_load_2d(kd + cb * Lay::BOX, &tmK, 64 * cb, row, full + st);
          tma_load_2d(kd + Lay::KV + cb * Lay::BOX, &tmV, 64 * cb, row, full + st);
        }
      }
      issued = gi + 1;
      cur = nxt;
    }
    if (flags[0] && lane == 0) {
      // the copies in flight land before the CTA can exit
      for (int g = max(0, issued - PF_S); g < issued; ++g)
        mbar_wait_bounded(full + g % PF_S, (uint32_t)(g / PF_S) & 1u, 100000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------- MMA issuer -------------------------------
    if (lane == 0) {
      constexpr uint32_t ID_QK = umma_idesc_f16<DT>(128, 128, 0, 0);
      constexpr uint32_t ID_PV = umma_idesc_f16<DT>(128, 128, 0, 1);
      const uint32_t stage0 = smem_u32(sm);
      int pv_seen = 0;  // PV completions observed (in order: at most one unobserved)
      auto see_pv = [&](int upto) -> bool {
        while (pv_seen < upto) {
          if (!wait(pvdone, (uint32_t)pv_seen & 1u)) return false;
          ++pv_seen;
        }
        return true;
      };
      auto issue_pv = [&](int g, bool first) -> bool {
        if (!wait(pfull + (g & 1), (uint32_t)(g >> 1) & 1u) || !see_pv(g)) return false;
        tc_fence_after();
        const uint32_t vb = stage0 + (g % PF_S) * Lay::STAGE + Lay::KV;
        const uint32_t pa = tbase + TM_S + (g & 1) * 128;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          // keys 16 kk .. 16 kk + 15: softmax set kk / 4 wrote their P hi words at
          // 64 (kk / 4) + 8 (kk % 4) and lo words 32 columns further
          const uint32_t ph = pa + 64 * (kk >> 2) + 8 * (kk & 3);
          const uint64_t bd = umma_desc_sw128(vb + kk * 2048, Lay::BOX, 1024);
          umma_f16_tmem_a(tbase + TM_O, ph, bd, ID_PV, (first && kk == 0) ? 0u : 1u);
          umma_f16_tmem_a(tbase + TM_O, ph + 32, bd, ID_PV, 1u);
        }
        umma_commit(empty + g % PF_S);
        umma_commit(pvdone);
        return true;
      };
      int gi = 0, piece = 0, pend = -1;
      bool pend_first = false, ok = true;
      for (int u = b0; u < b1 && ok;) {
        w.seek(a, u);
        const PfPiece pc = pf_piece(w, u, b1);
        for (int j = 0; u < pc.u1; ++u, ++j, ++gi) {
          const int st = gi % PF_S;
          if (j == 0) {
            // the previous piece's last PV before this piece's Q (the softmax warps copy the
            // new Q rows only after reading that piece's O out)
            if (pend >= 0 && !(ok = issue_pv(pend, pend_first))) break;
            pend = -1;
            if (!(ok = wait(tq, (uint32_t)piece & 1u))) break;
            ++piece;
          }
          // S[gi & 1] is free once PV(gi - 2) has read the P over it
          if (!(ok = wait(full + st, (uint32_t)(gi / PF_S) & 1u) && see_pv(gi - 1))) break;
          tc_fence_after();
          const uint32_t kb = stage0 + st * Lay::STAGE, d = tbase + TM_S + (gi & 1) * 128;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t bd = umma_desc_sw128(kb + (kk >> 2) * Lay::BOX + (kk & 3) * 32, 16, 1024);
            umma_f16_tmem_a(d, tbase + TM_QHI + kk * 8, bd, ID_QK, kk > 0 ? 1u : 0u);
            umma_f16_tmem_a(d, tbase + TM_QLO + kk * 8, bd, ID_QK, 1u);
          }
          umma_commit(sfull + (gi & 1));
          if (u + 1 == pc.u1) umma_commit(qfree);  // Q may be replaced once these QKs are done
          if (pend >= 0 && !(ok = issue_pv(pend, pend_first))) break;
          pend = gi;
          pend_first = j == 0;
        }
      }
      if (ok && pend >= 0) issue_pv(pend, pend_first);
      // every MMA complete before tensor memory and shared memory are released
      umma_commit(done);
      if (!mbar_wait_bounded(done, 0, 100000000ull)) {
        report(a.status, KVINJ_ST_TIMEOUT);
        flags[0] = 1;
      }
    }
    __syncwarp();
  } else if (warp < 4) {
    // warps 2-3: no role
  } else {
    // -------------------------------- softmax --------------------------------
    // two sets on the same rows: set 0 (warps 4-7) keys 0-63 of each chunk and O columns
    // 0-63, set 1 (warps 8-11) keys 64-127 and O columns 64-127; they exchange the rows'
    // maxima per unit and their sums per piece. Each set also copies its half of the next
    // piece's prepared query rows (set 0 the hi words, set 1 the lo words).
    regs_inc<PF_REG_SOFTMAX>();
    const int set = warp >= 8 ? 1 : 0;
    const int qd = warp & 3;
    const int m = 32 * qd + lane;  // tile row = tensor-memory lane
    const int tr = m / G, g = m % G;
    float *mxb = reinterpret_cast<float *>(sm + Lay::off_mx);  // [2 parities][2 sets][128]
    float *lxb = mxb + 4 * 128;                                 // [2 sets][128]
    // the prepared query row of this thread in a piece: 16 words-quads (its set's half)
    auto q_src = [&](const PfWalk &wk, const PfPiece &pq) {
      const bool r_ok = tr < wk.t.z;
      const int64_t row = (int64_t)(r_ok ? wk.t.y + tr : 0) * a.Hq + (int64_t)pq.h * G + g;
      return r_ok ? reinterpret_cast<const uint4 *>(a.qhl + row * PF_D) + 16 * set : nullptr;
    };
    auto q_store = [&](const uint4 (&v)[16]) {
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        uint32_t wv[16];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          wv[4 * e] = v[4 * q4 + e].x;
          wv[4 * e + 1] = v[4 * q4 + e].y;
          wv[4 * e + 2] = v[4 * q4 + e].z;
          wv[4 * e + 3] = v[4 * q4 + e].w;
        }
        tmem_st16_nw(tmem_addr(tbase, 32 * qd, (set ? TM_QLO : TM_QHI) + 16 * q4), wv);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tq);
    };
    // Every thread of both sets runs the same sequence of named barriers whatever happens: a
    // wait that gave up (the abort flag; later waits return at once) only skips work.
    int gi = 0, piece = 0;
    bool ok = true;
    {
      // the first piece's query rows
      w.seek(a, b0);
      const PfPiece pq = pf_piece(w, b0, b1);
      const uint4 *src = q_src(w, pq);
      uint4 v[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) v[e] = src ? __ldg(src + e) : make_uint4(0, 0, 0, 0);
      q_store(v);
    }
    for (int u = b0; u < b1; ++piece) {
      w.seek(a, u);
      const PfPiece pc = pf_piece(w, u, b1);
      const int i0 = w.t.y, nt = w.t.z, mp = w.t.w;
      const bool rv = tr < nt;
      const int tok = i0 + tr;
      const int p = rv ? __ldg(a.pos + tok) : -1;
      const bool wlive = __any_sync(0xffffffffu, rv);
      float m_run = -INFINITY, l_run = 0.f;
      for (int j = 0, c = pc.c0; u < pc.u1; ++u, ++j, ++c, ++gi) {
        const int st = gi % PF_S, par = gi & 1;
        ok = ok && wait(full + st, (uint32_t)(gi / PF_S) & 1u) &&
             wait(sfull + par, (uint32_t)(gi >> 1) & 1u);
        ok = __all_sync(0xffffffffu, ok);  // it gates warp-wide tensor-memory operations
        const bool work = ok && wlive;
        tc_fence_after();
        const int vb = valid[st];
        // this set's keys 64 set + e, e < 64, are attended to when at or before the row's
        // position and in a page in the cache
        const int lim = p - c * 128 - 64 * set;
        const uint32_t ts = tmem_addr(tbase, 32 * qd, TM_S + par * 128);
        float mu_own = -INFINITY;
        uint32_t mw[2] = {0u, 0u};
        // a warp whose rows hold no token (a tile of fewer than 128 / G tokens) skips the
        // math (tensor-memory loads and stores are warp-wide): its P and O rows are never
        // read out, and an O row depends on its own P row only
        if (work) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int nk = min(max(lim - 32 * q + 1, 0), 32);
            const uint32_t keys = nk >= 32 ? 0xFFFFFFFFu : ((1u << nk) - 1u);
            const int pg = 4 * set + 2 * q;  // pages of keys 32 q .. 32 q + 31 of this set
            const uint32_t pages = (((vb >> pg) & 1) ? 0x0000FFFFu : 0u) |
                                   (((vb >> (pg + 1)) & 1) ? 0xFFFF0000u : 0u);
            mw[q] = keys & pages;
          }
          // this set's 64 columns of S, 32 at a time (read again below for P)
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t x[32];
            tmem_ld<32>(ts + 64 * set + 32 * q, x);
            float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if ((mw[q] >> e) & 1u) mx4[e & 3] = fmaxf(mx4[e & 3], __uint_as_float(x[e]));
            mu_own = fmaxf(mu_own, fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])));
          }
        }
        // the row's maximum over both sets' keys
        mxb[(par * 2 + set) * 128 + m] = mu_own;
        named_bar_sync(1, 256);
        const float mu = fmaxf(mu_own, mxb[(par * 2 + (set ^ 1)) * 128 + m]);
        float alpha = 1.f;
        bool resc = false;
        if (mu > m_run + 8.f) {  // lazy maximum (also the first finite one)
          alpha = exp2f(m_run - mu);
          m_run = mu;
          resc = true;
        }
        float sum = 0.f;
        if (work) {
          // P = 2^(S - m) <= 2^8 (0 for masked keys), hi + lo 16-bit parts, over this set's
          // own 64 columns of S: hi words (keys 2j, 2j + 1 of the set) at 64 set + j, lo
          // words at 64 set + 32 + j. The lo words of keys 0-31 wait until keys 32-63 are
          // read (their columns hold S of keys 32-63).
          float sum4[4] = {0.f, 0.f, 0.f, 0.f};
          uint32_t lo[2][16];
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t x[32], hi[16];
            tmem_ld<32>(ts + 64 * set + 32 * q, x);
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const bool k0 = (mw[q] >> (2 * e)) & 1u, k1 = (mw[q] >> (2 * e + 1)) & 1u;
              const float p0 = k0 ? ex2_approx(__uint_as_float(x[2 * e]) - m_run) : 0.f;
              const float p1 = k1 ? ex2_approx(__uint_as_float(x[2 * e + 1]) - m_run) : 0.f;
              sum4[e & 3] += p0 + p1;
              hi[e] = pack2<DT>(p0, p1);
              const float2 h = unpack2<DT>(hi[e]);
              lo[q][e] = pack2<DT>(p0 - h.x, p1 - h.y);
            }
            tmem_st16_nw(ts + 64 * set + 16 * q, hi);
          }
          tmem_st16_nw(ts + 64 * set + 32, lo[0]);
          tmem_st16_nw(ts + 64 * set + 48, lo[1]);
          tmem_wait_st();
          sum = (sum4[0] + sum4[1]) + (sum4[2] + sum4[3]);
        }
        l_run = __fmaf_rn(l_run, alpha, sum);
        // PV(gi - 1) is waited for at every unit, before this unit's P is announced: its
        // phase is then told apart from the others by parity (PV(gi - 2) is complete -- this
        // unit's QK waited for it -- and PV(gi) cannot be issued yet), and at the end of a
        // piece only PV(last) remains
        if (gi >= 1) {
          ok = __all_sync(0xffffffffu, ok && wait(pvdone, (uint32_t)(gi - 1) & 1u));
          tc_fence_after();
        }
        // this set's O columns times alpha before this unit's PV
        const bool any_resc = __any_sync(0xffffffffu, resc);
        if (j > 0 && ok && any_resc) {
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
            uint32_t o[32];
            const uint32_t ta = tmem_addr(tbase, 32 * qd, TM_O + 64 * set + 32 * q2);
            tmem_ld<32>(ta, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st<32>(ta, o);
          }
        }
        // V rows that no row of the tile attends to -- keys past the tile's last position
        // (the tail of its last page) and pages outside the cache (read from another
        // block) -- may hold anything, NaN bit patterns included: zeroed (each set one of
        // the row's two 64-column blocks), so that their zero probabilities contribute 0
        if (ok && (c * 128 + m > mp || !((vb >> (m / BLK)) & 1))) {
          const uint32_t vr = smem_u32(sm + st * Lay::STAGE + Lay::KV + set * Lay::BOX) + m * 128;
#pragma unroll
          for (int e = 0; e < 8; ++e) sts128_zero(vr + 16 * e);
        }
        fence_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(pfull + par);
      }
      // ---- end of piece ----
      // the next piece's query rows are loaded now; they go to tensor memory after the
      // readout, once this piece's last QK is done
      const bool more = pc.u1 < b1;
      const bool complete = pc.seg0 >= b0 && pc.u1 == pc.seg1;
      const int seg0 = pc.seg0, h = pc.h;
      uint4 vq[16];
      if (more) {
        w.seek(a, pc.u1);
        const PfPiece pn = pf_piece(w, pc.u1, b1);
        const uint4 *src = q_src(w, pn);
#pragma unroll
        for (int e = 0; e < 16; ++e) vq[e] = src ? __ldg(src + e) : make_uint4(0, 0, 0, 0);
      }
      // PV(last) (PV(last - 1) was waited for in the last unit)
      ok = __all_sync(0xffffffffu, ok && wait(pvdone, (uint32_t)(gi - 1) & 1u));
      tc_fence_after();
      lxb[set * 128 + m] = l_run;
      named_bar_sync(1, 256);
      const float l_tot = l_run + lxb[(set ^ 1) * 128 + m];
      const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
      uint4 *dst = reinterpret_cast<uint4 *>(
          a.out + ((int64_t)tok * a.Hq + (int64_t)h * G + g) * PF_D + 64 * set);
      // slot 0: the CTA's first piece (its segment began at or before the range), slot 1:
      // its last piece
      float *slot = a.partials + (size_t)(2 * blockIdx.x + (seg0 <= b0 ? 0 : 1)) * PF_SLOT;
#pragma unroll
      for (int q2 = 0; q2 < 2 && ok; ++q2) {
        uint32_t xo[32];
        tmem_ld<32>(tmem_addr(tbase, 32 * qd, TM_O + 64 * set + 32 * q2), xo);
        if (complete) {
          if (rv) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float *f = reinterpret_cast<const float *>(xo + 8 * e);
              dst[4 * q2 + e] = make_uint4(pack2<DT>(f[0] * inv, f[1] * inv),
                                           pack2<DT>(f[2] * inv, f[3] * inv),
                                           pack2<DT>(f[4] * inv, f[5] * inv),
                                           pack2<DT>(f[6] * inv, f[7] * inv));
            }
          }
        } else {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            slot[256 + (64 * set + 32 * q2 + e) * 128 + m] = __uint_as_float(xo[e]);
        }
      }
      if (ok && !complete && set == 0) {
        slot[m] = m_run;
        slot[128 + m] = l_tot;
      }
      tc_fence_before();
      if (more) {
        // this piece's QKs are done with the tensor-memory Q (its last S was read)
        ok = ok && wait(qfree, (uint32_t)piece & 1u);
        tc_fence_after();
        if (ok) q_store(vq);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// merges the pieces of every segment (tile, head) that range boundaries cut: per row
// M = max m_c, L = sum l_c 2^(m_c - M), out = sum O_c 2^(m_c - M) / L. Four threads per
// row, 32 dimensions each.
template <int G, int DT>
__global__ void __launch_bounds__(PF_COMBINE_THREADS) prefill_combine_kernel(PrefillArgs a) {
  const int n_tiles = a.hdr[0], total = a.hdr[1];
  if (total == 0) return;
  const int m = threadIdx.x & 127, d0 = 32 * (threadIdx.x >> 7), tr = m / G, g = m % G;
  const int ng = ranges(total, a.grid);
  auto cta_of = [&](int u) {
    int c = (int)((int64_t)u * ng / total);
    while (c + 1 < ng && range_start(c + 1, total, ng) <= u) ++c;
    while (c > 0 && range_start(c, total, ng) > u) --c;
    return c;
  };
  for (int64_t sg = blockIdx.x; sg < (int64_t)n_tiles * a.Hkv; sg += gridDim.x) {
    const int k = (int)(sg / a.Hkv), h = (int)(sg % a.Hkv);
    const int4 t = a.tiles[k];
    const int nch = t.w / PF_D + 1;
    const int seg0 = a.tile_pre[k] + h * nch, seg1 = seg0 + nch;
    const int ca = cta_of(seg0), cb = cta_of(seg1 - 1);
    if (ca == cb || tr >= t.z) continue;
    // slot of CTA c's piece: 1 only for the first CTA when the segment began after its
    // range's start (that piece is the CTA's last), else 0 (the CTA's first piece)
    const int sel0 = seg0 > range_start(ca, total, ng) ? 1 : 0;
    float mm = -INFINITY;
    for (int c = ca; c <= cb; ++c)
      mm = fmaxf(mm, a.partials[(size_t)(2 * c + (c == ca ? sel0 : 0)) * PF_SLOT + m]);
    float o[32], L = 0.f;
#pragma unroll
    for (int e = 0; e < 32; ++e) o[e] = 0.f;
    if (mm != -INFINITY) {
      for (int c = ca; c <= cb; ++c) {
        const float *sl = a.partials + (size_t)(2 * c + (c == ca ? sel0 : 0)) * PF_SLOT;
        const float mc = sl[m];
        if (mc == -INFINITY) continue;
        const float f = exp2f(mc - mm);
        L = __fmaf_rn(sl[128 + m], f, L);
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = __fmaf_rn(sl[256 + (d0 + e) * 128 + m], f, o[e]);
      }
    }
    const float inv = L > 0.f ? 1.f / L : 0.f;
    uint4 *dst = reinterpret_cast<uint4 *>(
        a.out + ((int64_t)(t.y + tr) * a.Hq + (int64_t)h * G + g) * PF_D + d0);
#pragma unroll
    for (int e = 0; e < 4; ++e)
      dst[e] = make_uint4(pack2<DT>(o[8 * e] * inv, o[8 * e + 1] * inv),
                          pack2<DT>(o[8 * e + 2] * inv, o[8 * e + 3] * inv),
                          pack2<DT>(o[8 * e + 4] * inv, o[8 * e + 5] * inv),
                          pack2<DT>(o[8 * e + 6] * inv, o[8 * e + 7] * inv));
  }
}

template <int G, int DT>
cudaError_t launch_prefill_t(const PrefillArgs &a, const CUtensorMap &tmK,
                             const CUtensorMap &tmV, cudaStream_t s) {
  // one CTA for the tiles, one warp per query row in the others (two per SM at most)
  const int64_t qctas = ((int64_t)a.n * a.Hq + PF_TB / 32 - 1) / (PF_TB / 32);
  const int setup = 1 + (int)(qctas < 2 * (int64_t)a.grid ? qctas : 2 * (int64_t)a.grid);
  prefill_setup_kernel<DT><<<setup, PF_TB, 0, s>>>(a, 128 / G);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  auto kern = prefill_umma_kernel<G, DT>;
  // the warpgroups' setmaxnreg split adds up to the registers of a launch at
  // PF_REG_LAUNCH per thread; any other count could leave an increase waiting
  cudaFuncAttributes fa;
  if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
  if (fa.numRegs != PF_REG_LAUNCH) return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PfLayout::bytes);
  if (e != cudaSuccess) return e;
  kern<<<a.grid, PF_THREADS, PfLayout::bytes, s>>>(tmK, tmV, a);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  prefill_combine_kernel<G, DT><<<a.grid, PF_COMBINE_THREADS, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace

size_t prefill_partial_floats() { return PF_SLOT; }

cudaError_t launch_prefill(const PrefillArgs &a, const CUtensorMap &tmK, const CUtensorMap &tmV,
                           int G, int dtype, cudaStream_t s) {
  switch (G * 2 + dtype) {
    case 2: return launch_prefill_t<1, 0>(a, tmK, tmV, s);
    case 3: return launch_prefill_t<1, 1>(a, tmK, tmV, s);
    case 4: return launch_prefill_t<2, 0>(a, tmK, tmV, s);
    case 5: return launch_prefill_t<2, 1>(a, tmK, tmV, s);
    case 8: return launch_prefill_t<4, 0>(a, tmK, tmV, s);
    case 9: return launch_prefill_t<4, 1>(a, tmK, tmV, s);
    case 16: return launch_prefill_t<8, 0>(a, tmK, tmV, s);
    case 17: return launch_prefill_t<8, 1>(a, tmK, tmV, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kvinj
