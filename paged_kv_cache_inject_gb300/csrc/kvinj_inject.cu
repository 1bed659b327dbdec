// kvinj_inject.cu -- slot mapping, inject (gather pre-RoPE chunk rows, rotate
// K at the assigned absolute position, scatter into paged blocks) and append.
//
// "InferScale: GPU-Native KV Injection for Personalized LLM Serving" §3.3
// (compose retrieved pre-RoPE facts, RoPE applied at the assigned positions)
// and §3.4 (the worker scatter-copies the composed KV into the allocated
// blocks via the slot mapping, a same-device copy); §5.1 Theorem 1 (the
// relocation is exact, so rotating stored keys at injection time is valid).
// "LLM Inference: KV Caching", "The fix": each decode step appends one
// token's K/V per layer; "Paged attention": block table -> physical blocks.
//
// Design (GB300): the path is a gather-rotate-scatter of 2*D-byte rows, bound
// by HBM bandwidth. A warp takes one unit = (chunk, layer, token): all Hkv K
// rows and all Hkv V rows of that token. Each 16-lane half-warp handles one
// row; lane k owns elements [E*k, E*k+E) of the first half of the row and the
// same offsets of the second half (E = D/32), so the rotate-half partner of
// every element sits in the same lane: no shuffles, and every load/store
// instruction of the warp covers two full 128-byte lines (D = 128). All loads
// of a unit are issued before its stores (4 row pairs per batch) to keep
// enough bytes in flight. The cos/sin table row of the token's position is
// loaded once per unit and reused for its Hkv rows. The grid is persistent
// (a multiple of the SM count) and walks the units in pool order, so reads
// stream through each chunk's contiguous K (then V) block.
#include "kvinj_device.cuh"
#include "kvinj_internal.h"

namespace kvinj {

// ---------------------------------------------------------------------------
// slot mapping
// ---------------------------------------------------------------------------
__global__ void slot_mapping_kernel(const int32_t *__restrict__ bt, int max_blocks, int batch,
                                    int64_t num_blocks, int B, const int32_t *__restrict__ seq,
                                    const int32_t *__restrict__ pos, int64_t n,
                                    int64_t *__restrict__ out, int32_t *status) {
  int bad = 0;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n;
       i += (int64_t)gridDim.x * blockDim.x) {
    int r = seq[i], p = pos[i];
    int64_t slot = -1;
    if (r < 0 || r >= batch) {
      bad |= KVINJ_ST_BAD_SEQ;
    } else if (p < 0 || p / B >= max_blocks) {
      bad |= KVINJ_ST_BAD_POS;
    } else {
      int blk = bt[(int64_t)r * max_blocks + p / B];
      if (blk < 0 || blk >= num_blocks)
        bad |= KVINJ_ST_BAD_BLOCK;
      else
        slot = (int64_t)blk * B + p % B;
    }
    out[i] = slot;
  }
  if (bad) report(status, bad);
}

// ---------------------------------------------------------------------------
// row rotation + copy for one unit
// ---------------------------------------------------------------------------
template <int D>
struct RowVec {
  static constexpr int E = D / 32;  // elements per lane per half row
  static constexpr int W = E / 2;   // 32-bit words per lane per half row
  using T = typename Vec<E * 2>::T;
};

template <int W>
struct Words {
  uint32_t w[W];
};

template <int D>
__device__ __forceinline__ Words<RowVec<D>::W> load_half(const uint16_t *p) {
  using T = typename RowVec<D>::T;
  T v = ld_stream(reinterpret_cast<const T *>(p));
  Words<RowVec<D>::W> r;
  static_assert(sizeof(T) == sizeof(r), "vector width");
  memcpy(&r, &v, sizeof(T));
  return r;
}

template <int D>
__device__ __forceinline__ void store_half(uint16_t *p, const Words<RowVec<D>::W> &r) {
  using T = typename RowVec<D>::T;
  T v;
  memcpy(&v, &r, sizeof(T));
  st_global(reinterpret_cast<T *>(p), v);
}

// Process the Hkv K rows (rotated with `rot` = table row of the position, or
// copied when rot == nullptr) and Hkv V rows (copied) of one token.
// Source row of head h: sk + h*s_stride; destination: dk + h*d_stride.
template <int D, int DT>
__device__ __forceinline__ void process_token(const uint16_t *sk, const uint16_t *sv,
                                              int64_t s_stride, uint16_t *dk, uint16_t *dv,
                                              int64_t d_stride, int Hkv, const float4 *rot,
                                              int lane) {
  constexpr int E = RowVec<D>::E, W = RowVec<D>::W, HALF = D / 2, RB = 4;
  const int half = lane >> 4, k = lane & 15;
  float4 tab[E];
  if (rot) {
#pragma unroll
    for (int e = 0; e < E; ++e) tab[e] = __ldg(rot + k * E + e);
  }
  for (int h0 = 0; h0 < Hkv; h0 += 2 * RB) {
    Words<W> klo[RB], khi[RB], vlo[RB], vhi[RB];
#pragma unroll
    for (int i = 0; i < RB; ++i) {
      int h = h0 + 2 * i + half;
      if (h < Hkv) {
        const uint16_t *ks = sk + h * s_stride + k * E;
        const uint16_t *vs = sv + h * s_stride + k * E;
        klo[i] = load_half<D>(ks);
        khi[i] = load_half<D>(ks + HALF);
        vlo[i] = load_half<D>(vs);
        vhi[i] = load_half<D>(vs + HALF);
      }
    }
#pragma unroll
    for (int i = 0; i < RB; ++i) {
      int h = h0 + 2 * i + half;
      if (h < Hkv) {
        if (rot) {
#pragma unroll
          for (int w = 0; w < W; ++w) {
            float2 a = unpack2<DT>(klo[i].w[w]);
            float2 b = unpack2<DT>(khi[i].w[w]);
            float2 y0 = rope_pair(a.x, b.x, tab[2 * w]);
            float2 y1 = rope_pair(a.y, b.y, tab[2 * w + 1]);
            klo[i].w[w] = pack2<DT>(y0.x, y1.x);
            khi[i].w[w] = pack2<DT>(y0.y, y1.y);
          }
        }
        uint16_t *kd = dk + h * d_stride + k * E;
        uint16_t *vd = dv + h * d_stride + k * E;
        store_half<D>(kd, klo[i]);
        store_half<D>(kd + HALF, khi[i]);
        store_half<D>(vd, vlo[i]);
        store_half<D>(vd + HALF, vhi[i]);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// inject
// ---------------------------------------------------------------------------
template <int D, int DT>
__global__ void __launch_bounds__(256) inject_kernel(InjectArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t c = a.chunk_len;
  const int64_t n_units = (int64_t)a.n_inj * a.n_layers * c;
  const int64_t row = (int64_t)a.Hkv * D;
  const int64_t nslots = a.num_blocks * a.B;
  for (int64_t u = warp; u < n_units; u += nwarps) {
    const int t = (int)(u % c);
    const int64_t jl = u / c;
    const int l = a.layer_begin + (int)(jl % a.n_layers);
    const int j = (int)(jl / a.n_layers);
    const int id = a.chunk_ids[j];
    const int64_t slot = a.slot_mapping[(int64_t)j * c + t];
    const int pos = a.start_pos[j] + t;
    int bad = 0;
    if (id < 0 || id >= a.num_chunks) bad |= KVINJ_ST_BAD_CHUNK;
    if (slot < 0 || slot >= nslots) bad |= KVINJ_ST_BAD_SLOT;
    if (pos < 0 || pos >= a.max_pos) bad |= KVINJ_ST_BAD_POS;
    if (bad) {
      if (lane == 0) report(a.status, bad);
      continue;
    }
    const uint16_t *sk = a.pool + (((int64_t)id * a.L + l) * 2 * c + t) * row;
    const uint16_t *sv = sk + c * row;
    const int64_t dst = (((int64_t)l * a.num_blocks + slot / a.B) * a.Hkv * a.B + slot % a.B) * D;
    process_token<D, DT>(sk, sv, D, a.k + dst, a.v + dst, (int64_t)a.B * D, a.Hkv,
                         a.rope + (int64_t)pos * (D / 2), lane);
  }
}

// ---------------------------------------------------------------------------
// append
// ---------------------------------------------------------------------------
template <int D, int DT>
__global__ void __launch_bounds__(256) append_kernel(AppendArgs a) {
  const int lane = threadIdx.x & 31;
  const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
  const int64_t row = (int64_t)a.Hkv * D;
  const int64_t nslots = a.num_blocks * a.B;
  for (int64_t i = warp; i < a.n; i += nwarps) {
    const int pos = a.positions[i];
    int bad = 0;
    if (pos < 0 || (a.rope && pos >= a.max_pos)) bad |= KVINJ_ST_BAD_POS;
    int64_t slot;
    if (a.slot_mapping) {
      slot = a.slot_mapping[i];
    } else {  // token i of request i, slot from the request's block table
      const int pg = pos >= 0 ? pos / a.B : 0;
      const int64_t blk = pg < a.max_blocks ? a.block_tables[i * a.max_blocks + pg] : -1;
      slot = blk >= 0 && blk < a.num_blocks ? blk * a.B + (pos % a.B) : -1;
      if (slot < 0) bad |= KVINJ_ST_BAD_BLOCK;
    }
    if (!(bad & KVINJ_ST_BAD_BLOCK) && (slot < 0 || slot >= nslots)) bad |= KVINJ_ST_BAD_SLOT;
    if (bad) {
      if (lane == 0) report(a.status, bad);
      continue;
    }
    const int64_t dst =
        (((int64_t)a.layer * a.num_blocks + slot / a.B) * a.Hkv * a.B + slot % a.B) * D;
    process_token<D, DT>(a.k_new + i * row, a.v_new + i * row, D, a.k + dst, a.v + dst,
                         (int64_t)a.B * D, a.Hkv,
                         a.rope ? a.rope + (int64_t)pos * (D / 2) : nullptr, lane);
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------
static int persistent_grid(int64_t warps_of_work) {
  int64_t ctas = (warps_of_work + 7) / 8;
  int64_t cap = (int64_t)num_sms() * 8;
  if (ctas > cap) ctas = cap;
  return (int)(ctas < 1 ? 1 : ctas);
}

cudaError_t launch_slot_mapping(const int32_t *bt, int max_blocks, int batch, int64_t num_blocks,
                                int B, const int32_t *seq, const int32_t *pos, int64_t n,
                                int64_t *out, int32_t *status, cudaStream_t s) {
  int64_t ctas = (n + 255) / 256;
  int64_t cap = (int64_t)num_sms() * 8;
  if (ctas > cap) ctas = cap;
  slot_mapping_kernel<<<(int)ctas, 256, 0, s>>>(bt, max_blocks, batch, num_blocks, B, seq, pos,
                                                n, out, status);
  return cudaGetLastError();
}

template <int D, int DT>
static cudaError_t inject_dt(const InjectArgs &a, cudaStream_t s) {
  int64_t units = (int64_t)a.n_inj * a.n_layers * a.chunk_len;
  inject_kernel<D, DT><<<persistent_grid(units), 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_inject(const InjectArgs &a, int D, int dtype, cudaStream_t s) {
  switch (D * 2 + dtype) {
    case 64 * 2 + 0: return inject_dt<64, 0>(a, s);
    case 64 * 2 + 1: return inject_dt<64, 1>(a, s);
    case 128 * 2 + 0: return inject_dt<128, 0>(a, s);
    case 128 * 2 + 1: return inject_dt<128, 1>(a, s);
    case 256 * 2 + 0: return inject_dt<256, 0>(a, s);
    case 256 * 2 + 1: return inject_dt<256, 1>(a, s);
  }
  return cudaErrorInvalidValue;
}

template <int D, int DT>
static cudaError_t append_dt(const AppendArgs &a, cudaStream_t s) {
  append_kernel<D, DT><<<persistent_grid(a.n), 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_append(const AppendArgs &a, int D, int dtype, cudaStream_t s) {
  switch (D * 2 + dtype) {
    case 64 * 2 + 0: return append_dt<64, 0>(a, s);
    case 64 * 2 + 1: return append_dt<64, 1>(a, s);
    case 128 * 2 + 0: return append_dt<128, 0>(a, s);
    case 128 * 2 + 1: return append_dt<128, 1>(a, s);
    case 256 * 2 + 0: return append_dt<256, 0>(a, s);
    case 256 * 2 + 1: return append_dt<256, 1>(a, s);
  }
  return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// block copy (copy-on-write of a shared block)
// ---------------------------------------------------------------------------
// "LLM Inference: KV Caching", Paged attention: once blocks are first-class, two
// sequences can point at the same one and a block is duplicated only when one of them
// writes; "Inside LLM Inference Engines", PagedAttention item 4 (prefix blocks shared
// read-only, copy-on-write); "Latency Optimization > KV Cache Management" (beams share
// the prompt's pages, only diverging pages are copied). A record is one block of one
// layer of K or V: Hkv*B*D contiguous elements. A CTA copies one record at a time with
// 16-byte vectors, every load of its share issued before the stores (8 vectors per
// thread in flight); the grid is persistent and walks (pair, layer, K|V) records.
constexpr int COPY_THREADS = 256, COPY_VEC = 8;

__global__ void __launch_bounds__(COPY_THREADS) copy_blocks_kernel(CopyBlocksArgs a) {
  const int64_t nrec = a.n * a.n_layers * 2;
  const int64_t nvec = a.rec_bytes / 16;
  int bad = 0;
  for (int64_t r = blockIdx.x; r < nrec; r += gridDim.x) {
    const int kv = (int)(r & 1);
    const int64_t pl = r >> 1;
    const int l = a.layer_begin + (int)(pl % a.n_layers);
    const int64_t i = pl / a.n_layers;
    const int64_t sb = a.src[i], db = a.dst[i];
    if (sb < 0 || sb >= a.num_blocks || db < 0 || db >= a.num_blocks) {
      bad = KVINJ_ST_BAD_BLOCK;
      continue;
    }
    uint8_t *base = kv ? a.v : a.k;
    const uint4 *src = reinterpret_cast<const uint4 *>(base + ((int64_t)l * a.num_blocks + sb) *
                                                                  a.rec_bytes);
    uint4 *dst = reinterpret_cast<uint4 *>(base + ((int64_t)l * a.num_blocks + db) * a.rec_bytes);
    for (int64_t v0 = threadIdx.x; v0 < nvec; v0 += (int64_t)COPY_THREADS * COPY_VEC) {
      uint4 w[COPY_VEC];
#pragma unroll
      for (int k = 0; k < COPY_VEC; ++k) {
        const int64_t v = v0 + (int64_t)k * COPY_THREADS;
        if (v < nvec) w[k] = ld_stream(src + v);
      }
#pragma unroll
      for (int k = 0; k < COPY_VEC; ++k) {
        const int64_t v = v0 + (int64_t)k * COPY_THREADS;
        if (v < nvec) st_global(dst + v, w[k]);
      }
    }
  }
  if (bad && threadIdx.x == 0) report(a.status, bad);
}

cudaError_t launch_copy_blocks(const CopyBlocksArgs &a, cudaStream_t s) {
  const int64_t nrec = a.n * a.n_layers * 2;
  int64_t ctas = (int64_t)num_sms() * 8;
  if (ctas > nrec) ctas = nrec;
  copy_blocks_kernel<<<(int)(ctas < 1 ? 1 : ctas), COPY_THREADS, 0, s>>>(a);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// paged prefill: decode rows of query tokens
// ---------------------------------------------------------------------------
// "InferScale" §3.4 step 4: the query tokens are prefilled over the injected memory. Query
// token i of request r at position p (its K/V already in the cache) attends to r's tokens
// 0..p, which is the decode of a row whose context is p + 1 tokens under r's block table.
// One thread per entry of the rows' tables; the thread of page 0 also writes the row's
// context length and q position.
__global__ void prefill_rows_kernel(const int32_t *__restrict__ bt, int max_blocks, int batch,
                                    int B, const int32_t *__restrict__ seq,
                                    const int32_t *__restrict__ pos, int64_t i0, int rows,
                                    int32_t *row_bt, int32_t *row_ctx, int32_t *row_qpos,
                                    int32_t *status) {
  int bad = 0;
  const int64_t total = (int64_t)rows * max_blocks;
  for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
       e += (int64_t)gridDim.x * blockDim.x) {
    const int i = (int)(e / max_blocks), pg = (int)(e % max_blocks);
    const int r = seq[i0 + i], p = pos[i0 + i];
    const bool ok_r = r >= 0 && r < batch;
    row_bt[e] = ok_r ? bt[(int64_t)r * max_blocks + pg] : -1;
    if (pg == 0) {
      const bool ok_p = p >= 0 && (int64_t)p < (int64_t)max_blocks * B;
      if (!ok_r) bad |= KVINJ_ST_BAD_SEQ;
      else if (!ok_p) bad |= KVINJ_ST_BAD_POS;
      row_ctx[i] = (ok_r && ok_p) ? p + 1 : 0;
      row_qpos[i] = (ok_r && ok_p) ? p : 0;
    }
  }
  if (bad) report(status, bad);
}

cudaError_t launch_prefill_rows(const int32_t *bt, int max_blocks, int batch, int B,
                                const int32_t *seq, const int32_t *pos, int64_t i0, int rows,
                                int32_t *row_bt, int32_t *row_ctx, int32_t *row_qpos,
                                int32_t *status, cudaStream_t s) {
  int64_t ctas = ((int64_t)rows * max_blocks + 255) / 256;
  const int64_t cap = (int64_t)num_sms() * 8;
  if (ctas > cap) ctas = cap;
  prefill_rows_kernel<<<(int)(ctas < 1 ? 1 : ctas), 256, 0, s>>>(
      bt, max_blocks, batch, B, seq, pos, i0, rows, row_bt, row_ctx, row_qpos, status);
  return cudaGetLastError();
}

}  // namespace kvinj
