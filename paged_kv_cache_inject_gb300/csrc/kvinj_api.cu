// kvinj_api.cu -- the extern "C" entry points declared in include/kvinj.h:
// argument validation, the fp64 RoPE table, TMA tensor maps and dispatch to
// the kernels. Host code only.
#include <math.h>
#include <string.h>

#include <mutex>

#include "kvinj.h"
#include "kvinj_internal.h"

namespace kvinj {

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev < 0 || dev >= 64) dev = 0;
  if (cache[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = n > 0 ? n : 1;
  }
  return cache[dev];
}

size_t decode_partial_floats(int G, int D) { return (size_t)G * (size_t)(D + 2); }
int decode_max_ctas() { return 2 * num_sms(); }
int decode_head_group(int Hkv) {
  int hg = 8;
  while (hg > 1 && Hkv % hg) hg >>= 1;
  return hg;
}
size_t decode_desc_bytes() {
  return (((size_t)decode_max_ctas() * 8 * sizeof(int)) + 255) & ~size_t(255);
}

}  // namespace kvinj

using namespace kvinj;

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// The address under which the device reads p: p itself for device memory, the mapped
// address of page-locked host memory, nullptr for anything else (pageable host memory,
// an unknown pointer).
const void *device_view(const void *p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();  // the failed query's error is not sticky: clear it
    return nullptr;
  }
  if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) return p;
  if (at.type == cudaMemoryTypeHost) return at.devicePointer;
  return nullptr;
}

bool dtype_ok(int dt) { return dt == KVINJ_BF16 || dt == KVINJ_FP16; }

int check_cache(const kvinj_cache *c, bool decode) {
  if (!c || !c->k || !c->v) return KVINJ_EINVAL;
  if (!aligned16(c->k) || !aligned16(c->v)) return KVINJ_EINVAL;
  if (c->num_layers <= 0 || c->num_kv_heads <= 0 || c->num_blocks <= 0 || c->block_size <= 0)
    return KVINJ_EINVAL;
  if (!dtype_ok(c->dtype)) return KVINJ_EINVAL;
  if (decode) {
    if (c->head_dim != 64 && c->head_dim != 128) return KVINJ_EUNSUPPORTED;
    if (c->block_size != 16) return KVINJ_EUNSUPPORTED;
  } else if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256) {
    return KVINJ_EUNSUPPORTED;
  }
  return KVINJ_OK;
}

int check_rope(const kvinj_rope *r, int D) {
  if (!r) return KVINJ_OK;
  if (!r->table || r->max_pos <= 0 || r->head_dim != D) return KVINJ_EINVAL;
  if (!aligned16(r->table)) return KVINJ_EINVAL;
  return KVINJ_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D view of one cache array: rows of D elements, L*num_blocks*Hkv*16 rows;
// box 64 elements (128 bytes) x HG*16 rows (HG kv heads of one block),
// 128-byte swizzle
int make_cache_map(CUtensorMap *m, void *base, const kvinj_cache *c, int HG) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return KVINJ_ECUDA;
  const uint64_t rows = (uint64_t)c->num_layers * (uint64_t)c->num_blocks *
                        (uint64_t)c->num_kv_heads * (uint64_t)c->block_size;
  cuuint64_t dims[2] = {(cuuint64_t)c->head_dim, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)c->head_dim * 2};
  cuuint32_t box[2] = {64, (cuuint32_t)(c->block_size * HG)};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? KVINJ_OK : KVINJ_ECUDA;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? KVINJ_OK : KVINJ_ECUDA; }

int check_cache_i8(const kvinj_cache_i8 *c) {
  if (!c || !c->k || !c->v || !c->k_scale || !c->v_scale) return KVINJ_EINVAL;
  if (!aligned16(c->k) || !aligned16(c->v) || !aligned16(c->k_scale) || !aligned16(c->v_scale))
    return KVINJ_EINVAL;
  if (c->num_layers <= 0 || c->num_kv_heads <= 0 || c->num_blocks <= 0) return KVINJ_EINVAL;
  if (c->head_dim != 128 || c->block_size != 16) return KVINJ_EUNSUPPORTED;
  if ((int64_t)c->num_layers * c->num_blocks * c->num_kv_heads * 16 >= (int64_t)1 << 31)
    return KVINJ_EUNSUPPORTED;
  return KVINJ_OK;
}

// int8 codes as a 2-D tensor: rows of 128 bytes, box 128 bytes x `rows` rows, 128-byte
// swizzle (the converters read each row's 16-byte chunks at chunk ^ (row % 8))
int make_code_map(CUtensorMap *m, void *base, const kvinj_cache_i8 *c, int rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return KVINJ_ECUDA;
  const uint64_t n = (uint64_t)c->num_layers * (uint64_t)c->num_blocks *
                     (uint64_t)c->num_kv_heads * (uint64_t)c->block_size;
  cuuint64_t dims[2] = {(cuuint64_t)c->head_dim, (cuuint64_t)n};
  cuuint64_t strides[1] = {(cuuint64_t)c->head_dim};
  cuuint32_t box[2] = {128, (cuuint32_t)rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? KVINJ_OK : KVINJ_ECUDA;
}

// a rope for the int8 calls that rotate keys: both tables
int check_rope64(const kvinj_rope *r, int D) {
  int rc = check_rope(r, D);
  if (rc) return rc;
  if (!r->table64 || !aligned16(r->table64)) return KVINJ_EINVAL;
  return KVINJ_OK;
}

}  // namespace

extern "C" {

size_t kvinj_rope_table_bytes(int32_t head_dim, int32_t max_pos) {
  if (head_dim <= 0 || max_pos <= 0) return 0;
  return (size_t)max_pos * (size_t)(head_dim / 2) * 4 * sizeof(float);
}

int kvinj_rope_table_host(double theta, int32_t head_dim, int32_t max_pos, float *out) {
  if (!out || head_dim <= 0 || (head_dim & 1) || max_pos <= 0 || !(theta > 0.0))
    return KVINJ_EINVAL;
  const int half = head_dim / 2;
  for (int i = 0; i < half; ++i) {
    const double inv_freq = pow(theta, -(double)(2 * i) / (double)head_dim);
    for (int64_t p = 0; p < max_pos; ++p) {
      const double ang = (double)p * inv_freq;
      const double c = cos(ang), s = sin(ang);
      const float ch = (float)c, sh = (float)s;
      float *e = out + ((size_t)p * half + i) * 4;
      e[0] = ch;
      e[1] = sh;
      e[2] = (float)(c - (double)ch);
      e[3] = (float)(s - (double)sh);
    }
  }
  return KVINJ_OK;
}

size_t kvinj_rope_table64_bytes(int32_t head_dim, int32_t max_pos) {
  if (head_dim <= 0 || max_pos <= 0) return 0;
  return (size_t)max_pos * (size_t)(head_dim / 2) * 2 * sizeof(double);
}

int kvinj_rope_table64_host(double theta, int32_t head_dim, int32_t max_pos, double *out) {
  if (!out || head_dim <= 0 || (head_dim & 1) || max_pos <= 0 || !(theta > 0.0))
    return KVINJ_EINVAL;
  const int half = head_dim / 2;
  for (int i = 0; i < half; ++i) {
    const double inv_freq = pow(theta, -(double)(2 * i) / (double)head_dim);
    for (int64_t p = 0; p < max_pos; ++p) {
      const double ang = (double)p * inv_freq;
      double *e = out + ((size_t)p * half + i) * 2;
      e[0] = cos(ang);
      e[1] = sin(ang);
    }
  }
  return KVINJ_OK;
}

int kvinj_slot_mapping(const int32_t *block_tables, int32_t max_blocks, int32_t batch,
                       int64_t num_blocks, int32_t block_size, const int32_t *seq_ids,
                       const int32_t *positions, int64_t n, int64_t *slot_out,
                       int32_t *dev_status, kvinj_stream_t stream) {
  if (n < 0) return KVINJ_EINVAL;
  if (n == 0) return KVINJ_OK;
  if (!block_tables || !seq_ids || !positions || !slot_out) return KVINJ_EINVAL;
  if (max_blocks <= 0 || batch <= 0 || num_blocks <= 0 || block_size <= 0) return KVINJ_EINVAL;
  return cuda_rc(launch_slot_mapping(block_tables, max_blocks, batch, num_blocks, block_size,
                                     seq_ids, positions, n, slot_out, dev_status,
                                     (cudaStream_t)stream));
}

int kvinj_inject(const kvinj_pool *pool, const kvinj_cache *cache, const kvinj_rope *rope,
                 const int32_t *chunk_ids, const int32_t *start_pos,
                 const int64_t *slot_mapping, int32_t n_inj, int32_t layer_begin,
                 int32_t layer_end, int32_t *dev_status, kvinj_stream_t stream) {
  int rc = check_cache(cache, false);
  if (rc) return rc;
  if (!pool || !pool->data || !aligned16(pool->data)) return KVINJ_EINVAL;
  if (pool->num_layers != cache->num_layers || pool->num_kv_heads != cache->num_kv_heads ||
      pool->head_dim != cache->head_dim || pool->dtype != cache->dtype ||
      pool->chunk_len <= 0 || pool->num_chunks <= 0)
    return KVINJ_EINVAL;
  if (!rope) return KVINJ_EINVAL;
  if ((rc = check_rope(rope, cache->head_dim))) return rc;
  if (n_inj < 0 || layer_begin < 0 || layer_end > cache->num_layers || layer_begin > layer_end)
    return KVINJ_EINVAL;
  if (n_inj == 0 || layer_begin == layer_end) return KVINJ_OK;
  if (!chunk_ids || !start_pos || !slot_mapping) return KVINJ_EINVAL;
  // device memory, or page-locked host memory read in place over the host link
  const void *pool_dev = device_view(pool->data);
  if (!pool_dev || !aligned16(pool_dev)) return KVINJ_EINVAL;
  InjectArgs a;
  a.pool = static_cast<const uint16_t *>(pool_dev);
  a.L = cache->num_layers;
  a.Hkv = cache->num_kv_heads;
  a.chunk_len = pool->chunk_len;
  a.num_chunks = pool->num_chunks;
  a.k = static_cast<uint16_t *>(cache->k);
  a.v = static_cast<uint16_t *>(cache->v);
  a.num_blocks = cache->num_blocks;
  a.B = cache->block_size;
  a.rope = static_cast<const float4 *>(rope->table);
  a.max_pos = rope->max_pos;
  a.chunk_ids = chunk_ids;
  a.start_pos = start_pos;
  a.slot_mapping = slot_mapping;
  a.n_inj = n_inj;
  a.layer_begin = layer_begin;
  a.n_layers = layer_end - layer_begin;
  a.status = dev_status;
  return cuda_rc(launch_inject(a, cache->head_dim, cache->dtype, (cudaStream_t)stream));
}

int kvinj_copy_blocks(const kvinj_cache *cache, const int32_t *src, const int32_t *dst, int64_t n,
                      int32_t layer_begin, int32_t layer_end, int32_t *dev_status,
                      kvinj_stream_t stream) {
  int rc = check_cache(cache, false);
  if (rc) return rc;
  if (n < 0 || layer_begin < 0 || layer_end > cache->num_layers || layer_begin > layer_end)
    return KVINJ_EINVAL;
  if (n == 0 || layer_begin == layer_end) return KVINJ_OK;
  if (!src || !dst) return KVINJ_EINVAL;
  CopyBlocksArgs a;
  a.k = static_cast<uint8_t *>(cache->k);
  a.v = static_cast<uint8_t *>(cache->v);
  a.num_blocks = cache->num_blocks;
  a.rec_bytes = (int64_t)cache->num_kv_heads * cache->block_size * cache->head_dim * 2;
  a.src = src;
  a.dst = dst;
  a.n = n;
  a.layer_begin = layer_begin;
  a.n_layers = layer_end - layer_begin;
  a.status = dev_status;
  return cuda_rc(launch_copy_blocks(a, (cudaStream_t)stream));
}

int kvinj_append(const kvinj_cache *cache, const kvinj_rope *rope, int32_t layer,
                 const void *k_new, const void *v_new, const int32_t *positions,
                 const int64_t *slot_mapping, int64_t n, int32_t *dev_status,
                 kvinj_stream_t stream) {
  int rc = check_cache(cache, false);
  if (rc) return rc;
  if ((rc = check_rope(rope, cache->head_dim))) return rc;
  if (n < 0 || layer < 0 || layer >= cache->num_layers) return KVINJ_EINVAL;
  if (n == 0) return KVINJ_OK;
  if (!k_new || !v_new || !positions || !slot_mapping) return KVINJ_EINVAL;
  if (!aligned16(k_new) || !aligned16(v_new)) return KVINJ_EINVAL;
  AppendArgs a;
  a.k = static_cast<uint16_t *>(cache->k);
  a.v = static_cast<uint16_t *>(cache->v);
  a.Hkv = cache->num_kv_heads;
  a.num_blocks = cache->num_blocks;
  a.B = cache->block_size;
  a.layer = layer;
  a.k_new = static_cast<const uint16_t *>(k_new);
  a.v_new = static_cast<const uint16_t *>(v_new);
  a.positions = positions;
  a.slot_mapping = slot_mapping;
  a.block_tables = nullptr;
  a.max_blocks = 0;
  a.n = n;
  a.rope = rope ? static_cast<const float4 *>(rope->table) : nullptr;
  a.max_pos = rope ? rope->max_pos : 0;
  a.status = dev_status;
  return cuda_rc(launch_append(a, cache->head_dim, cache->dtype, (cudaStream_t)stream));
}

size_t kvinj_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim) {
  if (batch <= 0 || num_kv_heads <= 0 || num_q_heads <= 0 || num_q_heads % num_kv_heads ||
      head_dim <= 0)
    return 0;
  const int G = num_q_heads / num_kv_heads;
  const int HG = decode_head_group(num_kv_heads);
  return decode_desc_bytes() +
         (size_t)2 * decode_max_ctas() * HG * decode_partial_floats(G, head_dim) * sizeof(float);
}

int kvinj_decode_workspace_init(void *workspace, size_t ws_bytes, kvinj_stream_t stream) {
  if (!workspace && ws_bytes) return KVINJ_EINVAL;
  if (!ws_bytes) return KVINJ_OK;
  return cuda_rc(cudaMemsetAsync(workspace, 0, ws_bytes, (cudaStream_t)stream));
}

namespace {

// shared by the decode entry points: validate, pick the kernel, launch. With
// k_new/v_new (fused append), the token of request r at q_pos[r] is written
// first, at the slot its block table gives.
int decode_call(const kvinj_cache *cache, const kvinj_rope *rope, int32_t layer,
                int32_t num_q_heads, const void *q, const void *k_new, const void *v_new,
                const int32_t *q_pos, const int32_t *block_tables, int32_t max_blocks,
                const int32_t *context_lens, int32_t batch, float scale, void *out,
                void *workspace, size_t ws_bytes, int32_t *dev_status, kvinj_stream_t stream,
                int32_t variant, int32_t ctas, int32_t window = 0, int32_t flags = 0) {
  int rc = check_cache(cache, true);
  if (rc) return rc;
  const int D = cache->head_dim, Hkv = cache->num_kv_heads;
  if ((rc = check_rope(rope, D))) return rc;
  if (layer < 0 || layer >= cache->num_layers || batch < 0 || max_blocks <= 0) return KVINJ_EINVAL;
  if (num_q_heads <= 0 || num_q_heads % Hkv) return KVINJ_EINVAL;
  const int G = num_q_heads / Hkv;
  if (batch == 0) return KVINJ_OK;
  if (!q || !block_tables || !context_lens || !out || !workspace) return KVINJ_EINVAL;
  if (rope && !q_pos) return KVINJ_EINVAL;
  const bool append = k_new != nullptr || v_new != nullptr;
  if (append && (!k_new || !v_new || !q_pos || !aligned16(k_new) || !aligned16(v_new)))
    return KVINJ_EINVAL;
  if (!aligned16(q) || !aligned16(out)) return KVINJ_EINVAL;
  if (variant < 0 || variant > 3) return KVINJ_EINVAL;
  if (flags & ~KVINJ_DECODE_KV_READY) return KVINJ_EINVAL;
  const bool g_pow2_8 = G == 1 || G == 2 || G == 4 || G == 8;
  const bool umma_ok = D == 128 && decode_head_group(Hkv) == 8 && g_pow2_8;
  // automatic: tcgen05 wherever it applies (at G = 8 with units of two blocks of 4 kv
  // heads: 61.6 vs 69.6 us per layer for the mma.sync kernel at 8 requests x 8192
  // tokens, 64 q / 8 kv heads), else mma.sync from G = 4 up, else the FMA kernel
  if (variant == 0) variant = umma_ok ? 3 : (G >= 4 ? 2 : 1);
  if (window < 0) return KVINJ_EINVAL;
  if (window > 0 && variant != 3) return KVINJ_EUNSUPPORTED;  // the tcgen05 kernel only
  if (variant == 1 && !g_pow2_8) return KVINJ_EUNSUPPORTED;
  if (variant == 2 && !(g_pow2_8 || G == 16)) return KVINJ_EUNSUPPORTED;
  if (variant == 3 && !umma_ok) return KVINJ_EUNSUPPORTED;
  if ((int64_t)batch * Hkv * max_blocks >= (int64_t)1 << 31) return KVINJ_EUNSUPPORTED;
  if (batch > 4096) return KVINJ_EUNSUPPORTED;  // per-request prefix sums live in shared memory
  if ((int64_t)cache->num_layers * cache->num_blocks * Hkv * 16 >= (int64_t)1 << 31)
    return KVINJ_EUNSUPPORTED;
  if (ws_bytes < kvinj_decode_workspace_size(batch, num_q_heads, Hkv, D)) return KVINJ_EWORKSPACE;
  const int max_ctas = decode_max_ctas();
  if (ctas < 0 || ctas > max_ctas) return KVINJ_EINVAL;
  if (ctas == 0) ctas = num_sms();

  if (append && variant != 3) {
    // the other kernels take no fused append: the append kernel runs first
    AppendArgs p;
    p.k = static_cast<uint16_t *>(cache->k);
    p.v = static_cast<uint16_t *>(cache->v);
    p.Hkv = Hkv;
    p.num_blocks = cache->num_blocks;
    p.B = cache->block_size;
    p.layer = layer;
    p.k_new = static_cast<const uint16_t *>(k_new);
    p.v_new = static_cast<const uint16_t *>(v_new);
    p.positions = q_pos;
    p.slot_mapping = nullptr;
    p.block_tables = block_tables;
    p.max_blocks = max_blocks;
    p.n = batch;
    p.rope = rope ? static_cast<const float4 *>(rope->table) : nullptr;
    p.max_pos = rope ? rope->max_pos : 0;
    p.status = dev_status;
    if ((rc = cuda_rc(launch_append(p, D, cache->dtype, (cudaStream_t)stream)))) return rc;
  }

  const int HG = decode_head_group(Hkv);
  CUtensorMap tmK, tmV;
  // boxes of HG heads of one block; the tcgen05 kernel at G = 8 places one head of one
  // block per box (its units are two blocks of 4 kv heads)
  const int box_heads = (variant == 3 && G == 8) ? 1 : HG;
  if ((rc = make_cache_map(&tmK, cache->k, cache, box_heads))) return rc;
  if ((rc = make_cache_map(&tmV, cache->v, cache, box_heads))) return rc;

  DecodeArgs a;
  a.q = static_cast<const uint16_t *>(q);
  a.q_pos = q_pos;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.rope = rope ? static_cast<const float4 *>(rope->table) : nullptr;
  a.max_pos = rope ? rope->max_pos : 0;
  a.out = static_cast<uint16_t *>(out);
  a.desc = static_cast<int *>(workspace);
  a.partials = reinterpret_cast<float *>(static_cast<char *>(workspace) + decode_desc_bytes());
  a.k_new = append && variant == 3 ? static_cast<const uint16_t *>(k_new) : nullptr;
  a.v_new = append && variant == 3 ? static_cast<const uint16_t *>(v_new) : nullptr;
  a.k_cache = static_cast<uint16_t *>(cache->k);
  a.v_cache = static_cast<uint16_t *>(cache->v);
  a.status = dev_status;
  a.batch = batch;
  a.Hq = num_q_heads;
  a.Hkv = Hkv;
  a.max_blocks = max_blocks;
  a.layer = layer;
  a.num_blocks = cache->num_blocks;
  a.ctas = ctas;
  a.window = window;
  // early reads of pages, tables and lengths: the tcgen05 kernel only (the others wait
  // for the kernel ahead before anything)
  a.early = (flags & KVINJ_DECODE_KV_READY) && variant == 3 ? 1 : 0;
  const double sc = scale > 0.f ? (double)scale : 1.0 / sqrt((double)D);
  a.scale_log2 = (float)(sc * 1.4426950408889634);
  return cuda_rc(launch_decode(a, tmK, tmV, D, G, HG, cache->dtype, variant, ctas,
                               (cudaStream_t)stream));
}

}  // namespace

int kvinj_paged_decode_ex(const kvinj_cache *cache, const kvinj_rope *rope, int32_t layer,
                          int32_t num_q_heads, const void *q, const int32_t *q_pos,
                          const int32_t *block_tables, int32_t max_blocks,
                          const int32_t *context_lens, int32_t batch, float scale, void *out,
                          void *workspace, size_t ws_bytes, int32_t *dev_status,
                          kvinj_stream_t stream, int32_t variant, int32_t ctas, int32_t flags) {
  return decode_call(cache, rope, layer, num_q_heads, q, nullptr, nullptr, q_pos, block_tables,
                     max_blocks, context_lens, batch, scale, out, workspace, ws_bytes,
                     dev_status, stream, variant, ctas, 0, flags);
}

int kvinj_append_paged_decode_ex(const kvinj_cache *cache, const kvinj_rope *rope,
                                 int32_t layer, int32_t num_q_heads, const void *q,
                                 const void *k_new, const void *v_new, const int32_t *q_pos,
                                 const int32_t *block_tables, int32_t max_blocks,
                                 const int32_t *context_lens, int32_t batch, float scale,
                                 void *out, void *workspace, size_t ws_bytes,
                                 int32_t *dev_status, kvinj_stream_t stream, int32_t variant,
                                 int32_t ctas, int32_t flags) {
  if (!k_new || !v_new) return KVINJ_EINVAL;
  return decode_call(cache, rope, layer, num_q_heads, q, k_new, v_new, q_pos, block_tables,
                     max_blocks, context_lens, batch, scale, out, workspace, ws_bytes,
                     dev_status, stream, variant, ctas, 0, flags);
}

// query tokens per decode launch of a prefill
constexpr int PREFILL_CHUNK = 1024;
static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

namespace {

// the tensor-core prefill takes D = 128 and G in {1, 2, 4, 8}; other shapes run as decode rows
bool prefill_umma_ok(int D, int G) { return D == 128 && (G == 1 || G == 2 || G == 4 || G == 8); }

// workspace of the tensor-core prefill: header, tiles, unit prefix, first tile per CTA,
// partial states
struct PrefillWs {
  size_t hdr, tiles, tile_pre, cta_tile, partials, qhl, bytes;
};
PrefillWs prefill_umma_ws(int64_t n, int Hq) {
  const size_t grid = (size_t)num_sms();
  PrefillWs w;
  w.hdr = 0;
  w.tiles = 256;
  w.tile_pre = w.tiles + align256((size_t)n * 16);
  w.cta_tile = w.tile_pre + align256(((size_t)n + 1) * 4);
  w.partials = w.cta_tile + align256(grid * 4);
  w.qhl = w.partials + align256(2 * grid * prefill_partial_floats() * 4);
  w.bytes = w.qhl + align256((size_t)n * Hq * 128 * 4);
  return w;
}

}  // namespace

size_t kvinj_prefill_workspace_size(int32_t n, int32_t num_q_heads, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t max_blocks) {
  if (n <= 0 || max_blocks <= 0) return 0;
  const size_t dec = kvinj_decode_workspace_size(1, num_q_heads, num_kv_heads, head_dim);
  if (!dec) return 0;
  if (prefill_umma_ok(head_dim, num_q_heads / num_kv_heads)) return prefill_umma_ws(n, num_q_heads).bytes;
  const size_t rows = (size_t)(n < PREFILL_CHUNK ? n : PREFILL_CHUNK);
  return align256(dec) + align256(rows * max_blocks * 4) + 2 * align256(rows * 4);
}

int kvinj_paged_prefill(const kvinj_cache *cache, const kvinj_rope *rope, int32_t layer,
                        int32_t num_q_heads, const void *q, const int32_t *seq_ids,
                        const int32_t *positions, int32_t n, const int32_t *block_tables,
                        int32_t max_blocks, int32_t batch, float scale, void *out,
                        void *workspace, size_t ws_bytes, int32_t *dev_status,
                        kvinj_stream_t stream) {
  int rc = check_cache(cache, true);
  if (rc) return rc;
  if (n < 0 || batch < 0 || max_blocks <= 0 || num_q_heads <= 0) return KVINJ_EINVAL;
  if (n == 0) return KVINJ_OK;
  if (!q || !seq_ids || !positions || !block_tables || !out || !workspace) return KVINJ_EINVAL;
  if (!aligned16(workspace)) return KVINJ_EINVAL;
  const size_t need = kvinj_prefill_workspace_size(n, num_q_heads, cache->num_kv_heads,
                                                   cache->head_dim, max_blocks);
  if (!need) return KVINJ_EINVAL;
  if (ws_bytes < need) return KVINJ_EWORKSPACE;
  const int D = cache->head_dim, Hkv = cache->num_kv_heads;
  if (prefill_umma_ok(D, num_q_heads / Hkv)) {
    if ((rc = check_rope(rope, D))) return rc;
    if (layer < 0 || layer >= cache->num_layers) return KVINJ_EINVAL;
    // unit counts and cache rows stay below 2^31
    if ((int64_t)n * Hkv * ((int64_t)max_blocks * cache->block_size / 128 + 1) >= (int64_t)1 << 31 ||
        (int64_t)cache->num_layers * cache->num_blocks * Hkv * 16 >= (int64_t)1 << 31)
      return KVINJ_EUNSUPPORTED;
    if (!aligned16(q) || !aligned16(out)) return KVINJ_EINVAL;
    const PrefillWs wl = prefill_umma_ws(n, num_q_heads);
    char *w = static_cast<char *>(workspace);
    PrefillArgs p;
    p.q = static_cast<const uint16_t *>(q);
    p.seq = seq_ids;
    p.pos = positions;
    p.block_tables = block_tables;
    p.rope = rope ? static_cast<const float4 *>(rope->table) : nullptr;
    p.max_pos = rope ? rope->max_pos : 0;
    p.out = static_cast<uint16_t *>(out);
    p.status = dev_status;
    p.n = n;
    p.batch = batch;
    p.Hq = num_q_heads;
    p.Hkv = Hkv;
    p.max_blocks = max_blocks;
    p.layer = layer;
    p.num_blocks = cache->num_blocks;
    const double sc = scale > 0.f ? (double)scale : 1.0 / sqrt((double)D);
    p.scale_log2 = (float)(sc * 1.4426950408889634);
    p.grid = num_sms();
    p.hdr = reinterpret_cast<int *>(w + wl.hdr);
    p.tiles = reinterpret_cast<int4 *>(w + wl.tiles);
    p.tile_pre = reinterpret_cast<int *>(w + wl.tile_pre);
    p.cta_tile = reinterpret_cast<int *>(w + wl.cta_tile);
    p.partials = reinterpret_cast<float *>(w + wl.partials);
    p.qhl = reinterpret_cast<uint32_t *>(w + wl.qhl);
    CUtensorMap tmK, tmV;  // boxes of one head of one block
    if ((rc = make_cache_map(&tmK, cache->k, cache, 1))) return rc;
    if ((rc = make_cache_map(&tmV, cache->v, cache, 1))) return rc;
    return cuda_rc(launch_prefill(p, tmK, tmV, num_q_heads / Hkv, cache->dtype,
                                  (cudaStream_t)stream));
  }
  const size_t dec = align256(kvinj_decode_workspace_size(1, num_q_heads, cache->num_kv_heads,
                                                          cache->head_dim));
  const int chunk = n < PREFILL_CHUNK ? n : PREFILL_CHUNK;
  char *w = static_cast<char *>(workspace);
  int32_t *row_bt = reinterpret_cast<int32_t *>(w + dec);
  int32_t *row_ctx = reinterpret_cast<int32_t *>(w + dec + align256((size_t)chunk * max_blocks * 4));
  int32_t *row_qpos = row_ctx + align256((size_t)chunk * 4) / 4;
  const size_t row_bytes = (size_t)num_q_heads * cache->head_dim * 2;
  for (int32_t i0 = 0; i0 < n; i0 += chunk) {
    const int rows = (n - i0) < chunk ? (n - i0) : chunk;
    rc = cuda_rc(launch_prefill_rows(block_tables, max_blocks, batch, cache->block_size, seq_ids,
                                     positions, i0, rows, row_bt, row_ctx, row_qpos, dev_status,
                                     (cudaStream_t)stream));
    if (rc) return rc;
    rc = decode_call(cache, rope, layer, num_q_heads,
                     static_cast<const char *>(q) + (size_t)i0 * row_bytes, nullptr, nullptr,
                     row_qpos, row_bt, max_blocks, row_ctx, rows, scale,
                     static_cast<char *>(out) + (size_t)i0 * row_bytes, workspace, dec, dev_status,
                     stream, 0, 0);
    if (rc) return rc;
  }
  return KVINJ_OK;
}

int kvinj_paged_decode_window(const kvinj_cache *cache, const kvinj_rope *rope, int32_t layer,
                              int32_t num_q_heads, const void *q, const void *k_new,
                              const void *v_new, const int32_t *q_pos,
                              const int32_t *block_tables, int32_t max_blocks,
                              const int32_t *context_lens, int32_t batch, int32_t window,
                              float scale, void *out, void *workspace, size_t ws_bytes,
                              int32_t *dev_status, kvinj_stream_t stream, int32_t flags) {
  if ((k_new == nullptr) != (v_new == nullptr)) return KVINJ_EINVAL;
  return decode_call(cache, rope, layer, num_q_heads, q, k_new, v_new, q_pos, block_tables,
                     max_blocks, context_lens, batch, scale, out, workspace, ws_bytes,
                     dev_status, stream, 0, 0, window, flags);
}

int kvinj_append_paged_decode(const kvinj_cache *cache, const kvinj_rope *rope, int32_t layer,
                              int32_t num_q_heads, const void *q, const void *k_new,
                              const void *v_new, const int32_t *q_pos,
                              const int32_t *block_tables, int32_t max_blocks,
                              const int32_t *context_lens, int32_t batch, float scale,
                              void *out, void *workspace, size_t ws_bytes, int32_t *dev_status,
                              kvinj_stream_t stream) {
  return kvinj_append_paged_decode_ex(cache, rope, layer, num_q_heads, q, k_new, v_new, q_pos,
                                      block_tables, max_blocks, context_lens, batch, scale, out,
                                      workspace, ws_bytes, dev_status, stream, 0, 0, 0);
}

int kvinj_paged_decode(const kvinj_cache *cache, const kvinj_rope *rope, int32_t layer,
                       int32_t num_q_heads, const void *q, const int32_t *q_pos,
                       const int32_t *block_tables, int32_t max_blocks,
                       const int32_t *context_lens, int32_t batch, float scale, void *out,
                       void *workspace, size_t ws_bytes, int32_t *dev_status,
                       kvinj_stream_t stream) {
  return kvinj_paged_decode_ex(cache, rope, layer, num_q_heads, q, q_pos, block_tables,
                               max_blocks, context_lens, batch, scale, out, workspace, ws_bytes,
                               dev_status, stream, 0, 0, 0);
}

int kvinj_inject_i8(const kvinj_pool *pool, const kvinj_cache_i8 *cache, const kvinj_rope *rope,
                    const int32_t *chunk_ids, const int32_t *start_pos,
                    const int64_t *slot_mapping, int32_t n_inj, int32_t layer_begin,
                    int32_t layer_end, int32_t *dev_status, kvinj_stream_t stream) {
  int rc = check_cache_i8(cache);
  if (rc) return rc;
  if (!pool || !pool->data || !aligned16(pool->data) || !dtype_ok(pool->dtype)) return KVINJ_EINVAL;
  if (pool->num_layers != cache->num_layers || pool->num_kv_heads != cache->num_kv_heads ||
      pool->head_dim != cache->head_dim || pool->chunk_len <= 0 || pool->num_chunks <= 0)
    return KVINJ_EINVAL;
  if ((rc = check_rope64(rope, cache->head_dim))) return rc;
  if (n_inj < 0 || layer_begin < 0 || layer_end > cache->num_layers || layer_begin > layer_end)
    return KVINJ_EINVAL;
  if (n_inj == 0 || layer_begin == layer_end) return KVINJ_OK;
  if (!chunk_ids || !start_pos || !slot_mapping) return KVINJ_EINVAL;
  const void *pool_dev = device_view(pool->data);
  if (pool_dev != pool->data) return KVINJ_EINVAL;  // device memory only
  I8Args a = {};
  a.src_k = static_cast<const uint16_t *>(pool->data);
  a.L = cache->num_layers;
  a.Hkv = cache->num_kv_heads;
  a.chunk_len = pool->chunk_len;
  a.num_chunks = pool->num_chunks;
  a.k = static_cast<int8_t *>(cache->k);
  a.v = static_cast<int8_t *>(cache->v);
  a.ks = cache->k_scale;
  a.vs = cache->v_scale;
  a.num_blocks = cache->num_blocks;
  a.B = cache->block_size;
  a.rope = static_cast<const float4 *>(rope->table);
  a.rope64 = static_cast<const double2 *>(rope->table64);
  a.max_pos = rope->max_pos;
  a.chunk_ids = chunk_ids;
  a.start_pos = start_pos;
  a.slot_mapping = slot_mapping;
  a.n = n_inj;
  a.layer_begin = layer_begin;
  a.n_layers = layer_end - layer_begin;
  a.status = dev_status;
  return cuda_rc(launch_inject_i8(a, pool->dtype, (cudaStream_t)stream));
}

int kvinj_append_i8(const kvinj_cache_i8 *cache, const kvinj_rope *rope, int32_t dtype,
                    int32_t layer, const void *k_new, const void *v_new,
                    const int32_t *positions, const int64_t *slot_mapping, int64_t n,
                    int32_t *dev_status, kvinj_stream_t stream) {
  int rc = check_cache_i8(cache);
  if (rc) return rc;
  if (!dtype_ok(dtype)) return KVINJ_EINVAL;
  if (rope && (rc = check_rope64(rope, cache->head_dim))) return rc;
  if (n < 0 || layer < 0 || layer >= cache->num_layers) return KVINJ_EINVAL;
  if (n == 0) return KVINJ_OK;
  if (!k_new || !v_new || !positions || !slot_mapping) return KVINJ_EINVAL;
  if (!aligned16(k_new) || !aligned16(v_new)) return KVINJ_EINVAL;
  I8Args a = {};
  a.src_k = static_cast<const uint16_t *>(k_new);
  a.src_v = static_cast<const uint16_t *>(v_new);
  a.Hkv = cache->num_kv_heads;
  a.k = static_cast<int8_t *>(cache->k);
  a.v = static_cast<int8_t *>(cache->v);
  a.ks = cache->k_scale;
  a.vs = cache->v_scale;
  a.num_blocks = cache->num_blocks;
  a.B = cache->block_size;
  a.rope = rope ? static_cast<const float4 *>(rope->table) : nullptr;
  a.rope64 = rope ? static_cast<const double2 *>(rope->table64) : nullptr;
  a.max_pos = rope ? rope->max_pos : 0;
  a.positions = positions;
  a.slot_mapping = slot_mapping;
  a.n = n;
  a.layer = layer;
  a.status = dev_status;
  return cuda_rc(launch_append_i8(a, dtype, (cudaStream_t)stream));
}

int kvinj_paged_decode_i8(const kvinj_cache_i8 *cache, const kvinj_rope *rope, int32_t dtype,
                          int32_t layer, int32_t num_q_heads, const void *q, const void *k_new,
                          const void *v_new, const int32_t *q_pos, const int32_t *block_tables,
                          int32_t max_blocks, const int32_t *context_lens, int32_t batch,
                          float scale, void *out, void *workspace, size_t ws_bytes,
                          int32_t *dev_status, kvinj_stream_t stream, int32_t ctas) {
  int rc = check_cache_i8(cache);
  if (rc) return rc;
  if (!dtype_ok(dtype)) return KVINJ_EINVAL;
  const int D = cache->head_dim, Hkv = cache->num_kv_heads;
  const bool append = k_new != nullptr || v_new != nullptr;
  if (append && (!k_new || !v_new || !q_pos || !aligned16(k_new) || !aligned16(v_new)))
    return KVINJ_EINVAL;
  if (rope) {
    if ((rc = append ? check_rope64(rope, D) : check_rope(rope, D))) return rc;
  }
  if (layer < 0 || layer >= cache->num_layers || batch < 0 || max_blocks <= 0) return KVINJ_EINVAL;
  if (num_q_heads <= 0 || num_q_heads % Hkv) return KVINJ_EINVAL;
  const int G = num_q_heads / Hkv;
  if (batch == 0) return KVINJ_OK;
  if (!q || !block_tables || !context_lens || !out || !workspace) return KVINJ_EINVAL;
  if (rope && !q_pos) return KVINJ_EINVAL;
  if (!aligned16(q) || !aligned16(out)) return KVINJ_EINVAL;
  if (decode_head_group(Hkv) != 8 || !(G == 1 || G == 2 || G == 4 || G == 8))
    return KVINJ_EUNSUPPORTED;
  if ((int64_t)batch * Hkv * max_blocks >= (int64_t)1 << 31) return KVINJ_EUNSUPPORTED;
  if (batch > 4096) return KVINJ_EUNSUPPORTED;
  if (ws_bytes < kvinj_decode_workspace_size(batch, num_q_heads, Hkv, D)) return KVINJ_EWORKSPACE;
  const int max_ctas = decode_max_ctas();
  if (ctas < 0 || ctas > max_ctas) return KVINJ_EINVAL;
  if (ctas == 0) ctas = num_sms();
  CUtensorMap tmK, tmV;
  const int box_rows = G == 8 ? 16 : 128;  // one head of one block, or a block of 8 heads
  if ((rc = make_code_map(&tmK, cache->k, cache, box_rows))) return rc;
  if ((rc = make_code_map(&tmV, cache->v, cache, box_rows))) return rc;
  DecodeArgs a = {};
  a.q = static_cast<const uint16_t *>(q);
  a.q_pos = q_pos;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.rope = rope ? static_cast<const float4 *>(rope->table) : nullptr;
  a.rope64 = rope ? static_cast<const double2 *>(rope->table64) : nullptr;
  a.max_pos = rope ? rope->max_pos : 0;
  a.out = static_cast<uint16_t *>(out);
  a.desc = static_cast<int *>(workspace);
  a.partials = reinterpret_cast<float *>(static_cast<char *>(workspace) + decode_desc_bytes());
  a.k_new = static_cast<const uint16_t *>(k_new);
  a.v_new = static_cast<const uint16_t *>(v_new);
  a.k_cache = static_cast<uint16_t *>(cache->k);
  a.v_cache = static_cast<uint16_t *>(cache->v);
  a.k_scale = cache->k_scale;
  a.v_scale = cache->v_scale;
  a.status = dev_status;
  a.batch = batch;
  a.Hq = num_q_heads;
  a.Hkv = Hkv;
  a.max_blocks = max_blocks;
  a.layer = layer;
  a.num_blocks = cache->num_blocks;
  a.ctas = ctas;
  a.window = 0;
  a.early = 0;
  const double sc = scale > 0.f ? (double)scale : 1.0 / sqrt((double)D);
  a.scale_log2 = (float)(sc * 1.4426950408889634);
  return cuda_rc(launch_decode_i8(a, tmK, tmV, G, dtype, ctas, (cudaStream_t)stream));
}

int64_t kvinj_kv_bytes(int32_t layers, int32_t heads, int32_t head_dim, int64_t tokens,
                       int32_t bytes_per_elem) {
  return (int64_t)2 * layers * heads * head_dim * tokens * bytes_per_elem;
}

const char *kvinj_strerror(int code) {
  switch (code) {
    case KVINJ_OK: return "ok";
    case KVINJ_EINVAL: return "invalid argument (null or misaligned pointer, inconsistent shape)";
    case KVINJ_EUNSUPPORTED: return "unsupported shape for this build";
    case KVINJ_EWORKSPACE: return "decode workspace too small";
    case KVINJ_ECUDA: return "CUDA launch or driver call failed";
  }
  return "unknown error code";
}

}  // extern "C"

namespace kvinj {
cudaError_t launch_decode(const DecodeArgs &a, const CUtensorMap &tmK, const CUtensorMap &tmV,
                          int D, int G, int HG, int dtype, int variant, int ctas, cudaStream_t s) {
  if (variant == 1) return launch_decode_ffma(a, tmK, tmV, D, G, HG, dtype, ctas, s);
  if (variant == 2) return launch_decode_mma(a, tmK, tmV, D, G, HG, dtype, ctas, s);
  if (variant == 3) return launch_decode_umma(a, tmK, tmV, D, G, HG, dtype, ctas, s);
  return cudaErrorInvalidValue;
}
}  // namespace kvinj
