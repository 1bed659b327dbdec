// kvinj_internal.h -- declarations shared by the library's translation units
// (kernel argument blocks and launchers). Not part of the C ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace kvinj {

int num_sms();  // SMs of the current device (cached per device)

struct InjectArgs {
  const uint16_t *pool;
  int L, Hkv, chunk_len;
  int64_t num_chunks;
  uint16_t *k, *v;
  int64_t num_blocks;
  int B;
  const float4 *rope;
  int max_pos;
  const int32_t *chunk_ids, *start_pos;
  const int64_t *slot_mapping;
  int n_inj, layer_begin, n_layers;
  int32_t *status;
};

struct AppendArgs {
  uint16_t *k, *v;
  int Hkv;
  int64_t num_blocks;
  int B, layer;
  const uint16_t *k_new, *v_new;
  const int32_t *positions;
  const int64_t *slot_mapping;  // nullptr: slot of token i from its block table (below)
  const int32_t *block_tables;  // [n][max_blocks] when slot_mapping is nullptr
  int max_blocks;
  int64_t n;
  const float4 *rope;  // nullptr: keys already rotated
  int max_pos;
  int32_t *status;
};

struct DecodeArgs {
  const uint16_t *q;           // [batch][Hq][D]
  const int32_t *q_pos;        // [batch]
  const int32_t *block_tables; // [batch][max_blocks]
  const int32_t *context_lens; // [batch]
  const float4 *rope;          // nullptr: q already rotated
  int max_pos;
  uint16_t *out;               // [batch][Hq][D]
  float *partials;             // [2*max_ctas][HG][G][D+2]
  int *desc;                   // [max_ctas][8] reserved
  const uint16_t *k_new, *v_new;  // [batch][Hkv][D]: token appended at q_pos (nullptr: none)
  uint16_t *k_cache, *v_cache;    // cache bases, written by the append
  int32_t *status;
  int batch, Hq, Hkv, max_blocks, layer;
  int ctas;                    // split-K grid size (set for the combine pass)
  int window;                  // sliding window in tokens (0: the whole context)
  int early;                   // context lengths, q positions, block tables and cache pages
                               // may be read before the dependency wait (KVINJ_DECODE_KV_READY)
  int64_t num_blocks;
  float scale_log2;            // softmax scale times log2(e)
  // int8 cache (kvinj_paged_decode_i8): k_cache/v_cache hold int8 codes, these the scales
  float *k_scale, *v_scale;    // [L][num_blocks][Hkv][16]
  const double2 *rope64;       // fp64 table: exact rounding of the appended key
};

// decode workspace: descriptors first, then the partial slots
size_t decode_partial_floats(int G, int D);  // floats per head of a slot
int decode_max_ctas();                        // slots/2 the workspace is sized for
size_t decode_desc_bytes();

// int8 cache (inject / append): codes [L][NB][Hkv][B][D], scales [L][NB][Hkv][B]
struct I8Args {
  const uint16_t *src_k, *src_v;  // inject: the pool; append: k_new, v_new [n][Hkv][D]
  int L, Hkv, chunk_len;          // inject: pool geometry
  int64_t num_chunks;
  int8_t *k, *v;
  float *ks, *vs;
  int64_t num_blocks;
  int B;
  const float4 *rope;             // nullptr (append only): keys stored as given
  const double2 *rope64;          // fp64 {cos, sin} of the same positions
  int max_pos;
  const int32_t *chunk_ids, *start_pos;  // inject
  const int32_t *positions;              // append
  const int64_t *slot_mapping;
  int64_t n;                      // inject: injected chunks; append: tokens
  int layer, layer_begin, n_layers;
  int32_t *status;
};

cudaError_t launch_slot_mapping(const int32_t *bt, int max_blocks, int batch, int64_t num_blocks,
                                int B, const int32_t *seq, const int32_t *pos, int64_t n,
                                int64_t *out, int32_t *status, cudaStream_t s);
cudaError_t launch_inject(const InjectArgs &a, int D, int dtype, cudaStream_t s);
cudaError_t launch_append(const AppendArgs &a, int D, int dtype, cudaStream_t s);

// block copies for copy-on-write: record (pair i, layer, K|V) of rec_bytes bytes each
struct CopyBlocksArgs {
  uint8_t *k, *v;            // cache base pointers
  int64_t num_blocks;        // physical blocks per layer
  int64_t rec_bytes;         // bytes of one block of one layer: Hkv * B * D * 2
  const int32_t *src, *dst;  // [n] physical block ids
  int64_t n;
  int layer_begin, n_layers;
  int32_t *status;
};
cudaError_t launch_copy_blocks(const CopyBlocksArgs &a, cudaStream_t s);

// paged prefill as decode rows: row i of a chunk is query token i0 + i, with its request's
// block-table row, context length position + 1 (0 when the token is invalid) and q position
// paged prefill on the tensor cores (kvinj_prefill.cu): D = 128, G in {1, 2, 4, 8}
struct PrefillArgs {
  const uint16_t *q;            // [n][Hq][D]
  const int32_t *seq, *pos;     // [n]
  const int32_t *block_tables;  // [batch][max_blocks]
  const float4 *rope;           // nullptr: q already rotated
  int max_pos;
  uint16_t *out;                // [n][Hq][D]
  int32_t *status;
  int n, batch, Hq, Hkv, max_blocks, layer;
  int64_t num_blocks;
  float scale_log2;             // softmax scale times log2(e)
  int grid;                     // CTAs of the tensor-core pass
  // workspace: {tiles, units}; tiles [n] {request, first token, tokens, largest position};
  // tile_pre [n + 1]; cta_tile [grid]; partial states [2 grid][prefill_partial_floats()];
  // prepared query rows
  int *hdr;
  int4 *tiles;
  int *tile_pre, *cta_tile;
  float *partials;
  uint32_t *qhl;                // [n][Hq][128]: prepared query rows (hi words, then lo)
};
size_t prefill_partial_floats();
cudaError_t launch_prefill(const PrefillArgs &a, const CUtensorMap &tmK, const CUtensorMap &tmV,
                           int G, int dtype, cudaStream_t s);

cudaError_t launch_prefill_rows(const int32_t *bt, int max_blocks, int batch, int B,
                                const int32_t *seq, const int32_t *pos, int64_t i0, int rows,
                                int32_t *row_bt, int32_t *row_ctx, int32_t *row_qpos,
                                int32_t *status, cudaStream_t s);
// HG: kv heads per work unit (a power of two <= 8 dividing Hkv)
int decode_head_group(int Hkv);
cudaError_t launch_decode_ffma(const DecodeArgs &a, const CUtensorMap &tmK,
                               const CUtensorMap &tmV, int D, int G, int HG, int dtype, int ctas,
                               cudaStream_t s);
cudaError_t launch_decode_mma(const DecodeArgs &a, const CUtensorMap &tmK, const CUtensorMap &tmV,
                              int D, int G, int HG, int dtype, int ctas, cudaStream_t s);
// tcgen05 kernel: D = 128, HG = 8, G in {1, 2, 4, 8}
cudaError_t launch_decode_umma(const DecodeArgs &a, const CUtensorMap &tmK,
                               const CUtensorMap &tmV, int D, int G, int HG, int dtype, int ctas,
                               cudaStream_t s);
// int8 cache: inject / append (D = 128), decode (tcgen05; D = 128, HG = 8, G in {1,2,4,8})
cudaError_t launch_inject_i8(const I8Args &a, int dtype, cudaStream_t s);
cudaError_t launch_append_i8(const I8Args &a, int dtype, cudaStream_t s);
cudaError_t launch_decode_i8(const DecodeArgs &a, const CUtensorMap &tmK, const CUtensorMap &tmV,
                             int G, int dtype, int ctas, cudaStream_t s);
// variant: 1 = CUDA-core FMA kernel, 2 = mma.sync kernel, 3 = tcgen05 kernel
cudaError_t launch_decode(const DecodeArgs &a, const CUtensorMap &tmK, const CUtensorMap &tmV,
                          int D, int G, int HG, int dtype, int variant, int ctas, cudaStream_t s);

}  // namespace kvinj
