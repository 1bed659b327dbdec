/*
 * kvinj.h -- C ABI of the GB300 (sm_103a) paged KV-injection library.
 *
 * The hot path of InferScale-style KV injection and of paged GQA decode:
 *
 *   kvinj_slot_mapping  position -> physical slot through a block table
 *   kvinj_inject        gather pre-RoPE chunk K/V from a resident chunk pool,
 *                       rotate K at each chunk's assigned absolute position,
 *                       scatter K/V into a request's paged blocks
 *   kvinj_append        write one step's new K (rotated) / V at their slots
 *   kvinj_paged_decode  softmax(q K^T * scale) V of one query per request over
 *                       the request's non-contiguous blocks (split-K over the
 *                       context, online softmax, in-kernel combine)
 *
 * and around them: the append fused into the decode (kvinj_append_paged_decode),
 * a sliding-window decode (kvinj_paged_decode_window), block copies for
 * copy-on-write (kvinj_copy_blocks), the paged prefill of query tokens
 * (kvinj_paged_prefill), an int8 cache (kvinj_inject_i8, kvinj_append_i8,
 * kvinj_paged_decode_i8), and a decode with no caller workspace
 * (kvinj_paged_decode_static).
 *
 * Sources (web pages, by title and section):
 *   "InferScale: GPU-Native KV Injection for Personalized LLM Serving":
 *     §2.3 RoPE, R_a^T R_b = R_{b-a}; §3.1 keys stored before RoPE;
 *     §3.3 composition applies RoPE to stored keys at the assigned positions;
 *     §3.4 the worker scatter-copies the composed KV into the allocated paged
 *     blocks via the slot mapping; per-fact size 2*L*c*h*d*b; §5.1 Theorem 1.
 *   "LLM Inference: KV Caching": "First, what K and V are" (attention),
 *     "The fix" (append), "What the cache costs", "Paged attention".
 *   "Inside LLM Inference Engines: KV Caching, PagedAttention, and Continuous
 *     Batching": "PagedAttention: Virtual Memory for LLM Generation".
 *   "Latency Optimization > KV Cache Management": 16-token pages read through
 *     a page table by the attention kernel.
 *
 * Conventions (all entry points):
 *   - Every array pointer is a DEVICE pointer owned by the caller, except the
 *     outputs of kvinj_rope_table_host / kvinj_rope_table64_host (host memory)
 *     and a chunk pool in page-locked host memory. The library allocates and
 *     frees nothing and keeps no global state (the one exception is the fixed
 *     device scratch array of kvinj_paged_decode_static), and never
 *     synchronises: each call enqueues its kernels on `stream` (NULL = legacy
 *     default stream) and returns. Results are visible to later work on the
 *     same stream.
 *   - Return value: KVINJ_OK, or an error code for arguments the host can see
 *     are wrong (nothing is launched then), or KVINJ_ECUDA when a launch fails.
 *   - Bad indices that only the device sees (chunk id, slot, block-table
 *     entry, position, context length) never trap: the element is skipped (a
 *     decode page with a bad block is treated as masked) and a KVINJ_ST_* bit
 *     is OR-ed into *dev_status (a caller-owned device int32; may be NULL).
 *   - Element types: 16-bit floats (bf16 or fp16), the same type for pool,
 *     cache, queries and outputs (an int8 cache holds codes and fp32 scales
 *     instead; see kvinj_cache_i8). Pointers to 16-bit data must be 16-byte
 *     aligned.
 *   - Layouts (row-major, innermost last):
 *       pool   [num_chunks][L][2 (K, V)][chunk_len][Hkv][D]   keys pre-RoPE
 *       cache  k, v: [L][num_blocks][Hkv][block_size][D]       keys post-RoPE
 *              (one (block, head) page of block_size*D elements is contiguous)
 *       rope table (device) float4 [max_pos][D/2]
 *              {cos_hi, sin_hi, cos_lo, sin_lo}: cos/sin of pos*theta^(-2i/D)
 *              evaluated in fp64 and split into two fp32 parts (hi + lo).
 *   - RoPE is rotate-half: pair (x_i, x_{i+D/2}) turns by pos*theta^(-2i/D).
 */
#ifndef KVINJ_H
#define KVINJ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *kvinj_stream_t; /* a cudaStream_t */

/* element types */
#define KVINJ_BF16 0
#define KVINJ_FP16 1

/* return codes */
#define KVINJ_OK 0
#define KVINJ_EINVAL 1       /* null/misaligned pointer, inconsistent shapes */
#define KVINJ_EUNSUPPORTED 2 /* a shape this build has no kernel for */
#define KVINJ_EWORKSPACE 3   /* decode workspace too small */
#define KVINJ_ECUDA 4        /* a CUDA launch or driver call failed */

/* device status bits, OR-ed into *dev_status */
#define KVINJ_ST_BAD_CHUNK 0x01 /* chunk id outside [0, num_chunks)            */
#define KVINJ_ST_BAD_SLOT 0x02  /* slot outside [0, num_blocks*block_size)     */
#define KVINJ_ST_BAD_BLOCK 0x04 /* block-table entry outside [0, num_blocks)   */
#define KVINJ_ST_BAD_POS 0x08   /* position < 0, beyond the table or the rope table */
#define KVINJ_ST_BAD_CTX 0x10   /* context length <= 0 or > max_blocks*block_size */
#define KVINJ_ST_BAD_SEQ 0x20   /* sequence id outside [0, batch)              */
#define KVINJ_ST_TIMEOUT 0x40   /* a pipeline wait gave up (kernel returned early) */
#define KVINJ_ST_INTERNAL 0x80  /* a launch precondition failed on the device (no output) */

/* paged KV cache of one model (all layers) */
typedef struct {
  int32_t num_layers;   /* L */
  int32_t num_kv_heads; /* Hkv */
  int32_t head_dim;     /* D: 64 or 128 (inject/append also 256) */
  int32_t block_size;   /* tokens per block (decode: 16) */
  int64_t num_blocks;   /* physical blocks per layer */
  int32_t dtype;        /* KVINJ_BF16 / KVINJ_FP16 */
  void *k;              /* device [L][num_blocks][Hkv][block_size][D] */
  void *v;              /* device, same layout */
} kvinj_cache;

/* resident pool of pre-RoPE memory chunks ("facts"), one contiguous record
 * of 2*L*chunk_len*Hkv*D elements per chunk (InferScale §3.4). The pool may
 * also live in page-locked host memory (InferScale §6.7, Table 6: the store
 * kept in pinned host DRAM when GPU memory cannot hold it): the inject kernel
 * then reads the records in place over the host link (no staging copy). */
typedef struct {
  int32_t num_layers, num_kv_heads, head_dim;
  int32_t chunk_len;  /* c: tokens per chunk */
  int64_t num_chunks; /* records in the pool */
  int32_t dtype;
  const void *data; /* [num_chunks][L][2][c][Hkv][D]: device memory, or host
                       memory page-locked with cudaHostAlloc / cudaHostRegister
                       (mapped); other host memory is refused (KVINJ_EINVAL) */
} kvinj_pool;

/* RoPE table on the device (layout in the header comment) */
typedef struct {
  const void *table; /* device float4 [max_pos][head_dim/2] */
  int32_t max_pos;   /* positions 0 .. max_pos-1 are valid */
  int32_t head_dim;
  const void *table64; /* optional device double2 [max_pos][head_dim/2] {cos, sin} in fp64
                          (kvinj_rope_table64_host); required by the int8 calls that rotate
                          keys, ignored by the others (may be NULL there) */
} kvinj_rope;

/* int8 paged KV cache ("Latency Optimization > KV Cache Management", KV cache
 * quantization: int8 halves the cache's bytes). Every stored row (one token of
 * one kv head, D values) is quantized on its own, symmetrically: scale s =
 * max|x| / 127 as fp32, code = x / s rounded to nearest even and clamped to
 * [-127, 127] (a row of zeros: s = 0, codes 0); the value read back is code *
 * s. Keys are rotated first and rounded once to the call's 16-bit type, then
 * quantized, so a code is the one the fp64 rotation rounded to 16 bits
 * quantizes to. Same block structure as kvinj_cache; head_dim 128, block_size
 * 16. */
typedef struct {
  int32_t num_layers;   /* L */
  int32_t num_kv_heads; /* Hkv */
  int32_t head_dim;     /* D: 128 */
  int32_t block_size;   /* 16 */
  int64_t num_blocks;   /* physical blocks per layer */
  void *k;              /* device int8 codes [L][num_blocks][Hkv][block_size][D], 16-byte aligned */
  void *v;              /* device int8 codes, same layout */
  float *k_scale;       /* device fp32 [L][num_blocks][Hkv][block_size], 16-byte aligned */
  float *v_scale;       /* device fp32, same layout */
} kvinj_cache_i8;

/* Bytes of the RoPE table for (head_dim, max_pos): max_pos*head_dim/2*16. */
size_t kvinj_rope_table_bytes(int32_t head_dim, int32_t max_pos);

/* Fill a HOST buffer of kvinj_rope_table_bytes() bytes: entry [p][i] holds
 * cos and sin of p * theta^(-2i/head_dim), computed in fp64, each split into
 * hi = (float)x and lo = (float)(x - hi). The caller copies it to the device.
 * InferScale §2.3 (R_p) and §3.3 (RoPE applied with the rotary tables).
 * Returns KVINJ_EINVAL for head_dim odd or <= 0, max_pos <= 0, theta <= 0,
 * out == NULL. */
int kvinj_rope_table_host(double theta, int32_t head_dim, int32_t max_pos, float *out);

/* Bytes of the fp64 RoPE table for (head_dim, max_pos): max_pos*head_dim/2*16. */
size_t kvinj_rope_table64_bytes(int32_t head_dim, int32_t max_pos);

/* Fill a HOST buffer of kvinj_rope_table64_bytes() bytes: entry [p][i] holds
 * {cos, sin} of p * theta^(-2i/head_dim) in fp64 -- the values the float
 * table's hi/lo pairs are split from. The int8 calls use it where a rotated key
 * lies so close to a 16-bit rounding boundary that only the fp64 rotation
 * decides its rounding. Errors as kvinj_rope_table_host. */
int kvinj_rope_table64_host(double theta, int32_t head_dim, int32_t max_pos, double *out);

/* Slot mapping (InferScale §3.4; "LLM Inference: KV Caching", Paged
 * attention): slot_out[i] = block_tables[seq_ids[i]][positions[i] / B] * B
 * + positions[i] % B, as int64. block_tables [batch][max_blocks] int32.
 * Invalid sequence id, position or block entry: slot_out[i] = -1 and the
 * matching KVINJ_ST_* bit. n == 0 is a no-op. */
int kvinj_slot_mapping(const int32_t *block_tables, int32_t max_blocks, int32_t batch,
                       int64_t num_blocks, int32_t block_size, const int32_t *seq_ids,
                       const int32_t *positions, int64_t n, int64_t *slot_out,
                       int32_t *dev_status, kvinj_stream_t stream);

/* Inject (InferScale §3.3, §3.4, §5.1). For the j-th injected chunk
 * (j < n_inj) and each layer l in [layer_begin, layer_end): token t < c of
 * pool record chunk_ids[j] takes absolute position start_pos[j] + t and slot
 * slot_mapping[j*c + t]; its K row of each kv head is rotated there (fp32
 * arithmetic with the fp64-derived table, rounded once, nearest-even) and
 * written to k[l][slot / B][h][slot % B][:], its V row is copied bit for bit
 * to v. Pool and cache must agree in L, Hkv, D and dtype; rope->head_dim ==
 * D. Chunks that overlap in slots race (undefined which one wins). A pool in
 * page-locked host memory gives the same results; the call reads it through
 * its device mapping. KVINJ_EINVAL when pool->data is neither device memory
 * nor page-locked host memory mapped into the device's address space. */
int kvinj_inject(const kvinj_pool *pool, const kvinj_cache *cache, const kvinj_rope *rope,
                 const int32_t *chunk_ids, const int32_t *start_pos,
                 const int64_t *slot_mapping, int32_t n_inj, int32_t layer_begin,
                 int32_t layer_end, int32_t *dev_status, kvinj_stream_t stream);

/* Copy-on-write of shared blocks ("LLM Inference: KV Caching", Paged attention:
 * two sequences may point at one physical block, which is duplicated only when
 * one of them writes; "Inside LLM Inference Engines", PagedAttention: prefix
 * blocks shared read-only with copy-on-write; "Latency Optimization > KV Cache
 * Management": beams share the prompt's pages, diverging pages are copied).
 * For i < n and each layer l in [layer_begin, layer_end): block src[i] of layer
 * l is copied to block dst[i] of layer l, in k and in v (Hkv*B*D elements each,
 * bit for bit). src, dst: device int32 [n] physical block ids; the caller then
 * points the writer's block-table entry at dst[i]. A pair with an id outside
 * [0, num_blocks) is skipped and sets KVINJ_ST_BAD_BLOCK. Pairs whose dst is
 * another pair's src or dst race (undefined which copy wins). n == 0 or an
 * empty layer range is a no-op. */
int kvinj_copy_blocks(const kvinj_cache *cache, const int32_t *src, const int32_t *dst, int64_t n,
                      int32_t layer_begin, int32_t layer_end, int32_t *dev_status,
                      kvinj_stream_t stream);

/* Append ("LLM Inference: KV Caching", The fix): token i < n writes
 * k_new[i][h][:] rotated at positions[i] (copied as given when rope == NULL)
 * and v_new[i][h][:] to layer `layer` at slot_mapping[i].
 * k_new, v_new: device [n][Hkv][D] in the cache dtype. */
int kvinj_append(const kvinj_cache *cache, const kvinj_rope *rope, int32_t layer,
                 const void *k_new, const void *v_new, const int32_t *positions,
                 const int64_t *slot_mapping, int64_t n, int32_t *dev_status,
                 kvinj_stream_t stream);

/* Workspace bytes kvinj_paged_decode needs for this shape on the current
 * device: per CTA slot of the split-K grid, two partial softmax states (m, l
 * and the unnormalised output of every query head of a head group), after a
 * small reserved header. */
size_t kvinj_decode_workspace_size(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim);

/* Zero a decode workspace. Optional: every decode call writes each partial
 * state before reading it, so the workspace may hold anything; zeroing only
 * makes its contents deterministic for inspection. */
int kvinj_decode_workspace_init(void *workspace, size_t ws_bytes, kvinj_stream_t stream);

/* Paged decode attention ("LLM Inference: KV Caching", attention and Paged
 * attention; "Latency Optimization > KV Cache Management"). For request r <
 * batch and query head qh < Hq (kv head h = qh / (Hq/Hkv), consecutive
 * groups), with C = context_lens[r] tokens at positions 0..C-1 read from
 * k/v[layer][block_tables[r][p / 16]][h][p % 16]:
 *   q' = R_{q_pos[r]} q[r][qh]   (q taken as given when rope == NULL)
 *   out[r][qh] = sum_p softmax_p(scale * q'.K_p) V_p
 * scale <= 0 means 1/sqrt(D). q, out: device [batch][Hq][D] in the cache
 * dtype; accumulation is fp32. workspace: device, at least
 * kvinj_decode_workspace_size() bytes, any contents; calls sharing one
 * workspace must not overlap in time. A request with an invalid context gets
 * a zero output and KVINJ_ST_BAD_CTX; a block-table entry out of range is
 * treated as a block of masked tokens (KVINJ_ST_BAD_BLOCK); a q position out
 * of the RoPE table leaves q unrotated (KVINJ_ST_BAD_POS). Requires
 * block_size 16, D 64 or 128, Hq % Hkv == 0, Hq/Hkv <= 16 and batch <= 4096
 * (KVINJ_EUNSUPPORTED otherwise). Launches two kernels on `stream`: the
 * split-K pass and the combine of the segments it cut (a programmatic
 * dependent of the first). */
int kvinj_paged_decode(const kvinj_cache *cache, const kvinj_rope *rope, int32_t layer,
                       int32_t num_q_heads, const void *q, const int32_t *q_pos,
                       const int32_t *block_tables, int32_t max_blocks,
                       const int32_t *context_lens, int32_t batch, float scale, void *out,
                       void *workspace, size_t ws_bytes, int32_t *dev_status,
                       kvinj_stream_t stream);

/* Paged prefill of query tokens over the injected cache ("InferScale" §3.4 step
 * 4: only the query tokens are prefilled, attending to the injected memory as
 * if it had been prefilled). Query token i < n of request seq_ids[i] sits at
 * positions[i]; its K/V must already be in the cache (kvinj_append), and it
 * attends causally to the request's tokens 0..positions[i]: out[i][qh] =
 * softmax(scale * q' . K) V over those tokens of kv head qh / G, q' = q[i][qh]
 * rotated at positions[i] (as given when rope == NULL). q, out: device
 * [n][num_q_heads][D] in the cache dtype; seq_ids, positions: device int32 [n];
 * block_tables: device int32 [batch][max_blocks].
 * At D = 128 and G = num_q_heads / num_kv_heads in {1, 2, 4, 8} the tokens run
 * on the tensor cores in tiles: up to 128 / G consecutive entries of the token
 * list that belong to one request share a tile, whose 128 rows are (token,
 * query head of a kv head's group) pairs, and K and V of the request's tokens
 * 0 .. (the tile's largest position) are read once per tile and kv head, in
 * chunks of 128 keys, each row masking the keys after its own position. List
 * the tokens of a request next to each other: a token whose neighbours belong
 * to other requests gets a tile of its own. Other shapes run as decode rows
 * (context positions[i] + 1 under the request's table, launches of up to 1024
 * tokens: every row reads its own causal context). workspace: device,
 * kvinj_prefill_workspace_size() bytes, 16-byte aligned, any contents; one call
 * at a time per workspace. A request id outside [0, batch) or a position
 * outside the table gives a zero output row, KVINJ_ST_BAD_SEQ or
 * KVINJ_ST_BAD_POS, and KVINJ_ST_BAD_CTX; a block-table entry outside the cache
 * is read as a page of masked keys (KVINJ_ST_BAD_BLOCK); a position outside the
 * RoPE table leaves that query unrotated (KVINJ_ST_BAD_POS). */
size_t kvinj_prefill_workspace_size(int32_t n, int32_t num_q_heads, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t max_blocks);
int kvinj_paged_prefill(const kvinj_cache *cache, const kvinj_rope *rope, int32_t layer,
                        int32_t num_q_heads, const void *q, const int32_t *seq_ids,
                        const int32_t *positions, int32_t n, const int32_t *block_tables,
                        int32_t max_blocks, int32_t batch, float scale, void *out,
                        void *workspace, size_t ws_bytes, int32_t *dev_status,
                        kvinj_stream_t stream);

/* Paged decode under a sliding window ("LLM Inference: KV Caching", sliding
 * window attention: a token attends only to the last W tokens). As
 * kvinj_paged_decode (with the new token's append fused when k_new and v_new
 * are both given, as kvinj_append_paged_decode), except that the query of
 * request r attends to the tokens [max(0, ctx - window), ctx) of its context
 * only; window == 0 is the whole context. Only blocks holding an attended token
 * are read, so table entries of pages wholly before the window may hold
 * anything. Runs the tcgen05 kernel: D = 128, Hkv a multiple of 8, G in
 * {1, 2, 4, 8}, else KVINJ_EUNSUPPORTED; window < 0 or only one of k_new,
 * v_new: KVINJ_EINVAL. `flags`: KVINJ_DECODE_* bits, as kvinj_paged_decode_ex. */
int kvinj_paged_decode_window(const kvinj_cache *cache, const kvinj_rope *rope, int32_t layer,
                              int32_t num_q_heads, const void *q, const void *k_new,
                              const void *v_new, const int32_t *q_pos,
                              const int32_t *block_tables, int32_t max_blocks,
                              const int32_t *context_lens, int32_t batch, int32_t window,
                              float scale, void *out, void *workspace, size_t ws_bytes,
                              int32_t *dev_status, kvinj_stream_t stream, int32_t flags);

/* Flags of the decode calls that take them (bit set).
 *
 * KVINJ_DECODE_KV_READY: the cache pages of `layer`, the block tables, the
 * context lengths and the q positions this call reads were all written by work
 * enqueued on the stream before the previous decode call on that stream, and
 * that previous call appended into another layer (or appended nothing). The
 * split-K pass may then start reading them -- its prologue and its first
 * stages of K/V pages -- while the kernels ahead of it on the stream are still
 * running (it is launched as their programmatic dependent); it waits for them
 * before it reads q, k_new, v_new or the RoPE table and before it writes
 * anything. Typical use: every layer's call of a decode step but the first
 * after the inject, when q comes from the kernel just before. Applies to the
 * tcgen05 kernel (ignored by the others); without it every read waits. A
 * call that sets it when the condition does not hold may read stale pages. */
#define KVINJ_DECODE_KV_READY 1

/* Same as kvinj_paged_decode with an explicit kernel choice (G = Hq/Hkv):
 * variant 0 = automatic (3 where it applies, else 2 for G >= 4, else 1),
 * 1 = CUDA-core FMA kernel (G in {1, 2, 4, 8}),
 * 2 = warp-level mma.sync kernel (G in {1, 2, 4, 8, 16}),
 * 3 = tcgen05 kernel, accumulators in tensor memory (D = 128, Hkv a multiple
 *     of 8, G in {1, 2, 4, 8}).
 * KVINJ_EUNSUPPORTED when the chosen variant does not cover the shape.
 * `ctas` > 0 overrides the grid size (1 .. 2 x the SM count, the workspace
 * slots); 0 = one CTA per SM. `flags`: KVINJ_DECODE_* bits (0: none; an
 * unknown bit is KVINJ_EINVAL). */
int kvinj_paged_decode_ex(const kvinj_cache *cache, const kvinj_rope *rope, int32_t layer,
                          int32_t num_q_heads, const void *q, const int32_t *q_pos,
                          const int32_t *block_tables, int32_t max_blocks,
                          const int32_t *context_lens, int32_t batch, float scale, void *out,
                          void *workspace, size_t ws_bytes, int32_t *dev_status,
                          kvinj_stream_t stream, int32_t variant, int32_t ctas, int32_t flags);

/* Append, then decode ([KC] "The fix": each step appends the new token's K
 * and V, then attends over the whole cache). For request r < batch the token
 * at position q_pos[r] -- k_new/v_new[r]: device [batch][Hkv][D], pre-RoPE K --
 * is written to k/v[layer] at slot block_tables[r][q_pos/16]*16 + q_pos%16
 * (K rotated at q_pos, as kvinj_append does), and then every request is
 * decoded exactly as kvinj_paged_decode does; context_lens[r] counts the new
 * token (normally q_pos[r] + 1). Same result as kvinj_append with those slots
 * followed by kvinj_paged_decode. With the tcgen05 kernel the append is part
 * of the split-K pass: the CTA that reads the new token's block writes it
 * first (no separate append launch). q_pos must be
 * given; a position outside the RoPE table or a block-table entry outside the
 * cache is skipped and flagged (KVINJ_ST_BAD_POS / KVINJ_ST_BAD_BLOCK).
 * Other arguments and errors as kvinj_paged_decode / kvinj_paged_decode_ex. */
int kvinj_append_paged_decode(const kvinj_cache *cache, const kvinj_rope *rope, int32_t layer,
                              int32_t num_q_heads, const void *q, const void *k_new,
                              const void *v_new, const int32_t *q_pos,
                              const int32_t *block_tables, int32_t max_blocks,
                              const int32_t *context_lens, int32_t batch, float scale,
                              void *out, void *workspace, size_t ws_bytes, int32_t *dev_status,
                              kvinj_stream_t stream);
int kvinj_append_paged_decode_ex(const kvinj_cache *cache, const kvinj_rope *rope,
                                 int32_t layer, int32_t num_q_heads, const void *q,
                                 const void *k_new, const void *v_new, const int32_t *q_pos,
                                 const int32_t *block_tables, int32_t max_blocks,
                                 const int32_t *context_lens, int32_t batch, float scale,
                                 void *out, void *workspace, size_t ws_bytes,
                                 int32_t *dev_status, kvinj_stream_t stream, int32_t variant,
                                 int32_t ctas, int32_t flags);

/* Paged decode without a caller-provided workspace (no counterpart in the
 * pages; an addition of this library). For callers that cannot allocate
 * device memory where they run -- an engine hook or plugin that must not call
 * cudaMalloc (it can implicitly synchronize the device), a process whose
 * memory is already handed out, a path that must not fail on memory
 * pressure mid-request. Same arguments and results as kvinj_paged_decode
 * (bit for bit: the same kernels on the same inputs); the scratch is a fixed
 * device array of KVINJ_STATIC_SCRATCH_BYTES that every GPU loading this
 * library holds until exit. Nothing is allocated or freed.
 * Size limit: a shape is accepted when kvinj_decode_workspace_size() for it
 * on the current device is at most KVINJ_STATIC_SCRATCH_BYTES, i.e. when
 *   header + 2 * (2 * SMs) * HG * G * (D + 2) * 4 <= 24 MiB
 * with HG = the largest power of two <= 8 dividing Hkv, G = Hq / Hkv and SMs
 * the device's multiprocessor count (the header is 2 * SMs * 32 bytes rounded
 * up to 256). On a 152-SM GPU that admits G = 8 at D = 128 with HG = 8 (about
 * 19.3 MiB); the requirement grows with the SM count, so call
 * kvinj_decode_workspace_size() to test a shape on the device at hand; larger
 * shapes return KVINJ_EWORKSPACE.
 * Every call looks up the array's device address in the current context (it
 * is not cached, so a device reset cannot leave a stale address behind); the
 * first call on a device may load the library's device code there. All calls
 * on a device share the array and leave their contents in it; nothing in it
 * needs to start at zero, but calls whose kernels overlap on the GPU race on
 * it. */
#define KVINJ_STATIC_SCRATCH_BYTES (24u << 20)
int kvinj_paged_decode_static(const kvinj_cache *cache, const kvinj_rope *rope, int32_t layer,
                              int32_t num_q_heads, const void *q, const int32_t *q_pos,
                              const int32_t *block_tables, int32_t max_blocks,
                              const int32_t *context_lens, int32_t batch, float scale, void *out,
                              int32_t *dev_status, kvinj_stream_t stream);

/* Inject into an int8 cache: as kvinj_inject, except that each rotated K row
 * (rounded once to the pool's 16-bit type, exactly as the fp64 rotation would
 * be) and each V row is stored as int8 codes with one fp32 scale (see
 * kvinj_cache_i8). rope->table64 is required (KVINJ_EINVAL without it). The
 * pool must be device memory; D = 128. */
int kvinj_inject_i8(const kvinj_pool *pool, const kvinj_cache_i8 *cache, const kvinj_rope *rope,
                    const int32_t *chunk_ids, const int32_t *start_pos,
                    const int64_t *slot_mapping, int32_t n_inj, int32_t layer_begin,
                    int32_t layer_end, int32_t *dev_status, kvinj_stream_t stream);

/* Append into an int8 cache: as kvinj_append (k_new, v_new: device [n][Hkv][D]
 * of 16-bit type `dtype`), the rows quantized as kvinj_inject_i8 stores them.
 * With rope, rope->table64 is required; rope == NULL stores K as given. */
int kvinj_append_i8(const kvinj_cache_i8 *cache, const kvinj_rope *rope, int32_t dtype,
                    int32_t layer, const void *k_new, const void *v_new,
                    const int32_t *positions, const int64_t *slot_mapping, int64_t n,
                    int32_t *dev_status, kvinj_stream_t stream);

/* Paged decode over an int8 cache ("Latency Optimization > KV Cache
 * Management", KV cache quantization; attention as kvinj_paged_decode), with
 * the new token's append fused when k_new and v_new are both given (as
 * kvinj_append_paged_decode: the token at q_pos[r] is quantized and written at
 * the slot its block table gives, then attended to). Each key and value is
 * read back as code * scale of its row: scores are (q' . codes) * k_scale,
 * and each probability is multiplied by its row's v_scale before the sum over
 * values, in fp32. q, out, k_new, v_new are of 16-bit type `dtype`
 * ([batch][Hq][D], [batch][Hkv][D]). Workspace as kvinj_paged_decode
 * (kvinj_decode_workspace_size). Requires D = 128, block_size 16, Hkv a
 * multiple of 8 and G = Hq/Hkv in {1, 2, 4, 8} (KVINJ_EUNSUPPORTED
 * otherwise); `ctas` as in kvinj_paged_decode_ex; with a fused append and a
 * rope, rope->table64 is required. Two kernels on `stream`: the split-K pass
 * (which turns each unit's codes into tensor-core operands on the chip) and
 * the combine pass. */
int kvinj_paged_decode_i8(const kvinj_cache_i8 *cache, const kvinj_rope *rope, int32_t dtype,
                          int32_t layer, int32_t num_q_heads, const void *q, const void *k_new,
                          const void *v_new, const int32_t *q_pos, const int32_t *block_tables,
                          int32_t max_blocks, const int32_t *context_lens, int32_t batch,
                          float scale, void *out, void *workspace, size_t ws_bytes,
                          int32_t *dev_status, kvinj_stream_t stream, int32_t ctas);

/* KV bytes of `tokens` tokens: 2 * layers * heads * head_dim * tokens *
 * bytes_per_elem ("LLM Inference: KV Caching", What the cache costs). */
int64_t kvinj_kv_bytes(int32_t layers, int32_t heads, int32_t head_dim, int64_t tokens,
                       int32_t bytes_per_elem);

/* Static description of a return code. */
const char *kvinj_strerror(int code);

#ifdef __cplusplus
}
#endif

#endif /* KVINJ_H */
