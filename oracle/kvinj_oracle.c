/*
 * kvinj_oracle.c -- plain, slow, fp64 CPU statement of the paged KV-injection
 * hot path: RoPE, slot mapping, inject (gather pre-RoPE chunk K/V, rotate K at
 * its assigned absolute position, scatter into paged blocks), append, and
 * paged decode attention softmax(q K^T / sqrt(d)) V.
 *
 * TEST INFRASTRUCTURE. This file is the parity oracle for the CUDA library. It
 * shares no code, header, table or constant generator with that library, and
 * only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load it. No product code path calls it.
 *
 * Every function follows its definition literally, in fp64, one output at a
 * time; there is no blocking, fusion or reordering beyond the definition.
 * Sources (web pages, by title and section):
 *   [IS]  "InferScale: GPU-Native KV Injection for Personalized LLM Serving"
 *         §2.3 RoPE (R_p block-diagonal, R_a^T R_b = R_{b-a});
 *         §3.1 keys stored before apply_rotary_pos_emb (pre-RoPE, W_K h);
 *         §3.3 composition: RoPE applied to stored keys at the assigned
 *              positions; §5.1 Theorem 1 (relocation is exact);
 *         §3.4 scatter-copy of composed KV into allocated paged blocks via
 *              the slot mapping; per-fact size 2 x L x c x h x d x b.
 *   [KC]  "LLM Inference: KV Caching" -- "First, what K and V are"
 *         (Attention(Q,K,V) = softmax(QK^T/sqrt d)V), "The fix" (append one
 *         entry per step), "What the cache costs" (kv_cache_bytes),
 *         "Paged attention" (block table, 16-token blocks).
 *   [IE]  "Inside LLM Inference Engines: KV Caching, PagedAttention, and
 *         Continuous Batching" -- M_KV formula; "PagedAttention" page table.
 *   [KM]  "Latency Optimization > KV Cache Management" -- size_KV formula;
 *         pages of 16 tokens read through a page table.
 *
 * Readings where the pages are silent:
 *   - RoPE pairing is rotate-half (i, i + D/2), the convention of the
 *     apply_rotary_pos_emb function [IS §3.1] names; inv_freq_i =
 *     theta^(-2i/D); angle = position * inv_freq_i; all in fp64 (libm).
 *   - Rounding to the 16-bit cache type is round-to-nearest-even, once.
 *   - Decode: the query sits at the position of the newest token and
 *     attends over every cached token of its request (no mask needed for a
 *     single query); GQA groups are consecutive query heads (kv head =
 *     q head / G); scale defaults to 1/sqrt(D).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_BF16 0
#define ORC_FP16 1

/* status bits reported by the oracle (its own; the tests map them) */
#define ORC_ST_CHUNK 1  /* chunk id outside the pool            */
#define ORC_ST_SLOT 2   /* slot outside the paged cache         */
#define ORC_ST_BLOCK 4  /* block-table entry outside the cache  */
#define ORC_ST_POS 8    /* negative position / beyond the table */
#define ORC_ST_CTX 16   /* context length <= 0 or beyond table  */
#define ORC_ST_SEQ 32   /* sequence id outside the batch        */

/* ------------------------------------------------------------------ */
/* 16-bit float formats, written out from the IEEE-754 definition.     */
/* p = significand bits (incl. hidden bit), emin/emax = normal range.   */
/* ------------------------------------------------------------------ */
typedef struct {
  int p, emin, emax;
  uint16_t inf_bits, nan_bits;
} fmt16;

static const fmt16 FMT_BF16 = {8, -126, 127, 0x7F80u, 0x7FC0u};
static const fmt16 FMT_FP16 = {11, -14, 15, 0x7C00u, 0x7E00u};

static const fmt16 *fmt_of(int dtype) { return dtype == ORC_FP16 ? &FMT_FP16 : &FMT_BF16; }

/* round x (fp64) to the nearest representable value, ties to even, and
 * return its bit pattern */
static uint16_t enc16(double x, const fmt16 *f) {
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  if (isnan(x)) return (uint16_t)(sign | f->nan_bits);
  double a = fabs(x);
  if (isinf(a)) return (uint16_t)(sign | f->inf_bits);
  if (a == 0.0) return sign;
  int k;
  frexp(a, &k); /* a = m * 2^k, m in [0.5, 1): a in [2^(k-1), 2^k) */
  int e = k - 1;
  if (e < f->emin) e = f->emin;         /* subnormal range: fixed quantum */
  double q = ldexp(1.0, e - (f->p - 1)); /* spacing of representable values */
  double n = nearbyint(a / q);           /* ties-to-even in the default mode */
  if (n >= ldexp(1.0, f->p)) {           /* rounded up into the next binade */
    e += 1;
    n = ldexp(1.0, f->p - 1);
  }
  if (e > f->emax) return (uint16_t)(sign | f->inf_bits);
  uint32_t ni = (uint32_t)n;
  if (ni < (1u << (f->p - 1))) return (uint16_t)(sign | ni); /* subnormal */
  uint32_t biased = (uint32_t)(e + f->emax);
  return (uint16_t)(sign | (biased << (f->p - 1)) | (ni - (1u << (f->p - 1))));
}

static double dec16(uint16_t b, const fmt16 *f) {
  int mbits = f->p - 1;
  uint32_t emask = (uint32_t)((1u << (15 - mbits)) - 1u);
  uint32_t e = ((uint32_t)b >> mbits) & emask;
  uint32_t m = (uint32_t)b & ((1u << mbits) - 1u);
  double s = (b & 0x8000u) ? -1.0 : 1.0;
  if (e == emask) return m ? NAN : s * INFINITY;
  if (e == 0) return s * ldexp((double)m, f->emin - mbits);
  return s * ldexp((double)((1u << mbits) + m), (int)e - f->emax - mbits);
}

uint16_t orc_encode(double x, int dtype) { return enc16(x, fmt_of(dtype)); }
double orc_decode(uint16_t b, int dtype) { return dec16(b, fmt_of(dtype)); }

void orc_encode_array(const double *x, int64_t n, int dtype, uint16_t *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = enc16(x[i], fmt_of(dtype));
}
void orc_decode_array(const uint16_t *b, int64_t n, int dtype, double *out) {
  for (int64_t i = 0; i < n; ++i) out[i] = dec16(b[i], fmt_of(dtype));
}

/* ------------------------------------------------------------------ */
/* RoPE [IS §2.3]: R_p rotates each pair (x_i, x_{i+D/2}) by the angle  */
/* p * theta^(-2i/D).                                                   */
/* ------------------------------------------------------------------ */
void orc_rope(const double *x, int D, double pos, double theta, double *y) {
  int half = D / 2;
  for (int i = 0; i < half; ++i) {
    double inv_freq = pow(theta, -(2.0 * (double)i) / (double)D);
    double ang = pos * inv_freq;
    double c = cos(ang), s = sin(ang);
    double a = x[i], b = x[i + half];
    y[i] = a * c - b * s;
    y[i + half] = b * c + a * s;
  }
}

/* one stored row -> rotated at `pos` -> rounded once to the cache type */
static void rope_round_row(const uint16_t *in, int D, double pos, double theta, int dtype,
                           uint16_t *out) {
  const fmt16 *f = fmt_of(dtype);
  double *x = (double *)malloc(sizeof(double) * 2 * (size_t)D), *y = x + D;
  for (int d = 0; d < D; ++d) x[d] = dec16(in[d], f);
  orc_rope(x, D, pos, theta, y);
  for (int d = 0; d < D; ++d) out[d] = enc16(y[d], f);
  free(x);
}

void orc_rope_round_rows(const uint16_t *in, int64_t n, int D, const int32_t *positions,
                         double theta, int dtype, uint16_t *out) {
  for (int64_t r = 0; r < n; ++r)
    rope_round_row(in + r * D, D, (double)positions[r], theta, dtype, out + r * D);
}

/* ------------------------------------------------------------------ */
/* KV-cache size [KC "What the cache costs"], [IE], [KM], per-fact      */
/* size [IS §3.4]: 2 * layers * heads * head_dim * tokens * bytes.      */
/* ------------------------------------------------------------------ */
int64_t orc_kv_bytes(int64_t layers, int64_t heads, int64_t head_dim, int64_t tokens,
                     int64_t bytes_per_elem) {
  return 2 * layers * heads * head_dim * tokens * bytes_per_elem;
}

/* ------------------------------------------------------------------ */
/* Slot mapping [IS §3.4; KC "Paged attention"]: token at position p of */
/* request r lives in physical block block_tables[r][p / B] at offset   */
/* p mod B; slot = block * B + offset. Invalid -> slot -1, status bit.  */
/* ------------------------------------------------------------------ */
int32_t orc_slot_mapping(const int32_t *block_tables, int max_blocks, int batch,
                         int64_t num_blocks, const int32_t *seq_ids, const int32_t *positions,
                         int64_t n, int B, int64_t *slot_out) {
  int32_t st = 0;
  for (int64_t i = 0; i < n; ++i) {
    int32_t r = seq_ids[i], p = positions[i];
    slot_out[i] = -1;
    if (r < 0 || r >= batch) { st |= ORC_ST_SEQ; continue; }
    if (p < 0 || p / B >= max_blocks) { st |= ORC_ST_POS; continue; }
    int32_t blk = block_tables[(int64_t)r * max_blocks + p / B];
    if (blk < 0 || blk >= num_blocks) { st |= ORC_ST_BLOCK; continue; }
    slot_out[i] = (int64_t)blk * B + p % B;
  }
  return st;
}

/* cache element offset of row (layer, slot, head); layout
 * cache[L][num_blocks][Hkv][B][D] (one (block, head) page contiguous) */
static int64_t cache_row(int64_t layer, int64_t slot, int64_t h, int64_t num_blocks, int Hkv,
                         int B, int D) {
  int64_t blk = slot / B, off = slot % B;
  return (((layer * num_blocks + blk) * Hkv + h) * B + off) * D;
}

/* ------------------------------------------------------------------ */
/* Inject [IS §3.3, §3.4, §5.1]. Pool layout                            */
/* pool[n_chunks][L][2 (K,V)][c][Hkv][D]: one chunk is one contiguous   */
/* record of 2*L*c*Hkv*D elements, keys stored pre-RoPE. Token t of the */
/* j-th injected chunk takes absolute position start_pos[j] + t and     */
/* slot slot_mapping[j*c + t]; K is rotated there and rounded once, V   */
/* is copied bit for bit.                                               */
/* ------------------------------------------------------------------ */
int32_t orc_inject(const uint16_t *pool, int L, int Hkv, int D, int c, int64_t n_chunks,
                   int dtype, const int32_t *chunk_ids, const int32_t *start_pos,
                   const int64_t *slot_mapping, int n_inj, int layer_begin, int layer_end,
                   double theta, uint16_t *k_cache, uint16_t *v_cache, int64_t num_blocks,
                   int B, int n_threads) {
  int32_t st = 0;
  int64_t row = (int64_t)Hkv * D;
  int64_t kv_half = (int64_t)c * row;
#pragma omp parallel for num_threads(n_threads) reduction(| : st) schedule(dynamic)
  for (int j = 0; j < n_inj; ++j) {
    int32_t id = chunk_ids[j];
    if (id < 0 || id >= n_chunks) { st |= ORC_ST_CHUNK; continue; }
    for (int l = layer_begin; l < layer_end; ++l) {
      const uint16_t *kp = pool + ((int64_t)id * L + l) * 2 * kv_half;
      const uint16_t *vp = kp + kv_half;
      for (int t = 0; t < c; ++t) {
        int64_t slot = slot_mapping[(int64_t)j * c + t];
        int64_t pos = (int64_t)start_pos[j] + t;
        if (slot < 0 || slot >= num_blocks * B) { st |= ORC_ST_SLOT; continue; }
        if (pos < 0) { st |= ORC_ST_POS; continue; }
        for (int h = 0; h < Hkv; ++h) {
          int64_t dst = cache_row(l, slot, h, num_blocks, Hkv, B, D);
          rope_round_row(kp + t * row + (int64_t)h * D, D, (double)pos, theta, dtype,
                         k_cache + dst);
          memcpy(v_cache + dst, vp + t * row + (int64_t)h * D, sizeof(uint16_t) * D);
        }
      }
    }
  }
  return st;
}

/* ------------------------------------------------------------------ */
/* Append [KC "The fix"]: the new token's K (rotated at its position   */
/* unless already rotated) and V are written at its slot in one layer.  */
/* k_new/v_new layout [n][Hkv][D].                                      */
/* ------------------------------------------------------------------ */
int32_t orc_append(uint16_t *k_cache, uint16_t *v_cache, int Hkv, int D, int64_t num_blocks,
                   int B, int dtype, int layer, const uint16_t *k_new, const uint16_t *v_new,
                   const int32_t *positions, const int64_t *slot_mapping, int64_t n,
                   int rotate, double theta) {
  int32_t st = 0;
  for (int64_t i = 0; i < n; ++i) {
    int64_t slot = slot_mapping[i];
    if (slot < 0 || slot >= num_blocks * B) { st |= ORC_ST_SLOT; continue; }
    if (positions[i] < 0) { st |= ORC_ST_POS; continue; }
    for (int h = 0; h < Hkv; ++h) {
      int64_t dst = cache_row(layer, slot, h, num_blocks, Hkv, B, D);
      const uint16_t *ks = k_new + (i * Hkv + h) * D;
      if (rotate)
        rope_round_row(ks, D, (double)positions[i], theta, dtype, k_cache + dst);
      else
        memcpy(k_cache + dst, ks, sizeof(uint16_t) * D);
      memcpy(v_cache + dst, v_new + (i * Hkv + h) * D, sizeof(uint16_t) * D);
    }
  }
  return st;
}

/* ------------------------------------------------------------------ */
/* Copy-on-write of a shared block [KC "Paged attention": a block two   */
/* sequences point at is duplicated when one of them writes; IE          */
/* "PagedAttention" item 4; KM (beams copy only diverging pages)]. For   */
/* each pair i and layer l in [l0, l1): every element of block src[i]    */
/* of layer l, K and V, is copied to block dst[i]. Pairs with an id      */
/* outside the cache are skipped (status bit).                           */
/* ------------------------------------------------------------------ */
int32_t orc_copy_blocks(uint16_t *k_cache, uint16_t *v_cache, int Hkv, int D, int64_t num_blocks,
                        int B, const int32_t *src, const int32_t *dst, int64_t n, int l0,
                        int l1) {
  int32_t st = 0;
  for (int64_t i = 0; i < n; ++i) {
    if (src[i] < 0 || src[i] >= num_blocks || dst[i] < 0 || dst[i] >= num_blocks) {
      st |= ORC_ST_BLOCK;
      continue;
    }
    for (int l = l0; l < l1; ++l)
      for (int h = 0; h < Hkv; ++h)
        for (int t = 0; t < B; ++t) {
          int64_t from = cache_row(l, (int64_t)src[i] * B + t, h, num_blocks, Hkv, B, D);
          int64_t to = cache_row(l, (int64_t)dst[i] * B + t, h, num_blocks, Hkv, B, D);
          for (int d = 0; d < D; ++d) {
            k_cache[to + d] = k_cache[from + d];
            v_cache[to + d] = v_cache[from + d];
          }
        }
  }
  return st;
}

/* ------------------------------------------------------------------ */
/* Textbook attention for one query over a contiguous key/value list    */
/* [KC "First, what K and V are"]: s_j = scale * q.K_j, w = softmax(s)  */
/* (max-subtracted), out = sum_j w_j V_j. Also returns sum_j w_j.        */
/* ------------------------------------------------------------------ */
double orc_attention(const double *q, const double *K, const double *V, int64_t n, int D,
                     double scale, double *out) {
  double *s = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double m = -INFINITY;
  for (int64_t j = 0; j < n; ++j) {
    double acc = 0.0;
    for (int d = 0; d < D; ++d) acc += q[d] * K[j * D + d];
    s[j] = scale * acc;
    if (s[j] > m) m = s[j];
  }
  double z = 0.0;
  for (int64_t j = 0; j < n; ++j) z += exp(s[j] - m);
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  double wsum = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    double w = exp(s[j] - m) / z;
    wsum += w;
    for (int d = 0; d < D; ++d) out[d] += w * V[j * D + d];
  }
  free(s);
  return wsum;
}

/* attention whose inputs are stored 16-bit rows: q is rotated at q_pos
 * (when rotate_q) in fp64, keys and values are taken as stored */
void orc_attention_bits(const uint16_t *q_bits, int rotate_q, double q_pos, double theta,
                        const uint16_t *K_bits, const uint16_t *V_bits, int64_t n, int D,
                        int dtype, double scale, double *out) {
  const fmt16 *f = fmt_of(dtype);
  double *q0 = (double *)malloc(sizeof(double) * 2 * (size_t)D), *q = q0 + D;
  for (int d = 0; d < D; ++d) q0[d] = dec16(q_bits[d], f);
  if (rotate_q) orc_rope(q0, D, q_pos, theta, q);
  else memcpy(q, q0, sizeof(double) * D);
  double *K = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * D);
  double *V = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * D);
  for (int64_t i = 0; i < n * D; ++i) {
    K[i] = dec16(K_bits[i], f);
    V[i] = dec16(V_bits[i], f);
  }
  orc_attention(q, K, V, n, D, scale, out);
  free(K);
  free(V);
  free(q0);
}

/* ------------------------------------------------------------------ */
/* Paged decode [KC "Paged attention"; KM; IE "PagedAttention"]: for    */
/* request r and query head qh (kv head qh / G), token j of the context */
/* is read from block block_tables[r][j / B] at offset j mod B; then    */
/* the textbook attention above. q [batch][Hq][D] pre-RoPE (rotated at  */
/* q_pos[r] when rotate_q). out [batch][Hq][D] fp64, zero for a request */
/* whose context is invalid.                                            */
/* ------------------------------------------------------------------ */
int32_t orc_paged_decode(const uint16_t *k_cache, const uint16_t *v_cache, int Hkv, int D,
                         int64_t num_blocks, int B, int dtype, int layer, int Hq,
                         const uint16_t *q, const int32_t *q_pos, int rotate_q, double theta,
                         const int32_t *block_tables, int max_blocks,
                         const int32_t *context_lens, int batch, double scale, double *out,
                         int n_threads, int window) {
  int32_t st = 0;
  int G = Hq / Hkv;
  if (scale <= 0.0) scale = 1.0 / sqrt((double)D);
#pragma omp parallel for num_threads(n_threads) reduction(| : st) schedule(dynamic)
  for (int64_t rq = 0; rq < (int64_t)batch * Hq; ++rq) {
    int r = (int)(rq / Hq), qh = (int)(rq % Hq), h = qh / G;
    double *o = out + rq * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    int64_t ctx = context_lens[r];
    if (ctx <= 0 || ctx > (int64_t)max_blocks * B) { st |= ORC_ST_CTX; continue; }
    /* sliding window [KC "sliding window attention"]: only the last `window` tokens of the */
    /* context are attended to (window <= 0: all of them); only their blocks are read      */
    int64_t j0 = (window > 0 && ctx > window) ? ctx - window : 0, n = ctx - j0;
    uint16_t *Kr = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)n * D);
    uint16_t *Vr = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)n * D);
    int bad = 0;
    for (int64_t j = j0; j < ctx; ++j) {
      int32_t blk = block_tables[(int64_t)r * max_blocks + j / B];
      if (blk < 0 || blk >= num_blocks) { bad = 1; break; }
      int64_t src = cache_row(layer, (int64_t)blk * B + j % B, h, num_blocks, Hkv, B, D);
      memcpy(Kr + (j - j0) * D, k_cache + src, sizeof(uint16_t) * D);
      memcpy(Vr + (j - j0) * D, v_cache + src, sizeof(uint16_t) * D);
    }
    if (bad) st |= ORC_ST_BLOCK;
    else
      orc_attention_bits(q + rq * D, rotate_q, (double)q_pos[r], theta, Kr, Vr, n, D, dtype,
                         scale, o);
    free(Kr);
    free(Vr);
  }
  return st;
}

/* ------------------------------------------------------------------ */
/* Paged prefill of the query tokens over the injected cache [IS §3.4  */
/* step 4: only the query tokens are prefilled, attending to the       */
/* injected memory as if it had been prefilled]. Query token i belongs */
/* to request seq[i] and sits at position pos[i]; its K/V are already  */
/* in the cache (write, then attend) and it attends causally to the    */
/* request's tokens 0..pos[i]: out[i][qh] = attention of q[i][qh]       */
/* (rotated at pos[i]) over those keys of kv head qh / G.               */
/* ------------------------------------------------------------------ */
int32_t orc_paged_prefill(const uint16_t *k_cache, const uint16_t *v_cache, int Hkv, int D,
                          int64_t num_blocks, int B, int dtype, int layer, int Hq,
                          const uint16_t *q, const int32_t *seq, const int32_t *pos, int64_t n,
                          double theta, const int32_t *block_tables, int max_blocks, int batch,
                          double scale, double *out, int n_threads) {
  int32_t st = 0;
  int G = Hq / Hkv;
  if (scale <= 0.0) scale = 1.0 / sqrt((double)D);
#pragma omp parallel for num_threads(n_threads) reduction(| : st) schedule(dynamic)
  for (int64_t iq = 0; iq < n * Hq; ++iq) {
    int64_t i = iq / Hq;
    int qh = (int)(iq % Hq), h = qh / G;
    double *o = out + iq * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    int r = seq[i];
    int64_t ctx = (int64_t)pos[i] + 1;
    if (r < 0 || r >= batch) { st |= ORC_ST_SEQ; continue; }
    if (pos[i] < 0 || ctx > (int64_t)max_blocks * B) { st |= ORC_ST_POS; continue; }
    uint16_t *Kr = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)ctx * D);
    uint16_t *Vr = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)ctx * D);
    int bad = 0;
    for (int64_t j = 0; j < ctx; ++j) {
      int32_t page_blk = block_tables[(int64_t)r * max_blocks + j / B];
      if (page_blk < 0 || page_blk >= num_blocks) { bad = 1; break; }
      int64_t src = cache_row(layer, (int64_t)page_blk * B + j % B, h, num_blocks, Hkv, B, D);
      memcpy(Kr + j * D, k_cache + src, sizeof(uint16_t) * D);
      memcpy(Vr + j * D, v_cache + src, sizeof(uint16_t) * D);
    }
    if (bad) st |= ORC_ST_BLOCK;
    else
      orc_attention_bits(q + iq * D, 1, (double)pos[i], theta, Kr, Vr, ctx, D, dtype, scale, o);
    free(Kr);
    free(Vr);
  }
  return st;
}

/* ------------------------------------------------------------------ */
/* int8 KV cache [KM "KV cache quantization": int8 halves the cache's  */
/* bytes]. The page fixes no scheme; the reading taken: every stored    */
/* row (token, kv head) is quantized symmetrically on its own, scale    */
/* s = max|x| / 127 (kept as fp32), code q = x / s rounded to nearest   */
/* even and clamped to [-127, 127]; a zero row has s = 0. The value     */
/* read back is q * s.                                                  */
/* ------------------------------------------------------------------ */
void orc_quantize_rows_i8(const uint16_t *in, int64_t n, int D, int dtype, int8_t *q,
                          float *scale) {
  const fmt16 *f = fmt_of(dtype);
  for (int64_t r = 0; r < n; ++r) {
    double amax = 0.0;
    for (int d = 0; d < D; ++d) {
      double x = fabs(dec16(in[r * D + d], f));
      if (x > amax) amax = x;
    }
    float s = (float)(amax / 127.0);
    scale[r] = s;
    for (int d = 0; d < D; ++d) {
      double v = s > 0.0f ? nearbyint(dec16(in[r * D + d], f) / (double)s) : 0.0;
      if (v > 127.0) v = 127.0;
      if (v < -127.0) v = -127.0;
      q[r * D + d] = (int8_t)v;
    }
  }
}

/* paged decode over an int8 cache: as orc_paged_decode, each key and   */
/* value row read back as code * its row's scale. Scales are laid out   */
/* like the rows: [L][num_blocks][Hkv][B].                              */
int32_t orc_paged_decode_i8(const int8_t *kq, const float *ks, const int8_t *vq, const float *vs,
                            int Hkv, int D, int64_t num_blocks, int B, int layer, int Hq,
                            const uint16_t *q, int q_dtype, const int32_t *q_pos, int rotate_q,
                            double theta, const int32_t *block_tables, int max_blocks,
                            const int32_t *context_lens, int batch, double scale, double *out) {
  int32_t st = 0;
  int G = Hq / Hkv;
  const fmt16 *f = fmt_of(q_dtype);
  if (scale <= 0.0) scale = 1.0 / sqrt((double)D);
  for (int64_t rq = 0; rq < (int64_t)batch * Hq; ++rq) {
    int r = (int)(rq / Hq), qh = (int)(rq % Hq), kvh = qh / G;
    double *o = out + rq * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    int64_t ctx = context_lens[r];
    if (ctx <= 0 || ctx > (int64_t)max_blocks * B) { st |= ORC_ST_CTX; continue; }
    double *K = (double *)malloc(sizeof(double) * (size_t)ctx * D);
    double *V = (double *)malloc(sizeof(double) * (size_t)ctx * D);
    int bad = 0;
    for (int64_t j = 0; j < ctx; ++j) {
      int32_t b8 = block_tables[(int64_t)r * max_blocks + j / B];
      if (b8 < 0 || b8 >= num_blocks) { bad = 1; break; }
      int64_t e = cache_row(layer, (int64_t)b8 * B + j % B, kvh, num_blocks, Hkv, B, D);
      for (int d = 0; d < D; ++d) {
        K[j * D + d] = (double)kq[e + d] * (double)ks[e / D];
        V[j * D + d] = (double)vq[e + d] * (double)vs[e / D];
      }
    }
    if (bad) {
      st |= ORC_ST_BLOCK;
    } else {
      double *q0 = (double *)malloc(sizeof(double) * 2 * (size_t)D), *qr = q0 + D;
      for (int d = 0; d < D; ++d) q0[d] = dec16(q[rq * D + d], f);
      if (rotate_q) orc_rope(q0, D, (double)q_pos[r], theta, qr);
      else memcpy(qr, q0, sizeof(double) * D);
      orc_attention(qr, K, V, ctx, D, scale, o);
      free(q0);
    }
    free(K);
    free(V);
  }
  return st;
}

int orc_has_openmp(void) {
#ifdef _OPENMP
  return 1;
#else
  return 0;
#endif
}
