/*
 * pa_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously-correct CPU restatement of what the batched
 * paged-attention path computes.  It exists to check the CUDA library and is
 * used only by the tests, the smoke check and the benchmark's CPU-baseline leg.
 * Nothing in the product path may link, load or call it, and it shares no code,
 * header or constant table with the CUDA sources.
 *
 * Arithmetic is fp32 throughout, as the pages fix it (the managed C# reference
 * and the CPU MLA-prefill reference both accumulate in float).  Softmax is the
 * deliberately different TWO-PASS form (max over the visible row, then the
 * exp-sum, then the weighted sum) that the vllm.cpp "cpu_mla_prefill.cpp" page
 * prescribes for its oracle (MlaPrefillAttentionKernel, "PASS 1"/"PASS 2"),
 * so that a bug in the GPU's streaming rescale cannot hide behind a matching
 * reference.
 *
 * Sources, by page and section:
 *  [MPA]  TensorSharp "ManagedPagedAttention.cs": class summary (layouts),
 *         Forward (visible range), ComputeSingleQueryAttention (block lookup,
 *         dot-then-scale, empty context -> zeros), WriteKvToPagedPool.
 *  [TL]   tinyllm "Paged attention for decode in C": 2.1 (where position j
 *         lives), 2.2 (visible set, GQA map), 2.6 (validation), 3 (worked example).
 *  [V2]   "paged_attention_v2_pytorch.py": partitions of 512 aligned to 0,
 *         (max_logit, exp_sum, tmp_output) partials, log-sum-exp reduction.
 *  [MLA]  vllm.cpp "cpu_mla_prefill.cpp": two-pass softmax, LSE layout
 *         [num_heads, num_tokens], GatherMlaCacheKernel, MergeAttnStatesKernel.
 *
 * Mutants: oracle_set_mutant(n) plants one known mistake (n > 0) so the tests can
 * show each pin fails on it.  0 (the default) is the correct oracle.
 */
#include <float.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Status codes of the tinyllm interface ([TL] section 4: TL_EINVAL, TL_ESHAPE;
 * section 2.6: TL_EUNSUPPORTED). */
enum { ORC_OK = 0, ORC_EINVAL = 1, ORC_ESHAPE = 2, ORC_EUNSUPPORTED = 3 };
/* Element types the pages use for q / K / V / out ([MLA] LoadF/StoreF), and fp8 (e4m3) K/V
 * pools ([V2] kv_cache_dtype "fp8" with k_scale / v_scale; [TL] "Going further": fp8 KV, with
 * scales per head or per block -- the *_per_head functions take one scale per kv head, the
 * *_per_block ones one per (pool block, kv head)). */
enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_FP8 = 2 };

static int g_mutant = 0;
#define MUTANT(n) (g_mutant == (n))

void oracle_set_mutant(int n) { g_mutant = n; }
int oracle_get_mutant(void) { return g_mutant; }

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* ---- element codecs ------------------------------------------------------ */

/* bfloat16 is the top half of an IEEE binary32: widening is exact. */
static float bf16_bits_to_float(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* binary32 -> bfloat16, round to nearest, ties to even; NaN stays NaN. */
static uint16_t float_to_bf16_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

/* fp8 e4m3 ("fn": no infinities): sign, 4 exponent bits with bias 7, 3 mantissa bits.
 * Exponent 0 holds the subnormals m * 2^-9; S.1111.111 is NaN; the largest finite value is
 * 1.75 * 2^8 = 448.  Widening is exact. */
static float fp8_bits_to_float(uint8_t b) {
  const int sign = b >> 7, e = (b >> 3) & 15, m = b & 7;
  float v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexpf((float)m, -9);
  else
    v = ldexpf(1.0f + (float)m / 8.0f, e - (MUTANT(70) ? 8 : 7)); /* s70: wrong bias */
  return sign ? -v : v;
}

/* binary32 -> e4m3: saturate to +-448, then round to nearest, ties to even, over the
 * representable values (subnormals included); NaN stays NaN. */
static uint8_t float_to_fp8_bits(float f) {
  if (isnan(f)) return 0x7f;
  const uint8_t sign = signbit(f) ? 0x80 : 0x00;
  float a = fabsf(f);
  if (a > 448.0f) a = 448.0f;
  /* candidates: the 127 non-negative finite codes are monotone in value */
  int lo = 0, hi = 126;
  while (lo < hi) { /* the largest code whose value is <= a */
    int mid = (lo + hi + 1) / 2;
    if (fp8_bits_to_float((uint8_t)mid) <= a) lo = mid; else hi = mid - 1;
  }
  int code = lo;
  if (code < 126) {
    float below = fp8_bits_to_float((uint8_t)code), above = fp8_bits_to_float((uint8_t)(code + 1));
    float d0 = a - below, d1 = above - a;
    if (MUTANT(71)) d1 = INFINITY; /* s71: truncation instead of rounding */
    if (d1 < d0 || (d1 == d0 && (code & 1))) code += 1;
  }
  return (uint8_t)(sign | code);
}

static float load_elem(const void* base, int dt, int64_t i) {
  if (dt == ORC_BF16) return bf16_bits_to_float(((const uint16_t*)base)[i]);
  if (dt == ORC_FP8) return fp8_bits_to_float(((const uint8_t*)base)[i]);
  return ((const float*)base)[i];
}

static void store_elem(void* base, int dt, int64_t i, float v) {
  if (dt == ORC_BF16)
    ((uint16_t*)base)[i] = float_to_bf16_bits(v);
  else if (dt == ORC_FP8)
    ((uint8_t*)base)[i] = float_to_fp8_bits(v);
  else
    ((float*)base)[i] = v;
}

static int elem_bytes(int dt) { return dt == ORC_FP8 ? 1 : dt == ORC_BF16 ? 2 : 4; }
/* q / out / new K-V rows: fp32 or bf16; pools: those or fp8 */
static int dtype_ok(int dt) { return dt == ORC_F32 || dt == ORC_BF16; }
static int pool_dtype_ok(int dt) { return dtype_ok(dt) || dt == ORC_FP8; }

/* ---- where position j of a sequence lives ([TL] 2.1; [MPA] kvBaseOffset) ---
 * Logical block j / b of the sequence is physical block table[j / b]; the row
 * inside it is j mod b.  Pool layout is [numBlocks, blockSize, numKvHeads, D]. */
static int64_t pool_row_offset(const int32_t* table_row, int64_t j, int32_t block_size,
                               int32_t num_kv_heads, int32_t head_dim, int32_t kv_head) {
  int64_t logical = j / block_size;
  int64_t slot_in_block = j % block_size;
  int64_t block_id = MUTANT(3) ? logical : (int64_t)table_row[logical]; /* s03 */
  int64_t head = MUTANT(4) ? 0 : kv_head;                                /* s04 */
  return ((block_id * block_size + slot_in_block) * num_kv_heads + head) * head_dim;
}

/* ---- slot mapping ---------------------------------------------------------
 * The physical slot of token t, which sits at position positions[t] of its
 * sequence s: slot = table[s][pos / b] * b + pos mod b ([MPA] class summary,
 * "slot = blockId * blockSize + offsetInBlock"; [TL] 2.1). */
int oracle_slot_mapping(const int32_t* query_start_loc, const int32_t* positions,
                        const int32_t* block_tables, int32_t num_seqs, int32_t max_blocks,
                        int32_t block_size, int64_t num_blocks, int32_t* slot_out) {
  if (!query_start_loc || !positions || !block_tables || !slot_out) return ORC_EINVAL;
  if (block_size <= 0 || max_blocks <= 0) return ORC_ESHAPE;
  int status = ORC_OK;
  for (int32_t s = 0; s < num_seqs; ++s) {
    const int32_t* row = block_tables + (int64_t)s * max_blocks;
    for (int32_t t = query_start_loc[s]; t < query_start_loc[s + 1]; ++t) {
      int32_t pos = positions[t];
      if (pos < 0 || pos / block_size >= max_blocks || row[pos / block_size] < 0 ||
          row[pos / block_size] >= num_blocks) {
        slot_out[t] = -1;
        status = ORC_EINVAL;
        continue;
      }
      int32_t blk = row[pos / block_size];
      int32_t off = pos % block_size;
      slot_out[t] = MUTANT(20) ? off * block_size + blk : blk * block_size + off;
    }
  }
  return status;
}

/* ---- scatter of the new tokens' K and V ([MPA] WriteKvToPagedPool) --------
 * k, v: [T, Hkv, D]; pools [NB, b, Hkv, D].  Every slot is checked before the
 * first byte is written; the copy itself is a plain serial loop over tokens, so
 * duplicate slots resolve last-writer-wins. */
int oracle_reshape_and_cache(const void* k, const void* v, void* k_blocks, void* v_blocks,
                             const int32_t* slot_mapping, int64_t num_tokens,
                             int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                             int64_t num_blocks, int32_t kv_dtype) {
  if (!k || !v || !k_blocks || !v_blocks || !slot_mapping) return ORC_EINVAL;
  if (!pool_dtype_ok(kv_dtype)) return ORC_EUNSUPPORTED;
  if (num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0) return ORC_ESHAPE;
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0 || slot >= num_blocks * block_size) return ORC_EINVAL;
  }
  const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * elem_bytes(kv_dtype);
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    int64_t blk = slot / block_size;
    int64_t off = slot % block_size;
    int64_t dst = (blk * block_size + off) * row_bytes;
    memcpy((char*)k_blocks + dst, (const char*)k + t * row_bytes, (size_t)row_bytes);
    memcpy((char*)v_blocks + dst, MUTANT(21) ? (const char*)k + t * row_bytes
                                             : (const char*)v + t * row_bytes,
           (size_t)row_bytes);
  }
  return ORC_OK;
}

/* ---- scatter with conversion: new rows of src_dtype into a pool of kv_dtype, the pool
 * holding x / k_scale (x / v_scale) rounded to its type; for an fp8 pool that is the e4m3
 * code of the quotient (saturated, round to nearest even).  Every slot is checked first. */
/* Per kv head scales: k_scales / v_scales hold num_kv_heads factors (NULL: the scalar for
 * every head); each must be finite and > 0. */
static int head_scales_ok(const float* s, int32_t n) {
  if (!s) return 1;
  for (int32_t g = 0; g < n; ++g)
    if (!(s[g] > 0.f && s[g] <= FLT_MAX)) return 0;
  return 1;
}
static float head_scale(const float* s, int32_t g, int32_t num_kv_heads, float scalar) {
  if (!s) return scalar;
  return MUTANT(75) ? s[0] : s[g % num_kv_heads];
}
/* A per-block factor is a finite, positive normal float: at least FLT_MIN (2^-126), so its
 * reciprocal is finite as well (the library's reading of per-block scales; the pages give
 * no range). */
static int block_factor_ok(float a) { return a >= FLT_MIN && a <= FLT_MAX; }
/* Per-block scales ([num_blocks, num_kv_heads], NULL: none): every factor of every block a
 * sequence reads -- the first ceil(seq_len / b) entries of its table row, of the sequences
 * with query tokens when qsl is given -- must pass block_factor_ok.  Called after the tables
 * themselves were checked. */
static int block_scales_ok(const float* kbs, const float* vbs, const int32_t* qsl,
                           const int32_t* seq_lens, const int32_t* block_tables,
                           int32_t num_seqs, int32_t num_kv_heads, int32_t block_size,
                           int32_t max_blocks) {
  for (int32_t s = 0; s < num_seqs; ++s) {
    if (qsl && qsl[s + 1] <= qsl[s]) continue;
    const int64_t need = ((int64_t)seq_lens[s] + block_size - 1) / block_size;
    for (int64_t i = 0; i < need; ++i) {
      const int64_t id = block_tables[(int64_t)s * max_blocks + i];
      for (int32_t g = 0; g < num_kv_heads; ++g) {
        if (kbs && !block_factor_ok(kbs[id * num_kv_heads + g])) return 0;
        if (vbs && !block_factor_ok(vbs[id * num_kv_heads + g])) return 0;
      }
    }
  }
  return 1;
}

static int scatter_convert(const void* k, const void* v, void* k_blocks, void* v_blocks,
                           const int32_t* slot_mapping, int64_t num_tokens, int32_t num_kv_heads,
                           int32_t head_dim, int32_t block_size, int64_t num_blocks,
                           int32_t src_dtype, int32_t kv_dtype, const float* k_scales,
                           const float* v_scales, float k_scale, float v_scale) {
  if (!k || !v || !k_blocks || !v_blocks || !slot_mapping) return ORC_EINVAL;
  if (!dtype_ok(src_dtype) || !pool_dtype_ok(kv_dtype)) return ORC_EUNSUPPORTED;
  if (num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0) return ORC_ESHAPE;
  if (!head_scales_ok(k_scales, num_kv_heads) || !head_scales_ok(v_scales, num_kv_heads))
    return ORC_EINVAL;
  for (int64_t t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0 || slot >= num_blocks * block_size) return ORC_EINVAL;
  }
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    for (int64_t i = 0; i < row; ++i) {
      const int32_t g = (int32_t)(i / head_dim);
      const float ks = head_scale(k_scales, g, num_kv_heads, k_scale);
      const float vs = head_scale(v_scales, g, num_kv_heads, v_scale);
      store_elem(k_blocks, kv_dtype, slot * row + i, load_elem(k, src_dtype, t * row + i) / ks);
      store_elem(v_blocks, kv_dtype, slot * row + i, load_elem(v, src_dtype, t * row + i) / vs);
    }
  }
  return ORC_OK;
}

int oracle_reshape_and_cache_ex(const void* k, const void* v, void* k_blocks, void* v_blocks,
                                const int32_t* slot_mapping, int64_t num_tokens,
                                int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                int64_t num_blocks, int32_t src_dtype, int32_t kv_dtype,
                                float k_scale, float v_scale) {
  return scatter_convert(k, v, k_blocks, v_blocks, slot_mapping, num_tokens, num_kv_heads,
                         head_dim, block_size, num_blocks, src_dtype, kv_dtype, NULL, NULL,
                         k_scale, v_scale);
}

/* Scatter with one scale per (pool block, kv head): head g of a new row written to slot s is
 * stored as x / k_bscales[(s / b) * Hkv + g] (x / v_bscales[...]); NULL arrays: 1.  A factor
 * of a block written to that is not finite and positive is EINVAL, before any write. */
int oracle_reshape_and_cache_per_block(const void* k, const void* v, void* k_blocks,
                                       void* v_blocks, const int32_t* slot_mapping,
                                       int64_t num_tokens, int32_t num_kv_heads,
                                       int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                       int32_t src_dtype, int32_t kv_dtype,
                                       const float* k_bscales, const float* v_bscales) {
  if (!k || !v || !k_blocks || !v_blocks || !slot_mapping) return ORC_EINVAL;
  if (!dtype_ok(src_dtype) || !pool_dtype_ok(kv_dtype)) return ORC_EUNSUPPORTED;
  if (num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0) return ORC_ESHAPE;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot < 0 || slot >= num_blocks * block_size) return ORC_EINVAL;
    const int64_t blk = slot / block_size;
    for (int32_t g = 0; g < num_kv_heads; ++g) {
      const float a = k_bscales ? k_bscales[blk * num_kv_heads + g] : 1.f;
      const float b = v_bscales ? v_bscales[blk * num_kv_heads + g] : 1.f;
      if (!block_factor_ok(a) || !block_factor_ok(b)) return ORC_EINVAL;
    }
  }
  const int64_t row = (int64_t)num_kv_heads * head_dim;
  for (int64_t t = 0; t < num_tokens; ++t) {
    const int64_t slot = slot_mapping[t];
    const int64_t blk = slot / block_size;
    for (int64_t i = 0; i < row; ++i) {
      const int32_t g = (int32_t)(i / head_dim);
      const float ks = k_bscales ? k_bscales[blk * num_kv_heads + g] : 1.f;
      const float vs = v_bscales ? v_bscales[blk * num_kv_heads + g] : 1.f;
      store_elem(k_blocks, kv_dtype, slot * row + i, load_elem(k, src_dtype, t * row + i) / ks);
      store_elem(v_blocks, kv_dtype, slot * row + i, load_elem(v, src_dtype, t * row + i) / vs);
    }
  }
  return ORC_OK;
}

/* The same with one scale per kv head: head g of a new row is stored as x / k_scales[g]
 * (x / v_scales[g]).  A scale that is not finite and positive is EINVAL, before any write. */
int oracle_reshape_and_cache_per_head(const void* k, const void* v, void* k_blocks,
                                      void* v_blocks, const int32_t* slot_mapping,
                                      int64_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                                      int32_t block_size, int64_t num_blocks, int32_t src_dtype,
                                      int32_t kv_dtype, const float* k_scales,
                                      const float* v_scales) {
  return scatter_convert(k, v, k_blocks, v_blocks, slot_mapping, num_tokens, num_kv_heads,
                         head_dim, block_size, num_blocks, src_dtype, kv_dtype, k_scales,
                         v_scales, 1.f, 1.f);
}

/* ---- gather of a sequence's rows into a dense buffer ([MLA] GatherMlaCache) --
 * Output rows [cu[s], cu[s+1]) of k_out/v_out ([rows, Hkv, D]) receive the pool
 * rows at positions (r - cu[s]) + seq_starts[s] of sequence s (seq_starts may be
 * NULL, meaning 0).  A position past the block-table row or a block id outside
 * the pool is EINVAL, checked before any write.  v_blocks/v_out may be NULL. */
int oracle_gather_kv(const void* k_blocks, const void* v_blocks, void* k_out, void* v_out,
                     const int32_t* cu_seq_lens, const int32_t* seq_starts,
                     const int32_t* block_tables, int32_t num_seqs, int32_t num_kv_heads,
                     int32_t head_dim, int32_t block_size, int64_t num_blocks,
                     int32_t max_blocks, int32_t kv_dtype) {
  if (!k_blocks || !k_out || !cu_seq_lens || !block_tables) return ORC_EINVAL;
  if ((v_blocks == NULL) != (v_out == NULL)) return ORC_EINVAL;
  if (!pool_dtype_ok(kv_dtype)) return ORC_EUNSUPPORTED;
  if (num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0) return ORC_ESHAPE;
  for (int32_t s = 0; s < num_seqs; ++s) {
    if (cu_seq_lens[s + 1] < cu_seq_lens[s]) return ORC_EINVAL;
    int64_t start = seq_starts ? seq_starts[s] : 0;
    if (start < 0) return ORC_EINVAL;
    for (int64_t r = cu_seq_lens[s]; r < cu_seq_lens[s + 1]; ++r) {
      int64_t pos = r - cu_seq_lens[s] + start;
      if (pos / block_size >= max_blocks) return ORC_EINVAL;
      int32_t blk = block_tables[(int64_t)s * max_blocks + pos / block_size];
      if (blk < 0 || blk >= num_blocks) return ORC_EINVAL;
    }
  }
  const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * elem_bytes(kv_dtype);
  for (int32_t s = 0; s < num_seqs; ++s) {
    int64_t start = seq_starts ? seq_starts[s] : 0;
    for (int64_t r = cu_seq_lens[s]; r < cu_seq_lens[s + 1]; ++r) {
      int64_t pos = r - cu_seq_lens[s] + start;
      if (MUTANT(22)) pos += 1;
      int64_t blk = block_tables[(int64_t)s * max_blocks + pos / block_size];
      int64_t src = (blk * block_size + pos % block_size) * row_bytes;
      memcpy((char*)k_out + r * row_bytes, (const char*)k_blocks + src, (size_t)row_bytes);
      if (v_out) memcpy((char*)v_out + r * row_bytes, (const char*)v_blocks + src, (size_t)row_bytes);
    }
  }
  return ORC_OK;
}

/* ---- one attention row, two-pass -------------------------------------------
 * Softmax attention of query row q (length D) over positions [start, end) of one
 * sequence's cache (kv head g), written to out_row in out_dtype.  Returns the
 * log-sum-exp (natural log) of the scaled scores, -inf for an empty range, and
 * stores the running max and exp-sum through m_out / l_out when asked
 * ([V2] max_logits / exp_sums).  `logits` is caller scratch of >= end-start
 * floats and `acc` of >= D floats. */
static float attend_two_pass(const void* q, int64_t q_off, int q_dtype, const void* k_blocks,
                             const void* v_blocks, int kv_dtype, const int32_t* table_row,
                             int64_t start, int64_t end, int32_t block_size,
                             int32_t num_kv_heads, int32_t head_dim, int32_t kv_head,
                             float scale, float* logits, float* acc, void* out,
                             int64_t out_off, int out_dtype, float* m_out, float* l_out,
                             float sink, float k_scale, float v_scale, const float* k_bscales,
                             const float* v_bscales) {
  const int64_t n = end > start ? end - start : 0;
  /* Per-block scales ([TL] "Going further": fp8 caches with scales per head or per block):
   * position j is dequantised with the factor of (its block, this kv head) instead of the
   * scalar; NULL arrays keep the scalar. */
#define KV_FACTOR(arr, scalar, j) \
  ((arr) ? (arr)[(int64_t)table_row[(j) / block_size] * num_kv_heads + (MUTANT(76) ? 0 : kv_head)] \
         : (scalar))
  /* An attention sink ([MPA] ForwardWithSinks) is one more, virtual, position whose score is
   * the sink logit and whose value is zero: it enters the max and the exp-sum, never the
   * weighted sum.  sink = -inf means none (and then changes nothing). */
  const int has_sink = sink > -INFINITY;

  /* PASS 1: raw dot (ascending d), then the scale, and the row max
   * ([MPA] "Compute Q . K" then score *= scale; [MLA] PASS 1). */
  float m = has_sink ? sink : -INFINITY;
  for (int64_t i = 0; i < n; ++i) {
    int64_t j = start + i;
    int64_t k_off = pool_row_offset(table_row, j, block_size, num_kv_heads, head_dim, kv_head);
    float dot = 0.0f;
    const float kf = KV_FACTOR(k_bscales, k_scale, j);
    for (int32_t d = 0; d < head_dim; ++d)
      dot += load_elem(q, q_dtype, q_off + d) *
             (MUTANT(72) ? load_elem(k_blocks, kv_dtype, k_off + d)
                         : load_elem(k_blocks, kv_dtype, k_off + d) * kf);
    float s = MUTANT(30) ? dot : dot * scale;
    logits[i] = s;
    if (s > m) m = s;
  }

  /* PASS 2: the exp-sum (the sink's term first, as [MPA] seeds its denominator with it), then
   * the weighted sum; no running rescale ([MLA] PASS 2). */
  float l = 0.0f;
  if (has_sink && !MUTANT(60)) l = MUTANT(61) ? 1.0f : expf(sink - m); /* s60 / s61 */
  for (int64_t i = 0; i < n; ++i) {
    float p = expf(MUTANT(31) ? m - logits[i] : logits[i] - m);
    logits[i] = p;
    l += p;
  }
  for (int32_t d = 0; d < head_dim; ++d) acc[d] = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    int64_t j = start + i;
    int64_t v_off = pool_row_offset(table_row, j, block_size, num_kv_heads, head_dim, kv_head);
    const void* vsrc = MUTANT(8) ? k_blocks : v_blocks; /* s08: V read from the K pool */
    float p = logits[i];
    const float vf = KV_FACTOR(v_bscales, v_scale, j);
    for (int32_t d = 0; d < head_dim; ++d)
      acc[d] += p * (MUTANT(73) ? load_elem(vsrc, kv_dtype, v_off + d)
                                : load_elem(vsrc, kv_dtype, v_off + d) * vf);
  }
#undef KV_FACTOR

  /* o = acc * (1/l); an empty range writes zeros ([MPA] "Empty context: write
   * zeros"; [MLA] inv = l > 0 ? 1/l : 0; [TL] 2.4 multiply by 1/l). */
  float inv = l > 0.0f ? 1.0f / l : 0.0f;
  if (MUTANT(32)) inv = 1.0f;
  if (out)
    for (int32_t d = 0; d < head_dim; ++d) store_elem(out, out_dtype, out_off + d, acc[d] * inv);
  if (m_out) *m_out = m;
  if (l_out) *l_out = l;
  return l > 0.0f ? m + logf(l) : -INFINITY;
}

/* ---- validation of the batched call ([TL] 2.6, section 4) ----------------
 * Shape errors first (ESHAPE), then the metadata of every sequence that has
 * query tokens (EINVAL): a non-monotone or inconsistent query_start_loc, an empty
 * context, a table too short for ceil(seq_len / b) blocks, a block id outside the
 * pool among those entries, or a query position outside [0, seq_len).  Sequences
 * with no query tokens are skipped. */
static int validate_varlen(const void* q, const void* k_blocks, const void* v_blocks,
                           const void* out, const int32_t* qsl, const int32_t* seq_lens,
                           const int32_t* positions, const int32_t* block_tables,
                           int32_t num_seqs, int64_t num_tokens, int32_t num_heads,
                           int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                           int64_t num_blocks, int32_t max_blocks, int32_t q_dtype,
                           int32_t kv_dtype) {
  if (num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0)
    return ORC_ESHAPE;
  if (num_heads % num_kv_heads != 0) return ORC_ESHAPE;
  if (!dtype_ok(q_dtype) || !pool_dtype_ok(kv_dtype)) return ORC_EUNSUPPORTED;
  if (!q || !k_blocks || !v_blocks || !out || !qsl || !seq_lens || !positions || !block_tables)
    return ORC_EINVAL;
  if (num_seqs < 0 || num_tokens < 0 || max_blocks < 0 || num_blocks < 0) return ORC_EINVAL;
  if (qsl[0] != 0 || qsl[num_seqs] != num_tokens) return ORC_EINVAL;
  for (int32_t s = 0; s < num_seqs; ++s) {
    if (qsl[s + 1] < qsl[s]) return ORC_EINVAL;
    if (qsl[s + 1] == qsl[s]) continue;
    int32_t n = seq_lens[s];
    if (n < 1 && !MUTANT(13)) return ORC_EINVAL;
    int64_t need = ((int64_t)n + block_size - 1) / block_size;
    if (need > max_blocks && !MUTANT(14)) return ORC_EINVAL;
    for (int64_t i = 0; i < need && i < max_blocks; ++i) {
      int32_t id = block_tables[(int64_t)s * max_blocks + i];
      if ((id < 0 || id >= num_blocks) && !MUTANT(15)) return ORC_EINVAL;
    }
    if (MUTANT(13)) continue; /* s13: an empty context slips through */
    for (int32_t t = qsl[s]; t < qsl[s + 1]; ++t)
      if (positions[t] < 0 || positions[t] >= n) return ORC_EINVAL;
  }
  return ORC_OK;
}

/* ---- batched varlen paged attention ([MPA] Forward) ------------------------
 * For token t of sequence s and head h, with g = h / (H / Hkv) ([MPA] kvHead;
 * [TL] 2.2):  end = causal ? pos_t + 1 : seq_len_s,  start = w > 0 ?
 * max(0, end - w) : 0  ([MPA] contextEndExclusive / contextStart), then softmax
 * attention over positions [start, end).  out is [T, H, D] in out_dtype; lse
 * (may be NULL) is [H, T] in natural log ([MLA] LSE layout). */
/* sinks: [num_heads] sink logits on the score scale ([MPA] ForwardWithSinks), or NULL.
 * k_scale / v_scale: the pool holds K / k_scale and V / v_scale ([V2]: "k_flat.float()
 * .mul_(k_scale)"), so attention uses K = k_scale * pool and V = v_scale * pool. */
static int varlen_core(const void* q, const void* k_blocks, const void* v_blocks, void* out,
                       float* lse, const int32_t* query_start_loc, const int32_t* seq_lens,
                       const int32_t* positions, const int32_t* block_tables, int32_t num_seqs,
                       int64_t num_tokens, int32_t num_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, int64_t num_blocks,
                       int32_t max_blocks, int32_t q_dtype, int32_t kv_dtype, int32_t out_dtype,
                       float scale, int32_t causal, int32_t sliding_window, const float* sinks,
                       const float* k_scales, const float* v_scales, float k_scale,
                       float v_scale, const float* k_bscales, const float* v_bscales) {
  if (num_kv_heads > 0 &&
      (!head_scales_ok(k_scales, num_kv_heads) || !head_scales_ok(v_scales, num_kv_heads)))
    return ORC_EINVAL;
  int st = validate_varlen(q, k_blocks, v_blocks, out, query_start_loc, seq_lens, positions,
                           block_tables, num_seqs, num_tokens, num_heads, num_kv_heads,
                           head_dim, block_size, num_blocks, max_blocks, q_dtype, kv_dtype);
  if (st != ORC_OK) return st;
  if (!dtype_ok(out_dtype)) return ORC_EUNSUPPORTED;
  if (!block_scales_ok(k_bscales, v_bscales, query_start_loc, seq_lens, block_tables, num_seqs,
                       num_kv_heads, block_size, max_blocks))
    return ORC_EINVAL;

  /* token -> sequence, and the longest context (for the per-thread scratch). */
  int32_t* tok_seq = (int32_t*)malloc(sizeof(int32_t) * (size_t)(num_tokens > 0 ? num_tokens : 1));
  int64_t max_ctx = 1;
  for (int32_t s = 0; s < num_seqs; ++s) {
    for (int32_t t = query_start_loc[s]; t < query_start_loc[s + 1]; ++t) tok_seq[t] = s;
    if (query_start_loc[s + 1] > query_start_loc[s] && seq_lens[s] > max_ctx) max_ctx = seq_lens[s];
  }
  const int32_t group = num_heads / num_kv_heads;
  const int64_t work = num_tokens * (int64_t)num_heads;

#pragma omp parallel
  {
    float* logits = (float*)malloc(sizeof(float) * (size_t)(max_ctx + 2));
    float* acc = (float*)malloc(sizeof(float) * (size_t)head_dim);
#pragma omp for schedule(dynamic, 8)
    for (int64_t w = 0; w < work; ++w) {
      int64_t t = w / num_heads;
      int32_t h = (int32_t)(w % num_heads);
      int32_t s = tok_seq[t];
      int32_t g = MUTANT(5) ? h % num_kv_heads : h / group; /* s05: round-robin GQA */
      int64_t pos = positions[t];
      if (MUTANT(7)) pos += 1; /* s07: query one past its position */
      int64_t end = causal ? pos + 1 : seq_lens[s];
      int64_t win = MUTANT(6) ? (int64_t)sliding_window + 1 : sliding_window; /* s06 */
      int64_t start = sliding_window > 0 ? (end - win > 0 ? end - win : 0) : 0;
      const int32_t* row = block_tables + (int64_t)s * max_blocks;
      const int32_t gs = MUTANT(74) ? h % num_kv_heads : g; /* s74: the query head's scale */
      float l_lse = attend_two_pass(q, (t * num_heads + h) * (int64_t)head_dim, q_dtype, k_blocks,
                                    v_blocks, kv_dtype, row, start, end, block_size, num_kv_heads,
                                    head_dim, g, scale, logits, acc, out,
                                    (t * num_heads + h) * (int64_t)head_dim, out_dtype, NULL, NULL,
                                    sinks ? sinks[h] : -INFINITY,
                                    head_scale(k_scales, gs, num_kv_heads, k_scale),
                                    head_scale(v_scales, gs, num_kv_heads, v_scale), k_bscales,
                                    v_bscales);
      if (lse) lse[(int64_t)h * num_tokens + t] = l_lse;
    }
    free(logits);
    free(acc);
  }
  free(tok_seq);
  return ORC_OK;
}

int oracle_varlen_attention_ex(const void* q, const void* k_blocks, const void* v_blocks,
                               void* out, float* lse, const int32_t* query_start_loc,
                               const int32_t* seq_lens, const int32_t* positions,
                               const int32_t* block_tables, int32_t num_seqs, int64_t num_tokens,
                               int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                               int32_t block_size, int64_t num_blocks, int32_t max_blocks,
                               int32_t q_dtype, int32_t kv_dtype, int32_t out_dtype, float scale,
                               int32_t causal, int32_t sliding_window, const float* sinks,
                               float k_scale, float v_scale) {
  return varlen_core(q, k_blocks, v_blocks, out, lse, query_start_loc, seq_lens, positions,
                     block_tables, num_seqs, num_tokens, num_heads, num_kv_heads, head_dim,
                     block_size, num_blocks, max_blocks, q_dtype, kv_dtype, out_dtype, scale,
                     causal, sliding_window, sinks, NULL, NULL, k_scale, v_scale, NULL, NULL);
}

/* One dequantisation scale per kv head: query head h (kv head g = h / G) attends over
 * K = k_scales[g] * pool and V = v_scales[g] * pool (NULL arrays: 1).  A scale that is not
 * finite and positive is EINVAL. */
int oracle_varlen_attention_per_head(const void* q, const void* k_blocks, const void* v_blocks,
                                     void* out, float* lse, const int32_t* query_start_loc,
                                     const int32_t* seq_lens, const int32_t* positions,
                                     const int32_t* block_tables, int32_t num_seqs,
                                     int64_t num_tokens, int32_t num_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                     int32_t max_blocks, int32_t q_dtype, int32_t kv_dtype,
                                     int32_t out_dtype, float scale, int32_t causal,
                                     int32_t sliding_window, const float* sinks,
                                     const float* k_scales, const float* v_scales) {
  return varlen_core(q, k_blocks, v_blocks, out, lse, query_start_loc, seq_lens, positions,
                     block_tables, num_seqs, num_tokens, num_heads, num_kv_heads, head_dim,
                     block_size, num_blocks, max_blocks, q_dtype, kv_dtype, out_dtype, scale,
                     causal, sliding_window, sinks, k_scales, v_scales, 1.f, 1.f, NULL, NULL);
}

/* One dequantisation scale per (pool block, kv head) ([TL] "Going further": scales per
 * block): position j of a sequence attends over K = k_bscales[id * Hkv + g] * pool and
 * V = v_bscales[id * Hkv + g] * pool, id = its block, g its kv head (NULL arrays: 1).  A
 * factor of a block some sequence reads that is not finite and positive is EINVAL. */
int oracle_varlen_attention_per_block(const void* q, const void* k_blocks, const void* v_blocks,
                                      void* out, float* lse, const int32_t* query_start_loc,
                                      const int32_t* seq_lens, const int32_t* positions,
                                      const int32_t* block_tables, int32_t num_seqs,
                                      int64_t num_tokens, int32_t num_heads,
                                      int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                      int64_t num_blocks, int32_t max_blocks, int32_t q_dtype,
                                      int32_t kv_dtype, int32_t out_dtype, float scale,
                                      int32_t causal, int32_t sliding_window, const float* sinks,
                                      const float* k_bscales, const float* v_bscales) {
  return varlen_core(q, k_blocks, v_blocks, out, lse, query_start_loc, seq_lens, positions,
                     block_tables, num_seqs, num_tokens, num_heads, num_kv_heads, head_dim,
                     block_size, num_blocks, max_blocks, q_dtype, kv_dtype, out_dtype, scale,
                     causal, sliding_window, sinks, NULL, NULL, 1.f, 1.f, k_bscales, v_bscales);
}

int oracle_varlen_attention(const void* q, const void* k_blocks, const void* v_blocks,
                            void* out, float* lse, const int32_t* query_start_loc,
                            const int32_t* seq_lens, const int32_t* positions,
                            const int32_t* block_tables, int32_t num_seqs, int64_t num_tokens,
                            int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                            int32_t block_size, int64_t num_blocks, int32_t max_blocks,
                            int32_t q_dtype, int32_t kv_dtype, int32_t out_dtype, float scale,
                            int32_t causal, int32_t sliding_window) {
  return oracle_varlen_attention_ex(q, k_blocks, v_blocks, out, lse, query_start_loc, seq_lens,
                                    positions, block_tables, num_seqs, num_tokens, num_heads,
                                    num_kv_heads, head_dim, block_size, num_blocks, max_blocks,
                                    q_dtype, kv_dtype, out_dtype, scale, causal, sliding_window,
                                    NULL, 1.0f, 1.0f);
}

/* ---- split-KV decode, phase 1 ([V2] partition loop) ------------------------
 * One decode query per sequence, q [S, H, D], at position seq_len - 1 (causal by
 * construction, [TL] 2.2).  Partition p covers positions [p*P, min((p+1)*P,
 * seq_len)) ([V2] start/end), intersected with the window [max(0, seq_len - w),
 * seq_len).  For each (s, h, p < max_parts) the oracle stores the partition's
 * max scaled score, its exp-sum and its NORMALISED output sum_j e^{s_j-m} v_j / l
 * (the reading taken of the page's reduction, which only makes sense when
 * tmp_output holds normalised partition outputs).  Partitions with no visible
 * position, including those at or past ceil(seq_len / P), get (-inf, 0, zeros).
 * k_scale / v_scale: the pools hold K / k_scale and V / v_scale, possibly as fp8
 * ([V2]: kv_cache_dtype, "Apply scales" before the partition loop). */
static int splitkv_core(const void* q, const void* k_blocks, const void* v_blocks,
                        float* max_logits, float* exp_sums, float* tmp_out,
                        const int32_t* seq_lens, const int32_t* block_tables, int32_t num_seqs,
                        int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                        int32_t block_size, int64_t num_blocks, int32_t max_blocks,
                        int32_t partition_size, int32_t max_parts, int32_t q_dtype,
                        int32_t kv_dtype, float scale, int32_t sliding_window,
                        const float* k_scales, const float* v_scales, float k_scale,
                        float v_scale, const float* k_bscales, const float* v_bscales) {
  if (num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      num_heads % num_kv_heads != 0 || partition_size <= 0 || max_parts <= 0)
    return ORC_ESHAPE;
  if (!dtype_ok(q_dtype) || !pool_dtype_ok(kv_dtype)) return ORC_EUNSUPPORTED;
  if (!q || !k_blocks || !v_blocks || !max_logits || !exp_sums || !tmp_out || !seq_lens ||
      !block_tables)
    return ORC_EINVAL;
  if (!head_scales_ok(k_scales, num_kv_heads) || !head_scales_ok(v_scales, num_kv_heads))
    return ORC_EINVAL;
  int64_t max_ctx = 1;
  for (int32_t s = 0; s < num_seqs; ++s) {
    int32_t n = seq_lens[s];
    if (n < 1) return ORC_EINVAL;
    int64_t need = ((int64_t)n + block_size - 1) / block_size;
    if (need > max_blocks) return ORC_EINVAL;
    if (((int64_t)n + partition_size - 1) / partition_size > max_parts) return ORC_EINVAL;
    for (int64_t i = 0; i < need; ++i) {
      int32_t id = block_tables[(int64_t)s * max_blocks + i];
      if (id < 0 || id >= num_blocks) return ORC_EINVAL;
    }
    if (n > max_ctx) max_ctx = n;
  }
  if (!block_scales_ok(k_bscales, v_bscales, NULL, seq_lens, block_tables, num_seqs, num_kv_heads,
                       block_size, max_blocks))
    return ORC_EINVAL;
  const int32_t group = num_heads / num_kv_heads;
  const int64_t work = (int64_t)num_seqs * num_heads * max_parts;
#pragma omp parallel
  {
    float* logits = (float*)malloc(sizeof(float) * (size_t)(partition_size + 2));
    float* acc = (float*)malloc(sizeof(float) * (size_t)head_dim);
#pragma omp for schedule(dynamic, 8)
    for (int64_t w = 0; w < work; ++w) {
      int32_t p = (int32_t)(w % max_parts);
      int32_t h = (int32_t)((w / max_parts) % num_heads);
      int32_t s = (int32_t)(w / ((int64_t)max_parts * num_heads));
      int64_t n = seq_lens[s];
      int64_t vis_lo = sliding_window > 0 ? (n - sliding_window > 0 ? n - sliding_window : 0) : 0;
      int64_t lo = (int64_t)p * partition_size;
      int64_t hi = lo + partition_size < n ? lo + partition_size : n;
      if (lo < vis_lo) lo = vis_lo;
      int64_t idx = ((int64_t)s * num_heads + h) * max_parts + p;
      float m, l;
      attend_two_pass(q, ((int64_t)s * num_heads + h) * head_dim, q_dtype, k_blocks, v_blocks,
                      kv_dtype, block_tables + (int64_t)s * max_blocks, lo, hi, block_size,
                      num_kv_heads, head_dim, h / group, scale, logits, acc, tmp_out,
                      idx * head_dim, ORC_F32, &m, &l, -INFINITY,
                      head_scale(k_scales, h / group, num_kv_heads, k_scale),
                      head_scale(v_scales, h / group, num_kv_heads, v_scale), k_bscales,
                      v_bscales);
      max_logits[idx] = m;
      exp_sums[idx] = l;
    }
    free(logits);
    free(acc);
  }
  return ORC_OK;
}

int oracle_splitkv_partials_ex(const void* q, const void* k_blocks, const void* v_blocks,
                               float* max_logits, float* exp_sums, float* tmp_out,
                               const int32_t* seq_lens, const int32_t* block_tables,
                               int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                               int32_t head_dim, int32_t block_size, int64_t num_blocks,
                               int32_t max_blocks, int32_t partition_size, int32_t max_parts,
                               int32_t q_dtype, int32_t kv_dtype, float scale,
                               int32_t sliding_window, float k_scale, float v_scale) {
  return splitkv_core(q, k_blocks, v_blocks, max_logits, exp_sums, tmp_out, seq_lens,
                      block_tables, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                      num_blocks, max_blocks, partition_size, max_parts, q_dtype, kv_dtype, scale,
                      sliding_window, NULL, NULL, k_scale, v_scale, NULL, NULL);
}

/* Split-KV partials with one scale per kv head (NULL arrays: 1; not finite and positive:
 * EINVAL). */
int oracle_splitkv_partials_per_head(const void* q, const void* k_blocks, const void* v_blocks,
                                     float* max_logits, float* exp_sums, float* tmp_out,
                                     const int32_t* seq_lens, const int32_t* block_tables,
                                     int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                     int32_t max_blocks, int32_t partition_size,
                                     int32_t max_parts, int32_t q_dtype, int32_t kv_dtype,
                                     float scale, int32_t sliding_window, const float* k_scales,
                                     const float* v_scales) {
  return splitkv_core(q, k_blocks, v_blocks, max_logits, exp_sums, tmp_out, seq_lens,
                      block_tables, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                      num_blocks, max_blocks, partition_size, max_parts, q_dtype, kv_dtype, scale,
                      sliding_window, k_scales, v_scales, 1.f, 1.f, NULL, NULL);
}

/* Split-KV partials with one scale per (pool block, kv head), as
 * oracle_varlen_attention_per_block (NULL arrays: 1). */
int oracle_splitkv_partials_per_block(const void* q, const void* k_blocks, const void* v_blocks,
                                      float* max_logits, float* exp_sums, float* tmp_out,
                                      const int32_t* seq_lens, const int32_t* block_tables,
                                      int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                      int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                      int32_t max_blocks, int32_t partition_size,
                                      int32_t max_parts, int32_t q_dtype, int32_t kv_dtype,
                                      float scale, int32_t sliding_window,
                                      const float* k_bscales, const float* v_bscales) {
  return splitkv_core(q, k_blocks, v_blocks, max_logits, exp_sums, tmp_out, seq_lens,
                      block_tables, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                      num_blocks, max_blocks, partition_size, max_parts, q_dtype, kv_dtype, scale,
                      sliding_window, NULL, NULL, 1.f, 1.f, k_bscales, v_bscales);
}

int oracle_splitkv_partials(const void* q, const void* k_blocks, const void* v_blocks,
                            float* max_logits, float* exp_sums, float* tmp_out,
                            const int32_t* seq_lens, const int32_t* block_tables,
                            int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                            int32_t head_dim, int32_t block_size, int64_t num_blocks,
                            int32_t max_blocks, int32_t partition_size, int32_t max_parts,
                            int32_t q_dtype, int32_t kv_dtype, float scale,
                            int32_t sliding_window) {
  return oracle_splitkv_partials_ex(q, k_blocks, v_blocks, max_logits, exp_sums, tmp_out,
                                    seq_lens, block_tables, num_seqs, num_heads, num_kv_heads,
                                    head_dim, block_size, num_blocks, max_blocks, partition_size,
                                    max_parts, q_dtype, kv_dtype, scale, sliding_window, 1.0f,
                                    1.0f);
}

/* ---- log-sum-exp of one partition ----------------------------------------
 * lse = m + log(l); an infinite max of either sign or a zero exp-sum means the
 * partition holds no mass and its lse is -inf (the +inf -> -inf normalisation of
 * [MLA] MergeAttnStates, applied to the partition's (m, l) pair). */
static float partition_lse(float m, float l) {
  if (MUTANT(40)) return m + logf(l);
  if (isinf(m) || !(l > 0.0f)) return -INFINITY;
  return m + logf(l);
}

/* ---- split-KV decode, phase 2 ([V2] "Phase 2: Cross-partition reduction") --
 * For (s, h): the partitions 0 .. ceil(seq_len / P) - 1 are combined with
 * weights w_p = exp(lse_p - M), M = max_p lse_p, out = sum_p w_p o_p * (1 / sum_p w_p).
 * When every lse_p is -inf the result is partition 0's output (the both -inf
 * branch of [MLA] MergeAttnStates, which emits its first input).  out is [S, H, D]. */
int oracle_splitkv_reduce(void* out, const float* max_logits, const float* exp_sums,
                          const float* tmp_out, const int32_t* seq_lens, int32_t num_seqs,
                          int32_t num_heads, int32_t head_dim, int32_t partition_size,
                          int32_t max_parts, int32_t out_dtype) {
  if (num_heads <= 0 || head_dim <= 0 || partition_size <= 0 || max_parts <= 0)
    return ORC_ESHAPE;
  if (!dtype_ok(out_dtype)) return ORC_EUNSUPPORTED;
  if (!out || !max_logits || !exp_sums || !tmp_out || !seq_lens) return ORC_EINVAL;
  for (int32_t s = 0; s < num_seqs; ++s) {
    int64_t n = seq_lens[s];
    if (n < 1 || (n + partition_size - 1) / partition_size > max_parts) return ORC_EINVAL;
  }
  float* lse = (float*)malloc(sizeof(float) * (size_t)max_parts);
  for (int32_t s = 0; s < num_seqs; ++s) {
    int32_t np = (int32_t)((seq_lens[s] + partition_size - 1) / partition_size);
    for (int32_t h = 0; h < num_heads; ++h) {
      int64_t base = ((int64_t)s * num_heads + h) * max_parts;
      float M = -INFINITY;
      for (int32_t p = 0; p < np; ++p) {
        lse[p] = partition_lse(max_logits[base + p], exp_sums[base + p]);
        if (lse[p] > M) M = lse[p];
      }
      int64_t o_off = ((int64_t)s * num_heads + h) * head_dim;
      if (isinf(M) && !MUTANT(41)) {
        for (int32_t d = 0; d < head_dim; ++d)
          store_elem(out, out_dtype, o_off + d, tmp_out[base * head_dim + d]);
        continue;
      }
      float wsum = 0.0f;
      for (int32_t p = 0; p < np; ++p) {
        float wp = MUTANT(42) ? expf(max_logits[base + p] - M) : expf(lse[p] - M);
        lse[p] = wp; /* reuse the buffer for the weights */
        wsum += wp;
      }
      float inv = 1.0f / wsum;
      for (int32_t d = 0; d < head_dim; ++d) {
        float acc = 0.0f;
        for (int32_t p = 0; p < np; ++p)
          if (lse[p] > 0.0f) acc += lse[p] * tmp_out[(base + p) * head_dim + d];
        store_elem(out, out_dtype, o_off + d, acc * inv);
      }
    }
  }
  free(lse);
  return ORC_OK;
}

/* ---- two-state merge ([MLA] MergeAttnStatesKernel) --------------------------
 * out/prefix/suffix are [T, H, D] in `dtype`; lse arrays are [H, T] fp32 (out_lse
 * may be NULL).  Tokens t >= prefill_tokens_with_context (when that is >= 0) copy
 * the suffix unchanged.  Otherwise: an infinite lse of either sign is taken as
 * -inf; if both are -inf the prefix output is emitted with lse -inf; else
 * p_scale = p_se / (p_se + s_se), s_scale likewise, and
 * out_lse = log(p_se + s_se) + max. */
int oracle_merge_attn_states(void* out, float* out_lse, const void* prefix_out,
                             const float* prefix_lse, const void* suffix_out,
                             const float* suffix_lse, int64_t num_tokens, int32_t num_heads,
                             int32_t head_dim, int64_t prefill_tokens_with_context,
                             int32_t dtype) {
  if (num_heads <= 0 || head_dim <= 0) return ORC_ESHAPE;
  if (!dtype_ok(dtype)) return ORC_EUNSUPPORTED;
  if (!out || !prefix_out || !prefix_lse || !suffix_out || !suffix_lse) return ORC_EINVAL;
  const int64_t prefix_tokens =
      prefill_tokens_with_context < 0 ? num_tokens : prefill_tokens_with_context;
  for (int64_t t = 0; t < num_tokens; ++t) {
    for (int32_t h = 0; h < num_heads; ++h) {
      const int64_t off = (t * num_heads + h) * (int64_t)head_dim;
      const int64_t li = (int64_t)h * num_tokens + t;
      if (t >= prefix_tokens) {
        for (int32_t d = 0; d < head_dim; ++d)
          store_elem(out, dtype, off + d, load_elem(suffix_out, dtype, off + d));
        if (out_lse) out_lse[li] = suffix_lse[li];
        continue;
      }
      float p_lse = prefix_lse[li];
      float s_lse = suffix_lse[li];
      if (!MUTANT(50)) {
        if (isinf(p_lse)) p_lse = -INFINITY;
        if (isinf(s_lse)) s_lse = -INFINITY;
      }
      const float max_lse = fmaxf(p_lse, s_lse);
      if (isinf(max_lse)) {
        const void* src = MUTANT(51) ? suffix_out : prefix_out;
        for (int32_t d = 0; d < head_dim; ++d)
          store_elem(out, dtype, off + d, load_elem(src, dtype, off + d));
        if (out_lse) out_lse[li] = max_lse;
        continue;
      }
      const float p_se = expf(p_lse - max_lse);
      const float s_se = expf(s_lse - max_lse);
      const float out_se = p_se + s_se;
      float p_scale = p_se / out_se;
      float s_scale = s_se / out_se;
      if (MUTANT(52)) {
        float tmp = p_scale;
        p_scale = s_scale;
        s_scale = tmp;
      }
      for (int32_t d = 0; d < head_dim; ++d) {
        float po = load_elem(prefix_out, dtype, off + d);
        float so = load_elem(suffix_out, dtype, off + d);
        store_elem(out, dtype, off + d, po * p_scale + so * s_scale);
      }
      if (out_lse) out_lse[li] = logf(out_se) + max_lse;
    }
  }
  return ORC_OK;
}

/* Codec entry points, so the tests can pin the rounding against known values. */
float oracle_fp8_to_f32(uint8_t b) { return fp8_bits_to_float(b); }
uint8_t oracle_f32_to_fp8(float f) { return float_to_fp8_bits(f); }

float oracle_bf16_to_f32(uint16_t b) { return bf16_bits_to_float(b); }
uint16_t oracle_f32_to_bf16(float f) { return float_to_bf16_bits(f); }
