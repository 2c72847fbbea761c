/*
 * pa.h -- batched paged attention over a block-pooled KV cache, for GB300 (sm_103a).
 *
 * C ABI of libpa.so.  Every pointer argument named *_blocks, q, k, v, out, lse, the
 * int32 metadata arrays and any workspace is a DEVICE pointer that the caller owns;
 * the library allocates no device memory.  Every call is asynchronous on `stream`
 * (0 = the legacy default stream) and returns after enqueueing its kernels.
 *
 * Stream order.  A call observes everything enqueued before it on `stream` and everything
 * after it observes the call.  The varlen calls' planning kernel is launched with
 * programmatic dependent launch and reads the metadata arrays (query_start_loc, seq_lens,
 * positions, block_tables, per-head scales, per-block factors) before the kernel ahead of it
 * on the stream has finished; it waits for that kernel before writing anything.  So the
 * metadata must not be written by a kernel of the caller's that itself releases its
 * programmatic dependents (griddepcontrol.launch_dependents) before those writes.  Copies,
 * ordinary kernels and this library's own kernels ahead of the call are all safe.
 *
 * Layouts (row-major, as the TensorSharp "ManagedPagedAttention.cs" class summary
 * states them):
 *   q, out               [num_tokens, num_heads, head_dim]
 *   k, v (new tokens)    [num_tokens, num_kv_heads, head_dim]
 *   k_blocks, v_blocks   [num_blocks, block_size, num_kv_heads, head_dim]
 *   block_tables         int32 [num_seqs, max_blocks_per_seq]: position j of sequence s
 *                        lives in row j mod block_size of block block_tables[s][j / block_size]
 *                        (tinyllm "Paged attention for decode in C", section 2.1)
 *   query_start_loc      int32 [num_seqs + 1], query_start_loc[0] = 0,
 *                        query_start_loc[num_seqs] = num_tokens
 *   seq_lens             int32 [num_seqs]: cached positions of the sequence, new tokens included
 *   positions            int32 [num_tokens]: absolute position of each token in its sequence
 *   lse                  fp32 [num_heads, num_tokens], natural log (vllm.cpp cpu_mla_prefill.cpp)
 *
 * Errors.  Argument and shape errors are returned immediately and nothing is enqueued.
 * Errors in the device-resident metadata (a block id outside the pool, a table too short,
 * an empty context, a position outside its context, a slot outside the pool) are found on
 * the device by a validation kernel that runs before any output is written: the call then
 * writes NO output, and the error is recorded in a per-device status word that
 * pa_device_status() returns.  The recorded error is sticky: until pa_device_status() reads
 * and clears it, every later call on that device also skips its writes.  A bounded wait
 * that runs out inside a kernel records PA_ETIMEOUT the same way.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes: the error classes of the tinyllm decode interface (section 4:
 * TL_EINVAL, TL_ESHAPE; section 2.6: TL_EUNSUPPORTED) plus the CUDA and timeout cases. */
typedef enum {
  PA_OK = 0,
  PA_EINVAL = 1,       /* NULL pointer, bad metadata, sizes out of range */
  PA_ESHAPE = 2,       /* num_heads % num_kv_heads != 0, non-positive dims */
  PA_EUNSUPPORTED = 3, /* dtype or shape this build does not implement */
  PA_ECUDA = 4,        /* a CUDA runtime call failed */
  PA_ETIMEOUT = 5      /* a bounded wait inside a kernel ran out */
} pa_status;

/* Element types (vllm.cpp cpu_mla_prefill.cpp LoadF/StoreF: f32 and bf16), and fp8 e4m3
 * for K/V pools only ("paged_attention_v2_pytorch.py": kv_cache_dtype "fp8" with k_scale /
 * v_scale; tinyllm "Going further": fp8 KV caches, half the bytes per token).  PA_FP8_E4M3
 * is the OCP e4m3 "fn" format: 1 sign, 4 exponent (bias 7) and 3 mantissa bits, no
 * infinities, S.1111.111 NaN, largest finite value 448.  q, out and new K/V rows are f32 or
 * bf16. */
typedef enum { PA_F32 = 0, PA_BF16 = 1, PA_FP8_E4M3 = 2 } pa_dtype;

/* Flags of pa_varlen_forward_ex. */
enum { PA_FLAG_BITWISE = 1u };

/* Library version, major * 10000 + minor * 100 + patch. */
int pa_version(void);

/* Human-readable name of a status code (static string). */
const char* pa_status_string(pa_status status);

/* Synchronises `stream`, then returns and clears this device's sticky status word
 * (PA_OK if no kernel recorded an error).  Returns PA_ECUDA if the synchronisation
 * itself fails. */
pa_status pa_device_status(cudaStream_t stream);

/*
 * pa_slot_mapping -- the physical slot of every new token.
 * slot_mapping[t] = block_tables[s][p / block_size] * block_size + p % block_size for
 * token t of sequence s at position p = positions[t] (TensorSharp class summary,
 * "slot = blockId * blockSize + offsetInBlock"; tinyllm section 2.1).
 * A token whose position lies outside its table row, or whose block id lies outside
 * [0, num_blocks), gets slot -1 and records PA_EINVAL.
 */
pa_status pa_slot_mapping(const int32_t* query_start_loc, const int32_t* positions,
                          const int32_t* block_tables, int32_t num_seqs, int64_t num_tokens,
                          int32_t max_blocks_per_seq, int32_t block_size, int64_t num_blocks,
                          int32_t* slot_mapping, cudaStream_t stream);

/*
 * pa_reshape_and_cache -- scatter the new tokens' K and V rows into the pool
 * (TensorSharp WriteKvToPagedPool): the num_kv_heads * head_dim elements of token t go to
 * block slot_mapping[t] / block_size, row slot_mapping[t] % block_size, of each pool.
 * A pure copy: bit-exact (for PA_FP8_E4M3 the new rows are e4m3 codes already; to quantise
 * f32 / bf16 rows into an fp8 pool use pa_reshape_and_cache_ex).  Every slot is checked on
 * the device before any row is written;
 * one slot outside [0, num_blocks * block_size) writes nothing and records PA_EINVAL.
 * Duplicate slots are undefined.
 */
pa_status pa_reshape_and_cache(const void* k, const void* v, void* k_blocks, void* v_blocks,
                               const int32_t* slot_mapping, int64_t num_tokens,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               int64_t num_blocks, pa_dtype kv_dtype, cudaStream_t stream);

/*
 * pa_slot_mapping_and_cache -- pa_slot_mapping followed by pa_reshape_and_cache on the same
 * stream, as one launch when num_tokens <= 2048 and num_seqs <= 2047 (a decode step; larger
 * batches take the two launches).  Writes slot_mapping [num_tokens] (-1 for an invalid token)
 * and scatters the new K/V rows of every token into its slot.  Every token's slot is computed
 * and checked before any row is written: a token that no sequence's range
 * [query_start_loc[s], query_start_loc[s + 1]) holds, a malformed query_start_loc, a position
 * outside its table row or a block id outside [0, num_blocks) writes no row and records
 * PA_EINVAL.  Layouts and dtypes as in pa_slot_mapping and pa_reshape_and_cache (a copy, so
 * bit-exact).  Duplicate slots are undefined.
 */
pa_status pa_slot_mapping_and_cache(const void* k, const void* v, void* k_blocks, void* v_blocks,
                                    const int32_t* query_start_loc, const int32_t* positions,
                                    const int32_t* block_tables, int32_t num_seqs,
                                    int64_t num_tokens, int32_t max_blocks_per_seq,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                    int64_t num_blocks, pa_dtype kv_dtype, int32_t* slot_mapping,
                                    cudaStream_t stream);

/*
 * pa_reshape_and_cache_ex -- the scatter of pa_reshape_and_cache with a conversion: new rows
 * of src_dtype (f32 or bf16) go into pools of kv_dtype (f32, bf16 or fp8 e4m3), element x of
 * K stored as x / k_scale and of V as x / v_scale, the quotient taken in fp32 (IEEE division)
 * and rounded to kv_dtype to nearest, ties to even; an fp8 store saturates to +-448
 * ("paged_attention_v2_pytorch.py": the pool holds K / k_scale, so that K = k_scale * pool).
 * k_scale and v_scale must be finite and positive (PA_EINVAL otherwise).  Slots are checked as
 * in pa_reshape_and_cache.  Same pool layout [num_blocks, block_size, num_kv_heads, head_dim].
 */
pa_status pa_reshape_and_cache_ex(const void* k, const void* v, void* k_blocks, void* v_blocks,
                                  const int32_t* slot_mapping, int64_t num_tokens,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                  int64_t num_blocks, pa_dtype src_dtype, pa_dtype kv_dtype,
                                  float k_scale, float v_scale, cudaStream_t stream);

/*
 * pa_reshape_and_cache_per_head -- pa_reshape_and_cache_ex with one dequantisation scale per
 * kv head (tinyllm "Going further": fp8 KV caches with scales per head): head g of a new row
 * is stored as x / k_scales[g] (x / v_scales[g]).  k_scales, v_scales: DEVICE arrays of
 * num_kv_heads floats owned by the caller, or NULL for 1 on every head.  A scale that is not
 * finite and positive is recorded as PA_EINVAL in the device status (it is only read on the
 * device) and nothing is written; other errors as pa_reshape_and_cache_ex.
 */
pa_status pa_reshape_and_cache_per_head(const void* k, const void* v, void* k_blocks,
                                        void* v_blocks, const int32_t* slot_mapping,
                                        int64_t num_tokens, int32_t num_kv_heads,
                                        int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                        pa_dtype src_dtype, pa_dtype kv_dtype,
                                        const float* k_scales, const float* v_scales,
                                        cudaStream_t stream);

/*
 * pa_reshape_and_cache_per_block -- pa_reshape_and_cache_ex with one dequantisation factor per
 * (pool block, kv head) (tinyllm "Going further": fp8 KV caches with scales per block): head g
 * of a new row written to slot s is stored as x / k_block_scales[(s / block_size) *
 * num_kv_heads + g] (x / v_block_scales[...]).  k_block_scales, v_block_scales: DEVICE arrays
 * [num_blocks, num_kv_heads] of floats owned by the caller, both required (NULL: PA_EINVAL).
 * A factor of a block some row is written to that is not a finite positive normal float (at
 * least 2^-126) is recorded as PA_EINVAL in the device status and nothing is written; other
 * errors as
 * pa_reshape_and_cache_ex.  The caller chooses the factors (for example from a block's
 * largest magnitude when it is allocated); the library does not change them.
 */
pa_status pa_reshape_and_cache_per_block(const void* k, const void* v, void* k_blocks,
                                         void* v_blocks, const int32_t* slot_mapping,
                                         int64_t num_tokens, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t block_size,
                                         int64_t num_blocks, pa_dtype src_dtype,
                                         pa_dtype kv_dtype, const float* k_block_scales,
                                         const float* v_block_scales, cudaStream_t stream);

/*
 * pa_varlen_forward_workspace_size -- bytes of device workspace pa_varlen_forward needs
 * for these sizes (the per-call plan of work items and split-KV partial states).
 */
size_t pa_varlen_forward_workspace_size(int32_t num_seqs, int64_t num_tokens, int32_t num_heads,
                                        int32_t num_kv_heads, int32_t head_dim,
                                        int32_t max_blocks_per_seq, int32_t block_size);

/*
 * pa_varlen_forward -- batched varlen paged attention (TensorSharp Forward /
 * ComputeSingleQueryAttention; tinyllm section 2.2).  One call serves any mix of prefill
 * chunks and decode tokens.  For token t of sequence s at position p and head h, with
 * kv head g = h / (num_heads / num_kv_heads):
 *     end   = causal ? p + 1 : seq_lens[s]
 *     start = sliding_window > 0 ? max(0, end - sliding_window) : 0
 *     out[t, h] = softmax_j(scale * q[t, h] . K_j) V_j   over positions j in [start, end)
 * where K_j, V_j are pool rows of kv head g found through the block table.  out has
 * q_dtype.  k_blocks/v_blocks have kv_dtype (PA_FP8_E4M3: the codes' values, i.e. scales 1;
 * see pa_varlen_forward_ex for scaled pools).
 * Validation (tinyllm section 2.6), for every sequence with at least one query token:
 * seq_lens[s] >= 1, ceil(seq_lens[s] / block_size) <= max_blocks_per_seq, those table
 * entries in [0, num_blocks), positions in [0, seq_lens[s]); query_start_loc starts at 0,
 * never decreases and ends at num_tokens.  Failures record PA_EINVAL and leave out
 * untouched.  workspace must hold pa_varlen_forward_workspace_size(...) bytes, 256-byte
 * aligned; it is scratch owned by the caller and must not be shared by calls that overlap
 * on the device.
 */
pa_status pa_varlen_forward(const void* q, const void* k_blocks, const void* v_blocks, void* out,
                            const int32_t* query_start_loc, const int32_t* seq_lens,
                            const int32_t* positions, const int32_t* block_tables,
                            int32_t num_seqs, int64_t num_tokens, int32_t num_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                            int64_t num_blocks, int32_t max_blocks_per_seq, pa_dtype q_dtype,
                            pa_dtype kv_dtype, float scale, int32_t causal,
                            int32_t sliding_window, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream);

/*
 * pa_varlen_forward_ex -- pa_varlen_forward with optional extras (with sinks and lse NULL and
 * both scales 1 the call is pa_varlen_forward):
 *   sinks  [num_heads] fp32, device.  Per-head attention sink logits on the score scale
 *          (TensorSharp ForwardWithSinks): a virtual position with score sinks[h] and value
 *          zero, so with the visible scores s_j
 *              out[t, h] = sum_j e^(s_j - m) V_j / (e^(sinks[h] - m) + sum_j e^(s_j - m)),
 *          m = max(sinks[h], max_j s_j).  -inf means no sink for that head.  Finite values
 *          and -inf are defined; NaN and +inf are not.
 *   lse    [num_heads, num_tokens] fp32, device, written (the vllm.cpp MLA-prefill layout):
 *              lse[h, t] = log(e^sinks[h] + sum_j e^(s_j))   (natural log, sink term when given)
 *          and -inf when the sum is empty (no visible position and no sink).  It is what
 *          pa_merge_attn_states takes to combine two partial attentions of the same queries.
 *   k_scale, v_scale  dequantisation scales of the pools ("paged_attention_v2_pytorch.py":
 *          K = k_scale * k_blocks, V = v_scale * v_blocks before the attention), finite and
 *          > 0 (PA_EINVAL otherwise).  The scores above are scale * q . K_j with the scaled K.
 *          kv_dtype PA_FP8_E4M3 (pools written by pa_reshape_and_cache_ex) is accepted here:
 *          the pool's codes widen exactly to f16; on the tensor-core path q (bf16) enters the
 *          products as f16, so q entries must lie within f16's range (|q| <= 65504; entries
 *          below 2^-14 keep f16's subnormal precision), and the softmax weights enter the PV
 *          product as f16 (2^-11 relative).  fp8 pools take the tensor-core kernels for head
 *          size 128 with 16-position blocks (warp-MMA for decode tokens, tcgen05 for prefill
 *          chunks, as bf16 pools do) and the generic kernel otherwise.
 *   flags  0, or PA_FLAG_BITWISE: every sequence runs on the 16-row warp-MMA kernel (bf16 or
 *          fp8 pools, head size 64 / 128, 16-position blocks), including prefill-class
 *          sequences that would otherwise take the tensor-core prefill kernel.  That kernel
 *          folds each query row over the same 16-position blocks, in the same order and
 *          grouping, whatever the other rows of the batch are, so a token's out row and lse
 *          have the same bits computed as a decode token (q_len 1) or inside a prefill chunk,
 *          alone or in any batch (tinyllm 2.4: decode equals FlashAttention bit for bit, so
 *          prefill with one kernel and decode with the other agree).  Without the flag this
 *          holds for every sequence of at most 64 query rows per kv head; longer ones take
 *          the tcgen05 kernel, whose 128-key tiles group the sums differently (results within
 *          the tolerance, not bitwise).  Other bits: PA_EINVAL.
 * sinks and lse are read or written only for tokens of sequences with query tokens, and lse
 * is left untouched on a validation failure, like out.
 */
pa_status pa_varlen_forward_ex(const void* q, const void* k_blocks, const void* v_blocks,
                               void* out, const int32_t* query_start_loc,
                               const int32_t* seq_lens, const int32_t* positions,
                               const int32_t* block_tables, int32_t num_seqs, int64_t num_tokens,
                               int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                               int32_t block_size, int64_t num_blocks,
                               int32_t max_blocks_per_seq, pa_dtype q_dtype, pa_dtype kv_dtype,
                               float scale, int32_t causal, int32_t sliding_window,
                               const float* sinks, float* lse, float k_scale, float v_scale,
                               uint32_t flags, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream);

/*
 * pa_varlen_forward_per_head -- pa_varlen_forward_ex with one dequantisation scale per kv
 * head instead of one per pool: query head h (kv head g = h / (num_heads / num_kv_heads))
 * attends over K = k_scales[g] * k_blocks and V = v_scales[g] * v_blocks (tinyllm "Going
 * further": scales per head).  k_scales, v_scales: DEVICE arrays of num_kv_heads floats owned
 * by the caller, or NULL for 1 on every head; a scale that is not finite and positive is
 * recorded as PA_EINVAL in the device status and out / lse are left untouched.  All other
 * arguments, kernels and errors as pa_varlen_forward_ex.
 */
pa_status pa_varlen_forward_per_head(const void* q, const void* k_blocks, const void* v_blocks,
                                     void* out, const int32_t* query_start_loc,
                                     const int32_t* seq_lens, const int32_t* positions,
                                     const int32_t* block_tables, int32_t num_seqs,
                                     int64_t num_tokens, int32_t num_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                     int32_t max_blocks_per_seq, pa_dtype q_dtype,
                                     pa_dtype kv_dtype, float scale, int32_t causal,
                                     int32_t sliding_window, const float* sinks, float* lse,
                                     const float* k_scales, const float* v_scales,
                                     uint32_t flags, void* workspace, size_t workspace_bytes,
                                     cudaStream_t stream);

/*
 * pa_varlen_forward_per_block -- pa_varlen_forward_ex over e4m3 pools with one dequantisation
 * factor per (pool block, kv head) (tinyllm "Going further": scales per block): position j of
 * a sequence, in pool block id = block_tables[s][j / block_size], is read by query head h (kv
 * head g = h / (num_heads / num_kv_heads)) as K = k_block_scales[id * num_kv_heads + g] *
 * k_blocks[...] and V = v_block_scales[...] * v_blocks[...].  k_block_scales, v_block_scales:
 * DEVICE arrays [num_blocks, num_kv_heads] of floats owned by the caller, both required (NULL:
 * PA_EINVAL).  The factors of every block a sequence with query tokens reads (the first
 * ceil(seq_lens[s] / block_size) entries of its table row) must be finite positive normal
 * floats (at least 2^-126), else PA_EINVAL is recorded in the device status and out / lse are left untouched.  kv_dtype must
 * be PA_FP8_E4M3 and the call must qualify for the warp-MMA path (q bf16, head_dim 128,
 * block_size 16, 16-byte aligned tensors), else PA_EUNSUPPORTED before anything is enqueued.
 * Both kernels multiply each block's scores by its K factor in fp32, exactly.  V: the
 * warp-MMA kernel (decode tokens) multiplies the block's softmax weights by the factor over
 * the largest factor the warp has met so far, before the weights are rounded to f16, and that
 * reference multiplies the warp's fp32 output; the tcgen05 kernel (prefill chunks) multiplies
 * the block's widened codes by the factor over its item's reference (the factor of the item's
 * first block), rounded to f16, and the reference multiplies the output.  An item with a V
 * ratio outside [2^-12, 146] is recomputed by the warp-MMA kernel.  So any finite positive
 * factors keep the f16 values in range.  Other arguments and errors as pa_varlen_forward_ex.
 */
pa_status pa_varlen_forward_per_block(const void* q, const void* k_blocks, const void* v_blocks,
                                      void* out, const int32_t* query_start_loc,
                                      const int32_t* seq_lens, const int32_t* positions,
                                      const int32_t* block_tables, int32_t num_seqs,
                                      int64_t num_tokens, int32_t num_heads,
                                      int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                      int64_t num_blocks, int32_t max_blocks_per_seq,
                                      pa_dtype q_dtype, pa_dtype kv_dtype, float scale,
                                      int32_t causal, int32_t sliding_window, const float* sinks,
                                      float* lse, const float* k_block_scales,
                                      const float* v_block_scales, uint32_t flags,
                                      void* workspace, size_t workspace_bytes,
                                      cudaStream_t stream);

/*
 * pa_cache_and_attend -- one decode / prefill step over the cache: pa_slot_mapping_and_cache
 * of the new tokens' rows (k_new, v_new [num_tokens, num_kv_heads, head_dim] of kv_dtype;
 * slot_mapping [num_tokens] written) followed by pa_varlen_forward of q over the updated pools,
 * with the same arguments, results and errors as those two calls made one after the other.
 * For batches of up to 2048 tokens and 2047 sequences the slot mapping and scatter run as one
 * kernel launched right after the attention's planning kernel, overlapping it (neither reads
 * what the other writes), instead of in front of it.
 */
pa_status pa_cache_and_attend(const void* k_new, const void* v_new, const void* q,
                              void* k_blocks, void* v_blocks, void* out,
                              const int32_t* query_start_loc, const int32_t* seq_lens,
                              const int32_t* positions, const int32_t* block_tables,
                              int32_t num_seqs, int64_t num_tokens, int32_t num_heads,
                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                              int64_t num_blocks, int32_t max_blocks_per_seq, pa_dtype q_dtype,
                              pa_dtype kv_dtype, float scale, int32_t causal,
                              int32_t sliding_window, int32_t* slot_mapping, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream);

/*
 * pa_varlen_forward_noalloc -- pa_varlen_forward for callers that cannot allocate device
 * memory.  The pages have no counterpart: it exists for the library's users, not for the
 * method.  Some callers cannot hand this library a workspace: a host framework that gives an
 * op only its input and output buffers and owns all other device memory, a runtime whose
 * allocator is out of reach of the calling code, or a serving step that must not risk the
 * device synchronisation of cudaMalloc / cudaFree.  This call computes exactly what
 * pa_varlen_forward computes (same arguments, minus the workspace) and keeps its per-call
 * plan in a 4 MiB array inside the library, one copy per device, held until the process
 * exits.  It allocates nothing and calls no allocating routine.
 *   - The first call on a device looks up that device's copy of the array (with the
 *     device current); make that first call before capturing the stream into a graph.
 *   - A batch whose pa_varlen_forward_workspace_size(...) exceeds 4 MiB returns PA_EINVAL
 *     at once and enqueues nothing.
 *   - All calls on a device share the array: calls that may overlap on the GPU (different
 *     streams without ordering between them) race and must not be issued.  Calls on one
 *     stream are ordered and safe.  Each call writes every word of the array it later reads,
 *     so nothing has to start at zero.
 */
pa_status pa_varlen_forward_noalloc(const void* q, const void* k_blocks, const void* v_blocks,
                                    void* out, const int32_t* query_start_loc,
                                    const int32_t* seq_lens, const int32_t* positions,
                                    const int32_t* block_tables, int32_t num_seqs,
                                    int64_t num_tokens, int32_t num_heads, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                    int32_t max_blocks_per_seq, pa_dtype q_dtype,
                                    pa_dtype kv_dtype, float scale, int32_t causal,
                                    int32_t sliding_window, cudaStream_t stream);

/*
 * pa_decode_splitkv_partials -- phase 1 of split-KV decode ("paged_attention_v2_pytorch.py",
 * partition loop).  One query per sequence, q [num_seqs, num_heads, head_dim], at position
 * seq_lens[s] - 1 (causal by construction).  Partition p covers positions
 * [p * partition_size, min((p + 1) * partition_size, seq_lens[s])), intersected with the
 * window [max(0, seq_lens[s] - sliding_window), seq_lens[s]) when sliding_window > 0.
 * For every (s, h, p < max_num_partitions):
 *     max_logits[s, h, p] = max_j scale * q . K_j            (-inf if no position)
 *     exp_sums[s, h, p]   = sum_j exp(scale * q . K_j - max)  (0 if no position)
 *     tmp_out[s, h, p, :] = sum_j exp(...) V_j / exp_sum      (zeros if no position)
 * tmp_out holds the NORMALISED partition output (the reading under which the page's
 * reduction is a log-sum-exp merge).  max_logits / exp_sums are fp32 [S, H, P]; tmp_out fp32
 * [S, H, P, D].  Validation: seq_lens[s] >= 1, the table covers ceil(seq_len / block_size)
 * blocks with ids in [0, num_blocks), ceil(seq_len / partition_size) <= max_num_partitions.
 * partition_size must be a positive multiple of block_size.
 */
pa_status pa_decode_splitkv_partials(const void* q, const void* k_blocks, const void* v_blocks,
                                     float* max_logits, float* exp_sums, float* tmp_out,
                                     const int32_t* seq_lens, const int32_t* block_tables,
                                     int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                     int32_t max_blocks_per_seq, int32_t partition_size,
                                     int32_t max_num_partitions, pa_dtype q_dtype,
                                     pa_dtype kv_dtype, float scale, int32_t sliding_window,
                                     cudaStream_t stream);

/*
 * pa_decode_splitkv_partials_ex -- pa_decode_splitkv_partials over scaled pools
 * ("paged_attention_v2_pytorch.py": kv_cache_dtype, k_scale, v_scale; K = k_scale * k_blocks
 * and V = v_scale * v_blocks, both finite and > 0, else PA_EINVAL).  kv_dtype may be
 * PA_FP8_E4M3 (bf16 q and head size 128 take the warp-MMA kernel, with the f16 operand
 * rounding described at pa_varlen_forward_ex).  pa_decode_splitkv_partials is this call with
 * both scales 1; the reduce step needs no scales.
 */
pa_status pa_decode_splitkv_partials_ex(
    const void* q, const void* k_blocks, const void* v_blocks, float* max_logits,
    float* exp_sums, float* tmp_out, const int32_t* seq_lens, const int32_t* block_tables,
    int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, int64_t num_blocks, int32_t max_blocks_per_seq, int32_t partition_size,
    int32_t max_num_partitions, pa_dtype q_dtype, pa_dtype kv_dtype, float scale,
    int32_t sliding_window, float k_scale, float v_scale, cudaStream_t stream);

/*
 * pa_decode_splitkv_partials_per_head -- pa_decode_splitkv_partials_ex with one scale per kv
 * head: k_scales, v_scales are DEVICE arrays of num_kv_heads floats (NULL: 1), validated on
 * the device as in pa_varlen_forward_per_head (PA_EINVAL recorded, partials untouched).
 */
pa_status pa_decode_splitkv_partials_per_head(
    const void* q, const void* k_blocks, const void* v_blocks, float* max_logits,
    float* exp_sums, float* tmp_out, const int32_t* seq_lens, const int32_t* block_tables,
    int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, int64_t num_blocks, int32_t max_blocks_per_seq, int32_t partition_size,
    int32_t max_num_partitions, pa_dtype q_dtype, pa_dtype kv_dtype, float scale,
    int32_t sliding_window, const float* k_scales, const float* v_scales, cudaStream_t stream);

/*
 * pa_decode_splitkv_partials_per_block -- pa_decode_splitkv_partials_ex with one factor per
 * (pool block, kv head), as pa_varlen_forward_per_block (both arrays required; factors of the
 * blocks the sequences read validated on the device: PA_EINVAL recorded, partials untouched;
 * e4m3 pools on the warp-MMA path only, else PA_EUNSUPPORTED).
 */
pa_status pa_decode_splitkv_partials_per_block(
    const void* q, const void* k_blocks, const void* v_blocks, float* max_logits,
    float* exp_sums, float* tmp_out, const int32_t* seq_lens, const int32_t* block_tables,
    int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, int64_t num_blocks, int32_t max_blocks_per_seq, int32_t partition_size,
    int32_t max_num_partitions, pa_dtype q_dtype, pa_dtype kv_dtype, float scale,
    int32_t sliding_window, const float* k_block_scales, const float* v_block_scales,
    cudaStream_t stream);

/*
 * pa_decode_splitkv_reduce -- phase 2 ("Phase 2: Cross-partition reduction").  For each
 * (s, h) over partitions p < ceil(seq_lens[s] / partition_size):
 *     lse_p = max_logits + log(exp_sums), or -inf when max_logits is +/-inf or exp_sums <= 0
 *     M = max_p lse_p;  w_p = exp(lse_p - M);  out = sum_p w_p tmp_out_p * (1 / sum_p w_p)
 * and when every lse_p is -inf, out = tmp_out of partition 0 (the both-minus-infinity rule of
 * vllm.cpp MergeAttnStatesKernel, extended to P partitions).  Partitions combine in
 * increasing p.  out is [num_seqs, num_heads, head_dim] in out_dtype.
 */
pa_status pa_decode_splitkv_reduce(void* out, const float* max_logits, const float* exp_sums,
                                   const float* tmp_out, const int32_t* seq_lens,
                                   int32_t num_seqs, int32_t num_heads, int32_t head_dim,
                                   int32_t partition_size, int32_t max_num_partitions,
                                   pa_dtype out_dtype, cudaStream_t stream);

/* pa_decode_splitkv -- pa_decode_splitkv_partials followed by pa_decode_splitkv_reduce on
 * the same stream; the partial buffers are caller-owned scratch. */
pa_status pa_decode_splitkv(const void* q, const void* k_blocks, const void* v_blocks, void* out,
                            float* max_logits, float* exp_sums, float* tmp_out,
                            const int32_t* seq_lens, const int32_t* block_tables,
                            int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                            int32_t head_dim, int32_t block_size, int64_t num_blocks,
                            int32_t max_blocks_per_seq, int32_t partition_size,
                            int32_t max_num_partitions, pa_dtype q_dtype, pa_dtype kv_dtype,
                            float scale, int32_t sliding_window, cudaStream_t stream);

/*
 * pa_merge_attn_states -- merge two attention states of the same queries (vllm.cpp
 * cpu_mla_prefill.cpp, MergeAttnStatesKernel).  out/prefix_out/suffix_out [T, H, D] in dtype;
 * lse arrays fp32 [H, T]; out_lse may be NULL.  Tokens t >= prefill_tokens_with_context
 * (when that is >= 0) copy the suffix and its lse.  Otherwise an infinite lse of either sign
 * counts as -inf; if both are -inf the prefix output is emitted with lse -inf; else
 *     p_scale = p_se / (p_se + s_se), s_scale = s_se / (p_se + s_se),
 *     p_se = exp(p_lse - max), s_se = exp(s_lse - max),
 *     out = prefix * p_scale + suffix * s_scale,  out_lse = log(p_se + s_se) + max.
 */
pa_status pa_merge_attn_states(void* out, float* out_lse, const void* prefix_out,
                               const float* prefix_lse, const void* suffix_out,
                               const float* suffix_lse, int64_t num_tokens, int32_t num_heads,
                               int32_t head_dim, int64_t prefill_tokens_with_context,
                               pa_dtype dtype, cudaStream_t stream);

/*
 * pa_gather_kv -- copy sequences' cached rows into dense buffers (vllm.cpp
 * GatherMlaCacheKernel).  Output rows [cu_seq_lens[s], cu_seq_lens[s + 1]) receive the pool
 * rows (all kv heads) at positions (r - cu_seq_lens[s]) + seq_starts[s] of sequence s;
 * seq_starts may be NULL (all 0).  k_out/v_out are [cu_seq_lens[num_seqs], num_kv_heads,
 * head_dim]; v_blocks and v_out may both be NULL.  A position past the table row or a block
 * id outside the pool records PA_EINVAL and writes nothing.  Bit-exact copy.
 */
pa_status pa_gather_kv(const void* k_blocks, const void* v_blocks, void* k_out, void* v_out,
                       const int32_t* cu_seq_lens, const int32_t* seq_starts,
                       const int32_t* block_tables, int32_t num_seqs, int64_t num_out_rows,
                       int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                       int64_t num_blocks, int32_t max_blocks_per_seq, pa_dtype kv_dtype,
                       cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
