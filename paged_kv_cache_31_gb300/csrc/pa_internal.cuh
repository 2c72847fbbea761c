// pa_internal.cuh -- shared device helpers and launch interfaces of libpa (sm_103a only).
//
// Nothing here is part of the public ABI (include/pa.h).  The helpers wrap the PTX the
// kernels use directly: mbarrier phases with bounded waits, 3-D TMA tile loads, ldmatrix,
// the bf16 m16n8k16 warp MMA, and the device status word.
#pragma once

#include <cuda.h>  // CUtensorMap (type only; the driver is reached through cudaGetDriverEntryPoint)
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

#if defined(__CUDA_ARCH__) && (__CUDA_ARCH__ < 1000)
#error "libpa is written for sm_103a (Blackwell) only"
#endif

namespace pa {

// ------------------------------------------------------------------------------------------
// device status word

__device__ __forceinline__ void record_error(int* status, int code) {
  atomicCAS(status, 0, code);  // the first error wins; later ones keep it
}

__device__ __forceinline__ bool status_set(const int* status) {
  return *reinterpret_cast<const volatile int*>(status) != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------------------------------
// shared memory, mbarriers, TMA

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for phase `parity` of `bar` to complete, for at most `limit_ns` of wall time.
// Returns false when the limit ran out (the caller records PA_ETIMEOUT and unwinds).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 31u) == 0 && globaltimer_ns() - t0 > limit_ns) return false;
  }
}

// Programmatic dependent launch.  A kernel launched with programmatic stream serialization
// may start while the kernel before it on the stream still runs; pdl_wait() returns once that
// kernel has finished and its writes are visible (at once when there is no such dependency).
// pdl_launch_dependents() lets the next such kernel be scheduled early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch `kern` with programmatic stream serialization: it may be scheduled while the kernel
// before it on the stream still runs, so it must call pdl_wait() before it touches anything an
// earlier kernel (of this library or the caller) may write.
template <typename... Exp, typename... Act>
inline cudaError_t launch_pdl(void (*kern)(Exp...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Act&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Act&&>(args)...);
}

// 3-D tiled TMA load global -> shared, completing `bytes` on `bar`.  c0 is the innermost
// coordinate; callers keep c0 * sizeof(element) a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_3d(void* smem_dst, const CUtensorMap* map, int32_t c0,
                                            int32_t c1, int32_t c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------------------------------
// warp-level tensor-core helpers (bf16 m16n8k16, fp32 accumulate)

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                              uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr)
               : "memory");
}

__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32"
      " {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// The same MMA with f16 operands (the fp8 pools' path: e4m3 widens to f16 exactly).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32"
      " {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Two e4m3 codes (the low byte is the element at the lower address) -> f16x2, exactly.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t codes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(codes));
  return r;
}
// Four codes of a 32-bit word -> two f16x2 words, in element order.
__device__ __forceinline__ void e4m3x4_to_f16(uint32_t w, uint32_t& lo, uint32_t& hi) {
  lo = e4m3x2_to_f16x2((uint16_t)(w & 0xffffu));
  hi = e4m3x2_to_f16x2((uint16_t)(w >> 16));
}
// Two floats -> two e4m3 codes (saturating to +-448, round to nearest even), a at the lower
// address.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

// ------------------------------------------------------------------------------------------
// element access for the generic kernels

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

// An e4m3 pool element (the code; its value widens exactly through f16).
struct e4m3_t {
  uint8_t bits;
};
template <>
__device__ __forceinline__ float to_f32<e4m3_t>(e4m3_t x) {
  const uint32_t h = e4m3x2_to_f16x2((uint16_t)x.bits);
  return __half2float(__ushort_as_half((unsigned short)(h & 0xffffu)));
}

template <typename T>
__device__ __forceinline__ T from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint64_t kWaitLimitNs = 4000000000ull;  // 4 s: a TMA that has not landed by then never will

// ------------------------------------------------------------------------------------------
// per-call plan kept in the caller's workspace (int32 words)
//   [0] number of warp-MMA tile items (16 query rows, 8 on e4m3 pools; decode-class sequences)
//   [1] number of 256-row items (prefill-class sequences, tcgen05 kernel)
//   [2] work counter of the warp-MMA kernel (zeroed by the plan)
//   [3] number of 256-row items the tcgen05 kernel marked for recomputing (zeroed by the plan)
//   [4] work counter of the warp-MMA kernel over those items (zeroed by the plan)
//   [5] CTA pairs of the tcgen05 kernel that take 256-row items (the others leave at once,
//       and their SMs run the warp-MMA kernel's decode tiles meanwhile)
//   [6..15] reserved
//   [tok_off, tok_off + T)        token -> sequence
//   [cost_off, cost_off + S)      per sequence: keys its query rows can see (work estimate;
//                                 written only for batches too large to keep it in smem)
//   [mma_off, + 8 * mma_cap)      warp-MMA tile records, longest first: two int4 each,
//                                 (seq, tile index, query start, seq_len) and (union of the
//                                 tile's rows' visible key ranges [lo, hi), q_len * G, 0)
//   [tc_off, + 4 * tc_cap)        int4 items (seq, 256-row item, kv lo, kv hi), longest first
//   [tc_tmp_off, + 4 * tc_cap)    the same items in sequence order (planning scratch)
//   [redo_off, + tc_cap)          per 256-row item: marked for recomputing (zeroed by the plan)
//   [redo_list_off, + tc_cap)     the marked items, in the order they were marked
constexpr int kPlanHeaderWords = 16;

struct PlanLayout {
  int64_t tok_off, cost_off, mma_off, tc_off, tc_tmp_off, redo_off, redo_list_off;
  int64_t mma_cap, tc_cap;
  int64_t words;
  int32_t use_tc;       // prefill-class sequences go to the tcgen05 kernel
  int32_t tc_min_rows;  // a sequence is prefill-class when q_len * G exceeds this
  // Split of the SMs between the tcgen05 kernel and the warp-MMA kernel that runs beside it
  // (plan word [5]): the plan picks the number of CTA pairs K for the 256-row items that
  // minimises max(margin * T_prefill(K), T_decode(num_sms - 2 K)), with
  //   T_prefill(K) = (128-key tiles of all items) * tile_ns / K   (tiles spread over K pairs)
  //   T_decode(m)  = decode K/V bytes / hbm_bytes_per_ns * max(1, decode_sat_sms / m)
  // (decode tiles stream K/V at the HBM rate on decode_sat_sms SMs or more).  Ties go to the
  // larger K: the prefill then ends first and its SMs join the decode tiles.
  int32_t tc_pairs;        // CTA pairs the tcgen05 kernel is launched with
  int32_t num_sms;
  int32_t force_pairs;     // > 0: use this many pairs (measurements), else the model
  int32_t decode_sat_sms;
  float tile_ns;           // one 128-key tile of a 256-row item on one pair
  float hbm_bytes_per_ns;  // decode tiles' K/V streaming rate on the whole GPU
  float margin;            // the prefill estimate is taken this much longer
  int32_t kv_elem_bytes;   // bytes of one pool element (2 bf16, 1 e4m3), for the decode bytes
  int32_t mma_tile_rows;   // query rows per warp-MMA tile: 16, or 8 on e4m3 pools
  int32_t need_tok_map;    // the scalar kernel runs: write the token -> sequence map
};

// Layout of the plan for a batch of num_tokens tokens over num_seqs sequences.
inline PlanLayout plan_layout(int32_t num_seqs, int64_t num_tokens, int32_t group) {
  PlanLayout L;
  L.tok_off = kPlanHeaderWords;
  L.mma_cap = (num_tokens * group + 7) / 8 + num_seqs + 1;  // room for 8-row tiles
  L.tc_cap = (num_tokens * group + 255) / 256 + num_seqs + 1;
  L.cost_off = L.tok_off + num_tokens;
  L.mma_off = (L.cost_off + num_seqs + 3) & ~int64_t(3);
  L.tc_off = (L.mma_off + 8 * L.mma_cap + 3) & ~int64_t(3);
  L.tc_tmp_off = L.tc_off + 4 * L.tc_cap;
  L.redo_off = L.tc_tmp_off + 4 * L.tc_cap;
  L.redo_list_off = L.redo_off + L.tc_cap;
  L.words = L.redo_list_off + L.tc_cap;
  L.use_tc = 0;
  L.tc_min_rows = 64;
  L.tc_pairs = 0;
  L.num_sms = 0;
  L.force_pairs = 0;
  L.decode_sat_sms = 80;
  L.tile_ns = 1300.f;
  L.hbm_bytes_per_ns = 6700.f;
  L.margin = 1.1f;
  L.kv_elem_bytes = 2;
  L.mma_tile_rows = 16;
  L.need_tok_map = 1;
  return L;
}

struct VarlenMeta {
  const int32_t* query_start_loc;
  const int32_t* seq_lens;
  const int32_t* positions;
  const int32_t* block_tables;
  int32_t num_seqs;
  int64_t num_tokens;
  int32_t num_heads;
  int32_t num_kv_heads;
  int32_t group;  // num_heads / num_kv_heads
  int32_t head_dim;
  int32_t block_size;
  int64_t num_blocks;
  int32_t max_blocks;
  int32_t causal;
  int32_t window;
  const float* sinks;  // [num_heads] sink logits on the score scale, or null (varlen only)
  float* lse;          // [num_heads, num_tokens] natural-log lse out, or null (varlen only)
  float v_scale;       // V = v_scale * pool: applied to the normalised output (1 = none)
  // one dequantisation scale per kv head (device, [num_kv_heads]), or null: K of kv head g is
  // k_scales[g] * pool (taken with the score scale), V is v_scales[g] * pool
  const float* k_scales;
  const float* v_scales;
  // one factor per (pool block, kv head) (device, [num_blocks, num_kv_heads]), or null:
  // position j of kv head g reads K = k_bscales[id * Hkv + g] * pool, id = its block (e4m3
  // pools, the warp-MMA kernel); checked by the planner's table checks
  const float* k_bscales;
  const float* v_bscales;
};

// The scale of kv head g from a per-head array, times the per-pool scalar; the scalar alone
// when there is no array (no extra rounding step then).
__device__ __forceinline__ float head_scale(const float* s, int g, float scalar) {
  return s ? scalar * __ldg(s + g) : scalar;
}

struct Mma16Params {
  const __nv_bfloat16* q;
  void* out;  // bf16 [T, H, D] (varlen) / [S, H, D]
  VarlenMeta m;
  const int32_t* plan;  // varlen: workspace plan; split: nullptr
  int64_t items_off;    // varlen: word offset of the tile records in the plan
  int* status;
  float scale_log2;  // scale * log2(e)
  // split-KV partial outputs (mode split)
  float* max_logits;
  float* exp_sums;
  float* tmp_out;
  int32_t partition_size;
  int32_t max_parts;
  uint64_t wait_limit_ns;
  uint32_t debug_stall;  // tests only: every block wait runs out (see mma_debug_stall)
  // varlen, launched behind the tcgen05 kernel: the decode tiles do not wait for that kernel
  // (the plan is complete once it has started), and the 256-row items it marked are
  // recomputed after it has finished, 16 rows x one kv head per unit
  int32_t after_tc;
  int64_t tc_off;         // word offset of the int4 256-row items
  int64_t redo_list_off;  // word offset of the list of marked items
};

struct SimtParams {
  const void* q;
  const void* k_blocks;
  const void* v_blocks;
  void* out;
  VarlenMeta m;
  const int32_t* plan;  // token -> seq at plan + kPlanHeaderWords
  int* status;
  float scale;  // includes k_scale
  int32_t q_bf16, kv_bf16, kv_fp8;
  // split-KV mode (out unused): one warp per (s, h, p)
  float* max_logits;
  float* exp_sums;
  float* tmp_out;
  int32_t partition_size;
  int32_t max_parts;
  int32_t split;
};

struct TcParams {
  void* out;  // bf16 [T, H, D]
  VarlenMeta m;
  const int32_t* plan;
  int64_t tc_off;  // word offset of the int4 item list
  int* status;
  float scale_log2;
  uint64_t wait_limit_ns;
  uint32_t debug_stall;  // tests only: the softmax waits run out (PA_DEBUG_STALL_NS)
  int32_t kv_fp8;        // e4m3 pools (tk: 128 x 1 x 16 byte boxes, tv: 64 x 1 x 16)
  // items whose V does not fit f16 (recomputed by the warp-MMA kernel afterwards): a flag per
  // 256-row item, the list of marked items and its length (all in the plan)
  int32_t* redo_flags;
  int32_t* redo_list;
  int32_t* redo_count;
};

// ---- launchers (defined next to their kernels) --------------------------------------------
cudaError_t launch_plan_varlen(const VarlenMeta& m, int32_t* plan, const PlanLayout& L,
                               int* status, cudaStream_t stream);
cudaError_t launch_tc_prefill(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const TcParams& p, int grid, cudaStream_t stream);
cudaError_t launch_validate_decode(const int32_t* seq_lens, const int32_t* block_tables,
                                   int32_t num_seqs, int32_t max_blocks, int32_t block_size,
                                   int64_t num_blocks, int32_t partition_size, int32_t max_parts,
                                   int check_tables, int* status, cudaStream_t stream,
                                   const float* k_bscales = nullptr,
                                   const float* v_bscales = nullptr, int32_t num_kv_heads = 0);
cudaError_t launch_slot_mapping(const int32_t* qsl, const int32_t* positions,
                                const int32_t* block_tables, int32_t num_seqs, int64_t num_tokens,
                                int32_t max_blocks, int32_t block_size, int64_t num_blocks,
                                int32_t* slots, int* status, cudaStream_t stream);
cudaError_t launch_reshape_and_cache(const void* k, const void* v, void* k_blocks, void* v_blocks,
                                     const int32_t* slots, int64_t num_tokens, int64_t row_bytes,
                                     int32_t block_size, int64_t num_blocks, int* status,
                                     cudaStream_t stream);
// pa_slot_mapping followed by pa_reshape_and_cache, in one launch for decode-sized batches.
cudaError_t launch_slot_mapping_and_cache(const void* k, const void* v, void* k_blocks,
                                          void* v_blocks, const int32_t* qsl,
                                          const int32_t* positions, const int32_t* tables,
                                          int32_t num_seqs, int64_t num_tokens,
                                          int32_t max_blocks, int32_t block_size,
                                          int64_t num_blocks, int64_t row_bytes, int32_t* slots,
                                          int* status, cudaStream_t stream);
// The same, launched right after an attention call's plan kernel so that the two overlap
// (decode-sized batches only: map_and_scatter_fits).
bool map_and_scatter_fits(int32_t num_seqs, int64_t num_tokens);
cudaError_t launch_map_and_scatter_after_plan(const void* k, const void* v, void* k_blocks,
                                              void* v_blocks, const int32_t* qsl,
                                              const int32_t* positions, const int32_t* tables,
                                              int32_t num_seqs, int64_t num_tokens,
                                              int32_t max_blocks, int32_t block_size,
                                              int64_t num_blocks, int64_t row_bytes,
                                              int32_t* slots, int* status, cudaStream_t stream);
// Scatter with conversion: element x of K (V) is stored as x / k_scale (x / v_scale), the
// quotient rounded to the pool's type.  src_bf16: new rows are bf16 (else f32); dst: the
// pool's pa_dtype.  row_elems = num_kv_heads * head_dim.
cudaError_t launch_reshape_and_cache_convert(const void* k, const void* v, void* k_blocks,
                                             void* v_blocks, const int32_t* slots,
                                             int64_t num_tokens, int64_t row_elems,
                                             int32_t block_size, int64_t num_blocks, int src_bf16,
                                             int dst, float k_scale, float v_scale,
                                             const float* k_scales, const float* v_scales,
                                             int32_t head_dim, int* status, cudaStream_t stream,
                                             const float* k_bscales = nullptr,
                                             const float* v_bscales = nullptr);
// Records PA_EINVAL when a per-head scale (either array may be null) is not finite and > 0.
cudaError_t launch_validate_scales(const float* k_scales, const float* v_scales,
                                   int32_t num_kv_heads, int* status, cudaStream_t stream);
cudaError_t launch_gather_kv(const void* k_blocks, const void* v_blocks, void* k_out, void* v_out,
                             const int32_t* cu, const int32_t* starts, const int32_t* tables,
                             int32_t num_seqs, int64_t num_rows, int64_t row_bytes,
                             int32_t block_size, int64_t num_blocks, int32_t max_blocks,
                             int* status, cudaStream_t stream);
cudaError_t launch_mma16_varlen(const CUtensorMap& tk, const CUtensorMap& tv, const Mma16Params& p,
                                int head_dim, int items_cap, cudaStream_t stream);
// The same kernel over e4m3 pools (head size 128; tk / tv are byte maps, box 128 x 1 x 16).
cudaError_t launch_mma16_varlen_fp8(const CUtensorMap& tk, const CUtensorMap& tv,
                                    const Mma16Params& p, int items_cap, cudaStream_t stream);
cudaError_t launch_mma16_split_fp8(const CUtensorMap& tk, const CUtensorMap& tv,
                                   const Mma16Params& p, cudaStream_t stream);
cudaError_t launch_mma16_split(const CUtensorMap& tk, const CUtensorMap& tv, const Mma16Params& p,
                               int head_dim, cudaStream_t stream);
cudaError_t launch_simt(const SimtParams& p, cudaStream_t stream);
cudaError_t launch_splitkv_reduce(void* out, int out_bf16, const float* max_logits,
                                  const float* exp_sums, const float* tmp_out,
                                  const int32_t* seq_lens, int32_t num_seqs, int32_t num_heads,
                                  int32_t head_dim, int32_t partition_size, int32_t max_parts,
                                  int* status, cudaStream_t stream);
cudaError_t launch_merge_attn_states(void* out, float* out_lse, const void* prefix_out,
                                     const float* prefix_lse, const void* suffix_out,
                                     const float* suffix_lse, int64_t num_tokens,
                                     int32_t num_heads, int32_t head_dim, int64_t prefix_tokens,
                                     int bf16, int* status, cudaStream_t stream);

int num_sms();  // SM count of the current device (cached)
void* current_context();  // the calling thread's current driver context (CUcontext), or null
// argument checks of the varlen attention calls (all but the workspace); see pa_api.cu
pa_status varlen_check(const void* q, const void* k_blocks, const void* v_blocks,
                       const void* out, const int32_t* query_start_loc, const int32_t* seq_lens,
                       const int32_t* positions, const int32_t* block_tables, int32_t num_seqs,
                       int64_t num_tokens, int32_t num_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, int64_t num_blocks,
                       int32_t max_blocks_per_seq, pa_dtype q_dtype, pa_dtype kv_dtype,
                       float k_scale, float v_scale, uint32_t flags, bool* empty);

}  // namespace pa
