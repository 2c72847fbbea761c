// pa_api.cu -- the C ABI of libpa (include/pa.h): argument checks, tensor-map encoding,
// path selection and kernel launches.  No device memory is allocated here.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "pa_internal.cuh"

// Sticky per-device status word (one copy per device context): the first error a kernel
// records stays until pa_device_status() reads and clears it.
__device__ int g_pa_status = 0;

namespace pa {

// The driver context current on this thread (CUcontext), or nullptr when there is none or the
// driver entry point cannot be had.
void* current_context() {
  static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
  });
  CUcontext c = nullptr;
  if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
  return c;
}

namespace {

constexpr int kMaxDevices = 64;

struct DeviceState {
  void* ctx = nullptr;  // the context the address below was looked up in
  int* status = nullptr;
  int sms = 0;
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Status-word address and SM count of the current device, looked up with that device
// current, and again whenever the current context is not the one of the last lookup (after
// cudaDeviceReset, or under another driver context, the module is loaded anew and its
// __device__ variables may sit elsewhere).
const DeviceState* device_state() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* ctx = current_context();
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& d = g_dev[dev];
  if (!d.status || !ctx || d.ctx != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pa_status) != cudaSuccess) return nullptr;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return nullptr;
    d.sms = sms;
    d.status = static_cast<int*>(p);
    // looked up again (the runtime may have just made the primary context current)
    d.ctx = current_context();
  }
  return &d;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// TMA descriptor of a bf16 pool [num_blocks, 16, Hkv, D] seen as the 3-D tensor
// (D, Hkv, num_blocks * 16) with a 64 x 1 x 16 box and the 128-byte swizzle.
bool pool_map(CUtensorMap* map, const void* base, int64_t num_blocks, int block_size, int hkv,
              int d) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)hkv, (cuuint64_t)(num_blocks * block_size)};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)hkv * d * 2};
  cuuint32_t box[3] = {64, 1, 16};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// TMA descriptor of an fp8 pool [num_blocks, 16, Hkv, 128] (one byte per element) seen as
// the 3-D byte tensor (128, Hkv, num_blocks * 16): one 128 x 1 x 16 box is a whole K (or V)
// block tile of one kv head, 2 KB, with the 128-byte swizzle.
bool pool_map_fp8(CUtensorMap* map, const void* base, int64_t num_blocks, int block_size,
                  int hkv, int d) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)hkv, (cuuint64_t)(num_blocks * block_size)};
  cuuint64_t strides[2] = {(cuuint64_t)d, (cuuint64_t)hkv * d};
  cuuint32_t box[3] = {128, 1, 16};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same byte tensor with a 64 x 1 x 16 box and no swizzle: the 64 dims of one half of a
// head size of 128 for one (block, kv head), 1 KB of plain 64-byte rows (the tcgen05 prefill
// kernel's V part of a CTA).
bool pool_map_fp8_half(CUtensorMap* map, const void* base, int64_t num_blocks, int block_size,
                       int hkv, int d) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)hkv, (cuuint64_t)(num_blocks * block_size)};
  cuuint64_t strides[2] = {(cuuint64_t)d, (cuuint64_t)hkv * d};
  cuuint32_t box[3] = {64, 1, 16};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// TMA descriptor of q [T, H, D] bf16 seen as the 3-D tensor (D, H, T): a 64 x G x 128/G box
// is the 64-dim half of a 128-row query tile whose rows are the G heads of one kv head for
// 128/G consecutive tokens.
bool query_map(CUtensorMap* map, const void* q, int64_t num_tokens, int h, int d, int group) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)h, (cuuint64_t)num_tokens};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)h * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)group, (cuuint32_t)(128 / group)};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The tcgen05 prefill kernel can be switched off with PA_DISABLE_TC=1 (the prefill-class
// sequences then run on the 16-row warp-MMA kernel), for A/B comparisons.
bool tc_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("PA_DISABLE_TC");
    return !(v && v[0] == '1');
  }();
  return on;
}

// Test hook of the attention kernels (PA_DEBUG_STALL_NS=<ns>, read at every call): every
// wait then has a bound of <ns>, and the warp-MMA kernels' block waits and the tcgen05
// kernel's softmax waits name a barrier that nothing signals, so they run out and the kernel
// records PA_ETIMEOUT and unwinds (waiting for its own copies and MMAs still in flight)
// exactly as from a copy or an MMA that never completed.  Unset: real waits, bounded at 4 s.
void stall_hook(uint64_t& limit, uint32_t& stall) {
  limit = kWaitLimitNs;
  stall = 0;
  const char* v = std::getenv("PA_DEBUG_STALL_NS");
  if (v && *v) {
    char* end = nullptr;
    const unsigned long long x = std::strtoull(v, &end, 10);
    if (end && *end == 0 && x > 0 && x <= kWaitLimitNs) {
      limit = x;
      stall = 1;
    }
  }
}
void mma_waits(Mma16Params& p) { stall_hook(p.wait_limit_ns, p.debug_stall); }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
bool dtype_ok(pa_dtype t) { return t == PA_F32 || t == PA_BF16; }  // q, out, new rows
bool pool_dtype_ok(pa_dtype t) { return dtype_ok(t) || t == PA_FP8_E4M3; }
int esize(pa_dtype t) { return t == PA_FP8_E4M3 ? 1 : t == PA_BF16 ? 2 : 4; }
// dequantisation scales: finite and positive
bool scale_ok(float s) { return s > 0.f && s <= 3.402823466e38f; }

pa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? PA_OK : PA_ECUDA; }

// Fast path of the attention kernels: bf16 q and pool, head size 64 or 128, 16-position
// blocks, TMA-compatible pool addresses.
bool mma_path(pa_dtype q_dtype, pa_dtype kv_dtype, int32_t head_dim, int32_t block_size,
              const void* q, const void* kb, const void* vb, const void* out) {
  return q_dtype == PA_BF16 && kv_dtype == PA_BF16 && (head_dim == 64 || head_dim == 128) &&
         block_size == 16 && aligned(kb, 16) && aligned(vb, 16) && aligned(q, 4) &&
         (out == nullptr || aligned(out, 16));
}

// The same kernel over fp8 pools: bf16 q, head size 128.
bool mma_path_fp8(pa_dtype q_dtype, pa_dtype kv_dtype, int32_t head_dim, int32_t block_size,
                  const void* q, const void* kb, const void* vb, const void* out) {
  return q_dtype == PA_BF16 && kv_dtype == PA_FP8_E4M3 && head_dim == 128 && block_size == 16 &&
         aligned(kb, 16) && aligned(vb, 16) && aligned(q, 4) &&
         (out == nullptr || aligned(out, 16));
}

}  // namespace

int num_sms() {
  const DeviceState* d = device_state();
  return d ? d->sms : 0;
}

// The argument checks of the varlen attention calls, in their order, except for the
// workspace: shapes (PA_ESHAPE), types (PA_EUNSUPPORTED), scales and flags (PA_EINVAL), head
// size (PA_EUNSUPPORTED), negative counts (PA_EINVAL), token count (PA_EUNSUPPORTED), then
// null pointers (PA_EINVAL).  *empty is set for a batch with no sequence and no token, which
// is PA_OK with nothing to launch (pointers unchecked).
pa_status varlen_check(const void* q, const void* k_blocks, const void* v_blocks,
                       const void* out, const int32_t* query_start_loc, const int32_t* seq_lens,
                       const int32_t* positions, const int32_t* block_tables, int32_t num_seqs,
                       int64_t num_tokens, int32_t num_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t block_size, int64_t num_blocks,
                       int32_t max_blocks_per_seq, pa_dtype q_dtype, pa_dtype kv_dtype,
                       float k_scale, float v_scale, uint32_t flags, bool* empty) {
  *empty = false;
  if (num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      num_heads % num_kv_heads != 0)
    return PA_ESHAPE;
  if (!dtype_ok(q_dtype) || !pool_dtype_ok(kv_dtype)) return PA_EUNSUPPORTED;
  if (!scale_ok(k_scale) || !scale_ok(v_scale)) return PA_EINVAL;
  if (flags & ~(uint32_t)PA_FLAG_BITWISE) return PA_EINVAL;
  if (head_dim > 256) return PA_EUNSUPPORTED;
  if (num_seqs < 0 || num_tokens < 0 || num_blocks < 0 || max_blocks_per_seq < 0) return PA_EINVAL;
  if (num_tokens > INT32_MAX / 2) return PA_EUNSUPPORTED;
  if (num_seqs == 0 && num_tokens == 0) {
    *empty = true;
    return PA_OK;
  }
  if (!q || !k_blocks || !v_blocks || !out || !query_start_loc || !seq_lens || !positions ||
      !block_tables)
    return PA_EINVAL;
  return PA_OK;
}


}  // namespace pa

using namespace pa;

extern "C" {

int pa_version(void) { return 100; }

const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "PA_OK";
    case PA_EINVAL: return "PA_EINVAL";
    case PA_ESHAPE: return "PA_ESHAPE";
    case PA_EUNSUPPORTED: return "PA_EUNSUPPORTED";
    case PA_ECUDA: return "PA_ECUDA";
    case PA_ETIMEOUT: return "PA_ETIMEOUT";
  }
  return "PA_UNKNOWN";
}

pa_status pa_device_status(cudaStream_t stream) {
  const DeviceState* d = device_state();
  if (!d) return PA_ECUDA;
  int v = 0;
  if (cudaMemcpyAsync(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return PA_ECUDA;
  if (cudaMemsetAsync(d->status, 0, sizeof(int), stream) != cudaSuccess) return PA_ECUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return PA_ECUDA;
  return static_cast<pa_status>(v);
}

pa_status pa_slot_mapping(const int32_t* query_start_loc, const int32_t* positions,
                          const int32_t* block_tables, int32_t num_seqs, int64_t num_tokens,
                          int32_t max_blocks_per_seq, int32_t block_size, int64_t num_blocks,
                          int32_t* slot_mapping, cudaStream_t stream) {
  if (num_seqs < 0 || num_tokens < 0 || max_blocks_per_seq < 0 || num_blocks < 0) return PA_EINVAL;
  if (block_size <= 0) return PA_ESHAPE;
  if (num_seqs == 0) return PA_OK;
  if (!query_start_loc || !positions || !block_tables || !slot_mapping) return PA_EINVAL;
  if (num_blocks * block_size > INT32_MAX) return PA_EUNSUPPORTED;  // slots are int32
  const DeviceState* d = device_state();
  if (!d) return PA_ECUDA;
  return from_cuda(launch_slot_mapping(query_start_loc, positions, block_tables, num_seqs,
                                       num_tokens, max_blocks_per_seq, block_size, num_blocks,
                                       slot_mapping, d->status, stream));
}

pa_status pa_reshape_and_cache(const void* k, const void* v, void* k_blocks, void* v_blocks,
                               const int32_t* slot_mapping, int64_t num_tokens,
                               int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                               int64_t num_blocks, pa_dtype kv_dtype, cudaStream_t stream) {
  if (num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0) return PA_ESHAPE;
  if (!pool_dtype_ok(kv_dtype)) return PA_EUNSUPPORTED;
  if (num_tokens < 0 || num_blocks < 0) return PA_EINVAL;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !k_blocks || !v_blocks || !slot_mapping) return PA_EINVAL;
  const DeviceState* d = device_state();
  if (!d) return PA_ECUDA;
  const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * esize(kv_dtype);
  return from_cuda(launch_reshape_and_cache(k, v, k_blocks, v_blocks, slot_mapping, num_tokens,
                                            row_bytes, block_size, num_blocks, d->status, stream));
}

pa_status pa_slot_mapping_and_cache(const void* k, const void* v, void* k_blocks, void* v_blocks,
                                    const int32_t* query_start_loc, const int32_t* positions,
                                    const int32_t* block_tables, int32_t num_seqs,
                                    int64_t num_tokens, int32_t max_blocks_per_seq,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                    int64_t num_blocks, pa_dtype kv_dtype, int32_t* slot_mapping,
                                    cudaStream_t stream) {
  if (num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0) return PA_ESHAPE;
  if (!pool_dtype_ok(kv_dtype)) return PA_EUNSUPPORTED;
  if (num_seqs < 0 || num_tokens < 0 || max_blocks_per_seq < 0 || num_blocks < 0)
    return PA_EINVAL;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !k_blocks || !v_blocks || !query_start_loc || !positions || !block_tables ||
      !slot_mapping)
    return PA_EINVAL;
  if (num_blocks * block_size > INT32_MAX) return PA_EUNSUPPORTED;  // slots are int32
  const DeviceState* d = device_state();
  if (!d) return PA_ECUDA;
  const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * esize(kv_dtype);
  return from_cuda(launch_slot_mapping_and_cache(
      k, v, k_blocks, v_blocks, query_start_loc, positions, block_tables, num_seqs, num_tokens,
      max_blocks_per_seq, block_size, num_blocks, row_bytes, slot_mapping, d->status, stream));
}

pa_status pa_reshape_and_cache_ex(const void* k, const void* v, void* k_blocks, void* v_blocks,
                                  const int32_t* slot_mapping, int64_t num_tokens,
                                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                                  int64_t num_blocks, pa_dtype src_dtype, pa_dtype kv_dtype,
                                  float k_scale, float v_scale, cudaStream_t stream) {
  if (num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0) return PA_ESHAPE;
  if (!dtype_ok(src_dtype) || !pool_dtype_ok(kv_dtype)) return PA_EUNSUPPORTED;
  if (num_tokens < 0 || num_blocks < 0) return PA_EINVAL;
  if (!scale_ok(k_scale) || !scale_ok(v_scale)) return PA_EINVAL;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !k_blocks || !v_blocks || !slot_mapping) return PA_EINVAL;
  const DeviceState* d = device_state();
  if (!d) return PA_ECUDA;
  return from_cuda(launch_reshape_and_cache_convert(
      k, v, k_blocks, v_blocks, slot_mapping, num_tokens, (int64_t)num_kv_heads * head_dim,
      block_size, num_blocks, src_dtype == PA_BF16, kv_dtype, k_scale, v_scale, nullptr, nullptr,
      head_dim, d->status, stream));
}

pa_status pa_reshape_and_cache_per_head(const void* k, const void* v, void* k_blocks,
                                        void* v_blocks, const int32_t* slot_mapping,
                                        int64_t num_tokens, int32_t num_kv_heads,
                                        int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                        pa_dtype src_dtype, pa_dtype kv_dtype,
                                        const float* k_scales, const float* v_scales,
                                        cudaStream_t stream) {
  if (num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0) return PA_ESHAPE;
  if (!dtype_ok(src_dtype) || !pool_dtype_ok(kv_dtype)) return PA_EUNSUPPORTED;
  if (num_tokens < 0 || num_blocks < 0) return PA_EINVAL;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !k_blocks || !v_blocks || !slot_mapping) return PA_EINVAL;
  const DeviceState* d = device_state();
  if (!d) return PA_ECUDA;
  if (launch_validate_scales(k_scales, v_scales, num_kv_heads, d->status, stream) != cudaSuccess)
    return PA_ECUDA;
  return from_cuda(launch_reshape_and_cache_convert(
      k, v, k_blocks, v_blocks, slot_mapping, num_tokens, (int64_t)num_kv_heads * head_dim,
      block_size, num_blocks, src_dtype == PA_BF16, kv_dtype, 1.f, 1.f, k_scales, v_scales,
      head_dim, d->status, stream));
}

pa_status pa_reshape_and_cache_per_block(const void* k, const void* v, void* k_blocks,
                                         void* v_blocks, const int32_t* slot_mapping,
                                         int64_t num_tokens, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t block_size,
                                         int64_t num_blocks, pa_dtype src_dtype,
                                         pa_dtype kv_dtype, const float* k_block_scales,
                                         const float* v_block_scales, cudaStream_t stream) {
  if (num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0) return PA_ESHAPE;
  if (!dtype_ok(src_dtype) || !pool_dtype_ok(kv_dtype)) return PA_EUNSUPPORTED;
  if (num_tokens < 0 || num_blocks < 0) return PA_EINVAL;
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !k_blocks || !v_blocks || !slot_mapping || !k_block_scales ||
      !v_block_scales)
    return PA_EINVAL;
  if (num_blocks * block_size > INT32_MAX) return PA_EUNSUPPORTED;  // slots are int32
  const DeviceState* d = device_state();
  if (!d) return PA_ECUDA;
  return from_cuda(launch_reshape_and_cache_convert(
      k, v, k_blocks, v_blocks, slot_mapping, num_tokens, (int64_t)num_kv_heads * head_dim,
      block_size, num_blocks, src_dtype == PA_BF16, kv_dtype, 1.f, 1.f, nullptr, nullptr,
      head_dim, d->status, stream, k_block_scales, v_block_scales));
}

size_t pa_varlen_forward_workspace_size(int32_t num_seqs, int64_t num_tokens, int32_t num_heads,
                                        int32_t num_kv_heads, int32_t head_dim,
                                        int32_t max_blocks_per_seq, int32_t block_size) {
  (void)head_dim;
  (void)max_blocks_per_seq;
  (void)block_size;
  if (num_seqs < 0 || num_tokens < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
      num_heads % num_kv_heads != 0)
    return 0;
  const PlanLayout L = plan_layout(num_seqs, num_tokens, num_heads / num_kv_heads);
  return (size_t)((L.words * 4 + 255) / 256 * 256);
}

pa_status pa_varlen_forward(const void* q, const void* k_blocks, const void* v_blocks, void* out,
                            const int32_t* query_start_loc, const int32_t* seq_lens,
                            const int32_t* positions, const int32_t* block_tables,
                            int32_t num_seqs, int64_t num_tokens, int32_t num_heads,
                            int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                            int64_t num_blocks, int32_t max_blocks_per_seq, pa_dtype q_dtype,
                            pa_dtype kv_dtype, float scale, int32_t causal,
                            int32_t sliding_window, void* workspace, size_t workspace_bytes,
                            cudaStream_t stream) {
  return pa_varlen_forward_ex(q, k_blocks, v_blocks, out, query_start_loc, seq_lens, positions,
                              block_tables, num_seqs, num_tokens, num_heads, num_kv_heads,
                              head_dim, block_size, num_blocks, max_blocks_per_seq, q_dtype,
                              kv_dtype, scale, causal, sliding_window, nullptr, nullptr, 1.f,
                              1.f, 0u, workspace, workspace_bytes, stream);
}

// The new tokens' rows of pa_cache_and_attend, scattered by the kernel launched right after
// the plan.
struct CacheArgs {
  const void* k;
  const void* v;
  int32_t* slots;
  int64_t row_bytes;
};

static pa_status varlen_impl(const void* q, const void* k_blocks, const void* v_blocks,
                             void* out, const int32_t* query_start_loc, const int32_t* seq_lens,
                             const int32_t* positions, const int32_t* block_tables,
                             int32_t num_seqs, int64_t num_tokens, int32_t num_heads,
                             int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                             int64_t num_blocks, int32_t max_blocks_per_seq, pa_dtype q_dtype,
                             pa_dtype kv_dtype, float scale, int32_t causal,
                             int32_t sliding_window, const float* sinks, float* lse,
                             float k_scale, float v_scale, const float* k_scales,
                             const float* v_scales, uint32_t flags, void* workspace,
                             size_t workspace_bytes, cudaStream_t stream,
                             const CacheArgs* cache, const float* k_bscales = nullptr,
                             const float* v_bscales = nullptr) {
  // per-block factors: both arrays, e4m3 pools, not together with per-head scales
  const bool per_block = k_bscales || v_bscales;
  if (per_block && (!k_bscales || !v_bscales || k_scales || v_scales)) return PA_EINVAL;
  if (per_block && kv_dtype != PA_FP8_E4M3) return PA_EUNSUPPORTED;
  bool empty = false;
  const pa_status chk = varlen_check(q, k_blocks, v_blocks, out, query_start_loc, seq_lens,
                                     positions, block_tables, num_seqs, num_tokens, num_heads,
                                     num_kv_heads, head_dim, block_size, num_blocks,
                                     max_blocks_per_seq, q_dtype, kv_dtype, k_scale, v_scale,
                                     flags, &empty);
  if (chk != PA_OK || empty) return chk;
  if (!workspace) return PA_EINVAL;
  const size_t need = pa_varlen_forward_workspace_size(num_seqs, num_tokens, num_heads,
                                                       num_kv_heads, head_dim, max_blocks_per_seq,
                                                       block_size);
  if (workspace_bytes < need || !aligned(workspace, 256)) return PA_EINVAL;
  const DeviceState* d = device_state();
  if (!d) return PA_ECUDA;

  VarlenMeta m{};
  m.query_start_loc = query_start_loc;
  m.seq_lens = seq_lens;
  m.positions = positions;
  m.block_tables = block_tables;
  m.num_seqs = num_seqs;
  m.num_tokens = num_tokens;
  m.num_heads = num_heads;
  m.num_kv_heads = num_kv_heads;
  m.group = num_heads / num_kv_heads;
  m.head_dim = head_dim;
  m.block_size = block_size;
  m.num_blocks = num_blocks;
  m.max_blocks = max_blocks_per_seq;
  m.causal = causal ? 1 : 0;
  m.window = sliding_window > 0 ? sliding_window : 0;
  m.sinks = sinks;
  m.lse = lse;
  m.v_scale = v_scale;
  m.k_scales = k_scales;
  m.v_scales = v_scales;
  m.k_bscales = k_bscales;
  m.v_bscales = v_bscales;
  scale *= k_scale;  // K = k_scale * pool: the scores take it with the softmax scale
  int32_t* plan = static_cast<int32_t*>(workspace);  // (the plan also checks per-head scales)
  PlanLayout L = plan_layout(num_seqs, num_tokens, m.group);
  const bool fast = mma_path(q_dtype, kv_dtype, head_dim, block_size, q, k_blocks, v_blocks, out);
  const bool fast8 =
      mma_path_fp8(q_dtype, kv_dtype, head_dim, block_size, q, k_blocks, v_blocks, out);
  // per-block factors: the e4m3 kernels only (warp-MMA, and tcgen05 for prefill-class rows)
  if (per_block && !fast8) return PA_EUNSUPPORTED;
  // prefill-class sequences (more than 64 query rows per kv head) go to the tcgen05 kernel:
  // head size 128 and a GQA group that divides the 128-row tile; bf16 or e4m3 pools
  // No sequence can have more than num_tokens - num_seqs + 1 query tokens: when even that
  // many rows fit the warp-MMA path, the tcgen05 kernel is not launched at all.
  const int64_t max_rows = (num_tokens - (num_seqs > 0 ? num_seqs : 1) + 1) * m.group;
  L.use_tc = (fast || fast8) && head_dim == 128 && m.group <= 128 && (128 % m.group) == 0 &&
             aligned(q, 16) && max_rows > L.tc_min_rows && scale > 0.f && tc_enabled() &&
             !(flags & PA_FLAG_BITWISE);

  // the tcgen05 kernel's launch: one CTA per SM, pairs, never more than there are items
  const int64_t tc_work = L.tc_cap * num_kv_heads;
  const int tc_grid = (int)std::max<int64_t>(2, std::min<int64_t>(tc_work, d->sms)) & ~1;
  L.tc_pairs = tc_grid / 2;
  L.num_sms = d->sms;
  L.kv_elem_bytes = esize(kv_dtype);
  if (fast8) L.mma_tile_rows = 8;  // the e4m3 warp-MMA kernel's tiles are one group of 8 rows
  L.need_tok_map = !(fast || fast8);  // only the scalar kernel reads the token map
  cudaError_t e = launch_plan_varlen(m, plan, L, d->status, stream);
  if (e != cudaSuccess) return PA_ECUDA;
  if (cache) {  // the new tokens' slots and rows, alongside the plan
    e = launch_map_and_scatter_after_plan(cache->k, cache->v, const_cast<void*>(k_blocks),
                                          const_cast<void*>(v_blocks), query_start_loc,
                                          positions, block_tables, num_seqs, num_tokens,
                                          max_blocks_per_seq, block_size, num_blocks,
                                          cache->row_bytes, cache->slots, d->status, stream);
    if (e != cudaSuccess) return PA_ECUDA;
  }

  if (fast8) {
    // fp8 pools: prefill-class sequences on the tcgen05 kernel (the codes widened to f16 in
    // shared memory), then the decode tiles on the warp-MMA kernel, as for bf16 pools
    CUtensorMap tk, tv;
    if (!pool_map_fp8(&tk, k_blocks, num_blocks, block_size, num_kv_heads, head_dim) ||
        !pool_map_fp8(&tv, v_blocks, num_blocks, block_size, num_kv_heads, head_dim))
      return PA_ECUDA;
    Mma16Params p;
    std::memset(&p, 0, sizeof p);
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.out = out;
    p.m = m;
    p.plan = plan;
    p.items_off = L.mma_off;
    p.status = d->status;
    p.scale_log2 = scale * kLog2e;
    mma_waits(p);
    if (L.use_tc) {
      CUtensorMap tq, tv_half;
      if (!query_map(&tq, q, num_tokens, num_heads, head_dim, m.group) ||
          !pool_map_fp8_half(&tv_half, v_blocks, num_blocks, block_size, num_kv_heads, head_dim))
        return PA_ECUDA;
      TcParams tp;
      std::memset(&tp, 0, sizeof tp);
      tp.out = out;
      tp.m = m;
      tp.plan = plan;
      tp.tc_off = L.tc_off;
      tp.status = d->status;
      tp.scale_log2 = scale * kLog2e;
      stall_hook(tp.wait_limit_ns, tp.debug_stall);
      tp.redo_flags = plan + L.redo_off;
      tp.redo_list = plan + L.redo_list_off;
      tp.redo_count = plan + 3;
      tp.kv_fp8 = 1;
      e = launch_tc_prefill(tq, tk, tv_half, tp, tc_grid, stream);
      if (e != cudaSuccess) return PA_ECUDA;
      p.after_tc = 1;
      p.tc_off = L.tc_off;
      p.redo_list_off = L.redo_list_off;
    }
    return from_cuda(
        launch_mma16_varlen_fp8(tk, tv, p, (int)std::min<int64_t>(L.mma_cap, 65535), stream));
  }
  if (fast) {
    CUtensorMap tk, tv;
    if (!pool_map(&tk, k_blocks, num_blocks, block_size, num_kv_heads, head_dim) ||
        !pool_map(&tv, v_blocks, num_blocks, block_size, num_kv_heads, head_dim))
      return PA_ECUDA;
    Mma16Params p;
    std::memset(&p, 0, sizeof p);
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.out = out;
    p.m = m;
    p.plan = plan;
    p.items_off = L.mma_off;
    p.status = d->status;
    p.scale_log2 = scale * kLog2e;
    mma_waits(p);
    if (L.use_tc) {
      // the tcgen05 kernel first, then the warp-MMA kernel: its decode tiles start as soon as
      // every tcgen05 CTA has found the plan complete (programmatic dependent launch), on the
      // SMs the tcgen05 kernel leaves free; after that kernel it recomputes the items the
      // tcgen05 kernel marked (V outside f16's range)
      CUtensorMap tq;
      if (!query_map(&tq, q, num_tokens, num_heads, head_dim, m.group)) return PA_ECUDA;
      TcParams tp;
      std::memset(&tp, 0, sizeof tp);
      tp.out = out;
      tp.m = m;
      tp.plan = plan;
      tp.tc_off = L.tc_off;
      tp.status = d->status;
      tp.scale_log2 = scale * kLog2e;
      stall_hook(tp.wait_limit_ns, tp.debug_stall);
      tp.redo_flags = plan + L.redo_off;
      tp.redo_list = plan + L.redo_list_off;
      tp.redo_count = plan + 3;
      e = launch_tc_prefill(tq, tk, tv, tp, tc_grid, stream);
      if (e != cudaSuccess) return PA_ECUDA;
      p.after_tc = 1;
      p.tc_off = L.tc_off;
      p.redo_list_off = L.redo_list_off;
    }
    return from_cuda(launch_mma16_varlen(tk, tv, p, head_dim,
                                         (int)std::min<int64_t>(L.mma_cap, 65535), stream));
  }
  SimtParams p;
  std::memset(&p, 0, sizeof p);
  p.q = q;
  p.k_blocks = k_blocks;
  p.v_blocks = v_blocks;
  p.out = out;
  p.m = m;
  p.plan = plan;
  p.status = d->status;
  p.scale = scale;
  p.q_bf16 = q_dtype == PA_BF16;
  p.kv_bf16 = kv_dtype == PA_BF16;
  p.kv_fp8 = kv_dtype == PA_FP8_E4M3;
  return from_cuda(launch_simt(p, stream));
}

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
                               cudaStream_t stream) {
  return varlen_impl(q, k_blocks, v_blocks, out, query_start_loc, seq_lens, positions,
                     block_tables, num_seqs, num_tokens, num_heads, num_kv_heads, head_dim,
                     block_size, num_blocks, max_blocks_per_seq, q_dtype, kv_dtype, scale, causal,
                     sliding_window, sinks, lse, k_scale, v_scale, nullptr, nullptr, flags,
                     workspace, workspace_bytes, stream, nullptr);
}

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
                                     cudaStream_t stream) {
  return varlen_impl(q, k_blocks, v_blocks, out, query_start_loc, seq_lens, positions,
                     block_tables, num_seqs, num_tokens, num_heads, num_kv_heads, head_dim,
                     block_size, num_blocks, max_blocks_per_seq, q_dtype, kv_dtype, scale, causal,
                     sliding_window, sinks, lse, 1.f, 1.f, k_scales, v_scales, flags, workspace,
                     workspace_bytes, stream, nullptr);
}

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
                                      cudaStream_t stream) {
  if (!k_block_scales || !v_block_scales) return PA_EINVAL;
  return varlen_impl(q, k_blocks, v_blocks, out, query_start_loc, seq_lens, positions,
                     block_tables, num_seqs, num_tokens, num_heads, num_kv_heads, head_dim,
                     block_size, num_blocks, max_blocks_per_seq, q_dtype, kv_dtype, scale, causal,
                     sliding_window, sinks, lse, 1.f, 1.f, nullptr, nullptr, flags, workspace,
                     workspace_bytes, stream, nullptr, k_block_scales, v_block_scales);
}

pa_status pa_cache_and_attend(const void* k_new, const void* v_new, const void* q,
                              void* k_blocks, void* v_blocks, void* out,
                              const int32_t* query_start_loc, const int32_t* seq_lens,
                              const int32_t* positions, const int32_t* block_tables,
                              int32_t num_seqs, int64_t num_tokens, int32_t num_heads,
                              int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                              int64_t num_blocks, int32_t max_blocks_per_seq, pa_dtype q_dtype,
                              pa_dtype kv_dtype, float scale, int32_t causal,
                              int32_t sliding_window, int32_t* slot_mapping, void* workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
  if (num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0) return PA_ESHAPE;
  if (!pool_dtype_ok(kv_dtype)) return PA_EUNSUPPORTED;
  if (num_seqs < 0 || num_tokens < 0 || num_blocks < 0 || max_blocks_per_seq < 0)
    return PA_EINVAL;
  if (num_tokens > 0 && (!k_new || !v_new || !slot_mapping)) return PA_EINVAL;
  if (num_blocks * block_size > INT32_MAX) return PA_EUNSUPPORTED;  // slots are int32
  if (!map_and_scatter_fits(num_seqs, num_tokens)) {  // larger batches: one call after the other
    const pa_status st = pa_slot_mapping_and_cache(
        k_new, v_new, k_blocks, v_blocks, query_start_loc, positions, block_tables, num_seqs,
        num_tokens, max_blocks_per_seq, num_kv_heads, head_dim, block_size, num_blocks, kv_dtype,
        slot_mapping, stream);
    if (st != PA_OK) return st;
    return pa_varlen_forward(q, k_blocks, v_blocks, out, query_start_loc, seq_lens, positions,
                             block_tables, num_seqs, num_tokens, num_heads, num_kv_heads,
                             head_dim, block_size, num_blocks, max_blocks_per_seq, q_dtype,
                             kv_dtype, scale, causal, sliding_window, workspace,
                             workspace_bytes, stream);
  }
  const CacheArgs cache{k_new, v_new, slot_mapping,
                        (int64_t)num_kv_heads * head_dim * esize(kv_dtype)};
  return varlen_impl(q, k_blocks, v_blocks, out, query_start_loc, seq_lens, positions,
                     block_tables, num_seqs, num_tokens, num_heads, num_kv_heads, head_dim,
                     block_size, num_blocks, max_blocks_per_seq, q_dtype, kv_dtype, scale, causal,
                     sliding_window, nullptr, nullptr, 1.f, 1.f, nullptr, nullptr, 0u, workspace,
                     workspace_bytes, stream, &cache);
}

static pa_status splitkv_partials(const void* q, const void* k_blocks, const void* v_blocks,
                                  float* max_logits, float* exp_sums, float* tmp_out,
                                  const int32_t* seq_lens, const int32_t* block_tables,
                                  int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                  int32_t max_blocks_per_seq, int32_t partition_size,
                                  int32_t max_num_partitions, pa_dtype q_dtype, pa_dtype kv_dtype,
                                  float scale, int32_t sliding_window, float k_scale,
                                  float v_scale, const float* k_scales, const float* v_scales,
                                  cudaStream_t stream, const float* k_bscales = nullptr,
                                  const float* v_bscales = nullptr) {
  if (num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      num_heads % num_kv_heads != 0 || partition_size <= 0 || max_num_partitions <= 0)
    return PA_ESHAPE;
  const bool per_block = k_bscales || v_bscales;
  if (per_block && (!k_bscales || !v_bscales || k_scales || v_scales)) return PA_EINVAL;
  if (per_block && kv_dtype != PA_FP8_E4M3) return PA_EUNSUPPORTED;
  if (!dtype_ok(q_dtype) || !pool_dtype_ok(kv_dtype)) return PA_EUNSUPPORTED;
  if (!scale_ok(k_scale) || !scale_ok(v_scale)) return PA_EINVAL;
  scale *= k_scale;
  if (head_dim > 256 || partition_size % block_size != 0) return PA_EUNSUPPORTED;
  if (num_seqs < 0 || num_blocks < 0 || max_blocks_per_seq < 0) return PA_EINVAL;
  if (num_seqs == 0) return PA_OK;
  if (!q || !k_blocks || !v_blocks || !max_logits || !exp_sums || !tmp_out || !seq_lens ||
      !block_tables)
    return PA_EINVAL;
  const DeviceState* d = device_state();
  if (!d) return PA_ECUDA;
  const bool fp8 =
      mma_path_fp8(q_dtype, kv_dtype, head_dim, block_size, q, k_blocks, v_blocks, nullptr);
  // per-block factors: the e4m3 warp-MMA kernel only
  if (per_block && !(fp8 && num_heads / num_kv_heads <= 16 && aligned(tmp_out, 16)))
    return PA_EUNSUPPORTED;
  if (launch_validate_scales(k_scales, v_scales, num_kv_heads, d->status, stream) != cudaSuccess)
    return PA_ECUDA;
  cudaError_t e = launch_validate_decode(seq_lens, block_tables, num_seqs, max_blocks_per_seq,
                                         block_size, num_blocks, partition_size,
                                         max_num_partitions, 1, d->status, stream, k_bscales,
                                         v_bscales, num_kv_heads);
  if (e != cudaSuccess) return PA_ECUDA;
  VarlenMeta m{};
  std::memset(&m, 0, sizeof m);
  m.seq_lens = seq_lens;
  m.block_tables = block_tables;
  m.num_seqs = num_seqs;
  m.num_tokens = num_seqs;
  m.num_heads = num_heads;
  m.num_kv_heads = num_kv_heads;
  m.group = num_heads / num_kv_heads;
  m.head_dim = head_dim;
  m.block_size = block_size;
  m.num_blocks = num_blocks;
  m.max_blocks = max_blocks_per_seq;
  m.causal = 1;
  m.window = sliding_window > 0 ? sliding_window : 0;
  m.v_scale = v_scale;
  m.k_scales = k_scales;
  m.v_scales = v_scales;
  m.k_bscales = k_bscales;
  m.v_bscales = v_bscales;
  if ((fp8 || mma_path(q_dtype, kv_dtype, head_dim, block_size, q, k_blocks, v_blocks, nullptr)) &&
      m.group <= 16 && aligned(tmp_out, 16)) {
    CUtensorMap tk, tv;
    const bool ok =
        fp8 ? pool_map_fp8(&tk, k_blocks, num_blocks, block_size, num_kv_heads, head_dim) &&
                  pool_map_fp8(&tv, v_blocks, num_blocks, block_size, num_kv_heads, head_dim)
            : pool_map(&tk, k_blocks, num_blocks, block_size, num_kv_heads, head_dim) &&
                  pool_map(&tv, v_blocks, num_blocks, block_size, num_kv_heads, head_dim);
    if (!ok) return PA_ECUDA;
    Mma16Params p;
    std::memset(&p, 0, sizeof p);
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.m = m;
    p.status = d->status;
    p.scale_log2 = scale * kLog2e;
    p.max_logits = max_logits;
    p.exp_sums = exp_sums;
    p.tmp_out = tmp_out;
    p.partition_size = partition_size;
    p.max_parts = max_num_partitions;
    mma_waits(p);
    return from_cuda(fp8 ? launch_mma16_split_fp8(tk, tv, p, stream)
                         : launch_mma16_split(tk, tv, p, head_dim, stream));
  }
  SimtParams p;
  std::memset(&p, 0, sizeof p);
  p.q = q;
  p.k_blocks = k_blocks;
  p.v_blocks = v_blocks;
  p.m = m;
  p.status = d->status;
  p.scale = scale;
  p.q_bf16 = q_dtype == PA_BF16;
  p.kv_bf16 = kv_dtype == PA_BF16;
  p.kv_fp8 = kv_dtype == PA_FP8_E4M3;
  p.max_logits = max_logits;
  p.exp_sums = exp_sums;
  p.tmp_out = tmp_out;
  p.partition_size = partition_size;
  p.max_parts = max_num_partitions;
  p.split = 1;
  return from_cuda(launch_simt(p, stream));
}

static pa_status splitkv_reduce(void* out, const float* max_logits, const float* exp_sums,
                                const float* tmp_out, const int32_t* seq_lens, int32_t num_seqs,
                                int32_t num_heads, int32_t head_dim, int32_t partition_size,
                                int32_t max_num_partitions, pa_dtype out_dtype, bool validate,
                                cudaStream_t stream) {
  if (num_heads <= 0 || head_dim <= 0 || partition_size <= 0 || max_num_partitions <= 0)
    return PA_ESHAPE;
  if (!dtype_ok(out_dtype)) return PA_EUNSUPPORTED;
  if (head_dim % 4 != 0 || !aligned(tmp_out, 16) || max_num_partitions > 16384)
    return PA_EUNSUPPORTED;
  if (num_seqs < 0) return PA_EINVAL;
  if (num_seqs == 0) return PA_OK;
  if (!out || !max_logits || !exp_sums || !tmp_out || !seq_lens) return PA_EINVAL;
  const DeviceState* d = device_state();
  if (!d) return PA_ECUDA;
  if (validate) {
    cudaError_t e = launch_validate_decode(seq_lens, nullptr, num_seqs, 0, 1, 0, partition_size,
                                           max_num_partitions, 0, d->status, stream);
    if (e != cudaSuccess) return PA_ECUDA;
  }
  return from_cuda(launch_splitkv_reduce(out, out_dtype == PA_BF16, max_logits, exp_sums, tmp_out,
                                         seq_lens, num_seqs, num_heads, head_dim, partition_size,
                                         max_num_partitions, d->status, stream));
}

pa_status pa_decode_splitkv_partials(const void* q, const void* k_blocks, const void* v_blocks,
                                     float* max_logits, float* exp_sums, float* tmp_out,
                                     const int32_t* seq_lens, const int32_t* block_tables,
                                     int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                                     int32_t head_dim, int32_t block_size, int64_t num_blocks,
                                     int32_t max_blocks_per_seq, int32_t partition_size,
                                     int32_t max_num_partitions, pa_dtype q_dtype,
                                     pa_dtype kv_dtype, float scale, int32_t sliding_window,
                                     cudaStream_t stream) {
  return splitkv_partials(q, k_blocks, v_blocks, max_logits, exp_sums, tmp_out, seq_lens,
                          block_tables, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                          num_blocks, max_blocks_per_seq, partition_size, max_num_partitions,
                          q_dtype, kv_dtype, scale, sliding_window, 1.f, 1.f, nullptr, nullptr,
                          stream);
}

pa_status pa_decode_splitkv_partials_ex(
    const void* q, const void* k_blocks, const void* v_blocks, float* max_logits,
    float* exp_sums, float* tmp_out, const int32_t* seq_lens, const int32_t* block_tables,
    int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, int64_t num_blocks, int32_t max_blocks_per_seq, int32_t partition_size,
    int32_t max_num_partitions, pa_dtype q_dtype, pa_dtype kv_dtype, float scale,
    int32_t sliding_window, float k_scale, float v_scale, cudaStream_t stream) {
  return splitkv_partials(q, k_blocks, v_blocks, max_logits, exp_sums, tmp_out, seq_lens,
                          block_tables, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                          num_blocks, max_blocks_per_seq, partition_size, max_num_partitions,
                          q_dtype, kv_dtype, scale, sliding_window, k_scale, v_scale, nullptr,
                          nullptr, stream);
}

pa_status pa_decode_splitkv_partials_per_head(
    const void* q, const void* k_blocks, const void* v_blocks, float* max_logits,
    float* exp_sums, float* tmp_out, const int32_t* seq_lens, const int32_t* block_tables,
    int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, int64_t num_blocks, int32_t max_blocks_per_seq, int32_t partition_size,
    int32_t max_num_partitions, pa_dtype q_dtype, pa_dtype kv_dtype, float scale,
    int32_t sliding_window, const float* k_scales, const float* v_scales, cudaStream_t stream) {
  return splitkv_partials(q, k_blocks, v_blocks, max_logits, exp_sums, tmp_out, seq_lens,
                          block_tables, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                          num_blocks, max_blocks_per_seq, partition_size, max_num_partitions,
                          q_dtype, kv_dtype, scale, sliding_window, 1.f, 1.f, k_scales, v_scales,
                          stream);
}

pa_status pa_decode_splitkv_partials_per_block(
    const void* q, const void* k_blocks, const void* v_blocks, float* max_logits,
    float* exp_sums, float* tmp_out, const int32_t* seq_lens, const int32_t* block_tables,
    int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
    int32_t block_size, int64_t num_blocks, int32_t max_blocks_per_seq, int32_t partition_size,
    int32_t max_num_partitions, pa_dtype q_dtype, pa_dtype kv_dtype, float scale,
    int32_t sliding_window, const float* k_block_scales, const float* v_block_scales,
    cudaStream_t stream) {
  if (!k_block_scales || !v_block_scales) return PA_EINVAL;
  return splitkv_partials(q, k_blocks, v_blocks, max_logits, exp_sums, tmp_out, seq_lens,
                          block_tables, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                          num_blocks, max_blocks_per_seq, partition_size, max_num_partitions,
                          q_dtype, kv_dtype, scale, sliding_window, 1.f, 1.f, nullptr, nullptr,
                          stream, k_block_scales, v_block_scales);
}

pa_status pa_decode_splitkv_reduce(void* out, const float* max_logits, const float* exp_sums,
                                   const float* tmp_out, const int32_t* seq_lens,
                                   int32_t num_seqs, int32_t num_heads, int32_t head_dim,
                                   int32_t partition_size, int32_t max_num_partitions,
                                   pa_dtype out_dtype, cudaStream_t stream) {
  return splitkv_reduce(out, max_logits, exp_sums, tmp_out, seq_lens, num_seqs, num_heads,
                        head_dim, partition_size, max_num_partitions, out_dtype, true, stream);
}

pa_status pa_decode_splitkv(const void* q, const void* k_blocks, const void* v_blocks, void* out,
                            float* max_logits, float* exp_sums, float* tmp_out,
                            const int32_t* seq_lens, const int32_t* block_tables,
                            int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                            int32_t head_dim, int32_t block_size, int64_t num_blocks,
                            int32_t max_blocks_per_seq, int32_t partition_size,
                            int32_t max_num_partitions, pa_dtype q_dtype, pa_dtype kv_dtype,
                            float scale, int32_t sliding_window, cudaStream_t stream) {
  if (!out) return PA_EINVAL;
  if (head_dim % 4 != 0 || !aligned(tmp_out, 16) || max_num_partitions > 16384)
    return PA_EUNSUPPORTED;
  pa_status st = splitkv_partials(q, k_blocks, v_blocks, max_logits, exp_sums, tmp_out, seq_lens,
                                  block_tables, num_seqs, num_heads, num_kv_heads, head_dim,
                                  block_size, num_blocks, max_blocks_per_seq, partition_size,
                                  max_num_partitions, q_dtype, kv_dtype, scale, sliding_window,
                                  1.f, 1.f, nullptr, nullptr, stream);
  if (st != PA_OK) return st;
  return splitkv_reduce(out, max_logits, exp_sums, tmp_out, seq_lens, num_seqs, num_heads,
                        head_dim, partition_size, max_num_partitions, q_dtype, false, stream);
}

pa_status pa_merge_attn_states(void* out, float* out_lse, const void* prefix_out,
                               const float* prefix_lse, const void* suffix_out,
                               const float* suffix_lse, int64_t num_tokens, int32_t num_heads,
                               int32_t head_dim, int64_t prefill_tokens_with_context,
                               pa_dtype dtype, cudaStream_t stream) {
  if (num_heads <= 0 || head_dim <= 0) return PA_ESHAPE;
  if (!dtype_ok(dtype)) return PA_EUNSUPPORTED;
  if (num_tokens < 0) return PA_EINVAL;
  if (num_tokens == 0) return PA_OK;
  if (!out || !prefix_out || !prefix_lse || !suffix_out || !suffix_lse) return PA_EINVAL;
  const DeviceState* d = device_state();
  if (!d) return PA_ECUDA;
  const int64_t prefix_tokens =
      prefill_tokens_with_context < 0 ? num_tokens : prefill_tokens_with_context;
  return from_cuda(launch_merge_attn_states(out, out_lse, prefix_out, prefix_lse, suffix_out,
                                            suffix_lse, num_tokens, num_heads, head_dim,
                                            prefix_tokens, dtype == PA_BF16, d->status, stream));
}

pa_status pa_gather_kv(const void* k_blocks, const void* v_blocks, void* k_out, void* v_out,
                       const int32_t* cu_seq_lens, const int32_t* seq_starts,
                       const int32_t* block_tables, int32_t num_seqs, int64_t num_out_rows,
                       int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                       int64_t num_blocks, int32_t max_blocks_per_seq, pa_dtype kv_dtype,
                       cudaStream_t stream) {
  if (num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0) return PA_ESHAPE;
  if (!pool_dtype_ok(kv_dtype)) return PA_EUNSUPPORTED;
  if (num_seqs < 0 || num_out_rows < 0 || num_blocks < 0 || max_blocks_per_seq < 0)
    return PA_EINVAL;
  if (num_seqs == 0) return PA_OK;
  if (!k_blocks || !k_out || !cu_seq_lens || !block_tables) return PA_EINVAL;
  if ((v_blocks == nullptr) != (v_out == nullptr)) return PA_EINVAL;
  const DeviceState* d = device_state();
  if (!d) return PA_ECUDA;
  const int64_t row_bytes = (int64_t)num_kv_heads * head_dim * esize(kv_dtype);
  return from_cuda(launch_gather_kv(k_blocks, v_blocks, k_out, v_out, cu_seq_lens, seq_starts,
                                    block_tables, num_seqs, num_out_rows, row_bytes, block_size,
                                    num_blocks, max_blocks_per_seq, d->status, stream));
}

}  // extern "C"
