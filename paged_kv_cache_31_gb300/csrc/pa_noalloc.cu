// pa_noalloc.cu -- pa_varlen_forward_noalloc: batched varlen paged attention for callers
// that cannot allocate device memory.
//
// pa_varlen_forward needs a few hundred KB of caller-owned scratch for its per-call plan
// (the token -> sequence map and the list of work items).  Some callers have no way to
// provide it: an op inside a host framework that hands the op only its input and output
// buffers and owns every other byte of device memory, a runtime whose allocator cannot be
// reached from the code that issues the call, or a caller that must not risk the implicit
// device synchronisation of cudaMalloc / cudaFree in the middle of a serving step.  This
// entry point keeps that scratch in a fixed-size array in the library itself instead.
//
// The array below is a file-scope __device__ variable: each GPU that loads the library
// holds its own copy (kNoAllocWorkspaceBytes) until the process exits.  Host code cannot
// use the symbol's name as a device address, so the first call on each device looks the
// address up with cudaGetSymbolAddress (with that device current) and caches it.
#include <mutex>

#include "pa_internal.cuh"

namespace {

constexpr size_t kNoAllocWorkspaceBytes = size_t(4) << 20;  // 4 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_workspace[kNoAllocWorkspaceBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[kMaxDevices] = {};

// Device address of this device's copy of the array; nullptr when the lookup fails.
void* noalloc_workspace() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess) return nullptr;
    g_noalloc_addr[dev] = p;
  }
  return g_noalloc_addr[dev];
}

}  // namespace

extern "C" pa_status pa_varlen_forward_noalloc(
    const void* q, const void* k_blocks, const void* v_blocks, void* out,
    const int32_t* query_start_loc, const int32_t* seq_lens, const int32_t* positions,
    const int32_t* block_tables, int32_t num_seqs, int64_t num_tokens, int32_t num_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int64_t num_blocks,
    int32_t max_blocks_per_seq, pa_dtype q_dtype, pa_dtype kv_dtype, float scale,
    int32_t causal, int32_t sliding_window, cudaStream_t stream) {
  const size_t need = pa_varlen_forward_workspace_size(num_seqs, num_tokens, num_heads,
                                                       num_kv_heads, head_dim, max_blocks_per_seq,
                                                       block_size);
  if (need > kNoAllocWorkspaceBytes) return PA_EINVAL;  // batch too large for the fixed array
  void* ws = noalloc_workspace();
  if (!ws) return PA_ECUDA;
  // Nothing in the array has to start at zero: the validation / planning kernel of this
  // call writes every word that the call's attention kernel later reads.
  return pa_varlen_forward(q, k_blocks, v_blocks, out, query_start_loc, seq_lens, positions,
                           block_tables, num_seqs, num_tokens, num_heads, num_kv_heads,
                           head_dim, block_size, num_blocks, max_blocks_per_seq, q_dtype,
                           kv_dtype, scale, causal, sliding_window, ws, kNoAllocWorkspaceBytes,
                           stream);
}
