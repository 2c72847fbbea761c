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
// address up with cudaGetSymbolAddress (with that device current) and caches it together
// with the driver context it was found in.  A call under another context (after
// cudaDeviceReset, or with a caller's own driver context current) looks it up again: the
// module, and with it the array, is loaded anew in each context.
#include <mutex>

#include "pa_internal.cuh"

namespace {

constexpr size_t kNoAllocWorkspaceBytes = size_t(4) << 20;  // 4 MiB per device
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_noalloc_workspace[kNoAllocWorkspaceBytes];

std::mutex g_noalloc_mu;
struct NoAllocSlot {
  void* ctx = nullptr;   // driver context of the lookup
  void* addr = nullptr;  // the array's device address in that context
};
NoAllocSlot g_noalloc[kMaxDevices];

// Device address of the current context's copy of the array; nullptr when the lookup fails.
void* noalloc_workspace() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* ctx = pa::current_context();
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoAllocSlot& e = g_noalloc[dev];
  if (!e.addr || !ctx || e.ctx != ctx) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_workspace) != cudaSuccess) return nullptr;
    e.addr = p;
    e.ctx = pa::current_context();  // the lookup may have made the primary context current
  }
  return e.addr;
}

}  // namespace

extern "C" pa_status pa_varlen_forward_noalloc(
    const void* q, const void* k_blocks, const void* v_blocks, void* out,
    const int32_t* query_start_loc, const int32_t* seq_lens, const int32_t* positions,
    const int32_t* block_tables, int32_t num_seqs, int64_t num_tokens, int32_t num_heads,
    int32_t num_kv_heads, int32_t head_dim, int32_t block_size, int64_t num_blocks,
    int32_t max_blocks_per_seq, pa_dtype q_dtype, pa_dtype kv_dtype, float scale,
    int32_t causal, int32_t sliding_window, cudaStream_t stream) {
  // pa_varlen_forward's own argument checks come first, so that a batch it rejects gets the
  // same status here; only then the size of the fixed array
  bool empty = false;
  const pa_status chk = pa::varlen_check(q, k_blocks, v_blocks, out, query_start_loc, seq_lens,
                                         positions, block_tables, num_seqs, num_tokens,
                                         num_heads, num_kv_heads, head_dim, block_size,
                                         num_blocks, max_blocks_per_seq, q_dtype, kv_dtype, 1.f,
                                         1.f, 0u, &empty);
  if (chk != PA_OK || empty) return chk;
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
