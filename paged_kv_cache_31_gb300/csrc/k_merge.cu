// k_merge.cu -- log-sum-exp combination of attention states.
//
//  * k_splitkv_reduce: phase 2 of PagedAttention V2 ("Cross-partition reduction"): per
//    (sequence, head), lse_p = m_p + log(l_p) for the partitions 0 .. ceil(seq_len / P) - 1,
//    an infinite m_p of either sign or l_p <= 0 counting as -inf; M = max lse_p;
//    out = sum_p exp(lse_p - M) o_p * (1 / sum_p exp(lse_p - M)); all -inf -> partition 0.
//  * k_merge_attn_states: the two-state merge of vllm.cpp MergeAttnStatesKernel, with its
//    +inf -> -inf normalisation, the both -inf -> prefix rule and the suffix pass-through of
//    tokens past prefill_tokens_with_context.
// Both are HBM-bound streaming kernels; sums run in a fixed order, so results are
// deterministic.
#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kReduceWarps = 8;

// Words of the partition-weight array in the reduce kernel's shared memory, rounded up to
// a multiple of 4 so that the float4 partial sums after it stay 16-byte aligned.
__host__ __device__ constexpr int weights_words(int max_parts) { return (max_parts + 3) & ~3; }

__device__ __forceinline__ float part_lse(float m, float l) {
  return (isinf(m) || !(l > 0.f)) ? -INFINITY : m + logf(l);
}

// One CTA per (sequence, head).  Dynamic smem: max_parts floats (weights) + 8 x D floats.
template <typename TO>
__global__ void __launch_bounds__(kReduceWarps * 32)
    k_splitkv_reduce(TO* __restrict__ out, const float* __restrict__ max_logits,
                     const float* __restrict__ exp_sums, const float* __restrict__ tmp_out,
                     const int32_t* __restrict__ seq_lens, int32_t num_heads, int32_t head_dim,
                     int32_t partition_size, int32_t max_parts, const int* status) {
  extern __shared__ __align__(16) float sm[];
  __shared__ float s_red[kReduceWarps];
  __shared__ int s_skip;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) s_skip = status_set(status);
  __syncthreads();
  if (s_skip) return;
  float* w = sm;                                 // [max_parts]
  float* part = sm + weights_words(max_parts);  // [kReduceWarps][D], 16-byte aligned
  const int s = blockIdx.x / num_heads, h = blockIdx.x % num_heads;
  const int D = head_dim;
  const int np = (seq_lens[s] + partition_size - 1) / partition_size;
  const int64_t base = ((int64_t)s * num_heads + h) * max_parts;

  float mx = -INFINITY;
  for (int p = threadIdx.x; p < np; p += blockDim.x) {
    const float l = part_lse(max_logits[base + p], exp_sums[base + p]);
    w[p] = l;
    mx = fmaxf(mx, l);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
  if (lane == 0) s_red[warp] = mx;
  __syncthreads();
  float M = -INFINITY;
#pragma unroll
  for (int i = 0; i < kReduceWarps; ++i) M = fmaxf(M, s_red[i]);
  TO* o = out + ((int64_t)s * num_heads + h) * D;
  if (M == -INFINITY) {  // no partition holds mass: partition 0 passes through
    for (int d = threadIdx.x; d < D; d += blockDim.x) o[d] = from_f32<TO>(tmp_out[base * D + d]);
    return;
  }
  __syncthreads();
  float ws = 0.f;
  for (int p = threadIdx.x; p < np; p += blockDim.x) {
    const float e = expf(w[p] - M);
    w[p] = e;
    ws += e;
  }
#pragma unroll
  for (int o2 = 16; o2 > 0; o2 >>= 1) ws += __shfl_xor_sync(kFull, ws, o2);
  if (lane == 0) s_red[warp] = ws;
  __syncthreads();
  float W = 0.f;
#pragma unroll
  for (int i = 0; i < kReduceWarps; ++i) W += s_red[i];
  const float inv = 1.f / W;

  // weighted sum: warp `warp` takes partitions warp, warp + 8, ... in that order; lanes take
  // 4 dims each.  Four partitions' loads are issued before their products (a grid of one
  // CTA per (sequence, head) is too small to hide the latency of one load at a time); a
  // partition without mass adds exactly nothing, whatever its tmp_out holds
  auto add = [](float4& acc, float wp, float4 v) {
    if (!(wp > 0.f)) v = make_float4(0.f, 0.f, 0.f, 0.f);
    acc.x += wp * v.x;
    acc.y += wp * v.y;
    acc.z += wp * v.z;
    acc.w += wp * v.w;
  };
  for (int d0 = lane * 4; d0 < D; d0 += 128) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int p = warp;
    for (; p + 3 * kReduceWarps < np; p += 4 * kReduceWarps) {
      float4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        v[u] = *reinterpret_cast<const float4*>(tmp_out + (base + p + u * kReduceWarps) * D + d0);
#pragma unroll
      for (int u = 0; u < 4; ++u) add(acc, w[p + u * kReduceWarps], v[u]);
    }
    for (; p < np; p += kReduceWarps)
      add(acc, w[p], *reinterpret_cast<const float4*>(tmp_out + (base + p) * D + d0));
    *reinterpret_cast<float4*>(part + warp * D + d0) = acc;
  }
  __syncthreads();
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < kReduceWarps; ++i) a += part[i * D + d];
    o[d] = from_f32<TO>(a * inv);
  }
}

// One warp per (token, head); lanes walk the head dimension.
template <typename T>
__global__ void __launch_bounds__(256)
    k_merge_attn_states(T* __restrict__ out, float* __restrict__ out_lse,
                        const T* __restrict__ prefix_out, const float* __restrict__ prefix_lse,
                        const T* __restrict__ suffix_out, const float* __restrict__ suffix_lse,
                        int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                        int64_t prefix_tokens, const int* status) {
  if (status_set(status)) return;
  const int lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (gw >= num_tokens * num_heads) return;
  const int64_t t = gw / num_heads;
  const int h = (int)(gw % num_heads);
  const int64_t off = gw * head_dim;  // (t * H + h) * D
  const int64_t li = (int64_t)h * num_tokens + t;
  if (t >= prefix_tokens) {
    for (int d = lane; d < head_dim; d += 32) out[off + d] = suffix_out[off + d];
    if (out_lse && lane == 0) out_lse[li] = suffix_lse[li];
    return;
  }
  float pl = prefix_lse[li], sl = suffix_lse[li];
  if (isinf(pl)) pl = -INFINITY;
  if (isinf(sl)) sl = -INFINITY;
  const float mx = fmaxf(pl, sl);
  if (isinf(mx)) {
    for (int d = lane; d < head_dim; d += 32) out[off + d] = prefix_out[off + d];
    if (out_lse && lane == 0) out_lse[li] = mx;
    return;
  }
  const float pse = expf(pl - mx), sse = expf(sl - mx);
  const float ose = pse + sse;
  const float ps = pse / ose, ss = sse / ose;
  for (int d = lane; d < head_dim; d += 32)
    out[off + d] = from_f32<T>(to_f32(prefix_out[off + d]) * ps + to_f32(suffix_out[off + d]) * ss);
  if (out_lse && lane == 0) out_lse[li] = logf(ose) + mx;
}

// The same merge with 16-byte accesses: a (token, head) row of head_dim values is C chunks
// of 16 bytes (C a power of two <= 256), and a thread takes CPT of them, chunks c and
// c + C / CPT, ... (so a CTA of 256 threads holds 256 CPT / C whole rows, and each thread
// has 2 CPT loads in flight).  Rows are taken head-major (row = h * num_tokens + t): the rows
// of a CTA read and write consecutive lse entries of one head.  Per element it computes what
// k_merge_attn_states does.
template <typename T, int CPT>
__global__ void __launch_bounds__(256)
    k_merge_attn_states_v(T* __restrict__ out, float* __restrict__ out_lse,
                          const T* __restrict__ prefix_out, const float* __restrict__ prefix_lse,
                          const T* __restrict__ suffix_out, const float* __restrict__ suffix_lse,
                          int64_t num_tokens, int32_t num_heads, int32_t head_dim,
                          int64_t prefix_tokens, int log2_tpr, const int* status) {
  if (status_set(status)) return;
  constexpr int kE = 16 / (int)sizeof(T);  // values per chunk
  const int tpr = 1 << log2_tpr;           // threads per row
  const int c = threadIdx.x & (tpr - 1);
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> log2_tpr;
  if (row >= num_tokens * num_heads) return;
  const int h = (int)(row / num_tokens);
  const int64_t t = row - (int64_t)h * num_tokens;
  const int64_t base = (t * num_heads + h) * head_dim;
  const int64_t li = row;  // h * num_tokens + t
  if (t >= prefix_tokens) {
#pragma unroll
    for (int k = 0; k < CPT; ++k) {
      const int64_t off = base + (int64_t)(c + k * tpr) * kE;
      *reinterpret_cast<uint4*>(out + off) = *reinterpret_cast<const uint4*>(suffix_out + off);
    }
    if (out_lse && c == 0) out_lse[li] = suffix_lse[li];
    return;
  }
  // all loads in flight together (the states do not wait for the lse values)
  uint4 pv[CPT], sv[CPT];
#pragma unroll
  for (int k = 0; k < CPT; ++k) {
    const int64_t off = base + (int64_t)(c + k * tpr) * kE;
    pv[k] = *reinterpret_cast<const uint4*>(prefix_out + off);
    sv[k] = *reinterpret_cast<const uint4*>(suffix_out + off);
  }
  float pl = prefix_lse[li], sl = suffix_lse[li];
  if (isinf(pl)) pl = -INFINITY;
  if (isinf(sl)) sl = -INFINITY;
  const float mx = fmaxf(pl, sl);
  if (isinf(mx)) {
#pragma unroll
    for (int k = 0; k < CPT; ++k)
      *reinterpret_cast<uint4*>(out + base + (int64_t)(c + k * tpr) * kE) = pv[k];
    if (out_lse && c == 0) out_lse[li] = mx;
    return;
  }
  const float pse = expf(pl - mx), sse = expf(sl - mx);
  const float ose = pse + sse;
  const float ps = pse / ose, ss = sse / ose;
#pragma unroll
  for (int k = 0; k < CPT; ++k) {
    const T* pe = reinterpret_cast<const T*>(&pv[k]);
    const T* se = reinterpret_cast<const T*>(&sv[k]);
    uint4 r;
    T* re = reinterpret_cast<T*>(&r);
#pragma unroll
    for (int i = 0; i < kE; ++i) re[i] = from_f32<T>(to_f32(pe[i]) * ps + to_f32(se[i]) * ss);
    *reinterpret_cast<uint4*>(out + base + (int64_t)(c + k * tpr) * kE) = r;
  }
  if (out_lse && c == 0) out_lse[li] = logf(ose) + mx;
}

}  // namespace

cudaError_t launch_splitkv_reduce(void* out, int out_bf16, const float* max_logits,
                                  const float* exp_sums, const float* tmp_out,
                                  const int32_t* seq_lens, int32_t num_seqs, int32_t num_heads,
                                  int32_t head_dim, int32_t partition_size, int32_t max_parts,
                                  int* status, cudaStream_t stream) {
  const int64_t ctas = (int64_t)num_seqs * num_heads;
  if (ctas <= 0) return cudaSuccess;
  const size_t smem =
      ((size_t)weights_words(max_parts) + (size_t)kReduceWarps * head_dim) * sizeof(float);
  if (out_bf16) {
    auto k = k_splitkv_reduce<__nv_bfloat16>;
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    k<<<(unsigned)ctas, kReduceWarps * 32, smem, stream>>>(
        (__nv_bfloat16*)out, max_logits, exp_sums, tmp_out, seq_lens, num_heads, head_dim,
        partition_size, max_parts, status);
  } else {
    auto k = k_splitkv_reduce<float>;
    if (smem > 48 * 1024) {
      cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
      if (e != cudaSuccess) return e;
    }
    k<<<(unsigned)ctas, kReduceWarps * 32, smem, stream>>>((float*)out, max_logits, exp_sums,
                                                           tmp_out, seq_lens, num_heads, head_dim,
                                                           partition_size, max_parts, status);
  }
  return cudaGetLastError();
}

cudaError_t launch_merge_attn_states(void* out, float* out_lse, const void* prefix_out,
                                     const float* prefix_lse, const void* suffix_out,
                                     const float* suffix_lse, int64_t num_tokens,
                                     int32_t num_heads, int32_t head_dim, int64_t prefix_tokens,
                                     int bf16, int* status, cudaStream_t stream) {
  const int64_t warps = num_tokens * num_heads;
  if (warps <= 0) return cudaSuccess;
  // whole 16-byte chunks per row, a power of two of them, and 16-byte aligned tensors: the
  // vectorised kernel (2.5 -> 6+ TB/s on bf16 states of head size 128)
  const int row_bytes = head_dim * (bf16 ? 2 : 4);
  const int chunks = row_bytes / 16;
  const bool vec = row_bytes % 16 == 0 && chunks >= 1 && chunks <= 256 &&
                   (chunks & (chunks - 1)) == 0 &&
                   ((reinterpret_cast<uintptr_t>(out) | reinterpret_cast<uintptr_t>(prefix_out) |
                     reinterpret_cast<uintptr_t>(suffix_out)) & 15) == 0;
  if (vec) {
    // two chunks per thread when the row has two or more
    const int cpt = chunks >= 2 ? 2 : 1;
    const int tpr = chunks / cpt;
    const int lg = 31 - __builtin_clz((unsigned)tpr);
    const int64_t vgrid = (warps * tpr + 255) / 256;
    auto go = [&](auto kern, auto* o, const auto* po, const auto* so) {
      kern<<<(unsigned)vgrid, 256, 0, stream>>>(o, out_lse, po, prefix_lse, so, suffix_lse,
                                                num_tokens, num_heads, head_dim, prefix_tokens,
                                                lg, status);
    };
    using B = __nv_bfloat16;
    if (bf16) {
      if (cpt == 2)
        go(k_merge_attn_states_v<B, 2>, (B*)out, (const B*)prefix_out, (const B*)suffix_out);
      else
        go(k_merge_attn_states_v<B, 1>, (B*)out, (const B*)prefix_out, (const B*)suffix_out);
    } else {
      if (cpt == 2)
        go(k_merge_attn_states_v<float, 2>, (float*)out, (const float*)prefix_out,
           (const float*)suffix_out);
      else
        go(k_merge_attn_states_v<float, 1>, (float*)out, (const float*)prefix_out,
           (const float*)suffix_out);
    }
    return cudaGetLastError();
  }
  const int64_t grid = (warps + 7) / 8;
  if (bf16)
    k_merge_attn_states<__nv_bfloat16><<<(unsigned)grid, 256, 0, stream>>>(
        (__nv_bfloat16*)out, out_lse, (const __nv_bfloat16*)prefix_out, prefix_lse,
        (const __nv_bfloat16*)suffix_out, suffix_lse, num_tokens, num_heads, head_dim,
        prefix_tokens, status);
  else
    k_merge_attn_states<float><<<(unsigned)grid, 256, 0, stream>>>(
        (float*)out, out_lse, (const float*)prefix_out, prefix_lse, (const float*)suffix_out,
        suffix_lse, num_tokens, num_heads, head_dim, prefix_tokens, status);
  return cudaGetLastError();
}

}  // namespace pa
