// k_simt.cu -- the general paged-attention kernel: any mix of fp32 / bf16 for q and the
// pool, any head size up to 256 and any block size.  One warp serves one (token, head)
// (or one (sequence, head, partition) in split-KV mode) and walks the visible positions in
// increasing order through the block table with the per-position online softmax of the
// TensorSharp ComputeSingleQueryAttention routine: the dot product is spread over the
// lanes and reduced with shuffles, the running max / denominator / numerator are rescaled
// when a larger score arrives, and the output is numerator * (1 / denominator).
//
// It serves the shapes the tensor-core kernels do not cover (fp32 caches, head sizes other
// than 64 / 128, block sizes other than 16, GQA groups above 16 in split-KV decode, fp8
// pools with fp32 q or head sizes other than 128).  fp8 pools: p.scale carries k_scale and
// the output is multiplied by v_scale ("paged_attention_v2_pytorch.py", "Apply scales").
#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr unsigned kFull = 0xffffffffu;

template <typename TQ, typename TKV, int DPL>
__global__ void __launch_bounds__(128) k_simt(const SimtParams p) {
  if (status_set(p.status)) return;  // no barriers in this kernel: per-warp exit is safe
  const int lane = threadIdx.x & 31;
  const int64_t gw = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  const VarlenMeta& m = p.m;
  const int H = m.num_heads, D = m.head_dim;
  int64_t t;
  int s, h, part = 0, start, end;
  if (p.split) {
    const int64_t total = (int64_t)m.num_seqs * H * p.max_parts;
    if (gw >= total) return;
    part = (int)(gw % p.max_parts);
    h = (int)((gw / p.max_parts) % H);
    s = (int)(gw / ((int64_t)p.max_parts * H));
    t = s;
    const int n = m.seq_lens[s];
    end = n;
    start = m.window > 0 ? max(0, n - m.window) : 0;
    start = max(start, part * p.partition_size);
    end = min(end, (part + 1) * p.partition_size);
  } else {
    const int64_t total = m.num_tokens * H;
    if (gw >= total) return;
    t = gw / H;
    h = (int)(gw % H);
    s = p.plan[kPlanHeaderWords + t];
    const int pos = m.positions[t];
    end = m.causal ? pos + 1 : m.seq_lens[s];
    start = m.window > 0 ? max(0, end - m.window) : 0;
  }
  const int g = h / m.group;
  const float psc = head_scale(m.k_scales, g, p.scale);   // K = k_scales[g] * pool
  const float vsc = head_scale(m.v_scales, g, m.v_scale);  // V = v_scales[g] * pool
  const TQ* q = reinterpret_cast<const TQ*>(p.q) + (t * H + h) * (int64_t)D;
  const TKV* kb = reinterpret_cast<const TKV*>(p.k_blocks);
  const TKV* vb = reinterpret_cast<const TKV*>(p.v_blocks);
  const int32_t* row = m.block_tables + (int64_t)s * m.max_blocks;

  float qr[DPL], acc[DPL];
#pragma unroll
  for (int i = 0; i < DPL; ++i) {
    const int d = lane + 32 * i;
    qr[i] = d < D ? to_f32(q[d]) : 0.f;
    acc[i] = 0.f;
  }
  float mx = -INFINITY, den = 0.f;
  // KC positions at a time: their K and V rows are all requested before the first is used,
  // so a chunk waits for memory once instead of once per position; each position is then
  // folded exactly as one at a time
  constexpr int KC = DPL >= 8 ? 2 : 16 / DPL;
  for (int j0 = start; j0 < end; j0 += KC) {
    float kr[KC][DPL], vr[KC][DPL];
#pragma unroll
    for (int u = 0; u < KC; ++u) {
      const int j = j0 + u;
      if (j < end) {
        const int64_t blk = row[j / m.block_size];
        const int64_t base = ((blk * m.block_size + j % m.block_size) * m.num_kv_heads + g) * D;
#pragma unroll
        for (int i = 0; i < DPL; ++i) {
          const int d = lane + 32 * i;
          kr[u][i] = d < D ? to_f32(kb[base + d]) : 0.f;
          vr[u][i] = d < D ? to_f32(vb[base + d]) : 0.f;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < KC; ++u) {
      if (j0 + u >= end) break;
      float dot = 0.f;
#pragma unroll
      for (int i = 0; i < DPL; ++i) {
        const int d = lane + 32 * i;
        if (d < D) dot += qr[i] * kr[u][i];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dot += __shfl_xor_sync(kFull, dot, o);
      const float sc = dot * psc;
      if (sc > mx) {
        const float r = expf(mx - sc);
        den *= r;
#pragma unroll
        for (int i = 0; i < DPL; ++i) acc[i] *= r;
        mx = sc;
      }
      const float e = expf(sc - mx);
      den += e;
#pragma unroll
      for (int i = 0; i < DPL; ++i) {
        const int d = lane + 32 * i;
        if (d < D) acc[i] += e * vr[u][i];
      }
    }
  }
  float inv = den > 0.f ? vsc / den : 0.f;
  if (!p.split) {
    // an attention sink (TensorSharp ForwardWithSinks): one more state with max = the sink
    // logit, exp-sum 1 and weighted sum 0
    const float sk = m.sinks ? m.sinks[h] : -INFINITY;
    if (sk > -INFINITY) {
      const float m2 = fmaxf(mx, sk);
      const float a = mx == -INFINITY ? 0.f : expf(mx - m2);
      den = den * a + expf(sk - m2);
      mx = m2;
      inv = a * vsc / den;
    }
    if (m.lse && lane == 0) m.lse[(int64_t)h * m.num_tokens + t] = den > 0.f ? mx + logf(den) : -INFINITY;
  }
  if (p.split) {
    const int64_t idx = ((int64_t)s * H + h) * p.max_parts + part;
#pragma unroll
    for (int i = 0; i < DPL; ++i) {
      const int d = lane + 32 * i;
      if (d < D) p.tmp_out[idx * D + d] = acc[i] * inv;
    }
    if (lane == 0) {
      p.max_logits[idx] = mx;
      p.exp_sums[idx] = den;
    }
  } else {
    TQ* out = reinterpret_cast<TQ*>(p.out) + (t * H + h) * (int64_t)D;
#pragma unroll
    for (int i = 0; i < DPL; ++i) {
      const int d = lane + 32 * i;
      if (d < D) out[d] = from_f32<TQ>(acc[i] * inv);
    }
  }
}

template <typename TQ, typename TKV>
cudaError_t launch_dtypes(const SimtParams& p, cudaStream_t stream) {
  const int64_t warps = p.split ? (int64_t)p.m.num_seqs * p.m.num_heads * p.max_parts
                                : p.m.num_tokens * p.m.num_heads;
  if (warps <= 0) return cudaSuccess;
  const int64_t grid = (warps + 3) / 4;
  if (grid > 0x7fffffffLL) return cudaErrorInvalidValue;
  const int D = p.m.head_dim;
  if (D <= 32)
    k_simt<TQ, TKV, 1><<<(unsigned)grid, 128, 0, stream>>>(p);
  else if (D <= 64)
    k_simt<TQ, TKV, 2><<<(unsigned)grid, 128, 0, stream>>>(p);
  else if (D <= 128)
    k_simt<TQ, TKV, 4><<<(unsigned)grid, 128, 0, stream>>>(p);
  else if (D <= 256)
    k_simt<TQ, TKV, 8><<<(unsigned)grid, 128, 0, stream>>>(p);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt(const SimtParams& p, cudaStream_t stream) {
  if (p.kv_fp8)
    return p.q_bf16 ? launch_dtypes<__nv_bfloat16, e4m3_t>(p, stream)
                    : launch_dtypes<float, e4m3_t>(p, stream);
  if (p.q_bf16 && p.kv_bf16) return launch_dtypes<__nv_bfloat16, __nv_bfloat16>(p, stream);
  if (p.q_bf16) return launch_dtypes<__nv_bfloat16, float>(p, stream);
  if (p.kv_bf16) return launch_dtypes<float, __nv_bfloat16>(p, stream);
  return launch_dtypes<float, float>(p, stream);
}

}  // namespace pa
