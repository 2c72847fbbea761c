// k_meta.cu -- metadata kernels: validation and work planning, slot mapping, the K/V
// scatter into the paged pool and the gather back out of it.
//
// Every kernel first looks at the device status word: when an earlier kernel (or an earlier
// call) recorded an error, it writes nothing.  Validation always runs as its own launch
// before the kernel that writes, so a bad table is found before the first byte of output.
#include <algorithm>
#include <climits>

#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr unsigned kFull = 0xffffffffu;

// Exclusive prefix sum of one int per thread across the block; *total receives the sum.
__device__ int block_exclusive_scan(int v, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(kFull, w, o);
      if (lane >= o) w += y;
    }
    s_warp[lane] = w;
  }
  __syncthreads();
  const int before = warp ? s_warp[warp - 1] : 0;
  *total = s_warp[nwarps - 1];
  __syncthreads();
  return before + x - v;
}

__device__ __forceinline__ unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ unsigned long long warp_min_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const unsigned long long y = __shfl_xor_sync(kFull, v, o);
    v = y < v ? y : v;
  }
  return v;
}

// Exclusive prefix sum, in place, of the kCostBuckets ints at h, by one warp (16 per lane);
// the total goes to *total.  Called by warp 0 between two __syncthreads.
template <int N>
__device__ void warp_scan_inplace(int* h, int* total) {
  static_assert(N % 32 == 0, "buckets per lane");
  constexpr int kPer = N / 32;
  const int lane = threadIdx.x & 31;
  int v[kPer], sum = 0;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    v[i] = h[lane * kPer + i];
    sum += v[i];
  }
  int x = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(kFull, x, o);
    if (lane >= o) x += y;
  }
  int run = x - sum;
#pragma unroll
  for (int i = 0; i < kPer; ++i) {
    h[lane * kPer + i] = run;
    run += v[i];
  }
  if (lane == 31) *total = x;
}

// The model of PlanLayout for K CTA pairs of the tcgen05 kernel (the warp-MMA kernel's decode
// tiles run beside it on the other SMs), as a key for atomicMin: the estimated time (a
// positive float: its bits order like its value) above, and ties broken towards the larger K
// below.  tiles: 128-key tiles of all 256-row items (all kv heads); dec_bytes: K/V bytes the
// decode tiles stream.  fp32 throughout (this GPU's fp64 rate is a small fraction of it).
__device__ __forceinline__ unsigned long long split_key(const PlanLayout& L, int k, float tiles,
                                                       float dec_bytes) {
  const int free_sms = L.num_sms - 2 * k;
  float t;
  if (dec_bytes <= 0.f) {
    t = L.margin * tiles * L.tile_ns / (float)k;  // no decode tiles: all pairs
  } else if (free_sms <= 0) {
    t = 3.0e38f;
  } else {
    const float pre = L.margin * tiles * L.tile_ns / (float)k;
    const float dec = dec_bytes / L.hbm_bytes_per_ns * fmaxf(1.f, (float)L.decode_sat_sms / free_sms);
    t = fmaxf(pre, dec);
  }
  return ((unsigned long long)__float_as_uint(t) << 32) | (0xffffffffu - (unsigned)k);
}

// Work buckets for ordering: a cost c > 0 maps to 16 sub-buckets per power of two
// (descending: the largest costs get the smallest bucket index).
constexpr int kCostBuckets = 512;
constexpr int kPlanCacheSeqs = 4096;    // sequences whose metadata the planner keeps in smem
constexpr int kPlanCacheTokens = 8192;  // tokens whose visible ranges it keeps there too
constexpr int kPlanTokPer = kPlanCacheTokens / 1024;  // tokens per planner thread, at most
constexpr int kPlanCacheItems = 2048;  // 256-row items the planner keeps in smem
// 256-row items the planner keeps in shared memory for this layout (else in the plan)
__host__ __device__ constexpr int plan_items_cached(const PlanLayout& L) {
  return (L.use_tc && L.tc_cap <= kPlanCacheItems) ? (int)L.tc_cap : 0;
}
// dynamic shared memory of the planner for s cached sequences and t tokens: int4 [items]
// 256-row items, then ints [s + 1] query starts, [s] seq_len, [s] visible keys, [s]
// visible-range start, [s] visible-range end, and, when t <= kPlanCacheTokens, [t]
// visible-range start and [t] end of each token
__host__ __device__ constexpr size_t plan_smem_bytes(int s, int64_t t, int items) {
  return 16 * (size_t)items + 4 * (5 * (size_t)s + 1 + (t <= kPlanCacheTokens ? 2 * (size_t)t : 0));
}

// Table check of one pa_varlen_forward call, in blocks 1 .. V of the planning launch, beside
// the planner (block 0): the entries [0, ceil(seq_len / b)) of every sequence with query
// tokens lie in [0, num_blocks) (tinyllm section 2.6).  Block c takes the sequences c,
// c + V, c + 2V, ...; their tables are cut into chunks of 256 entries, which the warps take
// two at a time (16 loads in flight per lane).  A bad entry records PA_EINVAL in the status
// word; the attention kernels wait for the whole launch, so this happens before anything is
// written.  Table lengths beyond max_blocks and the other per-sequence checks are the
// planner's; only existing entries are read here, whatever query_start_loc holds.
// The per-block K and V factors of pool block id (every kv head) are finite, positive
// normal floats (at least 2^-126, so that their reciprocals are finite too).
__device__ __forceinline__ bool block_factors_bad(const float* kbs, const float* vbs, int32_t id,
                                                  int32_t hkv) {
  bool bad = false;
  for (int g = 0; g < hkv; ++g) {
    const float a = kbs[(int64_t)id * hkv + g], b = vbs[(int64_t)id * hkv + g];
    bad |= !(a >= 1.17549435e-38f && a <= 3.402823466e38f) ||
           !(b >= 1.17549435e-38f && b <= 3.402823466e38f);
  }
  return bad;
}

__device__ void check_tables(const VarlenMeta& m, int* status) {
  __shared__ int v_off[1025];  // chunk offsets of this round's sequences
  __shared__ int v_need[1024];
  __shared__ int v_seq[1024];
  __shared__ int v_warp[32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  const int V = gridDim.x - 1, c = blockIdx.x - 1;
  const int K = c < m.num_seqs ? (m.num_seqs - c + V - 1) / V : 0;  // this block's sequences
  bool bad = false;
  for (int k0 = 0; k0 < K; k0 += blockDim.x) {
    const int k = k0 + tid;
    int nch = 0, need = 0, s = 0;
    if (k < K) {
      s = c + V * k;
      const int a = m.query_start_loc[s], b = m.query_start_loc[s + 1], n = m.seq_lens[s];
      if (a < b && n >= 1) {
        const int64_t full = ((int64_t)n + m.block_size - 1) / m.block_size;
        need = (int)(full < (int64_t)m.max_blocks ? full : (int64_t)m.max_blocks);
        nch = (need + 255) / 256;
      }
    }
    int total;
    const int off = block_exclusive_scan(nch, v_warp, &total);
    v_off[tid] = off;
    v_need[tid] = need;
    v_seq[tid] = s;
    if (tid == 0) v_off[blockDim.x] = total;
    __syncthreads();
    const int cnt = min((int)blockDim.x, K - k0);  // sequences of this round
    for (int j0 = warp; j0 < total; j0 += 2 * nwarps) {  // warp-uniform
      int32_t id[2][8];
      uint32_t real = 0;  // bit 8h + u: a table entry (not padding)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int j = j0 + h * nwarps;
        int t = 0;
        if (j < total) {  // the sequence owning chunk j: the last t with v_off[t] <= j
          int lo2 = 0, hi2 = cnt;
          while (hi2 - lo2 > 1) {
            const int mid = (lo2 + hi2) >> 1;
            if (v_off[mid] <= j) lo2 = mid; else hi2 = mid;
          }
          t = lo2;
        }
        const int base = (j - v_off[t]) * 256;
        const int32_t* row = m.block_tables + (int64_t)v_seq[t] * m.max_blocks;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = base + lane + 32 * u;
          const bool r = j < total && i < v_need[t];
          id[h][u] = r ? row[i] : 0;
          real |= (uint32_t)r << (8 * h + u);
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int u = 0; u < 8; ++u) bad |= (id[h][u] < 0 || (int64_t)id[h][u] >= m.num_blocks);
      if (m.k_bscales)  // per-block factors of the blocks the call reads (e4m3 pools)
        for (int e = 0; e < 16; ++e) {
          const int32_t b = id[e >> 3][e & 7];
          if (((real >> e) & 1u) && b >= 0 && (int64_t)b < m.num_blocks)
            bad |= block_factors_bad(m.k_bscales, m.v_bscales, b, m.num_kv_heads);
        }
    }
    __syncthreads();  // the next round reuses the arrays
  }
  if (__any_sync(kFull, bad) && lane == 0) {
    pdl_wait();  // the planner may run before the kernels ahead of it have finished
    record_error(status, PA_EINVAL);
  }
}
__device__ __forceinline__ int cost_bucket(int c) {
  if (c <= 0) return kCostBuckets - 1;
  const int lg = 31 - __clz(c);
  const int sub = lg >= 4 ? (c >> (lg - 4)) & 15 : (c << (4 - lg)) & 15;
  return kCostBuckets - 1 - (lg * 16 + sub);
}

// Validation and planning of one pa_varlen_forward call (tinyllm section 2.6 checks), in a
// single CTA so that the work list can be built with one block-wide scan:
//  A. per sequence (a warp each): query_start_loc[s] <= query_start_loc[s + 1] <= num_tokens,
//     query_start_loc[0] == 0 and query_start_loc[num_seqs] == num_tokens; for a sequence with
//     query tokens: seq_len >= 1, ceil(seq_len / b) <= max_blocks, those table entries inside
//     the pool, query positions inside [0, seq_len); the token -> sequence map and the keys the
//     sequence's rows can see (its work estimate);
//  B. the work lists: a sequence's q_len * G query rows (token major, head minor within the
//     kv group) are cut into tiles of 16 rows (8 on e4m3 pools) for the warp-MMA kernel, or,
//     for prefill-class sequences, into 256-row items for the tcgen05 kernel; both lists are
//     ordered by the number of keys their rows see, longest first, so the kernels' last units
//     are short.
// The kernel is bound by the latency of its loads, not by bandwidth: every sequence's query
// start and length come into shared memory in one coalesced pass, phase A then issues each
// sequence's table and position loads together, and the work estimates stay in shared memory
// (up to kPlanCacheSeqs sequences; larger batches read everything from global memory).  The
// bucket scans run in one warp, and the prefill-item pass only when the tcgen05 kernel runs.
// TOK: the batch's sequences and tokens fit the planner's shared memory; TC: the tcgen05
// kernel runs (L.use_tc).  Each instance holds only the code its batches run: the kernel's
// time is mostly latency, and instruction fetches from a cold L2 are part of it.
template <bool TOK, bool TC>
__global__ void __launch_bounds__(1024)
    k_plan_varlen(VarlenMeta m, int32_t* plan, const PlanLayout L, int* status) {
  __shared__ int s_err;
  __shared__ int s_warp[32];
  __shared__ int s_hist[kCostBuckets];    // warp-MMA tiles per cost bucket
  __shared__ int s_hist_t[kCostBuckets];  // 256-row items per cost bucket
  __shared__ int s_tot;
  __shared__ unsigned long long s_dec_units;  // decode tiles x visible keys
  __shared__ unsigned int s_tc_tiles;         // 128-key tiles of the 256-row items
  __shared__ unsigned long long s_split;      // best split key (split_key)
  // when cached: [num_seqs + 1] query starts, [num_seqs] seq_len, [num_seqs] visible keys
  extern __shared__ __align__(16) int s_dyn[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  // early: everything the planner computes stays in shared memory until it writes the plan,
  // so it reads the batch and plans before the kernels ahead of it in the stream have
  // finished, and waits for them only before its first global write.  Its inputs are
  // complete when it starts: the kernel ahead of it is this library's (an attention kernel,
  // the planner or the scatter), which lets its dependents start only after its own wait for
  // the kernels before it, and none of those writes the batch's metadata; anything else ahead
  // of it (a copy, another kernel) has finished.  The grid still ends after the kernels ahead
  // of it, so the kernels behind it see the stream's order.
  const bool early = TOK && (!TC || L.tc_cap <= kPlanCacheItems);
  if (!early) pdl_wait();
  pdl_launch_dependents();  // the attention kernels' prologues may overlap this kernel
  if constexpr (TOK) {
    if (blockIdx.x > 0) {  // blocks 1 .. V check the block tables
      if (!status_set(status)) check_tables(m, status);
      return;
    }
  }
  const bool cached = TOK || m.num_seqs <= kPlanCacheSeqs;
  constexpr bool tok_cached = TOK;
  const int item_cap = cached ? plan_items_cached(L) : 0;
  int* s_qsl = s_dyn + 4 * item_cap;
  int* s_n = s_qsl + (cached ? m.num_seqs + 1 : 0);
  int* s_cost = s_n + (cached ? m.num_seqs : 0);
  int* s_lo = s_cost + (cached ? m.num_seqs : 0);
  int* s_hi = s_lo + (cached ? m.num_seqs : 0);
  int* s_ts = s_hi + (cached ? m.num_seqs : 0);  // when tok_cached: per token visible start
  int* s_te = s_ts + (tok_cached ? m.num_tokens : 0);  // ... and end
  // each thread's run of tpt consecutive query positions is loaded now, together with the
  // query starts and lengths below
  const int tpt = (int)((m.num_tokens + blockDim.x - 1) / blockDim.x);  // <= kPlanTokPer
  const int t_first = tid * tpt;
  int32_t pos0[kPlanTokPer];
  if constexpr (tok_cached) {
#pragma unroll
    for (int u = 0; u < kPlanTokPer; ++u)
      pos0[u] = (u < tpt && t_first + u < m.num_tokens) ? m.positions[t_first + u] : 0;
  }
  if (tid == 0) {
    s_err = status_set(status) ? -1 : 0;
    s_dec_units = 0;
    s_tc_tiles = 0;
    s_split = ~0ull;
  }
  for (int i = tid; i < kCostBuckets; i += blockDim.x) {
    s_hist[i] = 0;
    s_hist_t[i] = 0;
  }
  if (cached)
    for (int i = tid; i <= m.num_seqs; i += blockDim.x) {
      s_qsl[i] = m.query_start_loc[i];
      if (i < m.num_seqs) s_n[i] = m.seq_lens[i];
    }
  __syncthreads();
  if (s_err == 0) {
    if (m.num_seqs == 0 && tid == 0 && (int64_t)m.query_start_loc[0] != m.num_tokens)
      atomicCAS(&s_err, 0, PA_EINVAL);
    // per kv head dequantisation scales, when given, are finite and positive
    if (m.k_scales || m.v_scales)
      for (int g = tid; g < m.num_kv_heads; g += blockDim.x) {
        const float ks = m.k_scales ? m.k_scales[g] : 1.f, vs = m.v_scales ? m.v_scales[g] : 1.f;
        if (!(ks > 0.f && ks <= 3.402823466e38f) || !(vs > 0.f && vs <= 3.402823466e38f))
          atomicCAS(&s_err, 0, PA_EINVAL);
      }
    if constexpr (tok_cached) {
      // A1: per sequence (a thread each): the query-start order, a table long enough for
      // seq_len, and an empty visible range to fill in (the entries themselves are checked
      // by the other blocks of this launch)
      for (int q = tid; q < m.num_seqs; q += blockDim.x) {
        const int a = s_qsl[q], b = s_qsl[q + 1], n = s_n[q];
        bool bad = a < 0 || b < a || (int64_t)b > m.num_tokens || (q == 0 && a != 0) ||
                   (q == m.num_seqs - 1 && (int64_t)b != m.num_tokens);
        if (!bad && a < b) {
          const int64_t need = n >= 1 ? ((int64_t)n + m.block_size - 1) / m.block_size : 0;
          bad = n < 1 || need > m.max_blocks;
        }
        s_lo[q] = INT_MAX;
        s_hi[q] = 0;
        if (bad) atomicCAS(&s_err, 0, PA_EINVAL);
      }
      __syncthreads();
      if (s_err == 0 && m.num_seqs > 0) {
        // A2: each thread's run of consecutive query tokens: their sequence (the last q with
        // query_start_loc[q] <= t, found once and then advanced), the position check, the
        // token -> sequence map, each token's visible range [start, end) and, per sequence,
        // [min start, max end): folded in registers along the run, then (when the warp's
        // lanes end on one sequence) across the warp, with few shared-memory atomics
        bool bad = false;
        int q = -1, run_st = INT_MAX, run_e = 0;
        if (t_first < m.num_tokens) {
          int lo2 = 0, hi2 = m.num_seqs;  // s_qsl[lo2] <= t < s_qsl[hi2]
          while (hi2 - lo2 > 1) {
            const int mid = (lo2 + hi2) >> 1;
            if (s_qsl[mid] <= t_first) lo2 = mid; else hi2 = mid;
          }
          q = lo2;
        }
#pragma unroll
        for (int u = 0; u < kPlanTokPer; ++u) {
          const int t = t_first + u;
          if (u >= tpt || t >= m.num_tokens) break;
          while (s_qsl[q + 1] <= t) {  // the run crosses into the next sequence
            if (run_e > 0) {
              atomicMin(&s_lo[q], run_st);
              atomicMax(&s_hi[q], run_e);
            }
            ++q;
            run_st = INT_MAX;
            run_e = 0;
          }
          const int n = s_n[q];
          bad |= (pos0[u] < 0 || pos0[u] >= n);
          if (!early) plan[L.tok_off + t] = q;
          const int e = m.causal ? pos0[u] + 1 : n;
          const int st = m.window > 0 ? max(0, e - m.window) : 0;
          s_ts[t] = st;
          s_te[t] = e;
          run_st = min(run_st, st);
          run_e = max(run_e, e);
        }
        const int q_l0 = __shfl_sync(kFull, q, 0);
        if (__all_sync(kFull, q == q_l0)) {
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            run_st = min(run_st, __shfl_xor_sync(kFull, run_st, o));
            run_e = max(run_e, __shfl_xor_sync(kFull, run_e, o));
          }
          if (lane == 0 && q >= 0 && run_e > 0) {
            atomicMin(&s_lo[q], run_st);
            atomicMax(&s_hi[q], run_e);
          }
        } else if (q >= 0 && run_e > 0) {
          atomicMin(&s_lo[q], run_st);
          atomicMax(&s_hi[q], run_e);
        }
        if (__any_sync(kFull, bad) && lane == 0) atomicCAS(&s_err, 0, PA_EINVAL);
        __syncthreads();
        for (int q = tid; q < m.num_seqs; q += blockDim.x) s_cost[q] = max(0, s_hi[q] - s_lo[q]);
      }
    } else {
    for (int s = warp; s < m.num_seqs; s += nwarps) {
        const int a = cached ? s_qsl[s] : m.query_start_loc[s];
        const int b = cached ? s_qsl[s + 1] : m.query_start_loc[s + 1];
        const int n = cached ? s_n[s] : m.seq_lens[s];
        bool bad = a < 0 || b < a || (int64_t)b > m.num_tokens || (s == 0 && a != 0) ||
                   (s == m.num_seqs - 1 && (int64_t)b != m.num_tokens);
        int lo = INT_MAX, hi = 0;
        const int64_t need = n >= 1 ? ((int64_t)n + m.block_size - 1) / m.block_size : 0;
        if (!bad && a < b) {
          bad = n < 1 || need > m.max_blocks;
          if (!bad) {
            const int32_t* row = m.block_tables + (int64_t)s * m.max_blocks;
            // eight loads in flight per lane, table entries and positions together
            for (int64_t base = 0; base < need || base < b - a; base += 256) {
              int32_t id[8], pos[8];
  #pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int64_t i = base + lane + 32 * u;
                id[u] = i < need ? row[i] : 0;
                pos[u] = i < b - a ? m.positions[a + i] : 0;
              }
  #pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int64_t i = base + lane + 32 * u;
                bad |= (id[u] < 0 || (int64_t)id[u] >= m.num_blocks);
                if (i < b - a) {
                  bad |= (pos[u] < 0 || pos[u] >= n);
                  plan[L.tok_off + a + i] = s;
                  const int e = m.causal ? pos[u] + 1 : n;
                  lo = min(lo, m.window > 0 ? max(0, e - m.window) : 0);
                  hi = max(hi, e);
                }
              }
              if (m.k_bscales)  // per-block factors of the blocks the call reads
                for (int u = 0; u < 8; ++u)
                  if (base + lane + 32 * u < need && id[u] >= 0 && (int64_t)id[u] < m.num_blocks)
                    bad |= block_factors_bad(m.k_bscales, m.v_bscales, id[u], m.num_kv_heads);
            }
          }
        }
  #pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          lo = min(lo, __shfl_xor_sync(kFull, lo, o));
          hi = max(hi, __shfl_xor_sync(kFull, hi, o));
        }
        if (lane == 0) {
          const int cost = max(0, hi - lo);
          if (cached)
            s_cost[s] = cost;
          else
            plan[L.cost_off + s] = cost;
        }
        if (__any_sync(kFull, bad) && lane == 0) atomicCAS(&s_err, 0, PA_EINVAL);
      }
    }
  }
  __syncthreads();
  if (s_err != 0) {
    if (early) pdl_wait();
    if (tid == 0) {
      if (s_err > 0) record_error(status, s_err);
      plan[0] = 0;
      plan[1] = 0;
      plan[3] = 0;
      plan[4] = 0;
    }
    return;
  }
  // per-sequence q_len and visible keys, from shared memory when cached
  auto qlen_of = [&](int s) -> int {
    return cached ? s_qsl[s + 1] - s_qsl[s] : m.query_start_loc[s + 1] - m.query_start_loc[s];
  };
  auto cost_of = [&](int s) -> int { return cached ? s_cost[s] : plan[L.cost_off + s]; };
  int4* mma_recs = reinterpret_cast<int4*>(plan + L.mma_off);
  int4* tc_items = reinterpret_cast<int4*>(plan + L.tc_off);
  // the items in sequence order: in shared memory when they fit, else in the plan
  int4* tc_tmp = item_cap ? reinterpret_cast<int4*>(s_dyn) : reinterpret_cast<int4*>(plan + L.tc_tmp_off);
  const int tok_per_item = 256 / m.group;  // used only when use_tc (group divides 128)
  // B1: 256-row items of prefill-class sequences, in sequence order, the last one (most keys
  // under a causal mask) first; the histogram of the warp-MMA tiles' costs
  int carry_t = 0;
  if constexpr (TC) {
    unsigned long long dec_units = 0;
    for (int base = 0; base < m.num_seqs; base += blockDim.x) {
      const int s = base + tid;
      int cm = 0, ct = 0;
      if (s < m.num_seqs) {
        const int64_t rows = (int64_t)qlen_of(s) * m.group;
        if (rows > L.tc_min_rows)
          ct = (int)((rows + 255) / 256);
        else
          cm = (int)((rows + L.mma_tile_rows - 1) / L.mma_tile_rows);
      }
      if (cm > 0) {
        atomicAdd(&s_hist[cost_bucket(cost_of(s))], cm);
        dec_units += (unsigned long long)cm * (unsigned long long)cost_of(s);
      }
      int tot_t;
      const int et = block_exclusive_scan(ct, s_warp, &tot_t);
      for (int i = 0; i < ct; ++i) tc_tmp[carry_t + et + i] = make_int4(s, ct - 1 - i, 0, 0);
      carry_t += tot_t;
    }
    dec_units = warp_sum_u64(dec_units);  // one shared-memory atomic per warp
    if (lane == 0 && dec_units) atomicAdd(&s_dec_units, dec_units);
  } else {
    for (int s = tid; s < m.num_seqs; s += blockDim.x) {
      const int cm = (int)(((int64_t)qlen_of(s) * m.group + L.mma_tile_rows - 1) / L.mma_tile_rows);
      if (cm > 0) atomicAdd(&s_hist[cost_bucket(cost_of(s))], cm);
    }
  }
  __syncthreads();
  // B2: each item's key range [lo, hi), the union of its tokens' visible ranges (a warp per
  // item), and the histogram of the items' costs (carry_t is the same in every thread)
  if (carry_t > 0) {
    for (int k = warp; k < carry_t; k += nwarps) {
      const int4 it = tc_tmp[k];
      const int qs = cached ? s_qsl[it.x] : m.query_start_loc[it.x];
      const int qe = cached ? s_qsl[it.x + 1] : m.query_start_loc[it.x + 1];
      const int n = cached ? s_n[it.x] : m.seq_lens[it.x];
      const int ta = qs + it.y * tok_per_item, tb = min(qe, ta + tok_per_item);
      int lo = INT_MAX, hi = 0;
      for (int t = ta + lane; t < tb; t += 32) {
        int e, st;
        if constexpr (tok_cached) {
          e = s_te[t];
          st = s_ts[t];
        } else {
          e = m.causal ? m.positions[t] + 1 : n;
          st = m.window > 0 ? max(0, e - m.window) : 0;
        }
        lo = min(lo, st);
        hi = max(hi, e);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(kFull, lo, o));
        hi = max(hi, __shfl_xor_sync(kFull, hi, o));
      }
      if (lane == 0) {
        tc_tmp[k] = make_int4(it.x, it.y, lo, hi);
        atomicAdd(&s_hist_t[cost_bucket(hi - lo)], 1);
        if (hi > lo) atomicAdd(&s_tc_tiles, (unsigned)((hi - (lo / 16) * 16 + 127) / 128));
      }
    }
    __syncthreads();
    // B3: the items ordered by cost, longest first (a counting sort over the cost buckets)
    if (warp == 0) warp_scan_inplace<kCostBuckets>(s_hist_t, &s_tot);  // bucket starts
    __syncthreads();
    if (early) pdl_wait();  // the first global write
    for (int k = tid; k < carry_t; k += blockDim.x) {
      const int4 it = tc_tmp[k];
      tc_items[atomicAdd(&s_hist_t[cost_bucket(it.w - it.z)], 1)] = it;
      plan[L.redo_off + k] = 0;  // not marked for recomputing (the tcgen05 kernel marks items)
    }
  }
  // warp-MMA tiles, the sequences with the most visible keys first (a counting sort over
  // logarithmic cost buckets), so the persistent kernel's last units are the short ones
  if (warp == 0) warp_scan_inplace<kCostBuckets>(s_hist, &s_tot);  // bucket starts
  __syncthreads();
  if (early) {
    pdl_wait();  // (again, when there were items) the plan is written from here on
    // the token -> sequence map, which only the scalar kernel reads
    if (L.need_tok_map)
      for (int t = tid; t < m.num_tokens; t += blockDim.x) {
        int lo2 = 0, hi2 = m.num_seqs;  // s_qsl[lo2] <= t < s_qsl[hi2]
        while (hi2 - lo2 > 1) {
          const int mid = (lo2 + hi2) >> 1;
          if (s_qsl[mid] <= t) lo2 = mid; else hi2 = mid;
        }
        plan[L.tok_off + t] = lo2;
      }
  }
  const int carry_m = s_tot;
  for (int s = tid; s < m.num_seqs; s += blockDim.x) {
    const int64_t rows = (int64_t)qlen_of(s) * m.group;
    if (rows == 0 || (TC && rows > L.tc_min_rows)) continue;
    const int tr = L.mma_tile_rows;
    const int cm = (int)((rows + tr - 1) / tr);
    const int at = atomicAdd(&s_hist[cost_bucket(cost_of(s))], cm);
    const int qs = cached ? s_qsl[s] : m.query_start_loc[s];
    const int n = cached ? s_n[s] : m.seq_lens[s];
    for (int i = 0; i < cm; ++i) {
      // the union of the visible key ranges of the tile's tokens, formed as the kernel would
      // from the rows' positions (rows that see nothing do not count)
      const int64_t ra = (int64_t)i * tr, rb = min(rows, ra + tr);
      int lo = INT_MAX, hi = 0;
      for (int64_t tl = ra / m.group; tl <= (rb - 1) / m.group; ++tl) {
        const int64_t t = qs + tl;
        int st, en;
        if constexpr (tok_cached) {
          st = s_ts[t];
          en = s_te[t];
        } else {
          const int e = m.causal ? m.positions[t] + 1 : n;
          st = m.window > 0 ? max(0, e - m.window) : 0;
          en = max(e, st);
        }
        if (en > st) {
          lo = min(lo, st);
          hi = max(hi, en);
        }
      }
      mma_recs[2 * (at + i)] = make_int4(s, i, qs, n);
      mma_recs[2 * (at + i) + 1] = make_int4(lo, hi, (int)rows, 0);
    }
  }
  // the tcgen05 kernel's working pairs: every candidate K evaluated by its own thread (with no
  // decode tiles the model picks all pairs, so it is not run)
  if (TC && L.force_pairs <= 0 && s_dec_units > 0) {
    const float tiles = (float)s_tc_tiles * m.num_kv_heads;
    const float dec_bytes =
        (float)s_dec_units * m.num_kv_heads * 2.f * L.kv_elem_bytes * m.head_dim;
    for (int k0 = warp * 32 + 1; k0 <= L.tc_pairs; k0 += blockDim.x) {
      const int k = k0 + lane;
      const unsigned long long key =
          warp_min_u64(k <= L.tc_pairs ? split_key(L, k, tiles, dec_bytes) : ~0ull);
      if (lane == 0) atomicMin(&s_split, key);  // one shared-memory atomic per warp
    }
  }
  __syncthreads();
  if (tid == 0) {
    plan[0] = carry_m;
    plan[1] = carry_t;
    plan[2] = 0;  // work counter of the warp-MMA kernel
    plan[3] = 0;  // items marked by the tcgen05 kernel
    plan[4] = 0;  // work counter over their units
    int pairs = 0;
    if (TC)
      pairs = L.force_pairs > 0  ? min(L.force_pairs, L.tc_pairs)
              : s_dec_units == 0 ? L.tc_pairs
                                 : (int)(0xffffffffu - (unsigned)(s_split & 0xffffffffull));
    plan[5] = max(0, min(pairs, L.tc_pairs));
  }
}

// Split-KV decode validation: one CTA per sequence.
__global__ void k_validate_decode(const int32_t* seq_lens, const int32_t* block_tables,
                                  int32_t max_blocks, int32_t block_size, int64_t num_blocks,
                                  int32_t partition_size, int32_t max_parts, int check_tables,
                                  const float* k_bscales, const float* v_bscales,
                                  int32_t num_kv_heads, int* status) {
  const int s = blockIdx.x;
  const int n = seq_lens[s];
  if (n < 1) {
    if (threadIdx.x == 0) record_error(status, PA_EINVAL);
    return;
  }
  if (partition_size > 0 && ((int64_t)n + partition_size - 1) / partition_size > max_parts) {
    if (threadIdx.x == 0) record_error(status, PA_EINVAL);
    return;
  }
  if (!check_tables) return;
  const int64_t need = ((int64_t)n + block_size - 1) / block_size;
  if (need > max_blocks) {
    if (threadIdx.x == 0) record_error(status, PA_EINVAL);
    return;
  }
  const int32_t* row = block_tables + (int64_t)s * max_blocks;
  bool bad = false;
  for (int64_t i = threadIdx.x; i < need; i += blockDim.x) {
    const int32_t id = row[i];
    bad |= (id < 0 || (int64_t)id >= num_blocks);
  }
  if (k_bscales)  // per-block factors of the blocks the sequence reads (a pass of its own)
    for (int64_t i = threadIdx.x; i < need; i += blockDim.x) {
      const int32_t id = row[i];
      if (id >= 0 && (int64_t)id < num_blocks)
        bad |= block_factors_bad(k_bscales, v_bscales, id, num_kv_heads);
    }
  if (__syncthreads_or(bad) && threadIdx.x == 0) record_error(status, PA_EINVAL);
}

// Slot mapping: one CTA per sequence.
__global__ void k_slot_mapping(const int32_t* qsl, const int32_t* positions,
                               const int32_t* block_tables, int32_t num_seqs, int64_t num_tokens,
                               int32_t max_blocks, int32_t block_size, int64_t num_blocks,
                               int32_t* slots, int* status) {
  pdl_wait();
  pdl_launch_dependents();
  if (status_set(status)) return;
  const int s = blockIdx.x;
  const int a = qsl[s], b = qsl[s + 1];
  if (a < 0 || b < a || (int64_t)b > num_tokens) {
    if (threadIdx.x == 0) record_error(status, PA_EINVAL);
    return;
  }
  const int32_t* row = block_tables + (int64_t)s * max_blocks;
  for (int t = a + threadIdx.x; t < b; t += blockDim.x) {
    const int32_t pos = positions[t];
    int32_t slot = -1;
    if (pos >= 0 && pos / block_size < max_blocks) {
      const int32_t id = row[pos / block_size];
      if (id >= 0 && (int64_t)id < num_blocks) slot = id * block_size + pos % block_size;
    }
    if (slot < 0) record_error(status, PA_EINVAL);
    slots[t] = slot;
  }
}

__global__ void k_validate_slots(const int32_t* slots, int64_t num_tokens, int64_t num_slots,
                                 const float* kbs, const float* vbs, int32_t block_size,
                                 int32_t num_kv_heads, int* status) {
  pdl_wait();
  pdl_launch_dependents();
  bool bad = false;
  for (int64_t t = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; t < num_tokens;
       t += (int64_t)gridDim.x * blockDim.x) {
    const int32_t s = slots[t];
    const bool out = s < 0 || (int64_t)s >= num_slots;
    bad |= out;
    // per-block factors of the block the row goes to
    if (kbs && !out) bad |= block_factors_bad(kbs, vbs, s / block_size, num_kv_heads);
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) record_error(status, PA_EINVAL);
}

// Scatter: one warp per token copies its K row and its V row (num_kv_heads * head_dim
// elements each, contiguous on both sides) with VEC-wide accesses.
template <typename VEC>
__global__ void k_reshape_and_cache(const VEC* __restrict__ k, const VEC* __restrict__ v,
                                    VEC* __restrict__ k_blocks, VEC* __restrict__ v_blocks,
                                    const int32_t* __restrict__ slots, int64_t num_tokens,
                                    int64_t row_vecs, const int* status) {
  pdl_wait();
  pdl_launch_dependents();
  if (status_set(status)) return;
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= num_tokens) return;
  const int64_t dst = (int64_t)slots[t] * row_vecs;  // pool row index == slot
  const int64_t src = t * row_vecs;
  for (int64_t i = lane; i < row_vecs; i += 32) {
    const VEC a = k[src + i];
    const VEC b = v[src + i];
    k_blocks[dst + i] = a;
    v_blocks[dst + i] = b;
  }
}

// Batches of up to kCheckedScatter tokens (the decode step): the slot check and the scatter in
// one kernel.  Every CTA checks all slots before it writes (the same data, so either every CTA
// writes or none does, with no grid-wide barrier) and then copies its own eight tokens, one
// warp per token as above.
constexpr int kCheckedScatter = 2048;
template <typename VEC>
__global__ void __launch_bounds__(256)
    k_scatter_checked(const VEC* __restrict__ k, const VEC* __restrict__ v,
                      VEC* __restrict__ k_blocks, VEC* __restrict__ v_blocks,
                      const int32_t* __restrict__ slots, int num_tokens, int64_t num_slots,
                      int64_t row_vecs, int* status) {
  __shared__ int s_skip;
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) s_skip = status_set(status) ? 1 : 0;  // one read for the whole CTA
  __syncthreads();
  if (s_skip) return;
  bool bad = false;
  for (int t = threadIdx.x; t < num_tokens; t += blockDim.x) {
    const int32_t sl = slots[t];
    bad |= (sl < 0 || (int64_t)sl >= num_slots);
  }
  if (__syncthreads_or(bad)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) record_error(status, PA_EINVAL);
    return;
  }
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= num_tokens) return;
  const int64_t dst = (int64_t)slots[t] * row_vecs, src = (int64_t)t * row_vecs;
  for (int64_t i = lane; i < row_vecs; i += 32) {
    const VEC a = k[src + i];
    const VEC b = v[src + i];
    k_blocks[dst + i] = a;
    v_blocks[dst + i] = b;
  }
}

// One token's row in the quantising scatter, 8 consecutive values per lane (one kv head:
// head_dim is a multiple of 8), 16-byte loads of bf16 rows; the same per-element arithmetic
// as the one-value-per-lane loop of k_scatter_convert.
template <typename TS, int DST>
__device__ __forceinline__ void scatter_row_vec8(
    const TS* __restrict__ k, const TS* __restrict__ v, void* __restrict__ kb,
    void* __restrict__ vb, int64_t src, int64_t dst, int32_t slot, int64_t row_elems,
    float k_scale, float v_scale, const float* __restrict__ k_scales,
    const float* __restrict__ v_scales, const float* __restrict__ kbs,
    const float* __restrict__ vbs, int32_t block_size, int32_t head_dim, int32_t hkv, int lane) {
  for (int64_t i = (int64_t)lane * 8; i < row_elems; i += 256) {
    const int g = (int)(i / head_dim);
    float ks = k_scales ? __ldg(k_scales + g) : k_scale;
    float vs = v_scales ? __ldg(v_scales + g) : v_scale;
    if (kbs) {
      const int64_t f = (int64_t)(slot / block_size) * hkv + g;
      ks = __ldg(kbs + f);
      vs = __ldg(vbs + f);
    }
    const uint4 kw = *reinterpret_cast<const uint4*>(k + src + i);
    const uint4 vw = *reinterpret_cast<const uint4*>(v + src + i);
    const TS* ke = reinterpret_cast<const TS*>(&kw);
    const TS* ve = reinterpret_cast<const TS*>(&vw);
    float a[8], b[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      a[e] = __fdiv_rn(to_f32(ke[e]), ks);
      b[e] = __fdiv_rn(to_f32(ve[e]), vs);
    }
    if constexpr (DST == PA_FP8_E4M3) {
      uint2 ko, vo;
      ko.x = f32x2_to_e4m3x2(a[0], a[1]) | ((uint32_t)f32x2_to_e4m3x2(a[2], a[3]) << 16);
      ko.y = f32x2_to_e4m3x2(a[4], a[5]) | ((uint32_t)f32x2_to_e4m3x2(a[6], a[7]) << 16);
      vo.x = f32x2_to_e4m3x2(b[0], b[1]) | ((uint32_t)f32x2_to_e4m3x2(b[2], b[3]) << 16);
      vo.y = f32x2_to_e4m3x2(b[4], b[5]) | ((uint32_t)f32x2_to_e4m3x2(b[6], b[7]) << 16);
      *reinterpret_cast<uint2*>(static_cast<uint8_t*>(kb) + dst + i) = ko;
      *reinterpret_cast<uint2*>(static_cast<uint8_t*>(vb) + dst + i) = vo;
    } else if constexpr (DST == PA_BF16) {
      uint4 ko, vo;
      __nv_bfloat16* kr = reinterpret_cast<__nv_bfloat16*>(&ko);
      __nv_bfloat16* vr = reinterpret_cast<__nv_bfloat16*>(&vo);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        kr[e] = __float2bfloat16_rn(a[e]);
        vr[e] = __float2bfloat16_rn(b[e]);
      }
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(kb) + dst + i) = ko;
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(vb) + dst + i) = vo;
    } else {
      float* kf = static_cast<float*>(kb) + dst + i;
      float* vf = static_cast<float*>(vb) + dst + i;
      *reinterpret_cast<float4*>(kf) = make_float4(a[0], a[1], a[2], a[3]);
      *reinterpret_cast<float4*>(kf + 4) = make_float4(a[4], a[5], a[6], a[7]);
      *reinterpret_cast<float4*>(vf) = make_float4(b[0], b[1], b[2], b[3]);
      *reinterpret_cast<float4*>(vf + 4) = make_float4(b[4], b[5], b[6], b[7]);
    }
  }
}

// Scatter with conversion ("paged_attention_v2_pytorch.py": the pool holds K / k_scale and
// V / v_scale in kv_cache_dtype).  One warp per token; every element is divided by its scale
// in fp32 (IEEE division, as written) and rounded to the pool's type to nearest even, fp8
// saturating to +-448.  CHECKED: every CTA first checks all slots (batches up to
// kCheckedScatter tokens), otherwise k_validate_slots ran before.
template <typename TS, int DST, bool CHECKED>
__global__ void __launch_bounds__(256)
    k_scatter_convert(const TS* __restrict__ k, const TS* __restrict__ v, void* __restrict__ kb,
                      void* __restrict__ vb, const int32_t* __restrict__ slots, int64_t num_tokens,
                      int64_t num_slots, int64_t row_elems, float k_scale, float v_scale,
                      const float* __restrict__ k_scales, const float* __restrict__ v_scales,
                      const float* __restrict__ kbs, const float* __restrict__ vbs,
                      int32_t block_size, int32_t head_dim, bool vec8, int* status) {
  const int32_t hkv = (int32_t)(row_elems / head_dim);
  __shared__ int s_skip;
  pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) s_skip = status_set(status) ? 1 : 0;  // one read for the whole CTA
  __syncthreads();
  if (s_skip) return;
  if constexpr (CHECKED) {
    bool bad = false;
    for (int64_t t = threadIdx.x; t < num_tokens; t += blockDim.x) {
      const int32_t sl = slots[t];
      const bool out = sl < 0 || (int64_t)sl >= num_slots;
      bad |= out;
      if (kbs && !out) bad |= block_factors_bad(kbs, vbs, sl / block_size, hkv);
    }
    if (__syncthreads_or(bad)) {
      if (blockIdx.x == 0 && threadIdx.x == 0) record_error(status, PA_EINVAL);
      return;
    }
  }
  const int lane = threadIdx.x & 31;
  const int64_t t = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= num_tokens) return;
  const int32_t slot = slots[t];
  const int64_t dst = (int64_t)slot * row_elems, src = t * row_elems;
  if constexpr (sizeof(TS) == 2) {
    if (vec8) {
      scatter_row_vec8<TS, DST>(k, v, kb, vb, src, dst, slot, row_elems, k_scale, v_scale,
                                k_scales, v_scales, kbs, vbs, block_size, head_dim, hkv, lane);
      return;
    }
  }
  for (int64_t i = lane; i < row_elems; i += 32) {
    // one scale per kv head (head i / head_dim of the row), or per (block, kv head), when the
    // arrays are given
    const int g = k_scales || v_scales || kbs ? (int)(i / head_dim) : 0;
    float ks = k_scales ? __ldg(k_scales + g) : k_scale;
    float vs = v_scales ? __ldg(v_scales + g) : v_scale;
    if (kbs) {
      const int64_t f = (int64_t)(slot / block_size) * hkv + g;
      ks = __ldg(kbs + f);
      vs = __ldg(vbs + f);
    }
    const float a = __fdiv_rn(to_f32(k[src + i]), ks);
    const float b = __fdiv_rn(to_f32(v[src + i]), vs);
    if constexpr (DST == PA_FP8_E4M3) {
      static_cast<uint8_t*>(kb)[dst + i] = (uint8_t)(f32x2_to_e4m3x2(a, 0.f) & 0xffu);
      static_cast<uint8_t*>(vb)[dst + i] = (uint8_t)(f32x2_to_e4m3x2(b, 0.f) & 0xffu);
    } else if constexpr (DST == PA_BF16) {
      static_cast<__nv_bfloat16*>(kb)[dst + i] = __float2bfloat16_rn(a);
      static_cast<__nv_bfloat16*>(vb)[dst + i] = __float2bfloat16_rn(b);
    } else {
      static_cast<float*>(kb)[dst + i] = a;
      static_cast<float*>(vb)[dst + i] = b;
    }
  }
}

template <typename TS, int DST>
cudaError_t convert_as(const void* k, const void* v, void* kb, void* vb, const int32_t* slots,
                       int64_t T, int64_t row_elems, int64_t num_slots, float k_scale,
                       float v_scale, const float* ks, const float* vs, const float* kbs,
                       const float* vbs, int32_t block_size, int32_t head_dim, int* status,
                       cudaStream_t stream) {
  const dim3 grid((unsigned)((T + 7) / 8)), block(256);
  // 8 values per lane: bf16 rows of whole 16-byte groups inside one kv head, and tensors
  // aligned for the 16-byte loads and the destination's stores
  const size_t dst_elem = DST == PA_FP8_E4M3 ? 1 : DST == PA_BF16 ? 2 : 4;
  const bool vec8 = sizeof(TS) == 2 && row_elems % 8 == 0 && head_dim % 8 == 0 &&
                    ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15) == 0 &&
                    ((reinterpret_cast<uintptr_t>(kb) | reinterpret_cast<uintptr_t>(vb)) &
                     (8 * dst_elem - 1)) == 0;
  if (T <= kCheckedScatter)
    return launch_pdl(k_scatter_convert<TS, DST, true>, grid, block, 0, stream, (const TS*)k,
                      (const TS*)v, kb, vb, slots, T, num_slots, row_elems, k_scale, v_scale,
                      ks, vs, kbs, vbs, block_size, head_dim, vec8, status);
  const int64_t vgrid = std::min<int64_t>((T + 255) / 256, 1024);
  cudaError_t e = launch_pdl(k_validate_slots, dim3((unsigned)vgrid), dim3(256), 0, stream, slots,
                             T, num_slots, kbs, vbs, block_size,
                             (int32_t)(row_elems / head_dim), status);
  if (e != cudaSuccess) return e;
  return launch_pdl(k_scatter_convert<TS, DST, false>, grid, block, 0, stream, (const TS*)k,
                    (const TS*)v, kb, vb, slots, T, num_slots, row_elems, k_scale, v_scale, ks,
                    vs, kbs, vbs, block_size, head_dim, vec8, status);
}

// Per kv head dequantisation scales must be finite and positive (tinyllm 2.6: reject before
// any write); the kernels launched after this one see the recorded status and write nothing.
__global__ void k_validate_scales(const float* k_scales, const float* v_scales,
                                  int32_t num_kv_heads, int* status) {
  pdl_wait();
  pdl_launch_dependents();
  bool bad = false;
  for (int g = threadIdx.x; g < num_kv_heads; g += blockDim.x) {
    const float a = k_scales ? k_scales[g] : 1.f, b = v_scales ? v_scales[g] : 1.f;
    bad |= !(a > 0.f && a <= 3.402823466e38f) || !(b > 0.f && b <= 3.402823466e38f);
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) record_error(status, PA_EINVAL);
}


// Slot mapping and scatter in one launch, for batches of up to kCheckedScatter tokens and
// kFusedSeqs sequences (a decode step): every CTA loads the query start locations into shared
// memory, finds each token's sequence by binary search, computes every token's slot by the rule
// of k_slot_mapping and checks it; only when all are valid does it copy its own eight tokens'
// rows (one warp per token).  CTA 0 writes the slot mapping (-1 for an invalid token).  A token
// that no sequence's range holds is invalid.
//
// AFTER_PLAN: launched right after the planning kernel of the same attention call, so it runs
// alongside the plan instead of before it.  Its inputs are complete when it starts (the
// planner's reasoning); its writes wait for the plan, which ends only after the kernels ahead
// of it (an attention kernel of the previous call may still read a block this scatter writes,
// when the caller reuses freed blocks).  The attention kernel behind it waits for this grid,
// so it finds both done.
constexpr int kFusedSeqs = 2047;
template <typename VEC, bool AFTER_PLAN>
__device__ __forceinline__ void map_and_scatter_body(
    const VEC* __restrict__ k, const VEC* __restrict__ v, VEC* __restrict__ k_blocks,
    VEC* __restrict__ v_blocks, const int32_t* __restrict__ qsl,
    const int32_t* __restrict__ positions, const int32_t* __restrict__ tables, int num_seqs,
    int num_tokens, int32_t max_blocks, int32_t block_size, int64_t num_blocks,
    int64_t row_vecs, int32_t* __restrict__ slots, int* status) {
  __shared__ int s_qsl[kFusedSeqs + 1];
  __shared__ int s_slot[kCheckedScatter];
  __shared__ int s_skip;
  if (!AFTER_PLAN) pdl_wait();
  pdl_launch_dependents();
  if (threadIdx.x == 0) s_skip = status_set(status) ? 1 : 0;  // one read for the whole CTA
  __syncthreads();
  if (s_skip) return;
  for (int i = threadIdx.x; i <= num_seqs; i += blockDim.x) s_qsl[i] = qsl[i];
  __syncthreads();
  bool bad = false;
  for (int i = threadIdx.x; i < num_seqs; i += blockDim.x) {
    const int a = s_qsl[i], b = s_qsl[i + 1];
    bad |= a < 0 || b < a || b > num_tokens;
  }
  for (int t = threadIdx.x; t < num_tokens; t += blockDim.x) {
    int lo = 0, hi = num_seqs - 1, s = -1;  // the last sequence starting at or before t
    while (lo <= hi) {
      const int mid = (lo + hi) >> 1;
      if (s_qsl[mid] <= t) {
        s = mid;
        lo = mid + 1;
      } else {
        hi = mid - 1;
      }
    }
    int32_t slot = -1;
    if (s >= 0 && t < s_qsl[s + 1]) {
      const int32_t pos = positions[t];
      if (pos >= 0 && pos / block_size < max_blocks) {
        const int32_t id = tables[(int64_t)s * max_blocks + pos / block_size];
        if (id >= 0 && (int64_t)id < num_blocks) slot = id * block_size + pos % block_size;
      }
    }
    s_slot[t] = slot;
    bad |= slot < 0;
  }
  bad = __syncthreads_or(bad);
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int64_t src = (int64_t)t * row_vecs;
  // the start of this warp's token's rows is loaded before the wait (they are inputs), so
  // only the stores follow it
  constexpr int kPre = 4;
  VEC ka[kPre], va[kPre];
  if (!bad && t < num_tokens)
#pragma unroll
    for (int j = 0; j < kPre; ++j)
      if (lane + 32 * j < row_vecs) {
        ka[j] = k[src + lane + 32 * j];
        va[j] = v[src + lane + 32 * j];
      }
  if (AFTER_PLAN) pdl_wait();  // the first global write
  if (blockIdx.x == 0)
    for (int t = threadIdx.x; t < num_tokens; t += blockDim.x) slots[t] = s_slot[t];
  if (bad) {
    if (blockIdx.x == 0 && threadIdx.x == 0) record_error(status, PA_EINVAL);
    return;
  }
  if (t >= num_tokens) return;
  const int64_t dst = (int64_t)s_slot[t] * row_vecs;
#pragma unroll
  for (int j = 0; j < kPre; ++j)
    if (lane + 32 * j < row_vecs) {
      k_blocks[dst + lane + 32 * j] = ka[j];
      v_blocks[dst + lane + 32 * j] = va[j];
    }
  for (int64_t i = lane + 32 * kPre; i < row_vecs; i += 32) {
    const VEC a = k[src + i];
    const VEC b = v[src + i];
    k_blocks[dst + i] = a;
    v_blocks[dst + i] = b;
  }
}

template <typename VEC, bool AFTER_PLAN>
__global__ void __launch_bounds__(256)
    k_map_and_scatter(const VEC* __restrict__ k, const VEC* __restrict__ v,
                      VEC* __restrict__ k_blocks, VEC* __restrict__ v_blocks,
                      const int32_t* __restrict__ qsl, const int32_t* __restrict__ positions,
                      const int32_t* __restrict__ tables, int num_seqs, int num_tokens,
                      int32_t max_blocks, int32_t block_size, int64_t num_blocks,
                      int64_t row_vecs, int32_t* __restrict__ slots, int* status) {
  map_and_scatter_body<VEC, AFTER_PLAN>(k, v, k_blocks, v_blocks, qsl, positions, tables,
                                        num_seqs, num_tokens, max_blocks, block_size,
                                        num_blocks, row_vecs, slots, status);
  if (AFTER_PLAN) pdl_wait();  // this grid ends only after the plan has (CTAs that skipped)
}

template <typename VEC, bool AFTER_PLAN = false>
cudaError_t map_and_scatter_as(const void* k, const void* v, void* kb, void* vb,
                               const int32_t* qsl, const int32_t* positions,
                               const int32_t* tables, int32_t S, int64_t T, int32_t max_blocks,
                               int32_t bs, int64_t nb, int64_t row_bytes, int32_t* slots,
                               int* status, cudaStream_t stream) {
  return launch_pdl(k_map_and_scatter<VEC, AFTER_PLAN>, dim3((unsigned)((T + 7) / 8)), dim3(256),
                    0, stream,
                    (const VEC*)k, (const VEC*)v, (VEC*)kb, (VEC*)vb, qsl, positions, tables,
                    (int)S, (int)T, max_blocks, bs, nb, row_bytes / (int64_t)sizeof(VEC), slots,
                    status);
}

// Gather validation: one CTA per sequence.
__global__ void k_validate_gather(const int32_t* cu, const int32_t* starts, const int32_t* tables,
                                  int64_t num_rows, int32_t block_size, int64_t num_blocks,
                                  int32_t max_blocks, int* status) {
  const int s = blockIdx.x;
  const int a = cu[s], b = cu[s + 1];
  const int64_t start = starts ? starts[s] : 0;
  if (a < 0 || b < a || (int64_t)b > num_rows || start < 0) {
    if (threadIdx.x == 0) record_error(status, PA_EINVAL);
    return;
  }
  const int32_t* row = tables + (int64_t)s * max_blocks;
  bool bad = false;
  for (int r = a + threadIdx.x; r < b; r += blockDim.x) {
    const int64_t pos = (r - a) + start;
    if (pos / block_size >= max_blocks) {
      bad = true;
      continue;
    }
    const int32_t id = row[pos / block_size];
    bad |= (id < 0 || (int64_t)id >= num_blocks);
  }
  if (__syncthreads_or(bad) && threadIdx.x == 0) record_error(status, PA_EINVAL);
}

// Gather: CTA (s, y) copies rows a + y * warps + warp, stepping by gridDim.y * warps.
template <typename VEC>
__global__ void k_gather_kv(const VEC* __restrict__ k_blocks, const VEC* __restrict__ v_blocks,
                            VEC* __restrict__ k_out, VEC* __restrict__ v_out,
                            const int32_t* __restrict__ cu, const int32_t* __restrict__ starts,
                            const int32_t* __restrict__ tables, int32_t block_size,
                            int32_t max_blocks, int64_t row_vecs, const int* status) {
  if (status_set(status)) return;
  const int s = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int a = cu[s], b = cu[s + 1];
  const int64_t start = starts ? starts[s] : 0;
  const int32_t* row = tables + (int64_t)s * max_blocks;
  for (int r = a + blockIdx.y * nwarps + warp; r < b; r += gridDim.y * nwarps) {
    const int64_t pos = (r - a) + start;
    const int64_t slot = (int64_t)row[pos / block_size] * block_size + pos % block_size;
    const int64_t src = slot * row_vecs, dst = (int64_t)r * row_vecs;
    // up to four K and four V loads in flight per lane before their stores
    constexpr int U = 4;
    for (int64_t i0 = lane; i0 < row_vecs; i0 += 32 * U) {
      VEC kv[U], vv[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t i = i0 + 32 * u;
        if (i < row_vecs) {
          kv[u] = k_blocks[src + i];
          if (v_out) vv[u] = v_blocks[src + i];
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int64_t i = i0 + 32 * u;
        if (i < row_vecs) {
          k_out[dst + i] = kv[u];
          if (v_out) v_out[dst + i] = vv[u];
        }
      }
    }
  }
}

template <typename VEC>
cudaError_t scatter_as(const void* k, const void* v, void* kb, void* vb, const int32_t* slots,
                       int64_t T, int64_t row_bytes, int64_t num_slots, int* status,
                       cudaStream_t stream) {
  const int64_t row_vecs = row_bytes / (int64_t)sizeof(VEC);
  if (T <= kCheckedScatter)
    return launch_pdl(k_scatter_checked<VEC>, dim3((unsigned)((T + 7) / 8)), dim3(256), 0, stream,
                      (const VEC*)k, (const VEC*)v, (VEC*)kb, (VEC*)vb, slots, (int)T, num_slots,
                      row_vecs, status);
  const int64_t vgrid = std::min<int64_t>((T + 255) / 256, 1024);
  cudaError_t e = launch_pdl(k_validate_slots, dim3((unsigned)vgrid), dim3(256), 0, stream, slots,
                             T, num_slots, (const float*)nullptr, (const float*)nullptr, 1, 0,
                             status);
  if (e != cudaSuccess) return e;
  const int warps = 8;
  const int64_t grid = (T + warps - 1) / warps;
  return launch_pdl(k_reshape_and_cache<VEC>, dim3((unsigned)grid), dim3(warps * 32), 0, stream,
                    (const VEC*)k, (const VEC*)v, (VEC*)kb, (VEC*)vb, slots, T, row_vecs,
                    (const int*)status);
}

template <typename VEC>
cudaError_t gather_as(const void* kb, const void* vb, void* ko, void* vo, const int32_t* cu,
                      const int32_t* starts, const int32_t* tables, int32_t S, int64_t row_bytes,
                      int32_t bs, int32_t max_blocks, const int* status, cudaStream_t stream) {
  // about 4096 CTAs whatever the number of sequences: several waves even out the SMs' loads
  // (64 sequences x 16 CTAs, under one wave, copied at 0.85 of the copy rate; x 64 at 0.90)
  dim3 grid(S, (unsigned)std::max(16, std::min(1024, 4096 / std::max(S, 1))));
  k_gather_kv<VEC><<<grid, 256, 0, stream>>>((const VEC*)kb, (const VEC*)vb, (VEC*)ko, (VEC*)vo,
                                             cu, starts, tables, bs, max_blocks,
                                             row_bytes / (int64_t)sizeof(VEC), status);
  return cudaGetLastError();
}

bool aligned(const void* p, size_t a) { return p == nullptr || (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

cudaError_t launch_plan_varlen(const VarlenMeta& m, int32_t* plan, const PlanLayout& L,
                               int* status, cudaStream_t stream) {
  // block 0 plans; when the batch's metadata fits the planner's shared memory, blocks 1 .. V
  // check the block tables beside it (V = min(num_seqs, 32)); otherwise block 0 checks them
  const bool cached = m.num_seqs <= kPlanCacheSeqs && m.num_tokens <= kPlanCacheTokens;
  const size_t dyn = m.num_seqs <= kPlanCacheSeqs
                         ? plan_smem_bytes(m.num_seqs, m.num_tokens, plan_items_cached(L))
                         : 0;
  const int validators = cached ? std::min(m.num_seqs, 32) : 0;
  auto kern = cached ? (L.use_tc ? k_plan_varlen<true, true> : k_plan_varlen<true, false>)
                     : (L.use_tc ? k_plan_varlen<false, true> : k_plan_varlen<false, false>);
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
      (int)plan_smem_bytes(kPlanCacheSeqs, kPlanCacheTokens, kPlanCacheItems));
  if (e != cudaSuccess) return e;
  return launch_pdl(kern, dim3(1 + validators), dim3(1024), dyn, stream, m, plan, L, status);
}

cudaError_t launch_validate_decode(const int32_t* seq_lens, const int32_t* block_tables,
                                   int32_t num_seqs, int32_t max_blocks, int32_t block_size,
                                   int64_t num_blocks, int32_t partition_size, int32_t max_parts,
                                   int check_tables, int* status, cudaStream_t stream,
                                   const float* k_bscales, const float* v_bscales,
                                   int32_t num_kv_heads) {
  if (num_seqs <= 0) return cudaSuccess;
  k_validate_decode<<<num_seqs, 256, 0, stream>>>(seq_lens, block_tables, max_blocks, block_size,
                                                  num_blocks, partition_size, max_parts,
                                                  check_tables, k_bscales, v_bscales,
                                                  num_kv_heads, status);
  return cudaGetLastError();
}

cudaError_t launch_slot_mapping(const int32_t* qsl, const int32_t* positions,
                                const int32_t* block_tables, int32_t num_seqs, int64_t num_tokens,
                                int32_t max_blocks, int32_t block_size, int64_t num_blocks,
                                int32_t* slots, int* status, cudaStream_t stream) {
  if (num_seqs <= 0) return cudaSuccess;
  return launch_pdl(k_slot_mapping, dim3(num_seqs), dim3(256), 0, stream, qsl, positions,
                    block_tables, num_seqs, num_tokens, max_blocks, block_size, num_blocks, slots,
                    status);
}

cudaError_t launch_reshape_and_cache(const void* k, const void* v, void* k_blocks, void* v_blocks,
                                     const int32_t* slots, int64_t num_tokens, int64_t row_bytes,
                                     int32_t block_size, int64_t num_blocks, int* status,
                                     cudaStream_t stream) {
  if (num_tokens <= 0) return cudaSuccess;
  const int64_t num_slots = num_blocks * block_size;
  if (row_bytes % 16 == 0 && aligned(k, 16) && aligned(v, 16) && aligned(k_blocks, 16) &&
      aligned(v_blocks, 16))
    return scatter_as<uint4>(k, v, k_blocks, v_blocks, slots, num_tokens, row_bytes, num_slots,
                             status, stream);
  if (row_bytes % 4 == 0 && aligned(k, 4) && aligned(v, 4) && aligned(k_blocks, 4) &&
      aligned(v_blocks, 4))
    return scatter_as<uint32_t>(k, v, k_blocks, v_blocks, slots, num_tokens, row_bytes,
                                num_slots, status, stream);
  if (row_bytes % 2 == 0 && aligned(k, 2) && aligned(v, 2) && aligned(k_blocks, 2) &&
      aligned(v_blocks, 2))
    return scatter_as<uint16_t>(k, v, k_blocks, v_blocks, slots, num_tokens, row_bytes,
                                num_slots, status, stream);
  return scatter_as<uint8_t>(k, v, k_blocks, v_blocks, slots, num_tokens, row_bytes, num_slots,
                             status, stream);
}

cudaError_t launch_slot_mapping_and_cache(const void* k, const void* v, void* k_blocks,
                                          void* v_blocks, const int32_t* qsl,
                                          const int32_t* positions, const int32_t* tables,
                                          int32_t num_seqs, int64_t num_tokens,
                                          int32_t max_blocks, int32_t block_size,
                                          int64_t num_blocks, int64_t row_bytes, int32_t* slots,
                                          int* status, cudaStream_t stream) {
  if (num_tokens <= 0) return cudaSuccess;
  if (num_tokens > kCheckedScatter || num_seqs > kFusedSeqs || num_seqs <= 0) {
    // larger batches: the two launches of pa_slot_mapping and pa_reshape_and_cache; slots
    // start at -1, so a token no sequence holds fails the scatter's check
    cudaError_t e = cudaMemsetAsync(slots, 0xff, (size_t)num_tokens * sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
    e = num_seqs > 0 ? launch_slot_mapping(qsl, positions, tables, num_seqs, num_tokens,
                                           max_blocks, block_size, num_blocks, slots, status,
                                           stream)
                     : cudaSuccess;
    if (e != cudaSuccess) return e;
    return launch_reshape_and_cache(k, v, k_blocks, v_blocks, slots, num_tokens, row_bytes,
                                    block_size, num_blocks, status, stream);
  }
  if (row_bytes % 16 == 0 && aligned(k, 16) && aligned(v, 16) && aligned(k_blocks, 16) &&
      aligned(v_blocks, 16))
    return map_and_scatter_as<uint4>(k, v, k_blocks, v_blocks, qsl, positions, tables, num_seqs,
                                     num_tokens, max_blocks, block_size, num_blocks, row_bytes,
                                     slots, status, stream);
  if (row_bytes % 4 == 0 && aligned(k, 4) && aligned(v, 4) && aligned(k_blocks, 4) &&
      aligned(v_blocks, 4))
    return map_and_scatter_as<uint32_t>(k, v, k_blocks, v_blocks, qsl, positions, tables,
                                        num_seqs, num_tokens, max_blocks, block_size, num_blocks,
                                        row_bytes, slots, status, stream);
  if (row_bytes % 2 == 0 && aligned(k, 2) && aligned(v, 2) && aligned(k_blocks, 2) &&
      aligned(v_blocks, 2))
    return map_and_scatter_as<uint16_t>(k, v, k_blocks, v_blocks, qsl, positions, tables,
                                        num_seqs, num_tokens, max_blocks, block_size, num_blocks,
                                        row_bytes, slots, status, stream);
  return map_and_scatter_as<uint8_t>(k, v, k_blocks, v_blocks, qsl, positions, tables, num_seqs,
                                     num_tokens, max_blocks, block_size, num_blocks, row_bytes,
                                     slots, status, stream);
}

bool map_and_scatter_fits(int32_t num_seqs, int64_t num_tokens) {
  return num_tokens > 0 && num_tokens <= kCheckedScatter && num_seqs > 0 &&
         num_seqs <= kFusedSeqs;
}

cudaError_t launch_map_and_scatter_after_plan(const void* k, const void* v, void* k_blocks,
                                              void* v_blocks, const int32_t* qsl,
                                              const int32_t* positions, const int32_t* tables,
                                              int32_t num_seqs, int64_t num_tokens,
                                              int32_t max_blocks, int32_t block_size,
                                              int64_t num_blocks, int64_t row_bytes,
                                              int32_t* slots, int* status, cudaStream_t stream) {
  if (row_bytes % 16 == 0 && aligned(k, 16) && aligned(v, 16) && aligned(k_blocks, 16) &&
      aligned(v_blocks, 16))
    return map_and_scatter_as<uint4, true>(k, v, k_blocks, v_blocks, qsl, positions, tables,
                                           num_seqs, num_tokens, max_blocks, block_size,
                                           num_blocks, row_bytes, slots, status, stream);
  if (row_bytes % 4 == 0 && aligned(k, 4) && aligned(v, 4) && aligned(k_blocks, 4) &&
      aligned(v_blocks, 4))
    return map_and_scatter_as<uint32_t, true>(k, v, k_blocks, v_blocks, qsl, positions, tables,
                                              num_seqs, num_tokens, max_blocks, block_size,
                                              num_blocks, row_bytes, slots, status, stream);
  if (row_bytes % 2 == 0 && aligned(k, 2) && aligned(v, 2) && aligned(k_blocks, 2) &&
      aligned(v_blocks, 2))
    return map_and_scatter_as<uint16_t, true>(k, v, k_blocks, v_blocks, qsl, positions, tables,
                                              num_seqs, num_tokens, max_blocks, block_size,
                                              num_blocks, row_bytes, slots, status, stream);
  return map_and_scatter_as<uint8_t, true>(k, v, k_blocks, v_blocks, qsl, positions, tables,
                                           num_seqs, num_tokens, max_blocks, block_size,
                                           num_blocks, row_bytes, slots, status, stream);
}

cudaError_t launch_reshape_and_cache_convert(const void* k, const void* v, void* k_blocks,
                                             void* v_blocks, const int32_t* slots,
                                             int64_t num_tokens, int64_t row_elems,
                                             int32_t block_size, int64_t num_blocks, int src_bf16,
                                             int dst, float k_scale, float v_scale,
                                             const float* k_scales, const float* v_scales,
                                             int32_t head_dim, int* status, cudaStream_t stream,
                                             const float* k_bscales, const float* v_bscales) {
  if (num_tokens <= 0) return cudaSuccess;
  const int64_t ns = num_blocks * block_size;
#define PA_CONVERT(TS, DST)                                                                  \
  convert_as<TS, DST>(k, v, k_blocks, v_blocks, slots, num_tokens, row_elems, ns, k_scale,   \
                      v_scale, k_scales, v_scales, k_bscales, v_bscales, block_size,        \
                      head_dim, status, stream)
  cudaError_t e;
  if (src_bf16)
    e = dst == PA_FP8_E4M3 ? PA_CONVERT(__nv_bfloat16, PA_FP8_E4M3)
        : dst == PA_BF16   ? PA_CONVERT(__nv_bfloat16, PA_BF16)
                           : PA_CONVERT(__nv_bfloat16, PA_F32);
  else
    e = dst == PA_FP8_E4M3 ? PA_CONVERT(float, PA_FP8_E4M3)
        : dst == PA_BF16   ? PA_CONVERT(float, PA_BF16)
                           : PA_CONVERT(float, PA_F32);
#undef PA_CONVERT
  return e;
}

cudaError_t launch_gather_kv(const void* k_blocks, const void* v_blocks, void* k_out, void* v_out,
                             const int32_t* cu, const int32_t* starts, const int32_t* tables,
                             int32_t num_seqs, int64_t num_rows, int64_t row_bytes,
                             int32_t block_size, int64_t num_blocks, int32_t max_blocks,
                             int* status, cudaStream_t stream) {
  if (num_seqs <= 0) return cudaSuccess;
  k_validate_gather<<<num_seqs, 256, 0, stream>>>(cu, starts, tables, num_rows, block_size,
                                                  num_blocks, max_blocks, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (row_bytes % 16 == 0 && aligned(k_blocks, 16) && aligned(v_blocks, 16) && aligned(k_out, 16) &&
      aligned(v_out, 16))
    return gather_as<uint4>(k_blocks, v_blocks, k_out, v_out, cu, starts, tables, num_seqs,
                            row_bytes, block_size, max_blocks, status, stream);
  if (row_bytes % 4 == 0 && aligned(k_blocks, 4) && aligned(v_blocks, 4) && aligned(k_out, 4) &&
      aligned(v_out, 4))
    return gather_as<uint32_t>(k_blocks, v_blocks, k_out, v_out, cu, starts, tables, num_seqs,
                               row_bytes, block_size, max_blocks, status, stream);
  if (row_bytes % 2 == 0 && aligned(k_blocks, 2) && aligned(v_blocks, 2) && aligned(k_out, 2) &&
      aligned(v_out, 2))
    return gather_as<uint16_t>(k_blocks, v_blocks, k_out, v_out, cu, starts, tables, num_seqs,
                               row_bytes, block_size, max_blocks, status, stream);
  return gather_as<uint8_t>(k_blocks, v_blocks, k_out, v_out, cu, starts, tables, num_seqs,
                            row_bytes, block_size, max_blocks, status, stream);
}


cudaError_t launch_validate_scales(const float* k_scales, const float* v_scales,
                                   int32_t num_kv_heads, int* status, cudaStream_t stream) {
  if (!k_scales && !v_scales) return cudaSuccess;
  return launch_pdl(k_validate_scales, dim3(1), dim3(256), 0, stream, k_scales, v_scales,
                    num_kv_heads, status);
}

}  // namespace pa
