// k_decode_mma.cu -- paged attention for tiles of up to 16 query rows of one (sequence,
// kv head): decode tokens (one CTA serves the whole GQA group of a kv head) and the split-KV
// partitions of PagedAttention V2.
//
// Data path.  The pool is [num_blocks, 16, num_kv_heads, D] bf16.  One (block, kv head) K or
// V tile is 16 rows of D elements, rows 2 * num_kv_heads * D bytes apart.  Each warp of the
// CTA owns a private ring of NS stages; its lane 0 streams whole blocks into the ring with
// 3-D TMA tile loads (box 64 x 1 x 16, 128-byte swizzle, one 2 KB box per 64-dim half, K and
// V on one mbarrier).  Warps take the visible blocks round-robin, so every byte is read once
// per kv head and the reads stay 16-byte vectorised and coalesced.
//
// Math.  The tile's query rows are (token, head) pairs, token-major; q stays in registers as
// bf16 A fragments.  Per block: S = Q K^T on the m16n8k16 tensor-core MMA (fp32 accumulate),
// mask to each row's visible range [start, end), scale into the log2 domain, block max via
// quad shuffles, the online-softmax update m' = max(m, .), alpha = 2^(m - m'),
// l = alpha l + sum p, O = alpha O + P V (tinyllm section 2.2, applied per 16-key block).
// P enters the PV MMA as a bf16 hi/lo pair (two MMAs), so the weights keep ~17 bits; l sums
// the fp32 weights.  At the end the warps' (m, l, O) states are merged in fixed warp order
// and o = O * (1 / l).
//
// Why warp MMA here: these tiles are HBM-bound (one pass over K and V per kv head), so the
// tensor core only has to take the ~2 G D FMA per key off the FP32 pipe; with G = 8 the FMA
// path would need about half the chip's FP32 rate at full HBM bandwidth.
//
// fp8 (e4m3) pools, head size 128 ("paged_attention_v2_pytorch.py": kv_cache_dtype "fp8",
// K = k_scale * pool, V = v_scale * pool).  A tile is 16 rows of 128 one-byte codes, one TMA
// box of 2 KB with the 128-byte swizzle, so a stage is half the bf16 one and the ring is
// twice as deep.  The codes stay in shared memory as they arrived; each lane loads the
// bytes of its own MMA fragments with 16-byte loads and widens them in registers to f16
// (exact for e4m3), and the products run on the f16 m16n8k16 MMA.  The operands are swapped
// against the bf16 path: the block's 16 keys are the MMA's M and the tile's query rows its
// N, in groups of 8 (S^T = K Q^T, O^T = V^T P^T).  For a GQA group of up to 8 heads a decode
// token is one group: half the MMAs, exponentials and rescales of a 16-row tile.  Varlen
// tiles over e4m3 pools are therefore 8 rows (the plan cuts them so), and a split-KV
// partition of a larger group runs two groups with the same code per group, so a row's bits
// do not depend on the tile it sits in.  Both contractions read their dimensions in a
// permuted order, which leaves the sums alone and makes every lane's bytes contiguous:
//   S^T = K Q^T: in k-step kk, fragment column 2c + j (c = lane % 4) is dimension
//     32c + 4kk + j and column 2c + 8 + j is dimension 32c + 4kk + 2 + j, so the lane reads
//     bytes [32c, 32c + 32) of key rows g and g + 8 (g = lane / 4), and q is loaded in the
//     same order;
//   O^T = V^T P^T: in M-tile t = 2i + h, fragment row g is dimension 16g + 4i + 2h and row
//     g + 8 dimension 16g + 4i + 2h + 1, so the lane reads bytes [16g, 16g + 16) of its four
//     key rows 2c, 2c + 1, 2c + 8, 2c + 9 and pairs them with byte permutes before widening;
//     the accumulator rows are put back in order when the warps' states are merged.
// P^T reaches the B operand by transposing the two 8 x 8 halves of its accumulator layout
// across the warp (movmatrix).  k_scale is folded into the score scale and v_scale into the
// final normalisation.  P enters the PV product as one f16 fragment (11 significant bits)
// instead of the bf16 hi/lo pair.
#include <algorithm>

#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kBlk = 16;  // positions per pool block on this path

template <int D, bool FP8>
struct Geom {
  static_assert(!FP8 || D == 128, "fp8 tiles are one 128-byte-wide box");
  static constexpr int kHalves = FP8 ? 1 : D / 64;         // TMA boxes per tile
  static constexpr int kHalfBytes = kBlk * 128;            // 16 rows x 128 bytes
  static constexpr int kTileBytes = kHalves * kHalfBytes;  // one K (or V) block tile
  static constexpr int kStageBytes = 2 * kTileBytes;       // K + V
  static constexpr int kNT = D / 8;                        // n-tiles of the output
  static constexpr int kKS = D / 16;                       // k-steps of QK^T
};

template <int D, int NW, int NS, bool FP8>
constexpr size_t smem_bytes() {
  // ring | full barriers, one that no copy signals | merge m, l | fail flag, work unit | the
  // per-block K and V factors of each ring stage ; the O merge area aliases the ring
  return 1024 + (size_t)NW * NS * Geom<D, FP8>::kStageBytes + (NW * NS + 1) * 8 +
         NW * 16 * 4 * 2 + 16 + (size_t)NW * NS * 8;
}

// 4 bytes global -> shared without registers; the mbarrier's pending arrival count (set for
// it at initialisation) drops once every earlier cp.async of this thread has landed
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_arrive(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// bf16x2 -> f16x2 (exact inside f16's normal range)
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t w) {
  const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  return pack_f16x2(f.x, f.y);
}

// Transpose of an 8 x 8 matrix of 16-bit elements held in the accumulator layout (lane l:
// row l / 4, columns 2 (l % 4) and 2 (l % 4) + 1), returned in the same layout.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t r;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
  return r;
}

template <int N>
struct IntTag {
  static constexpr int value = N;
};

// Byte offset of 16-byte chunk `chunk` (along D) of row `row` inside a tile written by TMA
// with the 128-byte swizzle: halves of 64 dims are separate 2 KB boxes; inside a half the
// chunk index is XORed with row mod 8.
__device__ __forceinline__ uint32_t tile_off(int row, int chunk) {
  const int half = chunk >> 3, c = chunk & 7;
  return (uint32_t)(half * (kBlk * 128) + row * 128 + ((c ^ (row & 7)) << 4));
}

// PB (e4m3 pools only): one K and one V factor per (pool block, kv head), p.m.k_bscales /
// v_bscales [num_blocks, num_kv_heads].  The K factor multiplies the block's scores with the
// softmax scale.  The V factor, over the largest one the warp has met so far (its reference;
// O is rescaled when it rises) and times 2^15, multiplies the block's fp32 weights where they
// are rounded to f16 for P V, and the reference over 2^15 multiplies the warp's O where the
// warps are merged: the f16 weights stay in [0, 2^15] whatever the factors' magnitude (the
// row sum keeps the unscaled weights).  Lane 0 copies both factors into the stage's slot
// with cp.async when it issues the block's TMA copies, and the stage's barrier (two
// arrivals) completes only when they have landed too.
template <int D, int NW, int NS, bool SPLIT, bool FP8, bool PB = false>
__global__ void __launch_bounds__(NW * 32, 2)
    k_mma16(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
            const Mma16Params p) {
  static_assert(!PB || FP8, "per-block factors are for e4m3 pools");
  using G_ = Geom<D, FP8>;
  // query rows per tile: e4m3 varlen tiles are one group of 8 (one N of the swapped MMAs)
  constexpr int TR = (FP8 && !SPLIT) ? 8 : 16;
  extern __shared__ uint8_t smem_raw[];

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + (size_t)NW * NS * G_::kStageBytes);
  uint64_t* never = full + NW * NS;  // no copy ever signals it (the debug_stall test hook)
  float* mrg_m = reinterpret_cast<float*>(full + NW * NS + 1);
  float* mrg_l = mrg_m + NW * 16;
  int* fail = reinterpret_cast<int*>(mrg_l + NW * 16);
  float2* s_bs = reinterpret_cast<float2*>(fail + 2);  // [NW * NS] (K, V) factors (PB)
  float* mrg_o = reinterpret_cast<float*>(ring);  // [NW][16][D + 4], used after the ring drains
  constexpr int kOStride = D + 4;

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x <= NW * NS) mbar_init(&full[threadIdx.x], PB ? 2 : 1);  // the ring's, `never`
  if (threadIdx.x == 0) {
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
  }
  fence_mbar_init();
  // varlen launches overlap the kernels before them (programmatic dependent launch): the
  // plan, the status word and the inputs are read only after those have finished.  Behind
  // the tcgen05 kernel this kernel cannot start before every CTA of that kernel has passed
  // its own wait for the plan, so the plan (and all work before it) is complete already and
  // the decode tiles run alongside the prefill items; the wait for the tcgen05 kernel itself
  // comes before the recomputed items and before this kernel ends, so that whatever follows
  // on the stream finds both kernels finished.
  const bool after_tc = !SPLIT && p.after_tc != 0;
  if (!after_tc) pdl_wait();
  // failed validation or an earlier sticky error: the whole CTA writes nothing
  if (threadIdx.x == 0) *fail = status_set(p.status) ? 1 : 0;
  __syncthreads();
  if constexpr (!SPLIT) pdl_launch_dependents();  // the next kernel's prologue may start
  if (*reinterpret_cast<volatile int*>(fail)) {
    if (after_tc) pdl_wait();
    return;
  }

  const VarlenMeta& m = p.m;
  const int G = m.group;
  const int H = m.num_heads;
  uint32_t ring_pos = 0;  // blocks this warp has pushed through its ring so far

  // Split-KV: grid (partition x sequence, kv head), strided.  Varlen: a persistent 1-D grid
  // whose CTAs take (item, kv head) units from the plan's work counter, longest items first;
  // then (behind the tcgen05 kernel) the tiles of the 256-row items that kernel marked
  // (V outside f16's range), from a second counter.
  int n_units;
  int* unit_slot = fail + 1;
  int phase = 0;
  if constexpr (SPLIT) {
    n_units = m.num_seqs * p.max_parts;
  } else {
    n_units = p.plan[0] * m.num_kv_heads;
  }

  for (int it_no = 0;; ++it_no) {
    int item, kvh;
    if constexpr (SPLIT) {
      item = blockIdx.x + it_no * gridDim.x;
      if (item >= n_units) break;
      kvh = blockIdx.y;
    } else {
      if (threadIdx.x == 0) {
        const int u = atomicAdd(const_cast<int32_t*>(p.plan) + (phase ? 4 : 2), 1);
        *unit_slot = u < n_units ? u : -1;
      }
      __syncthreads();
      const int unit = *reinterpret_cast<volatile int*>(unit_slot);
      if (unit < 0) {
        if (phase == 1 || !after_tc) break;
        __syncthreads();  // every thread has read the slot before it is written again
        pdl_wait();       // the tcgen05 kernel has finished: its marks are final
        phase = 1;
        n_units = *reinterpret_cast<const volatile int32_t*>(p.plan + 3) * (256 / TR) * m.num_kv_heads;
        continue;
      }
      item = unit / m.num_kv_heads;
      kvh = unit % m.num_kv_heads;
    }
    // ---------------------------------------------------------------- item geometry
    int s, row0, rows_total, part = 0, qs, n;
    int lo = INT_MAX, hi = 0;  // the union of the tile's rows' visible key ranges
    bool have_range = false;   // the plan's tile record carries it
    if constexpr (SPLIT) {
      s = item / p.max_parts;
      part = item % p.max_parts;
      qs = s;
      row0 = 0;
      rows_total = G;
      n = m.seq_lens[s];
    } else if (phase == 0) {
      // the plan's record: (sequence, tile, query start, seq_len), (key range, rows): the
      // first copies can be issued without waiting for the positions
      const int4* rec = reinterpret_cast<const int4*>(p.plan + p.items_off) + 2 * item;
      const int4 r0 = rec[0], r1 = rec[1];
      s = r0.x;
      row0 = r0.y * TR;
      qs = r0.z;
      n = r0.w;
      lo = r1.x;
      hi = r1.y;
      rows_total = r1.z;
      have_range = true;
    } else {  // tile k of marked item j (item = j * 256 / TR + k): (sequence, tile index)
      const int4 t4 = reinterpret_cast<const int4*>(
          p.plan + p.tc_off)[p.plan[p.redo_list_off + item / (256 / TR)]];
      s = t4.x;
      row0 = (t4.y * (256 / TR) + item % (256 / TR)) * TR;
      qs = m.query_start_loc[s];
      rows_total = (m.query_start_loc[s + 1] - qs) * G;
      n = m.seq_lens[s];
    }
    // K = k_scales[kvh] * pool goes into the score scale (per kv head, when given)
    const float sl2 = head_scale(m.k_scales, kvh, p.scale_log2);

    // this lane's two rows: r0 = lane / 4 and r1 = r0 + 8 (their positions are loaded now and
    // used after the first copies are on their way)
    int st[2], en[2], tok[2], head[2], pos[2];
    bool valid[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int R = row0 + (lane >> 2) + 8 * i;
      valid[i] = (i == 0 || TR == 16) && R < rows_total;
      const int tl = valid[i] ? R / G : 0;
      tok[i] = qs + tl;
      head[i] = kvh * G + (valid[i] ? R % G : 0);
      pos[i] = (!SPLIT && valid[i]) ? m.positions[tok[i]] : 0;
    }
    auto row_ranges = [&]() {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        int e, b;
        if constexpr (SPLIT) {
          e = n;  // the decode query sits at n - 1: causal by construction
          b = m.window > 0 ? max(0, e - m.window) : 0;
          b = max(b, part * p.partition_size);
          e = min(e, (part + 1) * p.partition_size);
        } else {
          e = m.causal ? pos[i] + 1 : n;
          b = m.window > 0 ? max(0, e - m.window) : 0;
        }
        st[i] = valid[i] ? b : 0;
        en[i] = valid[i] ? max(e, b) : 0;
      }
    };
    if (!have_range) {
      row_ranges();
#pragma unroll
      for (int i = 0; i < 2; ++i)
        if (valid[i] && en[i] > st[i]) {
          lo = min(lo, st[i]);
          hi = max(hi, en[i]);
        }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        lo = min(lo, __shfl_xor_sync(kFull, lo, o));
        hi = max(hi, __shfl_xor_sync(kFull, hi, o));
      }
    }
    const int blk_lo = lo < hi ? lo / kBlk : 0;
    const int nblk = lo < hi ? (hi + kBlk - 1) / kBlk - blk_lo : 0;
    // warp w takes the blocks whose absolute index is w mod NW, so a row's arithmetic (which
    // blocks each warp folds, in which order, and the fixed-order merge of the warps) does
    // not depend on the other rows of its tile: a token gets the same bits as a decode token,
    // inside a prefill chunk, alone or in any batch.  Blocks a row cannot see add exact zeros.
    const int first = ((warp - blk_lo) % NW + NW) % NW;  // this warp's first block, relative
    const int my_count = nblk > first ? (nblk - first + NW - 1) / NW : 0;
    const int32_t* table_row = m.block_tables + (int64_t)s * m.max_blocks;

    // ---------------------------------------------------------------- streaming
    // bf16: this lane's rows g and g + 8 in [0], [1].  fp8: rows 8j + 2c + e in [2j + e].
    float mrow[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    float lrow[4] = {0.f, 0.f, 0.f, 0.f};
    // PB: the largest V factor of the blocks this warp has folded (0 until the first), and
    // its reciprocal: the warp's O is kept in units of vref / 2^15, so the f16 weights, at
    // most 2^15, keep 2^29 of range below their largest value before they turn subnormal
    float vref = 0.f, vinv = 0.f;
    float o[G_::kNT][4];
#pragma unroll
    for (int j = 0; j < G_::kNT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;

    int tbl_win = -1, tbl_val = 0;
    auto block_id = [&](int x) -> int {  // whole warp; x = this warp's block index
      const int win = x >> 5;
      if (win != tbl_win) {
        tbl_win = win;
        const int lb = first + (win * 32 + lane) * NW;
        tbl_val = lb < nblk ? table_row[blk_lo + lb] : 0;
      }
      return __shfl_sync(kFull, tbl_val, x & 31);
    };
    auto issue = [&](int x) {  // whole warp
      const int id = block_id(x);
      if (lane == 0) {
        const uint32_t slot = (ring_pos + x) % NS;
        uint64_t* bar = &full[warp * NS + slot];
        uint8_t* dst = ring + (size_t)(warp * NS + slot) * G_::kStageBytes;
        if constexpr (PB) {
          const int64_t f = (int64_t)id * m.num_kv_heads + kvh;
          cp_async4(&s_bs[warp * NS + slot].x, p.m.k_bscales + f);
          cp_async4(&s_bs[warp * NS + slot].y, p.m.v_bscales + f);
          cp_async_arrive(bar);
        }
        mbar_arrive_expect_tx(bar, G_::kStageBytes);
#pragma unroll
        for (int h = 0; h < G_::kHalves; ++h) {  // fp8: one 128-byte box per tile, x = 0
          tma_load_3d(dst + h * G_::kHalfBytes, &tk, h * 64, kvh, id * kBlk, bar);
          tma_load_3d(dst + G_::kTileBytes + h * G_::kHalfBytes, &tv, h * 64, kvh, id * kBlk, bar);
        }
      }
    };

    const int pro = my_count < NS ? my_count : NS;
    for (int x = 0; x < pro; ++x) issue(x);
    int issued = pro;
    bool timed_out = false;
    if (have_range) row_ranges();

    // ---------------------------------------------------------------- q fragments
    uint32_t qa[G_::kKS][4];
    {
      const uint32_t* q0 =
          reinterpret_cast<const uint32_t*>(p.q + ((int64_t)tok[0] * H + head[0]) * D);
      const uint32_t* q1 =
          reinterpret_cast<const uint32_t*>(p.q + ((int64_t)tok[1] * H + head[1]) * D);
      const int c = (lane & 3);
#pragma unroll
      for (int kk = 0; kk < G_::kKS; ++kk) {
        if constexpr (FP8) {  // f16, dimensions in the permuted order (header comment)
          const int w = 16 * c + 2 * kk;
          qa[kk][0] = valid[0] ? bf2_to_h2(q0[w]) : 0u;
          qa[kk][1] = valid[1] ? bf2_to_h2(q1[w]) : 0u;
          qa[kk][2] = valid[0] ? bf2_to_h2(q0[w + 1]) : 0u;
          qa[kk][3] = valid[1] ? bf2_to_h2(q1[w + 1]) : 0u;
          continue;
        }
        qa[kk][0] = valid[0] ? q0[kk * 8 + c] : 0u;
        qa[kk][1] = valid[1] ? q1[kk * 8 + c] : 0u;
        qa[kk][2] = valid[0] ? q0[kk * 8 + 4 + c] : 0u;
        qa[kk][3] = valid[1] ? q1[kk * 8 + 4 + c] : 0u;
      }
    }

    // fp8: the tile's query rows are the MMA's N, in groups of 8, and the block's 16 keys its
    // M.  A lane holds columns 2c, 2c + 1 of each group: their visible ranges come from the
    // lanes that loaded those rows above (row 8j + r sits in lane 4r, index j).
    const int nr = TR == 8 || rows_total - row0 <= 8 ? 1 : 2;  // row groups of this tile
    int cst[2][2], cen[2][2];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        cst[j][e] = __shfl_sync(kFull, st[j], (2 * (lane & 3) + e) * 4);
        cen[j][e] = __shfl_sync(kFull, en[j], (2 * (lane & 3) + e) * 4);
      }
    // keys every valid row of the tile sees: blocks inside that range need no mask
    int all_lo = 0, all_hi = INT_MAX;
#pragma unroll
    for (int i = 0; i < 2; ++i)
      if (valid[i]) {
        all_lo = max(all_lo, st[i]);
        all_hi = min(all_hi, en[i]);
      }
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      all_lo = max(all_lo, __shfl_xor_sync(kFull, all_lo, o));
      all_hi = min(all_hi, __shfl_xor_sync(kFull, all_hi, o));
    }
    auto fp8_step = [&](auto groups, const uint8_t* kt, const uint8_t* vt, int key_base,
                        float2 fac) {
      constexpr int NR = decltype(groups)::value;
      float sk = sl2;  // the block's score scale
      [[maybe_unused]] float fv = 1.f;  // PB: the weights' V factor, in vref / 2^15 units
      [[maybe_unused]] float beta = 1.f;  // PB: O's rescale when vref rises
      if constexpr (PB) {
        sk = sl2 * fac.x;
        if (fac.y > vref) {  // (the factors are the warp's own: uniform across it)
          beta = vref * __frcp_rn(fac.y);
          vref = fac.y;
          vinv = __frcp_rn(fac.y);  // finite: the factors are normal floats
        }
        fv = fac.y * vinv * 32768.f;
      }
      const int c = lane & 3, g = lane >> 2;
      // S^T = K Q^T: A = key rows g and g + 8, bytes [32c, 32c + 32) (chunks 2c, 2c + 1); B =
      // the q fragments of group j, qa[kk][j] and qa[kk][j + 2]
      const uint32_t kbase = smem_u32(kt);
      uint4 kw[2][2];
#pragma unroll
      for (int mt = 0; mt < 2; ++mt) {
        const int key = g + mt * 8;
        kw[mt][0] = lds128(kbase + key * 128 + (((2 * c) ^ (key & 7)) << 4));
        kw[mt][1] = lds128(kbase + key * 128 + (((2 * c + 1) ^ (key & 7)) << 4));
      }
      // two accumulators per group (even / odd k-steps)
      float sc[NR][4], sc2[NR][4];
#pragma unroll
      for (int j = 0; j < NR; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) sc[j][i] = sc2[j][i] = 0.f;
#pragma unroll
      for (int kk = 0; kk < G_::kKS; ++kk) {
        const uint4& k0 = kw[0][kk >> 2];
        const uint4& k1 = kw[1][kk >> 2];
        const int wsel = kk & 3;
        const uint32_t w0 = wsel == 0 ? k0.x : wsel == 1 ? k0.y : wsel == 2 ? k0.z : k0.w;
        const uint32_t w1 = wsel == 0 ? k1.x : wsel == 1 ? k1.y : wsel == 2 ? k1.z : k1.w;
        uint32_t a[4];  // (key g, dims 32c + 4kk + {0, 1}), (key g + 8, same), then dims + 2
        e4m3x4_to_f16(w0, a[0], a[2]);
        e4m3x4_to_f16(w1, a[1], a[3]);
#pragma unroll
        for (int j = 0; j < NR; ++j) mma_f16_16816((kk & 1) ? sc2[j] : sc[j], a, qa[kk][j], qa[kk][j + 2]);
      }
      // sc[j][i]: key g + 8 (i >> 1), row 8j + 2c + (i & 1); mask and scale to log2 units
      float alpha[NR][2];
      bool grew = false;  // a row's running max rose: its O needs the rescale (else alpha = 1)
#pragma unroll
      for (int j = 0; j < NR; ++j) {
        if (key_base >= all_lo && key_base + kBlk <= all_hi) {  // padding rows: unused values
#pragma unroll
          for (int i = 0; i < 4; ++i) sc[j][i] = (sc[j][i] + sc2[j][i]) * sk;
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int key = key_base + g + 8 * (i >> 1);
            const int e = i & 1;
            const bool vis = key >= cst[j][e] && key < cen[j][e];
            sc[j][i] = vis ? (sc[j][i] + sc2[j][i]) * sk : -INFINITY;
          }
        }
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          // the column's max over 16 keys: the lane's two, then the eight lanes of the column
          float mx = fmaxf(sc[j][e], sc[j][2 + e]);
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 16));
          const float mo = mrow[2 * j + e];
          const float mn = fmaxf(mo, mx);
          const float base = mn == -INFINITY ? 0.f : mn;
          alpha[j][e] = exp2f(mo - base);
          grew |= mn > mo;
          mrow[2 * j + e] = mn;
          sc[j][e] = exp2f(sc[j][e] - base);
          sc[j][2 + e] = exp2f(sc[j][2 + e] - base);
          // l per lane over its two keys of each block; the column's lanes are summed at the end
          lrow[2 * j + e] = lrow[2 * j + e] * alpha[j][e] + (sc[j][e] + sc[j][2 + e]);
        }
      }
      if constexpr (PB) {
        if (beta != 1.f) {  // O only: the row sums keep the unscaled weights
#pragma unroll
          for (int j = 0; j < NR; ++j) {
            alpha[j][0] *= beta;
            alpha[j][1] *= beta;
          }
          grew = true;
        }
      }
      if (__any_sync(kFull, grew)) {  // skipped, the factors are exactly 1
#pragma unroll
        for (int j = 0; j < NR; ++j)
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            o[8 * j + t][0] *= alpha[j][0];
            o[8 * j + t][1] *= alpha[j][1];
            o[8 * j + t][2] *= alpha[j][0];
            o[8 * j + t][3] *= alpha[j][1];
          }
      }
      // P^T as the B operand (k = keys, n = rows): each 8-key half of the f16 accumulator
      // layout, transposed across the warp, is the fragment of that half
      uint32_t pb[NR][2];
#pragma unroll
      for (int j = 0; j < NR; ++j) {
        auto vw = [&](float x) {  // the block's V factor on the weight (PB)
          if constexpr (PB) return x * fv;
          else return x;
        };
        pb[j][0] = movmatrix_trans(pack_f16x2(vw(sc[j][0]), vw(sc[j][1])));
        pb[j][1] = movmatrix_trans(pack_f16x2(vw(sc[j][2]), vw(sc[j][3])));
      }
      // O^T += V^T P^T.  A = V^T: M-tile t = 2i + h, row g is dimension 16g + 4i + 2h and row
      // g + 8 dimension 16g + 4i + 2h + 1; its k columns are keys 2c, 2c + 1, 2c + 8, 2c + 9,
      // so the lane reads bytes [16g, 16g + 16) of those four key rows
      const uint32_t vbase = smem_u32(vt);
      const int lim = n - key_base;  // rows at or past it were never written: zeros
      uint4 vr[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = 2 * c + (i & 1) + (i >> 1) * 8;
        vr[i] = lds128(vbase + r * 128 + ((g ^ (r & 7)) << 4));
        if (r >= lim) vr[i] = make_uint4(0u, 0u, 0u, 0u);
      }
      const uint32_t ra[4] = {vr[0].x, vr[0].y, vr[0].z, vr[0].w};
      const uint32_t rb[4] = {vr[1].x, vr[1].y, vr[1].z, vr[1].w};
      const uint32_t rc[4] = {vr[2].x, vr[2].y, vr[2].z, vr[2].w};
      const uint32_t rd[4] = {vr[3].x, vr[3].y, vr[3].z, vr[3].w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        // byte j of word i is dimension 16g + 4i + j: pair keys (2c, 2c + 1) and (2c + 8,
        // 2c + 9) byte by byte, lower key in the lower byte
        const uint32_t lo01 = __byte_perm(ra[i], rb[i], 0x5140);
        const uint32_t hi01 = __byte_perm(ra[i], rb[i], 0x7362);
        const uint32_t lo89 = __byte_perm(rc[i], rd[i], 0x5140);
        const uint32_t hi89 = __byte_perm(rc[i], rd[i], 0x7362);
        const uint32_t a0[4] = {e4m3x2_to_f16x2((uint16_t)(lo01 & 0xffffu)),
                                e4m3x2_to_f16x2((uint16_t)(lo01 >> 16)),
                                e4m3x2_to_f16x2((uint16_t)(lo89 & 0xffffu)),
                                e4m3x2_to_f16x2((uint16_t)(lo89 >> 16))};
        const uint32_t a1[4] = {e4m3x2_to_f16x2((uint16_t)(hi01 & 0xffffu)),
                                e4m3x2_to_f16x2((uint16_t)(hi01 >> 16)),
                                e4m3x2_to_f16x2((uint16_t)(hi89 & 0xffffu)),
                                e4m3x2_to_f16x2((uint16_t)(hi89 >> 16))};
#pragma unroll
        for (int j = 0; j < NR; ++j) {
          mma_f16_16816(o[8 * j + 2 * i], a0, pb[j][0], pb[j][1]);
          mma_f16_16816(o[8 * j + 2 * i + 1], a1, pb[j][0], pb[j][1]);
        }
      }
    };

    for (int x = 0; x < my_count; ++x) {
      const uint32_t cnt = ring_pos + x;
      const uint32_t slot = cnt % NS;
      // debug_stall: the wait names a barrier nothing signals, so it runs out after
      // wait_limit_ns and the kernel unwinds as from a copy that never landed
      uint64_t* const wb = p.debug_stall ? never : &full[warp * NS + slot];
      if (!mbar_wait(wb, p.debug_stall ? 0u : (cnt / NS) & 1u, p.wait_limit_ns)) {
        timed_out = true;
        break;
      }
      uint8_t* kt = ring + (size_t)(warp * NS + slot) * G_::kStageBytes;
      uint8_t* vt = kt + G_::kTileBytes;
      float2 fac = make_float2(1.f, 1.f);
      if constexpr (PB) fac = s_bs[warp * NS + slot];
      const int lb = blk_lo + first + x * NW;
      const int key_base = lb * kBlk;

      if constexpr (FP8 && TR == 8) {
        fp8_step(IntTag<1>{}, kt, vt, key_base, fac);
      } else if constexpr (FP8) {
        if (nr == 1)
          fp8_step(IntTag<1>{}, kt, vt, key_base, fac);
        else
          fp8_step(IntTag<2>{}, kt, vt, key_base, fac);
      } else {
        // rows of the sequence's last block past seq_len were never written: zero their V so
        // that 0-weight * garbage cannot turn into NaN
        if (key_base + kBlk > n) {
          const int first = n - key_base;  // 1..15
          for (int i = lane; i < (kBlk - first) * G_::kHalves * 8; i += 32) {
            const int r = first + i / (G_::kHalves * 8);
            const int rest = i % (G_::kHalves * 8);
            *reinterpret_cast<uint4*>(vt + (rest >> 3) * G_::kHalfBytes + r * 128 + (rest & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
          __syncwarp();
        }

        // S = Q K^T for 16 keys: two n-tiles of 8 keys
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
          const int mi = lane >> 3, rr = lane & 7;
          const int key = rr + ((mi >> 1) << 3);
          const uint32_t kbase = smem_u32(kt);
#pragma unroll
          for (int kk = 0; kk < G_::kKS; ++kk) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kbase + tile_off(key, kk * 2 + (mi & 1)), b0, b1, b2, b3);
            mma_bf16_16816(sc[0], qa[kk], b0, b1);
            mma_bf16_16816(sc[1], qa[kk], b2, b3);
          }
        }

        // mask, scale to log2 units, online softmax update
        const int kcol = key_base + (lane & 3) * 2;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const int key = kcol + nt * 8 + (c & 1);
            const int r = c >> 1;
            const bool vis = key >= st[r] && key < en[r];
            sc[nt][c] = vis ? sc[nt][c] * sl2 : -INFINITY;
          }
        float alpha[2];
        bool grew = false;  // a row's running max rose: its O needs the rescale (else alpha = 1)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          float mx = fmaxf(fmaxf(sc[0][2 * r], sc[0][2 * r + 1]), fmaxf(sc[1][2 * r], sc[1][2 * r + 1]));
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, 2));
          const float mn = fmaxf(mrow[r], mx);
          const float base = mn == -INFINITY ? 0.f : mn;
          alpha[r] = exp2f(mrow[r] - base);
          grew |= mn > mrow[r];
          mrow[r] = mn;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            sc[nt][2 * r] = exp2f(sc[nt][2 * r] - base);
            sc[nt][2 * r + 1] = exp2f(sc[nt][2 * r + 1] - base);
          }
        }
        // P as two bf16 A fragments, hi = bf16(p) and lo = bf16(p - hi): the PV product of
        // both keeps the weights to ~2^-17 relative, where bf16 P alone can be off by 2^-9 of
        // |v| when a row sees few keys.
        uint32_t ph[4], pl[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float a = sc[i >> 1][(i & 1) * 2], b = sc[i >> 1][(i & 1) * 2 + 1];
          ph[i] = pack_bf16x2(a, b);
          const float2 hv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ph[i]));
          pl[i] = pack_bf16x2(a - hv.x, b - hv.y);
        }
        lrow[0] = lrow[0] * alpha[0] + ((sc[0][0] + sc[0][1]) + (sc[1][0] + sc[1][1]));
        lrow[1] = lrow[1] * alpha[1] + ((sc[0][2] + sc[0][3]) + (sc[1][2] + sc[1][3]));
        if (__any_sync(kFull, grew)) {  // skipped, the factors are exactly 1
#pragma unroll
          for (int j = 0; j < G_::kNT; ++j) {
            o[j][0] *= alpha[0];
            o[j][1] *= alpha[0];
            o[j][2] *= alpha[1];
            o[j][3] *= alpha[1];
          }
        }
        // O += P V: V is the k-major B operand, read with transposing ldmatrix
        {
          const int mi = lane >> 3, rr = lane & 7;
          const int key = rr + ((mi & 1) << 3);
          const uint32_t vbase = smem_u32(vt);
#pragma unroll
          for (int dd = 0; dd < D / 16; ++dd) {
            uint32_t b0, b1, b2, b3;
            ldsm_x4_trans(vbase + tile_off(key, dd * 2 + (mi >> 1)), b0, b1, b2, b3);
            mma_bf16_16816(o[2 * dd], ph, b0, b1);
            mma_bf16_16816(o[2 * dd + 1], ph, b2, b3);
            mma_bf16_16816(o[2 * dd], pl, b0, b1);
            mma_bf16_16816(o[2 * dd + 1], pl, b2, b3);
          }
        }
      }
      __syncwarp();
      if (issued < my_count) {
        issue(issued);
        ++issued;
      }
    }

    if (timed_out) {
      if (lane == 0) {
        record_error(p.status, PA_ETIMEOUT);
        atomicExch(fail, 1);
      }
      // wait (bounded) for this warp's copies still in flight before the CTA leaves
      for (int x = 0; x < issued; ++x) {
        const uint32_t cnt = ring_pos + x;
        mbar_wait(&full[warp * NS + cnt % NS], (cnt / NS) & 1u, 100000000ull);
      }
    }
    ring_pos += issued;

    // ---------------------------------------------------------------- merge the warps
    if constexpr (FP8) {
#pragma unroll
      for (int r = 0; r < 4; ++r) {  // the column's eight lanes
        lrow[r] += __shfl_xor_sync(kFull, lrow[r], 4);
        lrow[r] += __shfl_xor_sync(kFull, lrow[r], 8);
        lrow[r] += __shfl_xor_sync(kFull, lrow[r], 16);
      }
    } else {
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        lrow[r] += __shfl_xor_sync(kFull, lrow[r], 1);
        lrow[r] += __shfl_xor_sync(kFull, lrow[r], 2);
      }
    }
    __syncthreads();  // every warp is done with its ring: the O area may alias it now
    if (*reinterpret_cast<volatile int*>(fail)) {
      if (after_tc) pdl_wait();
      return;
    }
    {
      float* ob = mrg_o + (size_t)warp * 16 * kOStride;
      if constexpr (FP8) {
        // group j, M-tile t = 2i + h: accumulator [e] is (dimension 16g + 4i + 2h, row
        // 8j + 2c + e), [2 + e] the next dimension
        const int c = lane & 3, g = lane >> 2;
        // PB: O back from units of vref / 2^15 (vref first: a tiny vref stays normal)
        auto u = [&](float x) { return PB ? x * vref * (1.f / 32768.f) : x; };
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          if (j >= nr) break;
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int row = 8 * j + 2 * c + e;
            if (g == 0) {
              mrg_m[warp * 16 + row] = mrow[2 * j + e];
              mrg_l[warp * 16 + row] = lrow[2 * j + e];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
              *reinterpret_cast<float4*>(ob + row * kOStride + 16 * g + 4 * i) =
                  make_float4(u(o[8 * j + 2 * i][e]), u(o[8 * j + 2 * i][2 + e]),
                              u(o[8 * j + 2 * i + 1][e]), u(o[8 * j + 2 * i + 1][2 + e]));
          }
        }
      } else {
        const int r0 = lane >> 2;
        if ((lane & 3) == 0) {
          mrg_m[warp * 16 + r0] = mrow[0];
          mrg_m[warp * 16 + r0 + 8] = mrow[1];
          mrg_l[warp * 16 + r0] = lrow[0];
          mrg_l[warp * 16 + r0 + 8] = lrow[1];
        }
#pragma unroll
        for (int j = 0; j < G_::kNT; ++j) {
          const int col = j * 8 + (lane & 3) * 2;
          *reinterpret_cast<float2*>(ob + r0 * kOStride + col) = make_float2(o[j][0], o[j][1]);
          *reinterpret_cast<float2*>(ob + (r0 + 8) * kOStride + col) =
              make_float2(o[j][2], o[j][3]);
        }
      }
    }
    __syncthreads();
    {
      constexpr int kSegs = NW * 32 / 16;  // threads per row
      constexpr int kSeg = D / kSegs;      // dims per thread
      static_assert(kSeg % 8 == 0, "epilogue writes 16-byte chunks");
      const int row = threadIdx.x / kSegs, seg = threadIdx.x % kSegs;
      const int R = row0 + row;
      if (row < TR && R < rows_total) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, mrg_m[w * 16 + row]);
        float wsc[NW];
        float L = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
          wsc[w] = M == -INFINITY ? 0.f : exp2f(mrg_m[w * 16 + row] - M);
          L += wsc[w] * mrg_l[w * 16 + row];
        }
        const int t = qs + R / G;
        const int h = kvh * G + R % G;
        if constexpr (!SPLIT) {
          // an attention sink (TensorSharp ForwardWithSinks) is one more state to merge: max
          // = the sink logit, exp-sum = 1, weighted sum = 0
          const float sk = p.m.sinks ? p.m.sinks[h] * kLog2e : -INFINITY;
          if (sk > -INFINITY) {
            const float M2 = fmaxf(M, sk);
            const float a = M == -INFINITY ? 0.f : exp2f(M - M2);
#pragma unroll
            for (int w = 0; w < NW; ++w) wsc[w] *= a;
            L = L * a + exp2f(sk - M2);
            M = M2;
          }
          if (p.m.lse && seg == 0)
            p.m.lse[(int64_t)h * p.m.num_tokens + t] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
        }
        const float inv = L > 0.f ? head_scale(p.m.v_scales, kvh, p.m.v_scale) / L : 0.f;
        float vals[kSeg];
#pragma unroll
        for (int d = 0; d < kSeg; ++d) {
          float acc = 0.f;
#pragma unroll
          for (int w = 0; w < NW; ++w)
            acc += wsc[w] * mrg_o[((size_t)w * 16 + row) * kOStride + seg * kSeg + d];
          vals[d] = acc * inv;
        }
        if constexpr (SPLIT) {
          const int64_t idx = ((int64_t)s * H + h) * p.max_parts + part;
          float* dst = p.tmp_out + idx * D + seg * kSeg;
#pragma unroll
          for (int d = 0; d < kSeg; d += 4)
            *reinterpret_cast<float4*>(dst + d) =
                make_float4(vals[d], vals[d + 1], vals[d + 2], vals[d + 3]);
          if (seg == 0) {
            p.max_logits[idx] = M == -INFINITY ? -INFINITY : M * kLn2;
            p.exp_sums[idx] = L;
          }
        } else {
          __nv_bfloat16* dst =
              reinterpret_cast<__nv_bfloat16*>(p.out) + ((int64_t)t * H + h) * D + seg * kSeg;
#pragma unroll
          for (int d = 0; d < kSeg; d += 8) {
            uint4 v;
            v.x = pack_bf16x2(vals[d], vals[d + 1]);
            v.y = pack_bf16x2(vals[d + 2], vals[d + 3]);
            v.z = pack_bf16x2(vals[d + 4], vals[d + 5]);
            v.w = pack_bf16x2(vals[d + 6], vals[d + 7]);
            *reinterpret_cast<uint4*>(dst + d) = v;
          }
        }
      }
    }
    __syncthreads();  // the merge area is the ring of the next item
  }
}

// Warps per CTA and ring stages per warp, two CTAs per SM in every case:
//   bf16: 4 warps x 3 stages of 8 KB (D = 128);
//   e4m3 split-KV partitions: 4 warps x 6 stages of 4 KB (the same bytes in flight);
//   e4m3 varlen: 8 warps x 3 stages of 4 KB (the same bytes again).  Its 8-row tiles keep a
//   thread within 128 registers, so 16 warps share an SM and each (sequence, kv head) is
//   served by twice the warps: this path is bound by each warp's chain of dependent
//   instructions (conversions, MMAs, the softmax), not by the bytes in flight.
template <int D, bool SPLIT, bool FP8>
struct Shape {
  static constexpr int NW = (FP8 && !SPLIT) ? 8 : 4;
  static constexpr int NS = FP8 ? (SPLIT ? 6 : 3) : 3;
};

template <int D, bool SPLIT, bool FP8 = false, bool PB = false>
cudaError_t launch(const CUtensorMap& tk, const CUtensorMap& tv, const Mma16Params& p, int grid_x,
                   cudaStream_t stream) {
  constexpr int NW = Shape<D, SPLIT, FP8>::NW, NS = Shape<D, SPLIT, FP8>::NS;
  auto kern = k_mma16<D, NW, NS, SPLIT, FP8, PB>;
  constexpr size_t smem = smem_bytes<D, NW, NS, FP8>();
  static_assert((size_t)NW * 16 * (D + 4) * 4 <= (size_t)NW * NS * Geom<D, FP8>::kStageBytes,
                "merge area must fit in the ring");
  static_assert(2 * (smem + 1024) <= 228 * 1024, "two CTAs per SM");
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_x, SPLIT ? p.m.num_kv_heads : 1);
  cfg.blockDim = dim3(NW * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = SPLIT ? 0 : 1;  // varlen: overlaps the plan (or prefill) kernel
  return cudaLaunchKernelEx(&cfg, kern, tk, tv, p);
}

}  // namespace

cudaError_t launch_mma16_varlen(const CUtensorMap& tk, const CUtensorMap& tv, const Mma16Params& p,
                                int head_dim, int items_cap, cudaStream_t stream) {
  // persistent: two resident CTAs per SM, never more than there can be units
  const int64_t units = (int64_t)items_cap * p.m.num_kv_heads;
  const int64_t resident = 2 * (int64_t)num_sms();
  const int grid_x = (int)std::max<int64_t>(1, std::min(units, resident));
  if (head_dim == 128) return launch<128, false>(tk, tv, p, grid_x, stream);
  if (head_dim == 64) return launch<64, false>(tk, tv, p, grid_x, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_mma16_varlen_fp8(const CUtensorMap& tk, const CUtensorMap& tv,
                                    const Mma16Params& p, int items_cap, cudaStream_t stream) {
  const int64_t units = (int64_t)items_cap * p.m.num_kv_heads;
  const int64_t resident = 2 * (int64_t)num_sms();
  const int grid_x = (int)std::max<int64_t>(1, std::min(units, resident));
  if (p.m.k_bscales) return launch<128, false, true, true>(tk, tv, p, grid_x, stream);
  return launch<128, false, true>(tk, tv, p, grid_x, stream);
}

cudaError_t launch_mma16_split_fp8(const CUtensorMap& tk, const CUtensorMap& tv,
                                   const Mma16Params& p, cudaStream_t stream) {
  const int64_t items = (int64_t)p.m.num_seqs * p.max_parts;
  const int grid_x = items > 65535 ? 65535 : (int)items;
  if (grid_x <= 0) return cudaSuccess;
  if (p.m.k_bscales) return launch<128, true, true, true>(tk, tv, p, grid_x, stream);
  return launch<128, true, true>(tk, tv, p, grid_x, stream);
}

cudaError_t launch_mma16_split(const CUtensorMap& tk, const CUtensorMap& tv, const Mma16Params& p,
                               int head_dim, cudaStream_t stream) {
  const int64_t items = (int64_t)p.m.num_seqs * p.max_parts;
  const int grid_x = items > 65535 ? 65535 : (int)items;
  if (grid_x <= 0) return cudaSuccess;
  if (head_dim == 128) return launch<128, true>(tk, tv, p, grid_x, stream);
  if (head_dim == 64) return launch<64, true>(tk, tv, p, grid_x, stream);
  return cudaErrorInvalidValue;
}

}  // namespace pa
