// k_prefill_tc.cu -- paged attention for prefill chunks on the 5th-generation tensor cores
// (tcgen05.mma, accumulators in tensor memory), sm_103a.
//
// Work item: (sequence, kv head, 128-row query tile).  The 128 rows are (token, head) pairs of
// one kv head's GQA group, token-major, so one K/V tile serves all G query heads.  Key tiles
// are 128 positions = 8 pool blocks, each block fetched by TMA from wherever the block table
// puts it (two 64-dim boxes of 16 rows per block, 128-byte swizzle); a block past the
// visible range is fetched at a negative row coordinate, which TMA fills with zeros.
//
// Work items are 256-row pairs of such tiles, run by a cluster of two CTAs on two SMs with the
// pair's 2-SM MMAs (tcgen05 cta_group::2, M = 256): CTA r holds query rows 128r .. 128r + 127,
// its own S, P and O in its tensor memory, and only its part of every K / V tile: keys
// 64r .. 64r + 63 of K (all 128 dims) and dims 64r .. 64r + 63 of V (all 128 keys), 16 KB each.
// The MMA splits A by rows and B by columns across the pair, so each SM's shared memory is
// filled with half of every K / V tile -- the fill rate of shared memory, not the tensor core,
// is what bounds this kernel.  CTA 0 (the leader) issues every MMA; its barriers also count
// the peer's arrivals (the peer's idle issuer warps forward "my part of this stage has landed"
// with remote mbarrier arrives), and the MMA completions are multicast to both CTAs.
//
// One CTA per SM, persistent over items, 16 warps; the producer / issuer and converter
// warpgroups give up registers to the two softmax warpgroups (setmaxnreg: 56, 200, 200, 56):
//   warp 0      TMA producer of Q (two buffers, so the next item's Q loads while this one
//               finishes) and of this CTA's part of K_j through a 3-stage ring; warp 2
//               produces its part of V_j through a 6-stage ring;
//   warp 1      TMEM owner and QK^T issuer; warp 3 issues PV.  In the leader lane 0 issues,
//               in warp-uniform code:
//                 S_j = Q K_j^T      (M 256, N 128, K 128: 8 MMAs, bf16, K-major operands)
//                 O  += P_j V_j      (f16 P read from TMEM, f16 V: 8 MMAs, V MN-major)
//               In the peer warp 1 forwards the Q / K arrivals to the leader.
//               TMEM columns: three S buffers at 0 / 128 / 384, O at 256.  P_j is written over
//               the S_j it came from, so S_{j+3} may only be issued once P_j V_j is done;
//   warps 4..11 softmax: two threads per query row (TMEM lane = row), one per 64-column
//               half; mask, row max (combined through shared memory), exp2, row sum, P to
//               tensor memory as f16, lazy O rescale, and the epilogue o = O * (1 / l) -> bf16.
//               A softmax thread waits for the previous P V only when it must rescale O,
//               so the exponentials of tile j run while the tensor core works on tile j - 1;
//   warps 12..15 V converters, one per SM sub-partition: each widens a quarter of every V
//               stage of its CTA (32 keys x 64 dims) from bf16 to f16 in place, zeroes the
//               never-written rows past the sequence's end, and arrives on the leader's
//               V-ready barrier, which the PV issuer waits for.
// P enters the PV product as one f16 value (11 significant bits; the row sum l adds the fp32
// weights), with V widened exactly to f16: a bf16 value converts without error when its
// magnitude is below 65520 (below 2^-14 it becomes an f16 subnormal, off by at most 2^-25).
// A stage holding a larger magnitude (or an inf / NaN) marks its 256-row item; the warp-MMA
// kernel that runs after this one recomputes every marked item from the bf16 pool (bf16 hi /
// lo weights), overwriting what this kernel wrote for it.
// The online softmax follows the per-tile update of the tinyllm decode page (section 2.2)
// with one change that leaves the result unchanged: the reference max m is only moved (and
// O, l rescaled by 2^(m_old - m_new)) when a tile's max exceeds it by more than 8 (log2
// units), so the weights stay <= 2^8 and most tiles need no O rescale.
//
// Every mbarrier wait is bounded; a wait that runs out records PA_ETIMEOUT, raises an abort
// flag that makes the other roles unwind, and the CTA still frees its tensor memory.  Before
// a CTA leaves, its producers wait (bounded) for the TMA copies they issued last, the MMA
// issuers for their last MMAs, and the pair meets at a cluster barrier, so no asynchronous
// write lands in the shared memory or tensor memory of a CTA that has gone.
#include "pa_internal.cuh"

namespace pa {
namespace {

constexpr unsigned kFull = 0xffffffffu;
constexpr int kBM = 128;          // query rows per tile
constexpr int kBN = 128;          // keys per tile (8 blocks of 16)
constexpr int kD = 128;           // head size on this path
constexpr int kHalf = 16384;      // one 64-dim half of a 128-row bf16 Q tile
constexpr int kTile = 2 * kHalf;  // 128 x 128 bf16 (this CTA's Q rows)
constexpr int kKVHalf = 8192;     // K part: one 64-dim half of this CTA's 64 keys
constexpr int kPart = 16384;      // this CTA's part of a K (or V) tile
constexpr int kSBufs = 3;    // S / P buffers in tensor memory (columns 0, 128 and 384)
constexpr int kStagesK = 3;  // K ring (a K tile is released as soon as its S MMAs finish)
constexpr int kStagesV = 6;  // V ring (held until P V, so it needs more stages in flight)
constexpr int kOffQ = 0;                          // two Q buffers (consecutive items)
constexpr int kOffK = kOffQ + 2 * kTile;
constexpr int kOffV = kOffK + kStagesK * kPart;
constexpr int kOffBar = kOffV + kStagesV * kPart;
constexpr int kNumBarsMax = 48;
constexpr int kOffTmem = kOffBar + kNumBarsMax * 8;
constexpr int kOffFlag = kOffTmem + 16;
// softmax pair exchange: [half][row] fp32 row max (or row sum), then [half][row] int failed-
// wait flags of the item's end (a tile's failure travels in the row max slot as kBadMax)
constexpr int kOffXchg = kOffFlag + 16;
constexpr int kSmemBytes = kOffXchg + 2 * 2 * 128 * 4 + 1024;  // + slack to align the base
constexpr uint32_t kBadMax = 0x7fc0dea1u;  // a NaN that no arithmetic produces (canonical 7fffffff)
static_assert(kSmemBytes <= 232448, "shared memory of one CTA");
constexpr int kSoftWarps = 8;   // two column halves x four lane quarters
constexpr int kConvWarps = 4;   // V converters, a quarter of each V stage each
constexpr int kThreads = 128 + kSoftWarps * 32 + kConvWarps * 32;
constexpr int kFirstConvWarp = 4 + kSoftWarps;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;    // O: columns 256..383
__device__ __forceinline__ uint32_t col_s(uint32_t b) { return b == 2 ? 384u : b * 128u; }
// Inside an S buffer, P_j of key half h (keys 64h .. 64h+63) is stored by the thread that read
// those scores, at columns 64h .. 64h+31 (two f16 per column); the MMA of key step k (keys
// 16k .. 16k+15) reads 8 columns from col_p(k).
__device__ __forceinline__ uint32_t col_p(int kstep) {
  return (uint32_t)((kstep >> 2) * 64 + (kstep & 3) * 8);
}

// barrier indices (the per-stage / per-buffer ones are consecutive)
enum : int {
  B_QFULL = 0,
  B_QEMPTY = B_QFULL + 2,
  B_KFULL = B_QEMPTY + 2,
  B_KEMPTY = B_KFULL + kStagesK,
  B_VFULL = B_KEMPTY + kStagesK,
  B_VEMPTY = B_VFULL + kStagesV,
  B_VCONV = B_VEMPTY + kStagesV,  // leader: the stage's V is f16 in both CTAs
  B_QCONV = B_VCONV + kStagesV,   // leader, fp8 pools: the Q buffer is f16 in both CTAs
  B_KCONV = B_QCONV + 2,          // leader, fp8 pools: the stage's K is f16 in both CTAs
  B_SFULL = B_KCONV + kStagesK,
  B_PFULL = B_SFULL + kSBufs,
  B_PVDONE = B_PFULL + kSBufs,
  B_OFREE = B_PVDONE + kSBufs,
  B_FIN = B_OFREE + 1,
  B_NEVER = B_FIN + 1,  // nothing arrives on it (the debug_stall test hook)
  kNumBars = B_NEVER + 1
};
static_assert(kNumBars <= kNumBarsMax, "barrier area");

// ---- tcgen05 / TMEM wrappers -----------------------------------------------------------------

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// The MMA issuers run as whole warps in uniform control flow (so the compiler keeps the
// descriptors in uniform registers; a lone thread in a divergent branch issues at about half
// the tensor core's rate), and only lane 0 executes the tcgen05 instructions: the wrappers
// below are predicated on %laneid inside the asm.  Every MMA and commit of a role therefore
// comes from the same thread, as tcgen05.commit requires.  All tcgen05 operations of this
// kernel are cta_group::2 (the pair): one MMA computes 256 rows, 128 in each CTA's tensor
// memory, with A taken from each CTA's own rows and B split by columns between the two CTAs'
// shared memory at the same offset.
__device__ __forceinline__ void tc_mma_l0(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .u32 l;\n\t.reg .pred e, p;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Same with the A operand in tensor memory (row r in lane r, two bf16 per 32-bit column).
__device__ __forceinline__ void tc_mma_ta_l0(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .u32 l;\n\t.reg .pred e, p;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr));
}
// Wait for this thread's outstanding TMEM loads; the register operands tie the loaded values
// to the wait so no use of them can be scheduled before it.
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]),
        "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]),
        "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]),
        "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]),
        "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]), "+r"(v[30]), "+r"(v[31])
      :
      : "memory");
}
// 64 consecutive fp32 columns of this thread's TMEM lane in one instruction (1.6% faster per
// prefill call than two 32-column loads for the softmax's half row of S).
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&v)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, "
      "%48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, [%64];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]),
        "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]),
        "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]),
        "=r"(v[32]), "=r"(v[33]), "=r"(v[34]), "=r"(v[35]), "=r"(v[36]), "=r"(v[37]),
        "=r"(v[38]), "=r"(v[39]), "=r"(v[40]), "=r"(v[41]), "=r"(v[42]), "=r"(v[43]),
        "=r"(v[44]), "=r"(v[45]), "=r"(v[46]), "=r"(v[47]), "=r"(v[48]), "=r"(v[49]),
        "=r"(v[50]), "=r"(v[51]), "=r"(v[52]), "=r"(v[53]), "=r"(v[54]), "=r"(v[55]),
        "=r"(v[56]), "=r"(v[57]), "=r"(v[58]), "=r"(v[59]), "=r"(v[60]), "=r"(v[61]),
        "=r"(v[62]), "=r"(v[63])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld64(uint32_t (&v)[64]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(v[0]), "+r"(v[1]), "+r"(v[2]), "+r"(v[3]), "+r"(v[4]), "+r"(v[5]), "+r"(v[6]),
        "+r"(v[7]), "+r"(v[8]), "+r"(v[9]), "+r"(v[10]), "+r"(v[11]), "+r"(v[12]), "+r"(v[13]),
        "+r"(v[14]), "+r"(v[15]), "+r"(v[16]), "+r"(v[17]), "+r"(v[18]), "+r"(v[19]),
        "+r"(v[20]), "+r"(v[21]), "+r"(v[22]), "+r"(v[23]), "+r"(v[24]), "+r"(v[25]),
        "+r"(v[26]), "+r"(v[27]), "+r"(v[28]), "+r"(v[29]), "+r"(v[30]), "+r"(v[31]),
        "+r"(v[32]), "+r"(v[33]), "+r"(v[34]), "+r"(v[35]), "+r"(v[36]), "+r"(v[37]),
        "+r"(v[38]), "+r"(v[39]), "+r"(v[40]), "+r"(v[41]), "+r"(v[42]), "+r"(v[43]),
        "+r"(v[44]), "+r"(v[45]), "+r"(v[46]), "+r"(v[47]), "+r"(v[48]), "+r"(v[49]),
        "+r"(v[50]), "+r"(v[51]), "+r"(v[52]), "+r"(v[53]), "+r"(v[54]), "+r"(v[55]),
        "+r"(v[56]), "+r"(v[57]), "+r"(v[58]), "+r"(v[59]), "+r"(v[60]), "+r"(v[61]),
        "+r"(v[62]), "+r"(v[63])
      :
      : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
      "%29, %30, %31, %32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]),
      "r"(v[15]), "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]),
      "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]),
      "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle (canonical layouts of 8-row, 1024-byte
// atoms).  K-major: rows of 128 B, 8-row groups `sbo` apart.  MN-major: 64-element MN blocks
// `lbo` apart, 8-row K groups `sbo` apart.
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16 with an fp32 accumulator; A and B both bf16 (bf16 = 1)
// or both f16 (bf16 = 0).
constexpr uint32_t idesc_f16kind(int M, int N, int b_mn_major, int bf16) {
  return (1u << 4) | ((uint32_t)bf16 << 7) | ((uint32_t)bf16 << 10) |
         ((uint32_t)b_mn_major << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
constexpr uint32_t kIdescQK = idesc_f16kind(256, 128, 0, 1);  // bf16 Q, K; M spans the pair
constexpr uint32_t kIdescPV = idesc_f16kind(256, 128, 1, 0);  // f16 P, V
constexpr uint32_t kIdescQK16 = idesc_f16kind(256, 128, 0, 0);  // fp8 pools: f16 Q, K

// ---- thread-block cluster (pairs of CTAs on two SMs) ------------------------------------------

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_id_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t num_clusters_x() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}
// Arrive on the barrier at this offset in every CTA of `mask` once this thread's MMAs are done.
__device__ __forceinline__ void tc_commit_mc_l0(uint64_t* bar, uint16_t mask) {
  asm volatile(
      "{\n\t.reg .u32 l;\n\t.reg .pred e;\n\tmov.u32 l, %%laneid;\n\tsetp.eq.u32 e, l, 0;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "h"(mask)
      : "memory");
}
// Arrive on the barrier at this offset in the leader CTA of the pair (default semantics: a
// cluster-scope release would fence every arrival; the data it announces is either written
// by the asynchronous proxy (TMA) or ordered by the tcgen05 fences around the arrive).
__device__ __forceinline__ void arrive_leader(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b32 ra;\n\tmapa.shared::cluster.u32 ra, %0, 0;\n\t"
      "mbarrier.arrive.shared::cluster.b64 _, [ra];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}


// 2^x with the SFU's approximate base-2 exponential (flush-to-zero; 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packed pairs of fp32 (Blackwell's two-wide FP32 instructions: one issue for two lanes of
// work).  A pair lives in one 64-bit register, .x in the low half.
__device__ __forceinline__ uint64_t f2_pack(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}

// ---- shared state -----------------------------------------------------------------------------

struct Ctx {
  uint8_t* sm;
  uint64_t* bar;
  volatile int* abort;
  int* status;
  uint64_t limit;
  uint32_t rank;       // this CTA's place in its pair (0: the leader, which issues the MMAs)
  int cluster;         // pair index
  int nclusters;       // number of pairs
};

__device__ __forceinline__ bool mbar_try_wait_cl(uint64_t* bar, uint32_t parity) {
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

// Bounded wait that also gives up when another role aborted.  The polls are plain try_waits
// (the hardware holds the thread briefly and resumes it when the phase completes): try_waits
// with a suspend-time hint, meant to leave the softmax warps more issue slots, woke up late
// enough to make the prefill chunks 6% slower (140.5 against 132.5 us per call); plain polls
// in the MMA issuers alone, or in the producers and converters alone, gave about half.
__device__ __forceinline__ bool wait_bar(const Ctx& c, int idx, uint32_t parity) {
  uint64_t* b = c.bar + idx;
  if (mbar_try_wait_cl(b, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cl(b, parity)) return true;
    if ((i & 31u) == 0) {
      if (*c.abort) return false;
      if (globaltimer_ns() - t0 > c.limit) {
        record_error(c.status, PA_ETIMEOUT);
        *c.abort = 1;
        return false;
      }
    }
  }
}

// The k-th item of this pair.  Items are ordered longest first; the pairs take them in snake
// order (round k runs over the pairs backwards when k is odd), which evens out their totals.
__device__ __forceinline__ int item_of(const Ctx& c, int k) {
  return k * c.nclusters + ((k & 1) ? c.nclusters - 1 - c.cluster : c.cluster);
}

struct Item {
  int s, kvh, qt, t0, n_tok, n, kv0, ntiles, nblk_vis;
};

// Item idx = (256-row pair, kv head); this CTA of the pair takes the 128-row tile `rank`.
__device__ __forceinline__ Item load_item(const TcParams& p, int idx, uint32_t rank) {
  const VarlenMeta& m = p.m;
  const int4 it = reinterpret_cast<const int4*>(p.plan + p.tc_off)[idx / m.num_kv_heads];
  Item r;
  r.s = it.x;
  r.qt = it.y;
  r.kvh = idx % m.num_kv_heads;
  const int tpt = kBM / m.group;
  const int qs = m.query_start_loc[r.s], qe = m.query_start_loc[r.s + 1];
  r.t0 = qs + (2 * r.qt + (int)rank) * tpt;
  r.n_tok = max(0, min(tpt, qe - r.t0));
  r.n = m.seq_lens[r.s];
  const int lo = it.z, hi = it.w;
  r.kv0 = (lo / 16) * 16;
  r.ntiles = (hi - r.kv0 + kBN - 1) / kBN;
  r.nblk_vis = (hi + 15) / 16;  // logical blocks [kv0 / 16, nblk_vis) hold visible keys
  return r;
}

// ---- roles ------------------------------------------------------------------------------------

// TMA producers of this CTA's parts.  The K warp also loads Q; the V warp runs its own copy of
// the loop, so a K tile is fetched as soon as its stage is free (gated only by the QK^T MMAs)
// and never waits behind a V stage that the slower PV MMAs still hold.  K part: blocks
// 4r .. 4r + 3 of the tile (keys 64r ..), both 64-dim halves, [half][64 keys][64 dims]; V part:
// all 8 blocks, dims 64r .. 64r + 63, [128 keys][64 dims].
// Wait, bounded and whatever the abort flag says, until the copies behind the last `issued`
// phases of a ring of `nst` full barriers have landed (all of them have, when their consumers
// saw them; after an abort the newest may still be in flight).
__device__ void drain_ring(const Ctx& c, int full, uint32_t nst, uint32_t issued) {
  if ((threadIdx.x & 31) != 0) return;
  for (uint32_t k = issued > nst ? issued - nst : 0; k < issued; ++k)
    mbar_wait(c.bar + full + k % nst, (k / nst) & 1u, c.limit);
}

template <bool FP8>
__device__ void producer_loop(const Ctx& c, const TcParams& p, const CUtensorMap* tq,
                              const CUtensorMap* tkv, bool is_v, int n_items, uint32_t& kv,
                              uint32_t& q_issued);

template <bool FP8>
__device__ void producer(const Ctx& c, const TcParams& p, const CUtensorMap* tq,
                         const CUtensorMap* tkv, bool is_v, int n_items) {
  uint32_t kv = 0, q_issued = 0;  // K (or V) stage loads and Q loads issued
  producer_loop<FP8>(c, p, tq, tkv, is_v, n_items, kv, q_issued);
  // normally every issued copy has been consumed and these return at once
  drain_ring(c, is_v ? B_VFULL : B_KFULL, is_v ? kStagesV : kStagesK, kv);
  if (!is_v) drain_ring(c, B_QFULL, 2, q_issued);
  __syncwarp();
}

template <bool FP8>
__device__ void producer_loop(const Ctx& c, const TcParams& p, const CUtensorMap* tq,
                              const CUtensorMap* tkv, bool is_v, int n_items, uint32_t& kv,
                              uint32_t& q_issued) {
  const int lane = threadIdx.x & 31;
  const VarlenMeta& m = p.m;
  const int full = is_v ? B_VFULL : B_KFULL, empty = is_v ? B_VEMPTY : B_KEMPTY;
  const int off = is_v ? kOffV : kOffK;
  const uint32_t nst = is_v ? kStagesV : kStagesK;
  uint32_t it_cnt = 0;
  for (int idx; (idx = item_of(c, (int)it_cnt)) < n_items; ++it_cnt) {
    const Item I = load_item(p, idx, c.rank);
    const int32_t* row = m.block_tables + (int64_t)I.s * m.max_blocks;
    const int blk0 = I.kv0 / 16;
    if (!is_v) {
      // Q: (D, H, T) tensor, box 64 x G x 128/G
      bool qok = true;
      if (lane == 0) {
        const uint32_t qb = it_cnt & 1u;
        qok = wait_bar(c, B_QEMPTY + qb, ((it_cnt >> 1) & 1u) ^ 1u);
        if (qok) {
          mbar_arrive_expect_tx(c.bar + B_QFULL + qb, kTile);
          uint8_t* dst = c.sm + kOffQ + qb * kTile;
          tma_load_3d(dst, tq, 0, I.kvh * m.group, I.t0, c.bar + B_QFULL + qb);
          tma_load_3d(dst + kHalf, tq, 64, I.kvh * m.group, I.t0, c.bar + B_QFULL + qb);
        }
      }
      if (!__shfl_sync(kFull, (int)qok, 0)) return;
      ++q_issued;
    }
    int next_id = (lane < 8 && blk0 + lane < I.nblk_vis) ? row[blk0 + lane] : -1;
    for (int j = 0; j < I.ntiles; ++j, ++kv) {
      const int id = next_id;
      if (j + 1 < I.ntiles) {  // prefetch the next tile's block ids
        const int lb = blk0 + 8 * (j + 1) + lane;
        next_id = (lane < 8 && lb < I.nblk_vis) ? row[lb] : -1;
      }
      // lane 0 claims the stage; then lanes 0..7 issue one box each (a TMA fill probe moved
      // these 16-row boxes faster with several issuing lanes than with one)
      const uint32_t st = kv % nst, ph = (kv / nst) & 1u;
      bool ok = true;
      if (lane == 0) {
        ok = wait_bar(c, empty + st, ph ^ 1u);
        if (ok) mbar_arrive_expect_tx(c.bar + full + st, FP8 ? kPart / 2 : kPart);
      }
      // K: lane l loads dim half l / 4 of block 4 * rank + l % 4; V: lane l loads block l
      const int my_id = __shfl_sync(kFull, id, is_v ? (lane & 7) : 4 * (int)c.rank + (lane & 3));
      __syncwarp();  // the stage's expected bytes are set before any box is issued
      if (__shfl_sync(kFull, (int)ok, 0) && lane < 8) {
        uint8_t* dst = c.sm + off + st * kPart;
        const int r = my_id >= 0 ? my_id * 16 : -16;
        if constexpr (FP8) {  // the codes go where the converters widen them in place
          if (!is_v && lane < 4)  // block 4 * rank + lane, all 128 dims (128 x 1 x 16 bytes)
            tma_load_3d(dst + kPart / 2 + lane * 2048, tkv, 0, I.kvh, r, c.bar + full + st);
          else if (is_v)  // block lane, dims 64 * rank .. (64 x 1 x 16 bytes), into the back
            tma_load_3d(dst + lane * 2048 + 1024, tkv, 64 * (int)c.rank, I.kvh, r,  // half of
                        c.bar + full + st);                                        // its rows
        } else if (!is_v) {
          tma_load_3d(dst + (lane >> 2) * kKVHalf + (lane & 3) * 2048, tkv, 64 * (lane >> 2),
                      I.kvh, r, c.bar + full + st);
        } else {
          tma_load_3d(dst + lane * 2048, tkv, 64 * (int)c.rank, I.kvh, r, c.bar + full + st);
        }
      }
      // kv counts the loads issued: the loop's increment is skipped for this unissued one
      if (!__shfl_sync(kFull, (int)ok, 0)) return;
    }
  }
}

// MMA issue runs on two threads of the leader (warps 1 and 3) so that one thread's
// instruction issue never delays the other chain: the QK^T issuer releases K and Q stages, the
// PV issuer releases V stages, S / P buffers and O.  In the peer warp 1 forwards the arrival
// of its Q / K parts to the leader's full barriers, which count two arrivals: the leader's own
// producer and the peer's forward; the V parts reach the leader through the converters.
//
// Tile counters run over all items of the CTA; tile s uses S / P buffer s % 3, and each
// per-buffer barrier completes once per use, so its phase parity is (s / 3) & 1.
__device__ __forceinline__ uint32_t buf_of(uint32_t s) { return s % kSBufs; }
__device__ __forceinline__ uint32_t use_par(uint32_t s) { return (s / kSBufs) & 1u; }

template <bool FP8>
__device__ void s_issuer(const Ctx& c, const TcParams& p, uint32_t tmem, int n_items) {
  const uint32_t sm = smem_u32(c.sm);
  const bool leader = c.rank == 0, fp8 = FP8;
  // fp8 pools: the converters tell the leader when both CTAs' Q and K parts are f16, and the
  // peer's warp has nothing to forward
  if (fp8 && !leader) return;
  const uint32_t idesc = fp8 ? kIdescQK16 : kIdescQK;
  const int qready = fp8 ? B_QCONV : B_QFULL, kready = fp8 ? B_KCONV : B_KFULL;
  uint32_t kv = 0, it_cnt = 0;
  for (int idx; (idx = item_of(c, (int)it_cnt)) < n_items; ++it_cnt) {
    const Item I = load_item(p, idx, c.rank);
    const uint32_t qb = it_cnt & 1u;
    if (!__all_sync(kFull, wait_bar(c, qready + qb, (it_cnt >> 1) & 1u))) return;
    if (!leader && (threadIdx.x & 31) == 0) arrive_leader(c.bar + B_QFULL + qb);
    const uint32_t qbase = sm + kOffQ + qb * kTile;
    for (int j = 0; j < I.ntiles; ++j) {
      const uint32_t s = kv + j, st = s % kStagesK, b = buf_of(s);
      if (!__all_sync(kFull, wait_bar(c, kready + st, (s / kStagesK) & 1u))) return;
      if (!leader) {
        if ((threadIdx.x & 31) == 0) arrive_leader(c.bar + B_KFULL + st);
        continue;
      }
      // the buffer's previous tile (s - 3): its P was consumed by its P V
      if (!__all_sync(kFull, wait_bar(c, B_PVDONE + b, use_par(s) ^ 1u))) return;
      tc_fence_after();
      const uint32_t kb = sm + kOffK + st * kPart;
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        tc_mma_l0(tmem + col_s(b), sdesc(qbase + (kk >> 2) * kHalf + (kk & 3) * 32, 16, 1024),
                  sdesc(kb + (kk >> 2) * kKVHalf + (kk & 3) * 32, 16, 1024), idesc,
                  kk > 0 ? 1u : 0u);
      tc_commit_mc_l0(c.bar + B_SFULL + b, 0x3);
      tc_commit_mc_l0(c.bar + B_KEMPTY + st, 0x3);
      if (j == I.ntiles - 1) tc_commit_mc_l0(c.bar + B_QEMPTY + qb, 0x3);
      __syncwarp();
    }
    kv += I.ntiles;
  }
}

// The leader's whole warp runs the PV loop (lane 0 issues): O += P_j V_j once P_j is in
// tensor memory and both CTAs' parts of V_j are f16.  The peer's warp has nothing to do.
__device__ void pv_issuer(const Ctx& c, const TcParams& p, uint32_t tmem, int n_items) {
  if (c.rank != 0) return;
  uint32_t kv = 0, it_cnt = 0;
  for (int idx; (idx = item_of(c, (int)it_cnt)) < n_items; ++it_cnt) {
    const Item I = load_item(p, idx, c.rank);
    for (int j = 0; j < I.ntiles; ++j) {
      const uint32_t s = kv + j, st = s % kStagesV, b = buf_of(s);
      if (j == 0 && !__all_sync(kFull, wait_bar(c, B_OFREE, (it_cnt & 1u) ^ 1u))) return;
      if (!__all_sync(kFull, wait_bar(c, B_PFULL + b, use_par(s)))) return;
      if (!__all_sync(kFull, wait_bar(c, B_VCONV + st, (s / kStagesV) & 1u))) return;
      tc_fence_after();
      const uint32_t vb = smem_u32(c.sm + kOffV + st * kPart), pb = tmem + col_s(b);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
        tc_mma_ta_l0(tmem + kColO, pb + col_p(kk), sdesc(vb + kk * 2048, 1024, 1024), kIdescPV,
                     (j > 0 || kk > 0) ? 1u : 0u);
      tc_commit_mc_l0(c.bar + B_PVDONE + b, 0x3);
      tc_commit_mc_l0(c.bar + B_VEMPTY + st, 0x3);
      __syncwarp();
    }
    kv += I.ntiles;
  }
}

// bf16x2 -> f16x2, each half through fp32 (the widening to fp32 is exact; the narrowing
// rounds to nearest even and is exact for magnitudes below 65520 down to f16's subnormal
// step).  The high element goes to the high half.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;"
      : "=r"(r)
      : "f"(__uint_as_float(w & 0xffff0000u)), "f"(__uint_as_float(w << 16)));
  return r;
}
// acc + h * 0 on f16 pairs: stays finite (+-0 added) until a half of h is infinite or NaN,
// then NaN for good -- one instruction per word tells whether any widening overflowed.
__device__ __forceinline__ uint32_t f16x2_poison(uint32_t acc, uint32_t h) {
  uint32_t r;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(h), "r"(0u), "r"(acc));
  return r;
}

// V converter warp w (0..3) of either CTA: for every V stage of its CTA, once the TMA has
// landed, the quarter holding keys 32w .. 32w + 31 (this CTA's 64 dims, 4 KB: rows of 128
// bytes, the 128-byte swizzle only permutes 16-byte chunks inside a row) is widened from bf16
// to f16 in place; rows at positions >= seq_len (never written: they may hold anything) become
// zeros.  Then the leader's V-ready barrier of the stage gets this warp's arrival.  A quarter
// with a value that f16 cannot hold (its magnitude rounds to infinity; an inf or NaN too)
// marks the item for the recompute after this kernel.
//
// The arrival is a plain remote arrive, as for the other forwards: a cluster-scope release
// on it stalls the warp on a memory barrier per stage, which measured 40% slower per call.
// The stores are to this CTA's own shared memory, and fence.proxy.async (shared::cta) makes
// them visible to the asynchronous proxy, through which the pair's MMAs read them.
__device__ void v_converter(const Ctx& c, const TcParams& p, int n_items) {
  const int lane = threadIdx.x & 31, w = (threadIdx.x >> 5) - kFirstConvWarp;
  uint32_t kv = 0, it_cnt = 0;
  for (int idx; (idx = item_of(c, (int)it_cnt)) < n_items; ++it_cnt) {
    const Item I = load_item(p, idx, c.rank);
    uint32_t poison = 0;  // f16 pair; NaN once a widened value overflowed
    for (int j = 0; j < I.ntiles; ++j) {
      const uint32_t s = kv + j, st = s % kStagesV;
      if (!__all_sync(kFull, wait_bar(c, B_VFULL + st, (s / kStagesV) & 1u))) return;
      uint8_t* q = c.sm + kOffV + st * kPart + w * 4096;
      const int pos0 = I.kv0 + j * kBN + 32 * w;  // position of the quarter's first row
      // two groups of four 16-byte chunks per lane (chunk lane + 32 i holds row (lane + 32 i) / 8)
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        uint4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          v[i] = *reinterpret_cast<const uint4*>(q + (lane + 32 * (4 * g + i)) * 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int ch = lane + 32 * (4 * g + i);
          if (pos0 + (ch >> 3) >= I.n) {
            v[i] = make_uint4(0u, 0u, 0u, 0u);
          } else {
            v[i].x = bf16x2_to_f16x2(v[i].x);
            v[i].y = bf16x2_to_f16x2(v[i].y);
            v[i].z = bf16x2_to_f16x2(v[i].z);
            v[i].w = bf16x2_to_f16x2(v[i].w);
            poison = f16x2_poison(f16x2_poison(poison, v[i].x), v[i].y);
            poison = f16x2_poison(f16x2_poison(poison, v[i].z), v[i].w);
          }
          *reinterpret_cast<uint4*>(q + ch * 16) = v[i];
        }
      }
      // the MMA (issued by the leader) reads V through the asynchronous proxy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) arrive_leader(c.bar + B_VCONV + st);
    }
    const bool over = (poison & 0x7fffu) > 0x7c00u || ((poison >> 16) & 0x7fffu) > 0x7c00u;
    if (__any_sync(kFull, over) && lane == 0) {
      const int pi = idx / p.m.num_kv_heads;  // the plan's 256-row item (all its kv heads)
      if (atomicCAS(p.redo_flags + pi, 0, 1) == 0) p.redo_list[atomicAdd(p.redo_count, 1)] = pi;
    }
    kv += I.ntiles;
  }
}


// Two e4m3 codes per 16-bit half of w -> four f16 in two words (element order kept), exactly.
__device__ __forceinline__ void widen4(uint32_t w, uint32_t& a, uint32_t& b) {
  a = e4m3x2_to_f16x2((uint16_t)(w & 0xffffu));
  b = e4m3x2_to_f16x2((uint16_t)(w >> 16));
}

// Converters over fp8 pools (e4m3 codes: K = k_scale * code, V = v_scale * code; the codes widen
// to f16 exactly).  TMA writes a stage's codes into part of its 16 KB slot, and each converter
// warp widens its own blocks into the f16 operand the MMAs read (rows of 128 bytes with the
// 128-byte swizzle):
//   K, warp w: block w of this CTA's four.  Its codes (16 rows x 128, swizzled like the
//     operand) sit where its second dim half goes, [8 KB + 2 KB w, + 2 KB); the warp loads all
//     of them, then writes dims 0..63 to [2 KB w, + 2 KB) and dims 64..127 over them.
//   V, warp w: blocks 2w and 2w + 1.  Block b's codes (16 rows x this CTA's 64 dims, plain
//     64-byte rows) sit in the back half of its own 2 KB output, [2 KB b + 1 KB, + 1 KB); the
//     warp loads them, then writes the 16 f16 rows of 128 bytes over the whole 2 KB.  Rows at
//     positions >= seq_len become zeros.
// Every byte a warp overwrites is one it loaded itself, so __syncwarp() orders the loads
// before the stores and the four warps need no barrier between them.  Q (bf16 from TMA) is
// widened to f16 in place once per item, a quarter per warp: exact in f16's normal range,
// which is how the warp-MMA fp8 path takes q as well.
// Per-block factors (p.m.k_bscales / v_bscales, [num_blocks, num_kv_heads]).  The softmax
// applies each block's K factor to its scores in fp32, exactly as the warp-MMA kernel does.
// V: the converter multiplies the widened codes of each block by the ratio of its factor to
// the item's reference, the factor of its first block (f16 product; the softmax multiplies
// the output by the reference), so the products stay in f16's normal range whatever the
// factors' magnitude.  A ratio outside [kRatioMin, kRatioMax] could not (a product past f16's
// range, or small values left with few bits): the item is then marked for the warp-MMA
// kernel behind this one, which keeps its f16 weights in range for any finite factors.
constexpr float kRatioMax = 146.0f;           // 65504 / 448, the largest e4m3 magnitude
constexpr float kRatioMin = 1.0f / 4096.0f;   // products of the smallest codes stay near 2^-21
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a),
                            *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ void hmul2x4(uint4& v, uint32_t f) {
  v.x = hmul2(v.x, f);
  v.y = hmul2(v.y, f);
  v.z = hmul2(v.z, f);
  v.w = hmul2(v.w, f);
}
__device__ __forceinline__ uint32_t half2_bits(float x) {
  const __half2 h = __float2half2_rn(x);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// The factors of NB consecutive 16-key blocks a thread applies in each 128-key tile of an
// item (logical blocks b0 + 8 j .. b0 + 8 j + NB - 1 in tile j), loaded ahead of their use:
// the table entries two tiles ahead, the factors one tile ahead, so the tile loop never waits
// for either.  Blocks past the last one with visible keys read nothing and take `dflt`.
template <int NB>
struct FactorPipe {
  const int32_t* trow;
  const float* f;
  int64_t H;
  int kvh, b0, lim;
  float dflt;
  int tb[NB];
  float cur[NB], nxt[NB];
  __device__ __forceinline__ void tables(int j) {
#pragma unroll
    for (int q = 0; q < NB; ++q) {
      const int lb = b0 + 8 * j + q;
      tb[q] = lb < lim ? trow[lb] : -1;
    }
  }
  __device__ __forceinline__ void factors() {
#pragma unroll
    for (int q = 0; q < NB; ++q) nxt[q] = tb[q] >= 0 ? f[tb[q] * H + kvh] : dflt;
  }
  // item start: the factors of tile 0 and the table entries of tile 1
  __device__ __forceinline__ void start() {
    tables(0);
    factors();
    tables(1);
  }
  // top of tile j: cur = the factors of tile j
  __device__ __forceinline__ void advance(int j) {
#pragma unroll
    for (int q = 0; q < NB; ++q) cur[q] = nxt[q];
    factors();
    tables(j + 2);
  }
};

// The item's V reference: the factor of its first block (1 when it has no visible keys).
__device__ __forceinline__ float v_reference(const VarlenMeta& m, const int32_t* trow,
                                             const Item& I) {
  const int b0 = I.kv0 / 16;
  return b0 < I.nblk_vis ? m.v_bscales[(int64_t)trow[b0] * m.num_kv_heads + I.kvh] : 1.f;
}

template <bool PB>
__device__ void fp8_converter(const Ctx& c, const TcParams& p, int n_items) {
  const int lane = threadIdx.x & 31, w = (threadIdx.x >> 5) - kFirstConvWarp;
  uint32_t kv = 0, it_cnt = 0;
  for (int idx; (idx = item_of(c, (int)it_cnt)) < n_items; ++it_cnt) {
    const Item I = load_item(p, idx, c.rank);
    FactorPipe<2> vf;  // PB: the V factors of blocks 2w, 2w + 1 of each tile
    float rref = 1.f;  // PB: 1 / the item's V reference
    bool out_of_range = false;  // PB: a ratio outside [kRatioMin, kRatioMax]
    if constexpr (PB) {
      const int32_t* trow = p.m.block_tables + (int64_t)I.s * p.m.max_blocks;
      const float vref = v_reference(p.m, trow, I);
      rref = __frcp_rn(vref);
      vf = FactorPipe<2>{trow, p.m.v_bscales, p.m.num_kv_heads, I.kvh, I.kv0 / 16 + 2 * w,
                         I.nblk_vis, vref};
      vf.start();
    }
    {  // Q: this warp's quarter of the 128 x 128 bf16 tile, 16 chunks of 16 bytes per lane
      const uint32_t qb = it_cnt & 1u;
      if (!__all_sync(kFull, wait_bar(c, B_QFULL + qb, (it_cnt >> 1) & 1u))) return;
      uint4* q = reinterpret_cast<uint4*>(c.sm + kOffQ + qb * kTile) + w * (kTile / 16 / 4);
#pragma unroll 4
      for (int i = 0; i < kTile / 16 / 4 / 32; ++i) {
        uint4 v = q[lane + 32 * i];
        v.x = bf16x2_to_f16x2(v.x);
        v.y = bf16x2_to_f16x2(v.y);
        v.z = bf16x2_to_f16x2(v.z);
        v.w = bf16x2_to_f16x2(v.w);
        q[lane + 32 * i] = v;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) arrive_leader(c.bar + B_QCONV + qb);
    }
    for (int j = 0; j < I.ntiles; ++j, ++kv) {
      uint32_t vr2a = 0, vr2b = 0;  // PB: the ratios of V blocks 2w, 2w + 1 (f16 pairs)
      if constexpr (PB) {
        vf.advance(j);
        const float r0 = vf.cur[0] * rref, r1 = vf.cur[1] * rref;
        out_of_range |= !(r0 >= kRatioMin && r0 <= kRatioMax && r1 >= kRatioMin &&
                          r1 <= kRatioMax);
        vr2a = half2_bits(r0);
        vr2b = half2_bits(r1);
      }
      {  // K block w
        const uint32_t st = kv % kStagesK;
        if (!__all_sync(kFull, wait_bar(c, B_KFULL + st, (kv / kStagesK) & 1u))) return;
        uint8_t* slot = c.sm + kOffK + st * kPart;
        const uint4* stg = reinterpret_cast<const uint4*>(slot + kPart / 2 + w * 2048);
        // four rounds of rows 4i .. 4i + 3: a round's stores overwrite only the staged codes
        // of its own rows, which all lanes have loaded before the __syncwarp
#pragma unroll 1
        for (int i = 0; i < 4; ++i) {
          const uint4 src = stg[lane + 32 * i];
          __syncwarp();
          const int q = lane + 32 * i;                // staged chunk: row q / 8, chunk q % 8
          const int r = q >> 3, L = (q & 7) ^ (r & 7);  // key row, dims 16 L .. 16 L + 15
          const int h = L >> 2, c0 = 2 * (L & 3);     // dim half, first output chunk
          uint4 lo, hi;
          widen4(src.x, lo.x, lo.y);
          widen4(src.y, lo.z, lo.w);
          widen4(src.z, hi.x, hi.y);
          widen4(src.w, hi.z, hi.w);
          uint8_t* row = slot + h * kKVHalf + w * 2048 + r * 128;
          *reinterpret_cast<uint4*>(row + ((c0 ^ (r & 7)) << 4)) = lo;
          *reinterpret_cast<uint4*>(row + (((c0 + 1) ^ (r & 7)) << 4)) = hi;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) arrive_leader(c.bar + B_KCONV + st);
      }
      {  // V blocks 2w, 2w + 1
        const uint32_t st = kv % kStagesV;
        if (!__all_sync(kFull, wait_bar(c, B_VFULL + st, (kv / kStagesV) & 1u))) return;
        uint8_t* slot = c.sm + kOffV + st * kPart;
        const int pos0 = I.kv0 + j * kBN;  // position of the tile's first key
        // per block, rows 0..7 first (their stores land in the block's front kilobyte, where
        // no codes are staged), then rows 8..15, whose stores overwrite the block's staged
        // codes: all loaded by then (__syncwarp)
#pragma unroll 1
        for (int i = 0; i < 4; ++i) {
          const int b = 2 * w + (i >> 1), q = lane + 32 * (i & 1);
          const uint4 src = reinterpret_cast<const uint4*>(slot + b * 2048 + 1024)[q];
          if (i & 1) __syncwarp();
          const int r = q >> 2, L = q & 3;  // key row, dims 16 L .. 16 L + 15
          uint4 lo = make_uint4(0u, 0u, 0u, 0u), hi = lo;
          if (pos0 + b * 16 + r < I.n) {  // rows past seq_len were never written
            widen4(src.x, lo.x, lo.y);
            widen4(src.y, lo.z, lo.w);
            widen4(src.z, hi.x, hi.y);
            widen4(src.w, hi.z, hi.w);
            if constexpr (PB) {
              const uint32_t r2 = (i >> 1) ? vr2b : vr2a;
              hmul2x4(lo, r2);
              hmul2x4(hi, r2);
            }
          }
          uint8_t* row = slot + b * 2048 + r * 128;
          *reinterpret_cast<uint4*>(row + (((2 * L) ^ (r & 7)) << 4)) = lo;
          *reinterpret_cast<uint4*>(row + (((2 * L + 1) ^ (r & 7)) << 4)) = hi;
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) arrive_leader(c.bar + B_VCONV + st);
      }
    }
    if (out_of_range && lane == 0) {  // (uniform across the warp)
      const int pi = idx / p.m.num_kv_heads;  // the plan's 256-row item (all its kv heads)
      if (atomicCAS(p.redo_flags + pi, 0, 1) == 0) p.redo_list[atomicAdd(p.redo_count, 1)] = pi;
    }
  }
}

// Named barrier of the two softmax warps that share 32 query rows (one per column half).  A
// softmax warp whose bounded wait fails does not leave at once: it carries the failure to
// the pair's next exchange (the tile's row max, or the item's end), where both warps read
// both flags and leave together, so neither is left waiting at this barrier.
__device__ __forceinline__ void pair_sync(int quad) {
  asm volatile("bar.sync %0, 64;" ::"r"(1 + quad) : "memory");
}

template <bool PB>
__device__ void softmax_role(const Ctx& c, const TcParams& p, uint32_t tmem, int n_items) {
  const VarlenMeta& m = p.m;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hf = (warp - 4) >> 2;  // column half of S / P / O this warp handles
  const int quad = warp & 3;       // TMEM lane quarter this warp may access
  const int r = 32 * quad + lane;  // this thread's query row == TMEM lane
  const int col0 = hf * 64;
  const uint32_t lane_addr = (uint32_t)(32 * quad) << 16;
  float* xchg = reinterpret_cast<float*>(c.sm + kOffXchg);  // [half][row]
  int* xbad_e = reinterpret_cast<int*>(xchg + 2 * 128);      // [half][row], item end
  bool bad = false;  // a wait of this warp ran out or another role aborted (warp-uniform)
  uint32_t kv = 0;
  // an item's metadata (plan entry, sequence bounds, this row's position) is a chain of
  // dependent loads: the next item's is fetched while the current one's last P V runs
  Item In{};
  int pos_n = 0;
  if (item_of(c, 0) < n_items) In = load_item(p, item_of(c, 0), c.rank);
  if (r / m.group < In.n_tok) pos_n = m.positions[In.t0 + r / m.group];
  for (int k = 0; item_of(c, k) < n_items; ++k) {
    const Item I = In;
    const int tl = r / m.group;
    const bool valid = tl < I.n_tok;
    const int t = I.t0 + (valid ? tl : 0);
    const int h = I.kvh * m.group + r % m.group;
    int start = 0, end = 0;
    if (valid) {
      end = m.causal ? pos_n + 1 : I.n;
      start = m.window > 0 ? max(0, end - m.window) : 0;
    }
    float m_ref = -INFINITY, l = 0.f;
    const float sl = head_scale(m.k_scales, I.kvh, p.scale_log2);  // K = k_scales[g] * pool
    // PB: the K factors of this thread's four blocks (64 columns) in each tile, and the V
    // reference the converters divided the factors by
    FactorPipe<4> kf;
    float vref = 1.f;
    if constexpr (PB) {
      const int32_t* trow = m.block_tables + (int64_t)I.s * m.max_blocks;
      kf = FactorPipe<4>{trow, m.k_bscales, m.num_kv_heads, I.kvh, I.kv0 / 16 + 4 * hf,
                         I.nblk_vis, 1.f};
      kf.start();
      vref = v_reference(m, trow, I);
    }
    for (int j = 0; j < I.ntiles; ++j) {
      if constexpr (PB) kf.advance(j);
      const uint32_t s = kv + j, b = buf_of(s);
      const uint32_t sbase = tmem + lane_addr + col_s(b) + col0;  // this thread's S / P columns
      // debug_stall (tests only): the wait names a barrier nothing arrives on, so it runs out
      // after the wait limit and the kernel unwinds as from an S that never completed
      if (!bad)
        bad = !__all_sync(kFull, p.debug_stall ? wait_bar(c, B_NEVER, 0u)
                                               : wait_bar(c, B_SFULL + b, use_par(s)));
      tc_fence_after();
      // after a failed wait the values read here only travel to the exchange below, where
      // the pair leaves (a read of allocated tensor memory is defined, whatever it holds)
      float x[64];
      {
        uint32_t v[64];
        tmem_ld64(sbase, v);
        tmem_wait_ld64(v);
#pragma unroll
        for (int i = 0; i < 64; ++i) x[i] = __uint_as_float(v[i]);
      }

      // mask the raw scores (scale > 0 on this path, so the max commutes with it); an
      // invalid row has start == end == 0 and masks everything
      const int key0 = I.kv0 + j * kBN + col0;
      if (!(key0 >= start && key0 + 64 <= end)) {
        // visible columns of this thread: [a, b) within its 64
        const int a = start - key0, bnd = end - key0;
#pragma unroll
        for (int i = 0; i < 64; ++i) x[i] = (i >= a && i < bnd) ? x[i] : -INFINITY;
      }
      float mx[8];
      float sq[4];  // PB: the score scale of each 16-column block, sl times its K factor
      float mine;
      if constexpr (PB) {
        // the factors are positive, so a block's max commutes with its scale: the max of
        // the scaled scores, exchanged as such
#pragma unroll
        for (int q = 0; q < 4; ++q) sq[q] = sl * kf.cur[q];
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = x[8 * k];
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (i & 7) mx[i >> 3] = fmaxf(mx[i >> 3], x[i]);
        mine = fmaxf(fmaxf(fmaxf(mx[0], mx[1]) * sq[0], fmaxf(mx[2], mx[3]) * sq[1]),
                     fmaxf(fmaxf(mx[4], mx[5]) * sq[2], fmaxf(mx[6], mx[7]) * sq[3]));
      } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) mx[k] = x[k];
#pragma unroll
        for (int i = 8; i < 64; ++i) mx[i & 7] = fmaxf(mx[i & 7], x[i]);
        mine = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                     fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      }
      // the row max over both column halves; a failed wait travels as kBadMax
      xchg[hf * 128 + r] = bad ? __uint_as_float(kBadMax) : mine;
      pair_sync(quad);
      const float other = xchg[(hf ^ 1) * 128 + r];
      const float mt = PB ? fmaxf(mine, other) : fmaxf(mine, other) * sl;
      const bool leave = __any_sync(kFull, bad || __float_as_uint(other) == kBadMax);
      pair_sync(quad);  // both read before either writes again
      if (leave) return;
      const float m_new = fmaxf(m_ref, mt);
      const bool resc = m_new > m_ref + 8.f;
      float alpha = 1.f;
      if (resc) {
        alpha = fast_exp2(m_ref - m_new);  // 0 when nothing was visible before
        m_ref = m_new;
        l *= alpha;
      }
      // p = 2^(x * scale_log2 - m_ref) two at a time (p <= 2^8), the row sum of the fp32
      // weights, and p rounded to f16 for the P V MMAs
      const float nbase = m_ref == -INFINITY ? 0.f : -m_ref;
      const uint64_t sl2 = f2_pack(sl, sl), nb2 = f2_pack(nbase, nbase);
      uint64_t sq2[4] = {sl2, sl2, sl2, sl2};
      if constexpr (PB) {
#pragma unroll
        for (int q = 0; q < 4; ++q) sq2[q] = f2_pack(sq[q], sq[q]);
      }
      uint32_t ph[32];
      {
        uint64_t rs2[4] = {0, 0, 0, 0};
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          float a, bb;
          f2_unpack(f2_fma(f2_pack(x[2 * e], x[2 * e + 1]), PB ? sq2[e >> 3] : sl2, nb2), a, bb);
          a = fast_exp2(a);
          bb = fast_exp2(bb);
          rs2[e & 3] = f2_add(rs2[e & 3], f2_pack(a, bb));
          ph[e] = pack_f16x2(a, bb);
        }
        float r0, r1, r2, r3, r4, r5, r6, r7;
        f2_unpack(rs2[0], r0, r1);
        f2_unpack(rs2[1], r2, r3);
        f2_unpack(rs2[2], r4, r5);
        f2_unpack(rs2[3], r6, r7);
        l += ((r0 + r1) + (r2 + r3)) + ((r4 + r5) + (r6 + r7));
      }

      // O rescale: only after P_{j-1} V_{j-1} is done (O stable); most tiles skip both
      if (j >= 1 && __any_sync(kFull, resc)) {
        // a failure here is carried to the next exchange (what this warp writes to tensor
        // memory until then is never read into the output)
        if (!bad) bad = !__all_sync(kFull, wait_bar(c, B_PVDONE + buf_of(s - 1), use_par(s - 1)));
        tc_fence_after();
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_addr + kColO + col0 + q * 32, o);
          tmem_wait_ld(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st32(tmem + lane_addr + kColO + col0 + q * 32, o);
        }
        tmem_wait_st();
      }
      // this half of P over the scores it came from
      tmem_st32(sbase, ph);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_leader(c.bar + B_PFULL + b);  // the leader issues this P's MMAs
    }

    if (item_of(c, k + 1) < n_items) {
      In = load_item(p, item_of(c, k + 1), c.rank);
      if (tl < In.n_tok) pos_n = m.positions[In.t0 + tl];
    }
    // epilogue: o = O / l, with l summed over both column halves; the pair's failure flags
    // travel with the second barrier, so both warps leave before any output is written
    const uint32_t last = kv + I.ntiles - 1;
    {
      xchg[hf * 128 + r] = l;
      pair_sync(quad);
      l += xchg[(hf ^ 1) * 128 + r];
      if (!bad) bad = !__all_sync(kFull, wait_bar(c, B_PVDONE + buf_of(last), use_par(last)));
      xbad_e[hf * 128 + r] = bad ? 1 : 0;
      pair_sync(quad);  // both read the sums before either writes again; the flags are read next
      if (__any_sync(kFull, bad || xbad_e[(hf ^ 1) * 128 + r] != 0)) return;
    }
    tc_fence_after();
    // an attention sink (TensorSharp ForwardWithSinks) is one more state to merge: max = the
    // sink logit, exp-sum = 1, weighted sum = 0
    float o_scale = 1.f;
    {
      const float sk = m.sinks ? m.sinks[h] * kLog2e : -INFINITY;
      if (sk > -INFINITY) {
        const float m2 = fmaxf(m_ref, sk);
        o_scale = m_ref == -INFINITY ? 0.f : fast_exp2(m_ref - m2);
        l = l * o_scale + fast_exp2(sk - m2);
        m_ref = m2;
      }
    }
    if (m.lse && hf == 0 && valid)
      m.lse[(int64_t)h * m.num_tokens + t] = l > 0.f ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
    const float inv =
        l > 0.f ? o_scale * head_scale(m.v_scales, I.kvh, m.v_scale) * vref / l : 0.f;
    __nv_bfloat16* dst =
        reinterpret_cast<__nv_bfloat16*>(p.out) + ((int64_t)t * m.num_heads + h) * kD + col0;
    // rows start 256 bytes apart and halves at 0 / 128: 32-byte aligned when the output is
    const bool st32 = (reinterpret_cast<uintptr_t>(p.out) & 31) == 0;
    uint32_t oo[64];
    tmem_ld64(tmem + lane_addr + kColO + col0, oo);
    tmem_wait_ld64(oo);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t* o = oo + 32 * q;
      if (valid) {
        uint32_t w[16];
#pragma unroll
        for (int i = 0; i < 16; ++i)
          w[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
        if (st32) {  // 32-byte stores: a whole sector each
#pragma unroll
          for (int i = 0; i < 16; i += 8)
            asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(
                             dst + q * 32 + 2 * i),
                         "r"(w[i]), "r"(w[i + 1]), "r"(w[i + 2]), "r"(w[i + 3]), "r"(w[i + 4]),
                         "r"(w[i + 5]), "r"(w[i + 6]), "r"(w[i + 7])
                         : "memory");
        } else {
#pragma unroll
          for (int i = 0; i < 16; i += 4)
            *reinterpret_cast<uint4*>(dst + q * 32 + 2 * i) =
                make_uint4(w[i], w[i + 1], w[i + 2], w[i + 3]);
        }
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) arrive_leader(c.bar + B_OFREE);
    kv += I.ntiles;
  }
}

template <bool FP8, bool PB>
__global__ void __launch_bounds__(kThreads, 1)
    k_tc_prefill(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, const TcParams p) {
  static_assert(!PB || FP8, "per-block factors are for e4m3 pools");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                           ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffTmem);
  int* flags = reinterpret_cast<int*>(sm + kOffFlag);  // [0] skip everything, [1] abort
  const int warp = threadIdx.x >> 5;

  const bool leader = cluster_rank() == 0;
  if (threadIdx.x == 0) {
    flags[1] = 0;
    // leader: q/k full count its producer and the peer's forward, v-ready one arrival per
    // converter warp of both CTAs, p_full / o_free one per softmax warp of both CTAs, fin one
    // per MMA-issuing warp; the empty / done barriers of both CTAs get one multicast commit
    // per phase; the rest (v full included: this CTA's own TMA) one arrival
    for (int i = 0; i < kNumBars; ++i) {
      uint32_t n = 1;
      if (leader) {
        // bf16 pools: q / k full count the leader's own TMA and the peer's forward; fp8 pools:
        // the own TMA only (the converters then arrive on q / k / v conv, from both CTAs)
        if ((i >= B_QFULL && i < B_QFULL + 2) || (i >= B_KFULL && i < B_KFULL + kStagesK))
          n = FP8 ? 1 : 2;
        if ((i >= B_VCONV && i < B_VCONV + kStagesV) || (i >= B_QCONV && i < B_QCONV + 2) ||
            (i >= B_KCONV && i < B_KCONV + kStagesK))
          n = 2 * kConvWarps;
        if ((i >= B_PFULL && i < B_PFULL + kSBufs) || i == B_OFREE) n = 2 * kSoftWarps;
        if (i == B_FIN) n = 2;
      }
      mbar_init(bar + i, n);
    }
    prefetch_tmap(&tq);
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
  }
  fence_mbar_init();
  if (warp == 1) {  // one warp of each CTA of the pair allocates, collectively
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync();  // the partner's barriers are initialised before any commit or arrive reaches them
  tc_fence_after();
  // everything above overlaps the planning kernel (programmatic dependent launch); the plan
  // and the status word are read only after it has finished
  pdl_wait();
  if (threadIdx.x == 0) flags[0] = status_set(p.status) ? 1 : 0;
  __syncthreads();
  pdl_launch_dependents();
  const uint32_t tmem = *tmem_slot;
  // the plan's number of working pairs: the others take no item and leave, and the warp-MMA
  // kernel launched behind this one runs its decode tiles on their SMs meanwhile
  const int pairs = max(1, min((int)num_clusters_x(), p.plan[5]));
  Ctx c{sm, bar, reinterpret_cast<volatile int*>(flags + 1), p.status, p.wait_limit_ns,
        cluster_rank(), (int)cluster_id_x(), pairs};
  const int n_items = (flags[0] || c.cluster >= pairs) ? 0 : p.plan[1] * p.m.num_kv_heads;

  // warps 0..3 (one warpgroup) produce and issue, warps 12..15 convert: both need few
  // registers; the two softmax warpgroups take theirs.  bf16 pools: 4 x 56 + 8 x 200 + 4 x 56,
  // e4m3 pools (the converters also widen K and Q): 4 x 64 + 8 x 184 + 4 x 80; both 16 x 128,
  // the launch's registers per thread (each branch ends the kernel itself, so no code runs
  // under two limits)
  static_assert(4 * 56 + 8 * 200 + 4 * 56 <= kThreads / 32 * 128, "register split, bf16");
  static_assert(4 * 64 + 8 * 184 + 4 * 80 <= kThreads / 32 * 128, "register split, e4m3");
  if (warp >= kFirstConvWarp) {
    if constexpr (FP8)
      asm volatile("setmaxnreg.dec.sync.aligned.u32 80;" ::: "memory");
    else
      asm volatile("setmaxnreg.dec.sync.aligned.u32 56;" ::: "memory");
    if constexpr (FP8)
      fp8_converter<PB>(c, p, n_items);
    else
      v_converter(c, p, n_items);
    tc_fence_before();
    cluster_sync();
  } else if (warp < 4) {
    if constexpr (FP8)
      asm volatile("setmaxnreg.dec.sync.aligned.u32 64;" ::: "memory");
    else
      asm volatile("setmaxnreg.dec.sync.aligned.u32 56;" ::: "memory");
    if (warp == 0) {
      producer<FP8>(c, p, &tq, &tk, false, n_items);
    } else if (warp == 2) {
      producer<FP8>(c, p, &tq, &tv, true, n_items);
    } else if (warp == 1 || warp == 3) {
      if (warp == 1)
        s_issuer<FP8>(c, p, tmem, n_items);
      else
        pv_issuer(c, p, tmem, n_items);
      __syncwarp();
      // every MMA issued by either warp of the leader has completed before the tensor memory is
      // released
      if (leader) {
        tc_commit_mc_l0(bar + B_FIN, 0x1);
        if ((threadIdx.x & 31) == 0) {
          uint64_t t0 = globaltimer_ns();
          while (!mbar_try_wait(bar + B_FIN, 0) && globaltimer_ns() - t0 < 1000000000ull) {
          }
        }
      }
      __syncwarp();
    }
    tc_fence_before();
    cluster_sync();  // neither CTA leaves while its partner may still write to its shared memory
    if (warp == 1) {  // collectively, like the allocation
      tc_fence_after();
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                   "r"(kTmemCols)
                   : "memory");
    }
  } else {
    if constexpr (FP8)
      asm volatile("setmaxnreg.inc.sync.aligned.u32 184;" ::: "memory");
    else
      asm volatile("setmaxnreg.inc.sync.aligned.u32 200;" ::: "memory");
    softmax_role<PB>(c, p, tmem, n_items);
    tc_fence_before();
    cluster_sync();
  }
}

}  // namespace

cudaError_t launch_tc_prefill(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const TcParams& p, int grid, cudaStream_t stream) {
  if (grid < 2) grid = 2;
  // per-block factors: e4m3 pools only (the caller checks)
  auto kern = !p.kv_fp8 ? k_tc_prefill<false, false>
              : p.m.k_bscales ? k_tc_prefill<true, true> : k_tc_prefill<true, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  // pairs of CTAs (a cluster of two SMs) run the 2-SM MMAs
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(grid & ~1), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlaps the plan kernel
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, p);
}

}  // namespace pa
