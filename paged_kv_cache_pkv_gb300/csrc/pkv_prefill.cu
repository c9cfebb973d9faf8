// pkv_prefill.cu -- chunked-prefill attention on the 5th-generation tensor
// cores (tcgen05 + TMEM + TMA) for sequences with many query rows.
//
// What is computed (llm-d blog post "What does production-grade LLM inference
// look like?", introduction: prefill is compute bound; with continuous
// batching a step carries prefill chunks next to decode rows): for query j of
// a chunk of n tokens in a sequence of L cached tokens, softmax attention over
// keys 0 .. L-n+j (bottom-right causal), query head h reading kv head h/G.
//
// Design (GB300):
//  * A Q tile is 128 query rows: TM = 128/G query tokens x the G query heads
//    of one kv head (row = token*G + head), so every K/V tile loaded serves
//    all G heads of the group.  One CTA holds two Q tiles (2*TM consecutive
//    tokens) and streams each K/V tile once for both: the copy engine's bytes
//    per tensor-core FLOP are halved, which is what limits a single tile.
//  * Q tiles: two TMA boxes each (64 dims, 128-byte swizzle) from q viewed as
//    [T][Hq][128].  K and V tiles of 128 keys = 8 pages, each page two TMA
//    boxes of 16 rows x 64 dims from the pool viewed as [NB*Hkv*16][128];
//    page ids come from the block table, pages past the sequence are skipped.
//    K/V tiles are double-buffered: tile i+1 loads while tile i computes.
//  * S = Q K^T: per Q tile 8 tcgen05.mma (M=128, N=128, K=16, bf16 in, fp32
//    out) into that tile's TMEM columns (0..127 / 128..255); both operands
//    K-major in shared memory.
//  * Softmax: threads t and t+128 own TMEM lane t%128 (query row t%128), 64
//    score columns each: tcgen05.ld, bottom-right causal mask, exp2 against
//    the running max in the log2 domain, row max exchanged through shared
//    memory.  The running max only moves when a score exceeds it by more than
//    kTau (then the pass is redone and O in TMEM is rescaled), so most tiles
//    take one pass.  P is stored into TMEM over the
//    thread's own S columns (two bf16 per 32-bit column, row = lane), where
//    the PV MMA reads its A operand: no shared-memory traffic for P.  P goes
//    in as two bf16 terms, the rounded value and the rounded remainder
//    (p - bf16(p), exact in fp32), each in half of the thread's 64 S columns,
//    so the rounding of P costs no accuracy (2^-16 of P instead of 2^-8).
//  * O += P V: per Q tile 16 tcgen05.mma (A from TMEM; 8 for each term of P)
//    into TMEM columns 256..383 / 384..511; V is the N-major (dims contiguous) operand in shared
//    memory.  V rows past the sequence end are zeroed in shared memory first
//    so stale pool contents cannot reach O.
//  * Warp roles: warps 0-7 run the softmax of the two Q tiles in turn; warp 8
//    loads K tiles, warp 9 loads V tiles (each refills a buffer as soon as
//    the MMAs that read it are done, with the next tiles' block ids
//    prefetched), warps 10 and 11 issue the tcgen05.mma of Q tile 0 and 1
//    (each whole warp runs its loop; one elected lane issues).
//    Pipeline per K/V tile i: PV(0, i) and S(0, i+1) run under the softmax of
//    Q tile 1, PV(1, i) and S(1, i+1) under the softmax of Q tile 0 for tile
//    i+1 (the S MMA that overwrites P is issued after the PV that reads it).  Hand-offs are
//    mbarriers: TMA complete_tx for K/V, tcgen05.commit for S done / PV
//    done, 256 softmax arrivals for P ready (one barrier per Q tile, so no
//    wait ever targets a phase more than one behind).
//  * Every mbarrier wait is bounded; on expiry the CTA flags
//    PKV_STATUS_TIMEOUT, lets its in-flight copies and MMAs land, frees TMEM
//    and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <climits>
#include <mutex>
#include <type_traits>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

constexpr int kPfSoftmaxThreads = 256;  // two threads per query row (64 score columns each)
constexpr int kPfThreads = kPfSoftmaxThreads + 128;  // + K-load, V-load and two MMA warps
// FP8 pages: four more warps, a second and a third widening warp for K and
// for V, so each operand's eight pages a tile are widened by three warps
// (pages 0-2, 3-5, 6-7).  The block's
// 512 threads launch with 128 registers each; the softmax warpgroups raise
// theirs to 160 and the other two lower theirs to 96 (2 x 128 x 160 +
// 2 x 128 x 96 = 65536, the launch's total, so the raise never waits on
// registers that are not there).
template <bool F8>
constexpr int kPfThreadsOf = F8 ? kPfThreads + 128 : kPfThreads;
constexpr int kPfPagesPerTile = kPfKeys / kPage;
constexpr uint32_t kTmemCols = 512;   // S/P of Q tile 0 [0,128), of tile 1 [128,256), O0 [256,384), O1 [384,512)
constexpr float kPfTau = 8.0f;

// Shared-memory map (offsets from a 1024-byte aligned base); P lives in TMEM.
constexpr uint32_t kHalfTile = 128 * 128;          // 128 rows x 64 bf16 = 16 KiB
// K and V tiles each have kKVBufs buffers: a tile's load is issued when the
// MMAs that read the same buffer kKVBufs tiles earlier are done, which covers
// the load latency of 8 random pages (about 1.3 us) at the tile cadence.
constexpr int kKVBufs = 2;
constexpr uint32_t kOffQ = 0;                                    // [2 Q tiles][2 halves]
constexpr uint32_t kOffK = kOffQ + 4 * kHalfTile;                // [bufs][2 halves]
constexpr uint32_t kOffV = kOffK + 2 * kKVBufs * kHalfTile;      // [bufs][2 halves]
constexpr uint32_t kOffMisc = kOffV + 2 * kKVBufs * kHalfTile;  // bf16 pages
// FP8 pages: one K/V tile of E4M3 codes (8 pages of 16 rows x 128 codes, as
// TMA lands them with 128-byte swizzle) and its 128 row scale bytes, for each
// of K and V, staged before the misc region.
constexpr uint32_t kStagePage = kPage * 128;
constexpr uint32_t kOffStageK = kOffMisc;
constexpr uint32_t kOffStageV = kOffStageK + kPfPagesPerTile * kStagePage;
constexpr uint32_t kOffScK = kOffStageV + kPfPagesPerTile * kStagePage;
constexpr uint32_t kOffScV = kOffScK + kPfPagesPerTile * kScaleBytes;
constexpr uint32_t kOffMiscF8 = kOffScV + kPfPagesPerTile * kScaleBytes;
template <bool F8>
constexpr uint32_t kMiscOf = F8 ? kOffMiscF8 : kOffMisc;
constexpr uint32_t kPfMisc = 1536;  // barriers, TMEM address, tile info, scan sums, row exchange
template <bool F8>
constexpr uint32_t kPfSmemOf = kMiscOf<F8> + kPfMisc + 1024;  // + alignment slack
static_assert(kPfSmemOf<true> <= 232448, "prefill shared memory above the 227 KiB per-CTA limit");

struct PrefillParams {
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* qsl;
  uint16_t* out;
  unsigned* status;
  int32_t B, T, Hkv, Hq, G, TM, max_blocks, num_blocks, split_max_q;
  float qscale;  // scale * log2(e)
  // shared-prefix pass: attend query rows to the first prefix_pages pages
  // (common to every block-table row) in chunks of chunk_tiles key tiles
  int32_t prefix_pages, chunk_tiles, chunks;
  float* prefix_part;  // [T][Hq][chunks] records of kPrefixRec floats
  // FP8 pages: row scale bytes [NB][Hkv][16] of K and V (null for bf16 pages)
  const uint8_t* k_scale;
  const uint8_t* v_scale;
  // Launched after the split-KV kernel of the same call, which runs on: every
  // CTA counts its exit here (the split-KV kernel stamped the word with this
  // epoch) and the last one waits for that kernel, so the call ends with
  // both.  Null when this pass runs first.
  unsigned long long* join;
  unsigned long long epoch;
};

// Exit of a CTA (thread 0): count it; the last of the grid waits for the
// split-KV kernel this pass was launched behind.
__device__ __forceinline__ void join_exit(const PrefillParams& p) {
  if (!p.join) return;
  const int total = int(gridDim.x * gridDim.y);  // < 32768 (checked on the host)
  const int before = arrive_stamped(p.join, p.epoch);
  if (before < 0) {
    flag_status(p.status, PKV_STATUS_TIMEOUT);
    return;
  }
  if (before + 1 == total) griddep_wait();
}

// ---------------------------------------------------------------------------
// tcgen05 / TMA helpers
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format: start
// address, leading and stride byte offsets in 16-byte units, version 1).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(b_mn_major) << 16) |
         (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// The MMA helpers are warp-collective: every lane of a converged warp runs
// them with the same operands and elect.sync picks the one lane that issues.
// Issued this way (the warp's loop uniform, the instruction predicated)
// rather than from one lane in a branch of its own, an MMA beside warps of
// FMA chains on the same sub-partition went from about 600 to about 190
// cycles, and beside a softmax-like mix from 70-76 to 64-66 (the tensor
// pipe's rate), in a one-SM probe.
__device__ __forceinline__ void umma(uint32_t tmem_d, uint64_t a, uint64_t b, uint32_t idesc,
                                     uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 l;\n\t"
      "elect.sync l|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem_d),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}

// Same, with the A operand (M rows x K, two bf16 per 32-bit column) in TMEM.
__device__ __forceinline__ void umma_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\t.reg .b32 l;\n\t"
      "elect.sync l|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(b), "r"(idesc), "r"(accumulate));
}

// Warp-collective too: the elected lane commits its MMAs to the barrier.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 l;\n\t"
      "elect.sync l|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31]));
}

__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Barrier over `threads` threads that also ORs a per-thread flag: every
// participant gets the same result.
__device__ __forceinline__ bool named_sync_or(int id, int threads, bool flag) {
  uint32_t res;
  asm volatile(
      "{\n\t.reg .pred pin, pout;\n\t"
      "setp.ne.u32 pin, %1, 0;\n\t"
      "bar.red.or.pred pout, %2, %3, pin;\n\t"
      "selp.u32 %0, 1, 0, pout;\n\t}"
      : "=r"(res)
      : "r"(uint32_t(flag)), "r"(id), "r"(threads)
      : "memory");
  return res != 0;
}

// Packed pairs of fp32 (element 0 in the low word) and the sm_100-family
// instructions that work on both lanes of a pair at once.
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_split(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
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
__device__ __forceinline__ uint64_t f2_sub(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
// Largest of three (NaN operands ignored, like fmaxf).
__device__ __forceinline__ float max3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// Bulk copy global -> shared (16-byte aligned, a multiple of 16 bytes).
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Four E4M3 codes (lowest byte first) -> two f16x2 (exact: E4M3 is a subset of f16).
__device__ __forceinline__ void e4m3x4_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

// f16 pair times a power of two -> bf16 pair (exact for E4M3 values under the
// row scales the FP8 write produces).
__device__ __forceinline__ uint32_t widen_pair(uint32_t h2, float sc) {
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
  return pack_bf16x2(f.x * sc, f.y * sc);
}

// Four E4M3 codes (lowest byte first) times 2^(scale-127) -> four bf16 (two
// pairs, lowest first), integer arithmetic only.  For a code with a nonzero
// exponent field E and mantissa m, the product is 2^(E-7) * (1 + m/8) *
// 2^(scale-127): bf16 exponent field E + scale - 7, mantissa m in its top
// three bits, the sign as is.  `adj` is (scale - 7) << 7 in both halves; it
// is exact for scale in [7, 246] (exponent fields 1..254) and codes with a
// nonzero exponent field (zero and subnormal codes take the f16 route).
__device__ __forceinline__ void widen4_int(uint32_t w, uint32_t adj, uint32_t& lo, uint32_t& hi) {
  const uint32_t p0 = __byte_perm(w, 0u, 0x1404u);  // codes 0, 1 in the high byte of each half
  const uint32_t p1 = __byte_perm(w, 0u, 0x3424u);  // codes 2, 3
  lo = (((p0 >> 4) & 0x07F007F0u) + adj) | (p0 & 0x80008000u);
  hi = (((p1 >> 4) & 0x07F007F0u) + adj) | (p1 & 0x80008000u);
}

// Nonzero when some code of w has a zero exponent field (zero or subnormal).
__device__ __forceinline__ uint32_t zero_field(uint32_t w) {
  const uint32_t t = w & 0x78787878u;
  return (t - 0x01010101u) & ~t & 0x80808080u;
}

// Same through f16 (exact for every finite code and any scale byte).
__device__ __forceinline__ void widen4_f16(uint32_t w, float sc, uint32_t& lo, uint32_t& hi) {
  uint32_t a0, a1;
  e4m3x4_f16x2(w, a0, a1);
  lo = widen_pair(a0, sc);
  hi = widen_pair(a1, sc);
}

// One lane's half row of an FP8 page: codes of dims 64h..64h+63 of row r (the
// staged page as TMA laid it out, 128-byte swizzle) times 2^(scale-127), as
// bf16 into row `drow` of the half-h block of a K/V tile (128-byte swizzle,
// row index = key within the tile, congruent to r mod 8).  The chunk order
// c = cc ^ 4h keeps each quarter-warp's 16-byte stores on distinct banks.
// One branch per lane: the integer route when the scale byte and every code
// allow it (nearly always), else the f16 route.  Words are picked with
// compile-time indices (a select on h), so w[] stays in registers.
__device__ __forceinline__ void widen_row_half(const uint8_t* spage, uint32_t sbyte, uint8_t* drow,
                                               int r, int h) {
  uint32_t w[16];  // codes of dims 64h + 4k .. 64h + 4k + 3
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 v = *reinterpret_cast<const uint4*>(spage + r * 128 + (((4 * h + i) ^ (r & 7)) << 4));
    w[4 * i] = v.x;
    w[4 * i + 1] = v.y;
    w[4 * i + 2] = v.z;
    w[4 * i + 3] = v.w;
  }
  uint32_t z = 0;
#pragma unroll
  for (int k = 0; k < 16; ++k) z |= zero_field(w[k]);
  if (z == 0u && sbyte >= 7u && sbyte <= 246u) {
    const uint32_t adj = ((sbyte - 7u) << 7) * 0x00010001u;
#pragma unroll
    for (int cc = 0; cc < 8; ++cc) {
      const int c = cc ^ (h << 2);  // dims 8c..8c+7 of the half
      const uint32_t wa = h ? w[2 * (cc ^ 4)] : w[2 * cc];
      const uint32_t wb = h ? w[2 * (cc ^ 4) + 1] : w[2 * cc + 1];
      uint4 o;
      widen4_int(wa, adj, o.x, o.y);
      widen4_int(wb, adj, o.z, o.w);
      *reinterpret_cast<uint4*>(drow + ((c ^ (r & 7)) << 4)) = o;
    }
  } else {
    const float sc = __uint_as_float(sbyte << 23);  // 2^(sbyte-127); byte 0 is never written
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint4 o;
      widen4_f16(w[2 * c], sc, o.x, o.y);
      widen4_f16(w[2 * c + 1], sc, o.z, o.w);
      *reinterpret_cast<uint4*>(drow + ((c ^ (r & 7)) << 4)) = o;
    }
  }
}

// ---------------------------------------------------------------------------
// kernel
// ---------------------------------------------------------------------------
// PREFIX = false: chunked prefill (bottom-right causal, normalised output).
// PREFIX = true: every query row against the shared prefix keys, written as
// log-sum-exp partial records that the split-KV kernel merges.
template <bool PREFIX, bool F8>
__global__ void __launch_bounds__(kPfThreadsOf<F8>, 1)
    pkv_prefill_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, PrefillParams p) {
  extern __shared__ uint8_t smem_raw[];
  // Run first (join == null): let the split-KV kernel that follows start on
  // the SMs this grid leaves free, beside this compute-bound pass (it reads
  // nothing this writes, and waits for this grid before it exits).  Mixed
  // step 329 -> 306 us.  Not for the shared-prefix pass: there it made the
  // step 6 % slower.  Run behind split-KV: no early start for what follows
  // (the next call's split-KV kernel would stamp its counters while this
  // call's still merges); it launches once every CTA here has exited, the
  // last of them after the split-KV kernel completed.
  if constexpr (!PREFIX) {
    if (!p.join) griddep_launch_dependents();
  }
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm + kOffQ;  // [tile u][2 halves]
  uint8_t* sK = sm + kOffK;
  uint8_t* sV = sm + kOffV;
  // misc region: barriers, TMEM address, tile info, scan sums, row exchange
  constexpr uint32_t kOffM = kMiscOf<F8>;
  constexpr int kNT = kPfThreadsOf<F8>;
  constexpr int kBars = 7 + 6 * kKVBufs + 6;
  static_assert(kBars * 8 <= 256 && 272 + 4 * (kNT / 32) <= 384 && 384 + 2 * 128 * 4 <= kPfMisc,
                "prefill misc region layout");
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + kOffM);
  uint64_t* bar_q = bars;                     // both Q tiles landed
  uint64_t* bar_s = bars + 1;                 // [2] S of Q tile u computed into its TMEM columns
  uint64_t* bar_o = bars + 3;                 // [2] PV of Q tile u done
  uint64_t* bar_p = bars + 5;                 // [2] P of Q tile u written by the softmax (256 arrivals)
  uint64_t* bar_k = bars + 7;                 // [kKVBufs] K tile landed in buffer b
  uint64_t* bar_v = bar_k + kKVBufs;          // [kKVBufs] V tile landed in buffer b
  uint64_t* bar_kfree = bar_v + kKVBufs;          // [kKVBufs][2] the S MMAs of Q tile u reading K buffer b are done
  uint64_t* bar_vfree = bar_kfree + 2 * kKVBufs;  // [kKVBufs][2] the PV MMAs of Q tile u reading V buffer b are done
  uint64_t* bar_kst = bar_vfree + 2 * kKVBufs;     // FP8: [3 slices] a K tile's codes and scales staged
  uint64_t* bar_vst = bar_kst + 3;                 // FP8: [3 slices] a V tile's codes and scales staged
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(sm + kOffM + 256);  // after 32 barrier slots
  int* s_info = reinterpret_cast<int*>(sm + kOffM + 264);  // b, t0
  int* s_scan = reinterpret_cast<int*>(sK);  // plan scratch (before any K tile lands)
  int* s_wsum = reinterpret_cast<int*>(sm + kOffM + 272);  // [warps] scan sums (up to 16 warps)

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = blockIdx.x;  // kv head; blockIdx.y = query group (real groups dispatch first)
  // query tokens of the CTA: two Q tiles of TM tokens x G heads (the shared-
  // prefix pass keeps one tile per CTA: its key windows are short chunks)
  const int TG = PREFIX ? p.TM : 2 * p.TM;

  // ---- plan: this CTA's query rows and key window ----------------------------
  int b = -1, t0 = 0, q_tok0 = 0, kbeg = 0, nkv = 0, key_end = 0, n = 0, L = 0, nt = 2;
  const int32_t* bt_row = p.block_tables;  // shared prefix: any row; row 0
  if constexpr (PREFIX) {
    const int qgroups = (p.T + TG - 1) / TG;
    const int i = int(blockIdx.y);
    if (i >= qgroups * p.chunks) return;
    const int qt = i / p.chunks, c = i - qt * p.chunks;
    const int ntiles = (p.prefix_pages * kPage + kPfKeys - 1) / kPfKeys;
    q_tok0 = qt * TG;
    nt = 1;
    kbeg = c * p.chunk_tiles;
    nkv = min(p.chunk_tiles, ntiles - kbeg);
    key_end = p.prefix_pages * kPage;
    b = c;  // chunk index (record slot)
    if (nkv <= 0) return;
  } else {
    const int per = (p.B + kNT - 1) / kNT;
    const int b0 = min(p.B, tid * per), b1 = min(p.B, b0 + per);
    int local = 0;
    for (int bb = b0; bb < b1; ++bb) {
      const int qq0 = __ldg(p.qsl + bb), q1 = __ldg(p.qsl + bb + 1), LL = __ldg(p.seq_lens + bb);
      const int nn = q1 - qq0;
      const bool bad = qq0 < 0 || nn < 0 || q1 > p.T || nn > LL || LL < 0 ||
                       (LL + kPage - 1) / kPage > p.max_blocks || (bb == 0 && qq0 != 0);
      const int groups = (!bad && nn > p.split_max_q) ? (nn + TG - 1) / TG : 0;
      s_scan[bb] = groups;
      local += groups;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_wsum[warp] = incl;
    __syncthreads();
    int base = 0, total = 0;
#pragma unroll
    for (int x = 0; x < kNT / 32; ++x) {
      if (x < warp) base += s_wsum[x];
      total += s_wsum[x];
    }
    int run = base + incl - local;
    for (int bb = b0; bb < b1; ++bb) {
      const int c = s_scan[bb];
      s_scan[bb] = run;
      run += c;
    }
    if (tid == 0) s_scan[p.B] = total;
    __syncthreads();
    if (tid == 0) {
      // heavier groups (later sequences, later query blocks) first
      const int i = total - 1 - int(blockIdx.y);
      int bb = -1, tt = 0;
      if (i >= 0) {
        int lo = 0, hi = p.B;  // last b with s_scan[b] <= i
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (s_scan[mid] <= i) lo = mid; else hi = mid;
        }
        bb = lo;
        tt = (i - s_scan[lo]) * TG;
      }
      s_info[0] = bb;
      s_info[1] = tt;
    }
    __syncthreads();
    b = s_info[0];
    if (b < 0) {  // no work for this CTA (before any TMEM is taken)
      if (tid == 0) join_exit(p);
      return;
    }
    t0 = s_info[1];
    const int q0 = __ldg(p.qsl + b);
    n = __ldg(p.qsl + b + 1) - q0;
    L = __ldg(p.seq_lens + b);
    q_tok0 = q0 + t0;
    nt = n - t0 > p.TM ? 2 : 1;
    key_end = L;
    const int max_pos = L - n + min(n, t0 + nt * p.TM) - 1;
    nkv = max_pos / kPfKeys + 1;
    bt_row = p.block_tables + int64_t(b) * p.max_blocks;
  }
  const int npages = (key_end + kPage - 1) / kPage;

  // ---- barriers and TMEM -----------------------------------------------------
  if (tid == 0) {
    // each barrier initialised once: P ready takes the 256 softmax arrivals,
    // a K or V tile on FP8 pages the arrivals of its three widening warps,
    // every other barrier one arrival (a TMA transaction or a commit)
    for (int i = 0; i < kBars; ++i) {
      const bool kv = bars + i >= bar_k && bars + i < bar_k + 2 * kKVBufs;
      mbar_init(bars + i, (bars + i == bar_p || bars + i == bar_p + 1) ? kPfSoftmaxThreads : (F8 && kv) ? 3 : 1);
    }
    fence_mbar_init();
  }
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(s_tmem)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t lane_off = uint32_t((warp & 3) * 32) << 16;  // warp w reads TMEM lanes 32*(w%4)..
  // Q tile u: S (fp32) and, over the same columns once S is consumed, P
  // (bf16 pairs; the half of the row a softmax thread owns starts its P at
  // the start of its own S columns); O of tile u at 256 + 128u
  auto tmem_s = [&](int u) { return tmem + uint32_t(u) * 128; };
  auto tmem_o = [&](int u) { return tmem + 256 + uint32_t(u) * 128; };
  const uint32_t idesc_s = idesc_bf16(128, 128, false);
  const uint32_t idesc_o = idesc_bf16(128, 128, true);
  // 0: K loads, 1: V loads, 2 + u: MMA of Q tile u; < 0 softmax; FP8 pages:
  // 4 and 5 the second K and V widening warps, 6 and 7 the third
  const int role = warp - kPfSoftmaxThreads / 32;
  // With FP8 pages the loader warps widen every tile and set the pace; the
  // softmax and MMA warps, which share their sub-partitions, sleep between
  // barrier tests instead of spinning.
  auto wait_idle = [&](uint64_t* bar, uint32_t parity) {
    return F8 ? mbar_wait_backoff(bar, parity, 256) : mbar_wait(bar, parity);
  };

  auto load_tile = [&](const CUtensorMap* map, uint8_t* base, uint64_t* bar, const int (&bids)[kPfPagesPerTile]) {
    int valid = 0;
#pragma unroll
    for (int j = 0; j < kPfPagesPerTile; ++j) valid += bids[j] >= 0;
    mbar_arrive_expect_tx(bar, uint32_t(valid) * 2 * 2048);
#pragma unroll
    for (int j = 0; j < kPfPagesPerTile; ++j) {
      if (bids[j] < 0) continue;  // past the window
      const int row = (bids[j] * p.Hkv + g) * kPage;
      tma_load_2d(base + j * 2048, map, 0, row, bar);
      tma_load_2d(base + kHalfTile + j * 2048, map, 64, row, bar);
    }
  };

  if (role >= 0) {
  // FP8 pages: the loader and MMA warps (two whole warpgroups) give up
  // registers here for the softmax warpgroups, which take them below
  if constexpr (F8) asm volatile("setmaxnreg.dec.sync.aligned.u32 96;");
  if (role == 0 || role == 1 || (F8 && role >= 4)) {
    // ===== K or V producer (lane 0 issues; the warp fetches block ids) =====
    // FP8 pages: slice 0 (roles 0, 1) widens pages 0-2 of each tile, slice 1
    // (roles 4, 5) pages 3-5, slice 2 (roles 6, 7) pages 6-7, each with its
    // own staging barrier; all three arrive on the tile's barrier.
    const int op = role & 1, slice = role < 2 ? 0 : (role - 2) >> 1;
    const int j0 = F8 ? (slice == 0 ? 0 : slice == 1 ? 3 : 6) : 0;
    const int j1 = F8 ? (slice == 0 ? 3 : slice == 1 ? 6 : kPfPagesPerTile) : kPfPagesPerTile;
    // Buffer kt % kKVBufs is free once the MMAs that read tile kt - kKVBufs
    // are done (the S of every Q tile for K, their PV for V; each buffer has
    // its own barrier, so no wait targets a phase more than one behind).
    // Block ids come in groups of four tiles, one page per lane, read a group
    // ahead: a tile's copies never wait on a block-table read.
    const CUtensorMap* map = op == 0 ? &tm_k : &tm_v;
    uint8_t* base0 = op == 0 ? sK : sV;
    uint64_t* bar_load = op == 0 ? bar_k : bar_v;
    uint64_t* bar_free = op == 0 ? bar_kfree : bar_vfree;
    if (role == 0 && lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tm_q)) : "memory");
      mbar_arrive_expect_tx(bar_q, uint32_t(nt) * 2 * kHalfTile);
      for (int u = 0; u < (kDropFirstCopy ? 0 : nt); ++u)
        for (int h = 0; h < 2; ++h)
          tma_load_3d(sQ + (u * 2 + h) * kHalfTile, &tm_q, h * 64, g * p.G, q_tok0 + u * p.TM, bar_q);
    }
    // lane l: page l % 8 of tile 4 * grp + l / 8 of this CTA's window; -1
    // past the window (no copy).  A table entry inside the window that is
    // not a page of the pool (negative, or num_blocks and up) is flagged and
    // page 0 is read in its place, so every id returned for a live page is
    // in the pool.
    auto group_id = [&](int grp) {
      const int kt = grp * 4 + lane / kPfPagesPerTile;
      const int pi = (kbeg + kt) * kPfPagesPerTile + lane % kPfPagesPerTile;
      if (kt >= nkv || pi >= npages) return -1;
      int bid = __ldg(bt_row + pi);
      if (bid < 0 || bid >= p.num_blocks) {
        flag_status(p.status, PKV_STATUS_BAD_BLOCK);
        bid = 0;
      }
      return bid;
    };
    int cur_g = group_id(0);
    int next_g = nkv > 4 ? group_id(1) : -1;
    int loaded = 0;
    bool ok = true;
    // FP8 pages: the tile's codes and scales go to a staging area first (lane
    // 0 issues), and the warp widens them into the bf16 tile buffer.
    uint8_t* stage = sm + (op == 0 ? kOffStageK : kOffStageV);
    uint8_t* ssc = sm + (op == 0 ? kOffScK : kOffScV);
    const uint8_t* scl = op == 0 ? p.k_scale : p.v_scale;
    uint64_t* bar_st = (op == 0 ? bar_kst : bar_vst) + slice;  // this slice's pages j0..j1-1
    int st_pending = -1;  // tile whose staging copies are out and not yet waited for
    auto arm_stage = [&](const int (&bids)[kPfPagesPerTile]) {
      int valid = 0;
#pragma unroll
      for (int j = 0; j < kPfPagesPerTile; ++j) valid += j >= j0 && j < j1 && bids[j] >= 0;
      mbar_arrive_expect_tx(bar_st, uint32_t(valid) * (kStagePage + kScaleBytes));
    };
    auto stage_page = [&](int j, int bid) {
      tma_load_2d(stage + j * kStagePage, map, 0, (bid * p.Hkv + g) * kPage, bar_st);
      bulk_copy(ssc + j * kScaleBytes, scl + (size_t(bid) * p.Hkv + g) * kScaleBytes, kScaleBytes, bar_st);
    };
    if constexpr (F8) {
      int ids0[kPfPagesPerTile];
#pragma unroll
      for (int j = 0; j < kPfPagesPerTile; ++j) ids0[j] = __shfl_sync(0xffffffffu, cur_g, j);
      if (lane == 0) {
        arm_stage(ids0);
        for (int j = j0; j < j1; ++j)
          if (ids0[j] >= 0) stage_page(j, ids0[j]);
      }
      st_pending = 0;
    }
    for (int kt = 0; kt < nkv; ++kt) {
      if (kt > 0 && (kt & 3) == 0) {
        cur_g = next_g;  // read four tiles ago
        next_g = kt + 4 < nkv ? group_id(kt / 4 + 1) : -1;
      }
      int ids[kPfPagesPerTile];
#pragma unroll
      for (int j = 0; j < kPfPagesPerTile; ++j) ids[j] = __shfl_sync(0xffffffffu, cur_g, (kt & 3) * 8 + j);
      const int kb = kt % kKVBufs;
      // the buffer is free once the MMA lane of every Q tile released it
      if (lane == 0 && kt >= kKVBufs)
        for (int u = 0; u < nt && ok; ++u) ok = mbar_wait(bar_free + kb * 2 + u, ((kt / kKVBufs) - 1) & 1);
      if (!__shfl_sync(0xffffffffu, int(ok), 0)) {
        ok = false;
        break;
      }
      if constexpr (!F8) {
        if (lane == 0) load_tile(map, base0 + kb * 2 * kHalfTile, bar_load + kb, ids);
      } else {
        // block ids of the next tile: its staging copies go out page by page
        // as this tile's pages are widened.  Ids come by shuffle inside the
        // (rolled) page loop, which keeps this role's code small.
        const int kn = kt + 1;
        const int src_g = (kn & 3) == 0 ? next_g : cur_g;
        const int cur_lane0 = (kt & 3) * 8, nxt_lane0 = (kn & 3) * 8;
        const uint32_t nvalid_mask = __ballot_sync(0xffffffffu, src_g >= 0);
        // every lane reads the staged bytes, so every lane waits
        if (!__all_sync(0xffffffffu, mbar_wait(bar_st, kt & 1))) {
          ok = false;
          break;
        }
        st_pending = -1;
        if (kn < nkv) {
          if (lane == 0) {
            const int valid = __popc((nvalid_mask >> (nxt_lane0 + j0)) & ((1u << (j1 - j0)) - 1u));
            mbar_arrive_expect_tx(bar_st, uint32_t(valid) * (kStagePage + kScaleBytes));
          }
          st_pending = kn;
        }
        uint8_t* dst = base0 + kb * 2 * kHalfTile;
        const int r = lane >> 1, h = lane & 1;
#pragma unroll 1
        for (int j = j0; j < j1; ++j) {
          const int idj = __shfl_sync(0xffffffffu, cur_g, cur_lane0 + j);
          const int nidj = __shfl_sync(0xffffffffu, src_g, nxt_lane0 + j);
          if (idj >= 0)
            widen_row_half(stage + j * kStagePage, ssc[j * kScaleBytes + r],
                           dst + h * kHalfTile + (j * kPage + r) * 128, r, h);
          __syncwarp();  // every lane has consumed the slot's codes: the copy may rewrite it
          if (lane == 0 && kn < nkv && nidj >= 0) stage_page(j, nidj);
        }
        fence_proxy_async_smem();  // widened rows -> visible to the tensor cores
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_load + kb);
      }
      ++loaded;
    }
    if (lane == 0) {
      // copies land before the CTA's shared memory is released
      for (int k = max(0, loaded - kKVBufs); k < loaded; ++k)
        mbar_wait(bar_load + k % kKVBufs, (k / kKVBufs) & 1, ok ? kLandLimitNs : kDrainLimitNs);
      if (F8 && st_pending >= 0) mbar_wait(bar_st, st_pending & 1, ok ? kLandLimitNs : kDrainLimitNs);
      if (!ok) flag_status(p.status, PKV_STATUS_TIMEOUT);
    }
    __syncwarp();
  } else if (role == 2 || role == 3) {
    // ===== MMA issuers: one warp per Q tile =====
    // Per K/V tile kt: PV(u, kt) as soon as P(u, kt) is written, then S(u,
    // kt+1) into the same TMEM columns (issued after the PV that reads P
    // there).  The two Q tiles have their own issuing warps, so one tile's
    // hand-offs never hold up the other's MMAs.  The whole warp runs the
    // loop and waits; one elected lane issues each MMA and commit.
    const int u = role - 2;
    // every lane waits; the warp goes on only if all of them saw the phase
    auto wait_all = [&](uint64_t* bar, uint32_t parity) {
      return __all_sync(0xffffffffu, wait_idle(bar, parity));
    };
    if (u < nt) {
      auto issue_s = [&](int kt) {
        const int kb = kt % kKVBufs;
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const int h = ks >> 2, kk = ks & 3;
          const uint64_t a = smem_desc(smem_u32(sQ + (u * 2 + h) * kHalfTile) + kk * 32, 16, 1024);
          const uint64_t bdesc = smem_desc(smem_u32(sK + (kb * 2 + h) * kHalfTile) + kk * 32, 16, 1024);
          umma(tmem_s(u), a, bdesc, idesc_s, ks > 0);
        }
        umma_commit(bar_s + u);
        umma_commit(bar_kfree + kb * 2 + u);
      };
      int ns = 0, npv = 0;  // S and PV groups issued (for the drain on failure)
      bool ok = wait_all(bar_q, 0) && wait_all(bar_k, 0);
      if (ok) {
        issue_s(0);
        ++ns;
      }
      for (int it = 0; ok && it < nkv; ++it) {
        const int vb = it % kKVBufs;
        // P(u, it) written by the softmax; V(it) landed
        if (!(ok = wait_all(bar_p + u, it & 1) && wait_all(bar_v + vb, (it / kKVBufs) & 1))) break;
        tc_fence_after();
        // 16 keys = 8 packed TMEM columns of P; the remainder term of the
        // same keys sits 32 columns on
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) {
          const int k16 = ks & 7;
          const uint64_t bdesc = smem_desc(smem_u32(sV + vb * 2 * kHalfTile) + k16 * 2048, kHalfTile, 1024);
          umma_ts(tmem_o(u), tmem_s(u) + (k16 >> 2) * 64 + (ks >> 3) * 32 + (k16 & 3) * 8, bdesc, idesc_o,
                  (it > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(bar_o + u);
        umma_commit(bar_vfree + vb * 2 + u);
        ++npv;
        if (it + 1 < nkv) {
          if (!(ok = wait_all(bar_k + (it + 1) % kKVBufs, ((it + 1) / kKVBufs) & 1))) break;
          issue_s(it + 1);
          ++ns;
        }
      }
      if (!ok && lane == 0) flag_status(p.status, PKV_STATUS_TIMEOUT);
      // this warp's newest commits land before TMEM is released, whatever
      // the softmax threads' waits saw (the warp stays converged, so
      // elect.sync picks the same lane for every MMA and commit, and each
      // commit covers all of that lane's earlier MMAs; at most one phase of
      // either barrier is pending)
      if (ns > 0) mbar_wait(bar_s + u, (ns - 1) & 1, ok ? kLandLimitNs : kDrainLimitNs);
      if (npv > 0) mbar_wait(bar_o + u, (npv - 1) & 1, ok ? kLandLimitNs : kDrainLimitNs);
    }
    __syncwarp();
  }
  } else {
    if constexpr (F8) asm volatile("setmaxnreg.inc.sync.aligned.u32 160;");
    // ===== softmax warps: Q tiles 0 and 1 in turn =====
    const int r = tid & 127;  // query row == TMEM lane
    const int ch = tid >> 7;  // which 64 of the 128 score columns
    const int t_rel = r / p.G;
    // keys visible to row r of tile u: the prefix pass sees the whole window
    bool row_valid[2];
    int pos[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int tu = u * p.TM + t_rel;
      row_valid[u] = u < nt && (PREFIX ? q_tok0 + tu < p.T : t0 + tu < n);
      pos[u] = PREFIX ? key_end - 1 : (row_valid[u] ? L - n + t0 + tu : L - 1);
    }
    // running max (same in both threads of a row) and half row sum, per tile
    float m0 = -INFINITY, l0 = 0.f, m1 = -INFINITY, l1 = 0.f;
    float* s_red = reinterpret_cast<float*>(sm + kOffM + 384);  // [2][128] exchange
    // ok: this thread's waits all succeeded.  stop: some softmax thread's
    // failed, decided at the same barrier by all 256 of them, so they leave
    // the loop together (the loop holds named barriers).
    bool ok = true, stop = false;
    for (int it = 0; it < nkv && !stop; ++it) {
      for (int u = 0; u < nt; ++u) {
        const int ph = it & 1;
        const int posu = u ? pos[1] : pos[0];
        float m = u ? m1 : m0;
        ok = wait_idle(bar_s + u, ph) && ok;
        tc_fence_after();
        // ---- this thread's 64 columns of row r ----
        const int kbase = (kbeg + it) * kPfKeys + ch * 64;
        // no masking in this half tile for any row of the warp: the pass below
        // runs warp-collective TMEM loads, so the choice must be warp-uniform
        const bool full = __all_sync(0xffffffffu, kbase + 63 <= posu);
        const uint32_t scol = tmem_s(u) + lane_off + ch * 64;
        uint32_t pk[2][16], pl[2][16];  // P as bf16 pairs, and the rounding remainders
        float mx = -INFINITY, rs = 0.f;
        // One pass over the 64 columns: exp2(s*scale - mref) packed to bf16,
        // optionally tracking the raw maximum.  FULL: no key of this half tile
        // is past the row's position (no masking work at all).
        // Key pairs go through packed fp32 instructions: one FMA for both
        // exponent arguments, one add into the pair of row sums, one
        // subtract for both remainders.
        auto pass = [&](float mref, auto full_t, auto track_t) {
          constexpr bool FULL = decltype(full_t)::value, TRACK = decltype(track_t)::value;
          const uint64_t qs2 = f2(p.qscale, p.qscale), nm2 = f2(-mref, -mref);
          uint64_t acc2[2] = {0ull, 0ull};  // (0, 0) pairs
          float mxl = -INFINITY;
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t sv[32];
            tmem_ld32(scol + c * 32, sv);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              float x0 = __uint_as_float(sv[2 * e]), x1 = __uint_as_float(sv[2 * e + 1]);
              if constexpr (!FULL) {
                const int k = kbase + c * 32 + 2 * e;
                if (k > posu) x0 = -INFINITY;
                if (k + 1 > posu) x1 = -INFINITY;
              }
              if constexpr (TRACK) mxl = max3(mxl, x0, x1);
              float t0, t1;
              f2_split(f2_fma(f2(x0, x1), qs2, nm2), t0, t1);
              const float a0 = ex2(t0), a1 = ex2(t1);  // exp2(-inf) = 0
              const uint64_t a2 = f2(a0, a1);
              acc2[e & 1] = f2_add(acc2[e & 1], a2);
              const uint32_t hi = pack_bf16x2(a0, a1);
              pk[c][e] = hi;
              float r0, r1;
              f2_split(f2_sub(a2, f2(bf_lo(hi), bf_hi(hi))), r0, r1);
              pl[c][e] = pack_bf16x2(r0, r1);
            }
          }
          float s0, s1, s2, s3;
          f2_split(acc2[0], s0, s1);
          f2_split(acc2[1], s2, s3);
          rs = (s0 + s1) + (s2 + s3);
          if constexpr (TRACK) mx = mxl;
        };
        if (full) pass(m, std::true_type{}, std::true_type{});
        else pass(m, std::false_type{}, std::true_type{});
        s_red[ch * 128 + r] = mx;
        named_sync(1, kPfSoftmaxThreads);
        const float row_mx = fmaxf(s_red[r], s_red[128 + r]) * p.qscale;
        // s_red may be rewritten next tile; a failed wait anywhere stops every
        // softmax thread here, together
        if (named_sync_or(2, kPfSoftmaxThreads, !ok)) {
          ok = false;
          stop = true;
          break;
        }
        const bool grow = row_mx > m + kPfTau;
        float alpha = 1.f;
        if (grow) {
          alpha = m == -INFINITY ? 0.f : ex2(m - row_mx);
          m = row_mx;
        }
        const bool warp_grow = __any_sync(0xffffffffu, grow);
        // redo the pass against the new maximum; warp-uniform (TMEM loads are
        // warp-collective), rows whose maximum did not move recompute the same P
        if (warp_grow) {
          // (the tracking variant again: one copy of the pass code less, and
          // its maximum is not used after the exchange)
          if (full) pass(m, std::true_type{}, std::true_type{});
          else pass(m, std::false_type{}, std::true_type{});
        }
        if (u) {
          m1 = m;
          l1 = l1 * alpha + rs;
        } else {
          m0 = m;
          l0 = l0 * alpha + rs;
        }
        // P (bf16 pairs) over this thread's own S columns: row r, keys
        // ch*64 .. ch*64+63 = 32 columns from the start of its half, and
        // their remainders in the next 32.  The other thread of the row may
        // still read its S half; this one is done with its own.
        {
          uint32_t pw[32];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            pw[e] = pk[0][e];
            pw[16 + e] = pk[1][e];
          }
          tmem_st32(scol, pw);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            pw[e] = pl[0][e];
            pw[16 + e] = pl[1][e];
          }
          tmem_st32(scol + 32, pw);
          tmem_wait_st();
        }
        // rescale this thread's 64 O columns when the running max moved; O is
        // final up to PV(u, it-1), which must have finished
        if (it > 0 && warp_grow) {
          const bool done = mbar_wait(bar_o + u, (it - 1) & 1);
          ok = ok && done;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t ov[32];
            tmem_ld32(tmem_o(u) + lane_off + ch * 64 + c * 32, ov);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) ov[e] = __float_as_uint(__uint_as_float(ov[e]) * alpha);
            tmem_st32(tmem_o(u) + lane_off + ch * 64 + c * 32, ov);
          }
          tmem_wait_st();
        }
        // keys past the sequence end: zero their V rows (after V landed, once
        // per K/V tile, before the first PV reads them) so stale pool contents
        // cannot leak through P = 0
        if (u == 0 && (kbeg + it + 1) * kPfKeys > key_end) {
          const int vb = it % kKVBufs;
          ok = mbar_wait(bar_v + vb, (it / kKVBufs) & 1) && ok;
          if ((kbeg + it) * kPfKeys + r >= key_end) {
            uint4* vrow = reinterpret_cast<uint4*>(sV + (vb * 2 + ch) * kHalfTile + r * 128);
#pragma unroll
            for (int q = 0; q < 8; ++q) vrow[q] = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar_p + u);  // P(u, it) is ready for the MMA warp
      }
    }
    // ---- epilogue per Q tile: O / l -> bf16, each thread its 64 columns of row r ----
    for (int u = 0; u < nt; ++u) {
      ok = ok && mbar_wait(bar_o + u, (nkv - 1) & 1);
      named_sync(1, kPfSoftmaxThreads);  // s_red of the previous use is read
      s_red[ch * 128 + r] = u ? l1 : l0;
      named_sync(1, kPfSoftmaxThreads);
      tc_fence_after();
      const float lsum = s_red[r] + s_red[128 + r];
      const int tok = q_tok0 + u * p.TM + t_rel;
      const bool valid = (u ? row_valid[1] : row_valid[0]) && ok;
      if constexpr (PREFIX) {
        // partial record: o (unnormalised, 128 floats), running max m, sum l
        float* rec = p.prefix_part + ((size_t(tok) * p.Hq + g * p.G + (r % p.G)) * p.chunks + b) * kPrefixRec;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t ov[32];
          tmem_ld32(tmem_o(u) + lane_off + ch * 64 + c * 32, ov);
          tmem_wait_ld();
          if (valid) {
            float4* dst = reinterpret_cast<float4*>(rec + ch * 64 + c * 32);
#pragma unroll
            for (int q = 0; q < 8; ++q)
              dst[q] = make_float4(__uint_as_float(ov[4 * q]), __uint_as_float(ov[4 * q + 1]),
                                   __uint_as_float(ov[4 * q + 2]), __uint_as_float(ov[4 * q + 3]));
          }
        }
        if (valid && ch == 0) {
          rec[128] = u ? m1 : m0;
          rec[129] = lsum;
        }
      } else {
        const float inv = 1.f / lsum;
        uint16_t* orow = p.out + (size_t(tok) * p.Hq + g * p.G + (r % p.G)) * kHeadDim + ch * 64;
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          uint32_t ov[32];
          tmem_ld32(tmem_o(u) + lane_off + ch * 64 + c * 32, ov);
          tmem_wait_ld();
          if (valid) {
            uint4* dst = reinterpret_cast<uint4*>(orow + c * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t w4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w4[e] = pack_bf16x2(__uint_as_float(ov[8 * q + 2 * e]) * inv,
                                    __uint_as_float(ov[8 * q + 2 * e + 1]) * inv);
              dst[q] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
          }
        }
      }
    }
    if (!ok && tid == 0) flag_status(p.status, PKV_STATUS_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
  }
  if (tid == 0) join_exit(p);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    else
      cudaGetLastError();
  });
  return fn;
}

bool encode(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides, const cuuint32_t* box) {
  return encode_tensor_map(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims, strides, box);
}

}  // namespace

bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int rank,
                       const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box) {
  auto fn = encode_fn();
  if (!fn) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, dtype, rank, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Query tokens per tile: 128 rows / G heads.
static int tile_tokens(const pkv_desc& d) { return 128 / (d.num_q_heads / d.num_kv_heads); }

int prefill_max_tiles(const pkv_desc& d, int32_t num_seqs, int32_t num_tokens) {
  // every sequence may end in a partial tile
  const int tm = tile_tokens(d);
  return (num_tokens + tm - 1) / tm + num_seqs;
}

template <bool PREFIX, bool F8>
static int ensure_prefill_attr(int device) {
  static bool done[64] = {};
  if (device < 0 || device >= 64) return PKV_ERR_DEVICE;
  if (!done[device]) {
    if (cudaFuncSetAttribute(pkv_prefill_kernel<PREFIX, F8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             int(kPfSmemOf<F8>)) != cudaSuccess) {
      cudaGetLastError();
      return PKV_ERR_LAUNCH;
    }
    if constexpr (F8) {
      // The warpgroups' register split (softmax up to 160, the rest down to
      // 96) needs the block launched with at least 128 registers a thread:
      // with fewer, the softmax warpgroups' raise would wait for registers
      // that never come.  Refuse to launch a build where that is not so.
      cudaFuncAttributes fa{};
      if (cudaFuncGetAttributes(&fa, pkv_prefill_kernel<PREFIX, F8>) != cudaSuccess) {
        cudaGetLastError();
        return PKV_ERR_LAUNCH;
      }
      if (fa.numRegs * kPfThreadsOf<F8> < 2 * 128 * 160 + 2 * 128 * 96) return PKV_ERR_LAUNCH;
    }
    done[device] = true;
  }
  return PKV_OK;
}

static int make_maps(const AttendArgs& a, CUtensorMap* tq, CUtensorMap* tk, CUtensorMap* tv) {
  const pkv_desc& d = a.desc;
  const int G = d.num_q_heads / d.num_kv_heads;
  {
    const cuuint64_t dims[3] = {cuuint64_t(kHeadDim), cuuint64_t(d.num_q_heads), cuuint64_t(a.num_tokens)};
    const cuuint64_t strides[2] = {cuuint64_t(kHeadDim) * 2, cuuint64_t(d.num_q_heads) * kHeadDim * 2};
    const cuuint32_t box[3] = {64, cuuint32_t(G), cuuint32_t(tile_tokens(d))};
    if (!encode(tq, a.q, 3, dims, strides, box)) return PKV_ERR_LAUNCH;
  }
  const cuuint64_t rows = cuuint64_t(d.num_blocks) * d.num_kv_heads * kPage;
  if (a.fp8) {
    // E4M3 codes as [rows][128]: one box = one page of 16 rows
    const cuuint64_t dims[2] = {cuuint64_t(kHeadDim), rows};
    const cuuint64_t strides[1] = {cuuint64_t(kHeadDim)};
    const cuuint32_t box[2] = {cuuint32_t(kHeadDim), cuuint32_t(kPage)};
    if (!encode_tensor_map(tk, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.k_cache, 2, dims, strides, box) ||
        !encode_tensor_map(tv, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.v_cache, 2, dims, strides, box))
      return PKV_ERR_LAUNCH;
    return PKV_OK;
  }
  const cuuint64_t dims[2] = {cuuint64_t(kHeadDim), rows};
  const cuuint64_t strides[1] = {cuuint64_t(kHeadDim) * 2};
  const cuuint32_t box[2] = {64, cuuint32_t(kPage)};
  if (!encode(tk, a.k_cache, 2, dims, strides, box)) return PKV_ERR_LAUNCH;
  if (!encode(tv, a.v_cache, 2, dims, strides, box)) return PKV_ERR_LAUNCH;
  return PKV_OK;
}

static PrefillParams make_params(const LaunchCtx& ctx, const AttendArgs& a, int split_max_q) {
  const pkv_desc& d = a.desc;
  PrefillParams pp{};
  pp.block_tables = a.block_tables;
  pp.seq_lens = a.seq_lens;
  pp.qsl = a.query_start_loc;
  pp.out = a.out;
  pp.status = ctx.status;
  pp.B = a.num_seqs;
  pp.T = a.num_tokens;
  pp.Hkv = d.num_kv_heads;
  pp.Hq = d.num_q_heads;
  pp.G = d.num_q_heads / d.num_kv_heads;
  pp.TM = tile_tokens(d);
  pp.max_blocks = d.max_blocks_per_seq;
  pp.num_blocks = d.num_blocks;
  pp.split_max_q = split_max_q;
  pp.qscale = a.scale * 1.4426950408889634f;
  pp.k_scale = a.k_scale;
  pp.v_scale = a.v_scale;
  return pp;
}

int prefill_groups(const pkv_desc& d, int32_t num_seqs, int32_t num_tokens, int max_tiles) {
  // one CTA per group of two Q tiles; every sequence may end in a partial group
  const int tg = 2 * tile_tokens(d);
  return min(max_tiles, (num_tokens + tg - 1) / tg + num_seqs);
}

int launch_prefill(const LaunchCtx& ctx, const AttendArgs& a, int split_max_q, int max_tiles,
                   unsigned long long* join, unsigned long long epoch) {
  if (int e = a.fp8 ? ensure_prefill_attr<false, true>(ctx.dev->device)
                    : ensure_prefill_attr<false, false>(ctx.dev->device))
    return e;
  CUtensorMap tq, tk, tv;
  if (int e = make_maps(a, &tq, &tk, &tv)) return e;
  PrefillParams pp = make_params(ctx, a, split_max_q);
  pp.join = join;
  pp.epoch = epoch;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.desc.num_kv_heads, prefill_groups(a.desc, a.num_seqs, a.num_tokens, max_tiles));
  cfg.blockDim = dim3(a.fp8 ? kPfThreadsOf<true> : kPfThreadsOf<false>);
  cfg.dynamicSmemBytes = a.fp8 ? kPfSmemOf<true> : kPfSmemOf<false>;
  cfg.stream = ctx.stream;
  // behind the split-KV kernel: start once its CTAs let it (their pool reads
  // begin after pkv_write completed, and so do this pass's)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = join ? 1 : 0;
  TraceScope ts(ctx.stream, PKV_K_PREFILL);
  if (a.fp8)
    cudaLaunchKernelEx(&cfg, pkv_prefill_kernel<false, true>, tq, tk, tv, pp);
  else
    cudaLaunchKernelEx(&cfg, pkv_prefill_kernel<false, false>, tq, tk, tv, pp);
  return ts.done();
}

int prefix_chunks(const pkv_desc& d, int32_t num_tokens, int32_t prefix_pages, int* chunk_tiles) {
  if (prefix_pages <= 0 || num_tokens <= 0) {
    *chunk_tiles = 0;
    return 0;
  }
  const int tg = tile_tokens(d);  // query tokens per CTA of the prefix pass (one Q tile)
  const int qgroups = (num_tokens + tg - 1) / tg;
  const int ntiles = (prefix_pages * kPage + kPfKeys - 1) / kPfKeys;
  // split the prefix keys into as many chunks as keep the pass to one wave
  // (one CTA per SM, 152 SMs), at most 16 (the split-KV merge holds one chunk
  // per lane of a half warp)
  const int want = min(16, max(1, 152 / (qgroups * d.num_kv_heads)));
  const int per = max(1, (ntiles + want - 1) / want);
  *chunk_tiles = per;
  return (ntiles + per - 1) / per;
}

int launch_prefix(const LaunchCtx& ctx, const AttendArgs& a, float* records, int chunks,
                  int chunk_tiles) {
  if (int e = a.fp8 ? ensure_prefill_attr<true, true>(ctx.dev->device)
                    : ensure_prefill_attr<true, false>(ctx.dev->device))
    return e;
  CUtensorMap tq, tk, tv;
  if (int e = make_maps(a, &tq, &tk, &tv)) return e;
  PrefillParams pp = make_params(ctx, a, 0);
  pp.prefix_pages = a.shared_prefix_pages;
  pp.chunk_tiles = chunk_tiles;
  pp.chunks = chunks;
  pp.prefix_part = records;
  const int qgroups = (a.num_tokens + pp.TM - 1) / pp.TM;
  TraceScope ts(ctx.stream, PKV_K_PREFILL);
  if (a.fp8)
    pkv_prefill_kernel<true, true><<<dim3(a.desc.num_kv_heads, qgroups * chunks), kPfThreadsOf<true>,
                                     kPfSmemOf<true>, ctx.stream>>>(tq, tk, tv, pp);
  else
    pkv_prefill_kernel<true, false><<<dim3(a.desc.num_kv_heads, qgroups * chunks), kPfThreadsOf<false>,
                                      kPfSmemOf<false>, ctx.stream>>>(tq, tk, tv, pp);
  return ts.done();
}

}  // namespace pkv
