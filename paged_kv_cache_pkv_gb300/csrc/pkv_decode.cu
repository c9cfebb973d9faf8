// pkv_decode.cu -- split-KV paged attention for decode rows, with the work
// plan and the log-sum-exp merge of split partials fused into the same kernel.
//
// What is computed (llm-d blog post "What does production-grade LLM inference
// look like?", introduction: paged attention over a paged KV cache; decode is
// memory-bandwidth bound): for every query row r of a sequence whose query
// count is small (decode, or a short speculative chunk) and every query head
// h, softmax(scale * q_r,h . K^T) V over the row's visible keys, with K/V read
// page by page through the sequence's block table.
//
// Design (GB300):
//  * Work unit = one (query row, group of GH query heads sharing a kv head,
//    page).  A unit moves exactly one K page and one V page of one kv head
//    (pool layout [NB, Hkv, 16, 128] makes each one contiguous block: 4 KiB
//    in bf16, 2 KiB of FP8 codes); the GH query heads reuse that read (GQA).
//  * Plan: every CTA reads seq_lens / query_start_loc (tiny) and builds the
//    per-sequence unit prefix in shared memory; units are numbered row-major
//    and each decode warp takes an equal contiguous range, so 16-token and
//    32768-token sequences are balanced to within one page.
//  * Each warp is an independent worker with its own ring (2 stages for bf16
//    pages, 3 for FP8): the whole warp runs the copy issue and the lane
//    elect.sync picks issues the copies (L2 evict-first) that complete on an
//    mbarrier; all 32 lanes compute.  No CTA barrier sits on the page loop.
//  * Page products on warp-level MMAs (mma.sync m16n8k16, f32 accumulators)
//    fed straight from registers: S^T[16 tokens x 8 columns] = K . Q^T, then
//    O^T[128 dims x 8 columns] += V^T . P^T.  Column c < GH is query head c
//    of the group; column GH + c repeats head c (the same scores) and carries
//    the rounding remainder of its P, so P enters the PV product as two terms
//    (rounded value + rounded remainder) at no extra MMA: the flush adds the
//    two columns.  The contraction index of both products is permuted so that
//    every lane's operands are whole 16-byte pieces of shared memory: lane
//    (g, t) reads dims 32t..32t+31 of K rows g and g+8 and dims 16g..16g+15
//    of V rows 2t, 2t+1, 2t+8, 2t+9.  A tcgen05 MMA needs M >= 64 and its
//    operands in shared memory or TMEM; this product has M = 16 and its
//    operands come from registers, so the warp-level MMA is the fit.  It needs
//    about a quarter of the instructions of packed FMAs, which lets a CTA run
//    12 warps (168 registers) and hide more latency.
//  * bf16 pages: bf16 operands as stored (q too), P as two bf16 terms; a page
//    is one TMA tensor copy (the pool viewed as rows of 128 bytes, 128-byte
//    swizzle: conflict-free fragment reads).  FP8 pages (template flag F8):
//    2 KiB pages of E4M3 codes by the same kind of copy, plus 16-byte blocks
//    of per-row scale bytes (scale = 2^(byte-127)) by bulk copies; codes are widened exactly to f16 (E4M3 is a subset of f16), q is
//    scaled by a power of two into f16 range (exact), P is two f16 terms.  Row scales:
//    the K one multiplies the finished score; the V one weights the
//    probability relative to the largest V scale of the segment (a running
//    exponent, like the softmax maximum).
//  * Online softmax in the log2 domain (scores scaled by scale*log2 e); the
//    running maximum only moves when a score exceeds it by more than kTau (a
//    warp vote), so most pages skip the max reduction and the rescale.  P
//    moves from the score fragment to the PV operand fragment with 4 shuffles.
//  * A warp that sees a whole (row, head group) writes bf16 output directly.
//    A split one writes (m, l, o) to one of its two partial slots and bumps
//    an epoch-tagged arrival counter; the last warp to arrive merges the
//    partials (log-sum-exp) and writes the output.  The epoch is new on every
//    call, so the workspace never needs clearing.
//  * Beside the tensor-core prefill pass of the same call: this kernel is
//    launched first and its plan leaves the pass part of the SMs (sized from
//    the pass's tile steps against this kernel's units); the pass, launched
//    behind it, runs on those SMs at the same time.
#include <atomic>
#include <chrono>
#include <climits>
#include <cmath>
#include <type_traits>

#include <cuda_fp16.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

struct DecodeParams {
  const uint16_t* q;
  const uint8_t* k_cache;  // bf16 pages, or E4M3 codes for the FP8 variant
  const uint8_t* v_cache;
  const uint8_t* k_scale;  // FP8 only: [NB][Hkv][16] scale bytes
  const uint8_t* v_scale;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* qsl;
  uint16_t* out;
  float* partials;
  unsigned long long* counters;  // [T * Hkv * nsub * warps per ring] arrival counters
  unsigned* status;
  int32_t B, T, num_blocks, Hkv, Hq, G, nsub, max_blocks, simt_max_q, nwarps;
  float qscale;  // scale * log2(e)
  unsigned long long epoch;  // 48-bit call tag, never 0
  // 0 when the kernel right before this one is this call's chunked-prefill
  // pass, whose results this kernel never reads (its own inputs were
  // complete before that pass started): then it runs beside the pass, and
  // waits for it only before it exits, so that the call ends with both
  int32_t wait_prev;
  // 1 when this call's chunked-prefill pass is launched right after this
  // kernel: the plan leaves the pass some of the SMs (its K/V tile steps
  // times pf_cost against this kernel's units), and once the pool writes are
  // complete every CTA lets the pass launch.  `join` is the pass's exit
  // counter, stamped with the epoch here.
  // lead_sat: SMs at which this kernel's page stream saturates HBM (0: it
  // never does, i.e. it is bound by the SMs it runs on)
  int32_t lead, pf_cost, lead_sat;
  unsigned long long* join;
  // shared prefix: the first np pages of every row were attended by the
  // prefix pass, whose partial records (chunks per row and head) are merged
  int32_t np, chunks;
  const float* prefix_part;  // [T][Hq][chunks][kPrefixRec]
};

struct StageDesc {
  int32_t row, item, item_start, nvis;
};

// Bytes of one (page, kv head) of K (or V) in the pool.
template <bool F8>
constexpr int kPageBytesOf = F8 ? kPageBytesF8 : kPageBytes;

// One warp's page ring: K and V pages of each stage, copied by TMA with
// 128-byte swizzle (stages 1024-byte aligned).  A bf16 page is 32 units of
// 128 bytes (token row r = units 2r, 2r+1), an FP8 page 16 units (one per row).
template <bool F8>
struct DecRing {
  uint8_t kv[F8 ? kDecStagesF8 : kDecStages][2][F8 ? kPageBytesF8 : kPageBytes];
};
static_assert(sizeof(DecRing<false>) % 1024 == 0 && sizeof(DecRing<true>) % 1024 == 0,
              "ring stages stay 1024-byte aligned");
// Per-warp ring bookkeeping, kept apart from the aligned pages.
template <bool F8>
struct DecMeta {
  uint4 sc[F8 ? kDecStagesF8 : 1][2];  // FP8: K and V row scale bytes of a stage
  StageDesc desc[F8 ? kDecStagesF8 : kDecStages];
  uint64_t bar[F8 ? kDecStagesF8 : kDecStages];
};

// 2^(byte - 127) for a scale byte in [1, 254]; 0 for byte 0.
__device__ __forceinline__ float scale_of(uint32_t byte) { return __uint_as_float(byte << 23); }

// Exact widening of the four E4M3 codes of a word to two f16x2 words: bytes
// 0, 1 -> lo (byte 0 in the low half), bytes 2, 3 -> hi.
__device__ __forceinline__ void e4m3x4_to_f16x2(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi)
      : "r"(w));
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// (a, b) minus their f16 pair `rounded` (exact in fp32), rounded to f16.
__device__ __forceinline__ uint32_t f16_remainder(uint32_t rounded, float a, float b) {
  const float2 r = __half22float2(*reinterpret_cast<const __half2*>(&rounded));
  return pack_f16x2(a - r.x, b - r.y);
}

// D += A . B, m16n8k16, f16 operands, f32 accumulators (warp-collective).
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D += A . B, m16n8k16, bf16 operands, f32 accumulators (warp-collective).
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Bytes t and t+8 (t < 8) of a 16-byte vector, as two scale bytes.
__device__ __forceinline__ void bytes_t_t8(const uint4& v, int t, uint32_t& b0, uint32_t& b1) {
  const int sh = (t & 3) * 8;
  b0 = (((t & 4) ? v.y : v.x) >> sh) & 0xFFu;
  b1 = (((t & 4) ? v.w : v.z) >> sh) & 0xFFu;
}

// 16-byte chunk c of 128-byte unit u of a page copied with 128-byte swizzle.
__device__ __forceinline__ const uint4& swz(const uint8_t* page, int u, int c) {
  return *reinterpret_cast<const uint4*>(page + u * 128 + ((c ^ (u & 7)) << 4));
}

// 2D TMA tile load with an L2 cache hint.
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* map, int c0, int c1,
                                                 uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// Warp-collective forms of a page's copy issue: every lane of a converged
// warp runs them with the same operands and the lane elect.sync picks acts,
// so the warp never runs the issue code in one lane's branch of its own.
__device__ __forceinline__ void tma_load_2d_hint_w(void* dst, const CUtensorMap* map, int c0, int c1,
                                                   uint64_t* bar, uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 l;\n\telect.sync l|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;\n\t}" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_g2s_w(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                           uint64_t policy) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 l;\n\telect.sync l|e, 0xffffffff;\n\t"
      "@e cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;\n\t}" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx_w(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .b32 l;\n\telect.sync l|e, 0xffffffff;\n\t"
      "@e mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

constexpr int kDecThreads = kDecWarps * 32;
constexpr float kTau = 8.0f;  // log2-domain slack before the running max moves
// Fewest pages a decode warp is given.  Only batches with fewer pages than
// 4 per warp feel it: on the 4-sequence batch (L up to 255) 4 / 2 / 1 pages
// gave a 22.3 / 19.4 / 21.1 us step (one page each: more partials to merge).
constexpr int kMinChunk = 2;
constexpr unsigned kFull = 0xffffffffu;

// Sum over positions p in (0, x] of ceil(p / 16): pages of rows with those
// visible-key counts.
__device__ __forceinline__ long long pages_prefix(long long x) {
  const long long a = x / kPage, r = x % kPage;
  return kPage * a * (a + 1) / 2 + r * (a + 1);
}

// Producer cursor over a warp's units (all lanes hold identical copies).
struct Cursor {
  int b, j, item, page;     // sequence, its query row, head group, page
  int q0, n, L;             // sequence facts
  int nvis, npages;         // row facts
  int item_start;           // global unit index of (row, item, page 0)
  int bid;                  // block id of the current unit
};

// Sequence facts come from the shared-memory copies the plan made.
struct SeqSmem {
  const int* start;  // [B+1] unit prefix
  const int* q0;     // [B+1] query_start_loc
  const int* len;    // [B]   seq_lens
};

__device__ __forceinline__ void cursor_seq(Cursor& c, const SeqSmem& sq, int b) {
  c.b = b;
  c.q0 = sq.q0[b];
  c.n = sq.q0[b + 1] - c.q0;
  c.L = sq.len[b];
}

// Visible keys of the row and its own (suffix) pages after the shared prefix.
__device__ __forceinline__ void cursor_row(Cursor& c, int np) {
  c.nvis = c.L - c.n + c.j + 1;
  c.npages = (c.nvis + kPage - 1) / kPage - np;
}

__device__ __forceinline__ void cursor_bid(Cursor& c, const DecodeParams& p) {
  int bid = __ldg(p.block_tables + int64_t(c.b) * p.max_blocks + p.np + c.page);
  if (bid < 0 || bid >= p.num_blocks) {
    flag_status(p.status, PKV_STATUS_BAD_BLOCK);
    bid = 0;
  }
  c.bid = bid;
}

// The cursor one unit on, without reading the new unit's block id.
__device__ __forceinline__ void cursor_step(Cursor& c, int np, const SeqSmem& sq, int per_row) {
  if (++c.page == c.npages) {
    c.page = 0;
    c.item_start += c.npages;
    if (++c.item == per_row) {
      c.item = 0;
      if (++c.j == c.n) {
        c.j = 0;
        int b = c.b + 1;
        while (sq.start[b + 1] == sq.start[b]) ++b;
        cursor_seq(c, sq, b);
      }
      cursor_row(c, np);
    }
  }
}

__device__ __forceinline__ void cursor_advance(Cursor& c, const DecodeParams& p,
                                               const SeqSmem& sq, int per_row) {
  if (++c.page == c.npages) {
    c.page = 0;
    c.item_start += c.npages;
    if (++c.item == per_row) {
      c.item = 0;
      if (++c.j == c.n) {
        c.j = 0;
        int b = c.b + 1;
        while (sq.start[b + 1] == sq.start[b]) ++b;
        cursor_seq(c, sq, b);
      }
      cursor_row(c, p.np);
    }
  }
  cursor_bid(c, p);
}

// Log-sum-exp merge of the partials of one (row, head group) over warps
// w0..w1.  Lane i reads partial w0+i's maxima and sums (32 partials per
// round, reduced across the warp), then every lane accumulates 4 dims of each
// of the GH heads over all partials with independent loads.
// Record of the shared-prefix pass for (row, query head, chunk c).
__device__ __forceinline__ const float* prefix_rec(const DecodeParams& p, int row, int head, int c) {
  return p.prefix_part + ((size_t(row) * p.Hq + head) * p.chunks + c) * kPrefixRec;
}

// Shared-prefix records of (row, heads h0..h0+NH-1), read lane-parallel:
// lane c < chunks holds chunk c's maximum and sum of every head.
template <int NH>
struct PrefixFold {
  float pm[NH], pl[NH], w[NH];
  __device__ __forceinline__ void load(const DecodeParams& p, int lane, int row, int h0) {
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      const bool mine = lane < p.chunks;
      const float* rec = prefix_rec(p, row, h0 + h, mine ? lane : 0);
      pm[h] = mine ? __ldcg(rec + 128) : -INFINITY;
      pl[h] = mine ? __ldcg(rec + 129) : 0.f;
    }
  }
  // raise M[h] to the records' maximum
  __device__ __forceinline__ void max_into(float (&M)[NH]) const {
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      float x = pm[h];
#pragma unroll
      for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
      M[h] = fmaxf(M[h], x);
    }
  }
  // per-lane weights against the final M; adds the records' sums into L
  __device__ __forceinline__ void weigh(const float (&M)[NH], float (&L)[NH]) {
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      w[h] = pm[h] == -INFINITY ? 0.f : ex2(pm[h] - M[h]);
      float x = w[h] * pl[h];
#pragma unroll
      for (int o = 16; o; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
      L[h] += x;
    }
  }
};

template <int GH>
__device__ __forceinline__ void merge_item(const DecodeParams& p, int lane, int row, int h0,
                                           int item_start, int npages, int chunk) {
  const int w0 = item_start / chunk, w1 = (item_start + npages - 1) / chunk;
  const int nparts = w1 - w0 + 1;
  const int npre = p.np > 0 ? p.chunks : 0;  // shared-prefix records to fold in
  auto base_of = [&](int w) {
    return p.partials + size_t(2 * w + (item_start <= w * chunk ? 0 : 1)) * partial_floats(GH);
  };
  float M[GH], L[GH];
#pragma unroll
  for (int h = 0; h < GH; ++h) {
    M[h] = -INFINITY;
    L[h] = 0.f;
  }
  for (int k0 = 0; k0 < nparts; k0 += 32) {
    const int k = k0 + lane;
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      float mk = k < nparts ? __ldcg(base_of(w0 + k) + h) : -INFINITY;
#pragma unroll
      for (int o = 16; o; o >>= 1) mk = fmaxf(mk, __shfl_xor_sync(kFull, mk, o));
      M[h] = fmaxf(M[h], mk);
    }
  }
  PrefixFold<GH> pf;
  if (npre) {
    pf.load(p, lane, row, h0);
    pf.max_into(M);
  }
  float4 acc[GH];
#pragma unroll
  for (int h = 0; h < GH; ++h) acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int k0 = 0; k0 < nparts; k0 += 32) {
    const int k = k0 + lane;
    float sc_mine[GH];
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      const float* b = base_of(w0 + min(k, nparts - 1));
      const float sc = k < nparts ? ex2(__ldcg(b + h) - M[h]) : 0.f;
      float lk = sc * (k < nparts ? __ldcg(b + 4 + h) : 0.f);
#pragma unroll
      for (int o = 16; o; o >>= 1) lk += __shfl_xor_sync(kFull, lk, o);
      L[h] += lk;
      sc_mine[h] = sc;
    }
    const int cnt = min(32, nparts - k0);
#pragma unroll 4
    for (int i = 0; i < cnt; ++i) {
      const float* b = base_of(w0 + k0 + i);
#pragma unroll
      for (int h = 0; h < GH; ++h) {
        const float sc = __shfl_sync(kFull, sc_mine[h], i);
        const float4 x = __ldcg(reinterpret_cast<const float4*>(b + kPartialHeader + h * kHeadDim) + lane);
        acc[h].x += sc * x.x;
        acc[h].y += sc * x.y;
        acc[h].z += sc * x.z;
        acc[h].w += sc * x.w;
      }
    }
  }
  if (npre) {
    pf.weigh(M, L);
#pragma unroll 4
    for (int c = 0; c < npre; ++c) {
#pragma unroll
      for (int h = 0; h < GH; ++h) {
        const float sc = __shfl_sync(kFull, pf.w[h], c);
        const float4 x = __ldcg(reinterpret_cast<const float4*>(prefix_rec(p, row, h0 + h, c)) + lane);
        acc[h].x += sc * x.x;
        acc[h].y += sc * x.y;
        acc[h].z += sc * x.z;
        acc[h].w += sc * x.w;
      }
    }
  }
#pragma unroll
  for (int h = 0; h < GH; ++h) {
    const float inv = 1.f / L[h];
    uint2 pk;
    pk.x = pack_bf16x2(acc[h].x * inv, acc[h].y * inv);
    pk.y = pack_bf16x2(acc[h].z * inv, acc[h].w * inv);
    *reinterpret_cast<uint2*>(p.out + (size_t(row) * p.Hq + h0 + h) * kHeadDim + lane * 4) = pk;
  }
}

// tmk / tmv: TMA descriptors of the FP8 pools viewed as [rows][128 codes]
// (unused by the bf16 variant).
template <int GH, bool F8>
__global__ void __launch_bounds__(F8 ? kDecWarpsF8 * 32 : kDecThreads, PKV_DEC_MIN_CTAS)
    pkv_decode_kernel(DecodeParams p, const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  using Ring = DecRing<F8>;
  using Meta = DecMeta<F8>;
  constexpr int NS = F8 ? kDecStagesF8 : kDecStages;  // ring stages
  constexpr int NW = F8 ? kDecWarpsF8 : kDecWarps;    // warps per CTA
  constexpr int NT = NW * 32;
  // swizzled pages need 1024-byte aligned stages
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ring& R = reinterpret_cast<Ring*>(smem)[wib];
  Meta& M = reinterpret_cast<Meta*>(smem + sizeof(Ring) * NW)[wib];
  int* s_start = reinterpret_cast<int*>(smem + (sizeof(Ring) + sizeof(Meta)) * NW);
  int* s_q0 = s_start + (p.B + 1);
  int* s_len = s_q0 + (p.B + 1);
  const SeqSmem sq{s_start, s_q0, s_len};
  __shared__ int s_wsum[NW];

  if (lane == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&M.bar[s], 1);
    fence_mbar_init();
  }
  // Under programmatic dependent launch everything up to griddep_wait() below
  // (plan, cursor, first block ids, L2 prefetch hints) overlaps the previous
  // kernel (pkv_write, the shared-prefix pass, or a chunked-prefill pass that
  // runs first).  It reads only seq_lens, query_start_loc and block_tables,
  // which none of them writes; the pools and the workspace records are read
  // only after the wait.

  // ---- plan: per-sequence unit counts and their exclusive prefix ----------
  const int per_row = p.Hkv * p.nsub;
  // Stamp this launch's epoch (count 0) into every arrival counter, a share
  // per thread, so that arrivals are single atomic adds.  A counter is first
  // hit when a warp finishes a split item, long after these stamps; an
  // arrival that still sees an old epoch adds again once it is stamped.
#ifndef PKV_TEST_NO_EPOCH_STAMP  // a test build leaves the counters unstamped: arrivals time out
  for (int i = blockIdx.x * NT + threadIdx.x; i < p.T * per_row; i += gridDim.x * NT)
    atomicExch(p.counters + i, p.epoch << 16);
#endif
  // the prefill pass launched after this kernel counts its exits here (it
  // launches only once this CTA has passed its trigger below, or exited)
  if (p.lead && blockIdx.x == 0 && threadIdx.x == 0) atomicExch(p.join, p.epoch << 16);
  __shared__ long long s_pfw[NW];
  long long lead_steps = 0;  // lead: K/V tile steps of the prefill pass, all its CTAs
  {
    const int tid = threadIdx.x;
    const int per = (p.B + NT - 1) / NT;
    const int b0 = min(p.B, tid * per), b1 = min(p.B, b0 + per);
    int local = 0;
    for (int b = b0; b < b1; ++b) {
      const int q0 = __ldg(p.qsl + b), q1 = __ldg(p.qsl + b + 1), L = __ldg(p.seq_lens + b);
      const int n = q1 - q0;
      s_q0[b] = q0;
      s_len[b] = L;
      if (b == p.B - 1) s_q0[p.B] = q1;
      const bool bad = q0 < 0 || n < 0 || q1 > p.T || n > L || L < 0 ||
                       (L + kPage - 1) / kPage > p.max_blocks || (b == 0 && q0 != 0);
      if (bad && blockIdx.x == 0) flag_status(p.status, PKV_STATUS_BAD_QUERY);
      int units = 0;
      if (!bad && n >= 1 && n <= p.simt_max_q) {
        if (p.np > 0 && L - n + 1 <= p.np * kPage) {
          // every split-KV row needs a key of its own past the shared prefix
          if (blockIdx.x == 0) flag_status(p.status, PKV_STATUS_BAD_QUERY);
        } else {
          units = int(pages_prefix(L) - pages_prefix(L - n) - int64_t(n) * p.np) * per_row;
        }
      }
      s_start[b] = units;
      local += units;
      if (p.lead && !bad && n > p.simt_max_q) {
        // the pass's CTAs: per kv head, groups of two Q tiles; a group's
        // steps are the K/V tiles up to its last query's position
        const int tg = 2 * (kPfRows / p.G);
        long long st = 0;
        for (int t0 = 0; t0 < n; t0 += tg) st += (L - n + min(n, t0 + tg) - 1) / kPfKeys + 1;
        lead_steps += st * p.Hkv;
      }
    }
    if (p.lead) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) lead_steps += __shfl_xor_sync(kFull, lead_steps, o);
      if (lane == 0) s_pfw[wib] = lead_steps;
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += v;
    }
    if (lane == 31) s_wsum[wib] = incl;
    __syncthreads();
    int base = 0, total = 0;
#pragma unroll
    for (int x = 0; x < NW; ++x) {
      if (x < wib) base += s_wsum[x];
      total += s_wsum[x];
    }
    int run = base + incl - local;
    for (int b = b0; b < b1; ++b) {
      const int c = s_start[b];
      s_start[b] = run;
      run += c;
    }
    if (tid == 0) s_start[p.B] = total;
    __syncthreads();
    if (p.lead) {
      lead_steps = 0;
#pragma unroll
      for (int x = 0; x < NW; ++x) lead_steps += s_pfw[x];
    }
  }
  const int U = s_start[p.B];
  // Warps that take part.  With the prefill pass launched after this kernel,
  // the last `psm` CTAs leave their SMs to it; every CTA computes the same
  // count.  The pass's work in this kernel's units is its tile steps times
  // pf_cost (the units this kernel streams, whole GPU, while one SM does one
  // step).  While at least lead_sat SMs stay here this kernel is bound by HBM
  // and takes about as long as on all of them: the pass gets the SMs that
  // finish its work in that time.  A larger pass leaves fewer SMs than that,
  // and then both kernels' times scale with their SM counts: the SMs are
  // split in proportion to the work (pass work : units x lead_sat / grid).
  // At least one SM goes to the pass and one stays here.
  int nw = p.nwarps;
  if (p.lead && lead_steps > 0) {
    const long long ncta = gridDim.x;
    const long long sat = p.lead_sat > 0 ? min(ncta, (long long)p.lead_sat) : ncta;
    const long long work = lead_steps * p.pf_cost;
    long long want = ncta - 1;
    if (U > 0) {
      want = (work + U - 1) / U;
      if (want > ncta - sat) want = (work * ncta + work + U * sat - 1) / (work + U * sat);
    }
    const int psm = int(min(ncta - 1, max(1ll, want)));
    nw = (int(ncta) - psm) * NW;
  }
  // equal contiguous ranges, at least kMinChunk pages so small batches do not
  // shatter into one-page partials
  const int chunk = max(kMinChunk, (U + nw - 1) / nw);
  const int w = blockIdx.x * NW + wib;
  if (w >= nw || int64_t(w) * chunk >= U) {
    // lead: this CTA's exit may let the prefill pass launch, which must not
    // happen before the pool writes are complete; beside the pass: the call
    // ends with this grid, so it must not end before the pass
    if (p.lead || !p.wait_prev) griddep_wait();
    return;
  }
  const int u_begin = w * chunk;
  const int n_units = min(U - u_begin, chunk);
  const uint64_t policy = l2_evict_first_policy();

  // ---- producer cursor at u_begin -------------------------------------------
  Cursor pc;
  {
    int lo = 0, hi = p.B;  // last b with s_start[b] <= u_begin
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_start[mid] <= u_begin) lo = mid; else hi = mid;
    }
    cursor_seq(pc, sq, lo);
    int local = u_begin - s_start[lo];
    pc.j = 0;
    cursor_row(pc, p.np);
    while (local >= pc.npages * per_row) {
      local -= pc.npages * per_row;
      ++pc.j;
      cursor_row(pc, p.np);
    }
    pc.item = local / pc.npages;
    pc.page = local - pc.item * pc.npages;
    pc.item_start = u_begin - pc.page;
    cursor_bid(pc, p);
  }
  // warp-collective (every lane holds the same cursor): one elected lane
  // arms the stage and issues its copies
  auto issue = [&](int stage) {
    constexpr int PB = kPageBytesOf<F8>;
    const int g = pc.item / p.nsub;
    const size_t ph = size_t(pc.bid) * p.Hkv + g;  // (page, kv head)
    if (lane == 0) M.desc[stage] = StageDesc{pc.q0 + pc.j, pc.item, pc.item_start, pc.nvis - p.np * kPage};
    // lane 0's store ordered before the arrival, whichever lane elect.sync picks
    __syncwarp();
    mbar_arrive_expect_tx_w(&M.bar[stage], 2 * PB + (F8 ? 2 * kScaleBytes : 0));
    if (kDropFirstCopy && pc.item_start + pc.page == u_begin) return;
    // one box per page: the pool viewed as [units][128 bytes]; the host
    // checks that unit indices fit int32
    const int unit0 = int(ph) * (PB / 128);
    tma_load_2d_hint_w(&R.kv[stage][0][0], &tmk, 0, unit0, &M.bar[stage], policy);
    tma_load_2d_hint_w(&R.kv[stage][1][0], &tmv, 0, unit0, &M.bar[stage], policy);
    if constexpr (F8) {
      bulk_g2s_w(&M.sc[stage][0], p.k_scale + ph * kScaleBytes, kScaleBytes, &M.bar[stage], policy);
      bulk_g2s_w(&M.sc[stage][1], p.v_scale + ph * kScaleBytes, kScaleBytes, &M.bar[stage], policy);
    }
  };
  // Each warp's first pages into L2 while the previous kernel (normally
  // pkv_write, whose step leaves HBM idle) is still running; the copies into
  // shared memory wait below.  bf16 pages: the ring's two pages and four more
  // (1824 warps x 6 pages x 8 KiB = 88 MB, under the 129 MB L2): the
  // 8B-shaped step 116 -> 112 us, the long-tail and mixed steps unchanged.
  // Behind a shared-prefix pass (which reads the prefix from L2) only the
  // ring's pages: six made that step 4 % slower; FP8 pages: none (2 % slower).
  // Lane s takes unit s: the block-id reads go out together.
  if constexpr (!F8) {
    const int npf = min(p.np > 0 ? NS : NS + 4, n_units);
    if (lane < npf) {
      Cursor c = pc;
      for (int s = 0; s < lane; ++s) cursor_step(c, p.np, sq, per_row);
      int bid = __ldg(p.block_tables + int64_t(c.b) * p.max_blocks + p.np + c.page);
      if (bid >= 0 && bid < p.num_blocks) {  // a bad id is flagged when its page is copied
        constexpr int PB = kPageBytesOf<F8>;
        const size_t ph = size_t(bid) * p.Hkv + c.item / p.nsub;
        prefetch_l2(p.k_cache + ph * PB, PB);
        prefetch_l2(p.v_cache + ph * PB, PB);
      }
    }
    __syncwarp();
  }
  if (p.wait_prev) griddep_wait();
  if (p.lead) griddep_launch_dependents();
  {
    const int prologue = min(NS, n_units);
    for (int s = 0; s < prologue; ++s) {
      issue(s);
      if (s + 1 < n_units) cursor_advance(pc, p, sq, per_row);
    }
  }

  // ---- consumer state ----------------------------------------------------------
  // MMA fragments: lane = (gq = lane/4, tq = lane%4).  qb: Q^T operand of head
  // gq, dims 32tq+4s+{0,1} / {2,3} for k-step s; oacc: O^T of dims
  // 16gq+2mb+{0,1} (M-block mb) for heads 2tq, 2tq+1; m2 / l2: the running
  // maximum (log2 domain) and sum of those two heads over this lane's tokens
  // gq, gq+8.  At a segment's end they move to the flush layout: o by lanes
  // (dc, par), m and l of every head on every lane.
  const int gq = lane >> 2, tq = lane & 3;
  const int dc = lane & 15, par = lane >> 4;
  uint32_t qb[8][2];
  float oacc[8][4];
  float m2[2], l2[2];
  float qmul = 0.f;  // scale * log2(e) (FP8: times 2^-kq)
  int eref = 0;      // FP8: largest V scale byte of the segment so far (0: none)
  float2 o[GH][4];   // flush layout: dims 8dc+2e, 8dc+2e+1 of head h
  float m[GH], lfin[GH];
  int cur_row = -1, cur_item = -1, cur_item_start = 0, cur_seg_start = 0, cur_nvis = 0, cur_h0 = 0;

  auto start_segment = [&](const StageDesc& d, int u) {
    cur_row = d.row;
    cur_item = d.item;
    cur_item_start = d.item_start;
    cur_nvis = d.nvis;
    cur_seg_start = u;
    const int g = d.item / p.nsub, sub = d.item - g * p.nsub;
    cur_h0 = g * p.G + sub * GH;
    const uint4* qrow = reinterpret_cast<const uint4*>(p.q + (size_t(d.row) * p.Hq + cur_h0) * kHeadDim);
    if constexpr (!F8) {
      // bf16 pages: the Q^T operand is q's own bf16 pairs; column gq is head
      // gq % GH for gq < 2 GH (the remainder columns repeat the heads), zero past
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 x = make_uint4(0, 0, 0, 0);
        if (gq < 2 * GH) x = __ldg(qrow + (gq & (GH - 1)) * 16 + tq * 4 + c);
        qb[2 * c][0] = x.x;
        qb[2 * c][1] = x.y;
        qb[2 * c + 1][0] = x.z;
        qb[2 * c + 1][1] = x.w;
      }
      qmul = p.qscale;
    } else {
      // column gq's dims 32tq..32tq+31: head gq % GH for gq < 2 GH, zero past
      float qv[32];
      float amax = 0.f;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint4 x = make_uint4(0, 0, 0, 0);
        if (gq < 2 * GH) x = __ldg(qrow + (gq & (GH - 1)) * 16 + tq * 4 + c);
        const uint32_t wq[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          qv[c * 8 + 2 * e] = bf_lo(wq[e]);
          qv[c * 8 + 2 * e + 1] = bf_hi(wq[e]);
          amax = fmaxf(amax, fmaxf(fabsf(qv[c * 8 + 2 * e]), fabsf(qv[c * 8 + 2 * e + 1])));
        }
      }
#pragma unroll
      for (int o2 = 1; o2 < 32; o2 <<= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o2));
      // power of two that puts the group's largest |q| in [2^14, 2^15): exact in f16
      int kq = 0;
      if (amax > 0.f) kq = 14 - (int((__float_as_uint(amax) >> 23) & 0xFF) - 127);
      kq = max(-100, min(kq, 64));
      const float up = __uint_as_float(uint32_t(127 + kq) << 23);
      qmul = p.qscale * __uint_as_float(uint32_t(127 - kq) << 23);
#pragma unroll
      for (int st = 0; st < 8; ++st) {
        qb[st][0] = pack_f16x2(qv[4 * st] * up, qv[4 * st + 1] * up);
        qb[st][1] = pack_f16x2(qv[4 * st + 2] * up, qv[4 * st + 3] * up);
      }
    }
#pragma unroll
    for (int mb = 0; mb < 8; ++mb)
#pragma unroll
      for (int e = 0; e < 4; ++e) oacc[mb][e] = 0.f;
    m2[0] = m2[1] = -INFINITY;
    l2[0] = l2[1] = 0.f;
    eref = 0;
  };

  // Fragment state -> flush layout.  Lane (dc, par 0) takes dims 8dc..8dc+7
  // of head h from the lane with tq = h/2 that holds them; par 1 lanes hold 0.
  // l is summed over the lanes of a tq.
  auto frag_to_common = [&]() {
    // add each remainder column into its head's column: column GH + c sits
    // in lane tq + GH/2 (GH = 2, 4), or next to column 0 in the same lane
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      if constexpr (GH == 1) {
        oacc[mb][0] += oacc[mb][1];
        oacc[mb][2] += oacc[mb][3];
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) oacc[mb][e] += __shfl_xor_sync(kFull, oacc[mb][e], GH / 2);
      }
    }
    const float os = F8 ? scale_of(uint32_t(eref)) : 1.f;
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      // bf16: dims 8dc.. live in lane gq = dc % 8, M-blocks 4(dc/8)..; FP8:
      // lane gq = dc/2, M-blocks 4(dc%2)..
      const int src = F8 ? 4 * (dc >> 1) + (h >> 1) : 4 * (dc & 7) + (h >> 1);
      const bool odd = F8 ? (dc & 1) : (dc >> 3);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float x0 = __shfl_sync(kFull, oacc[e][h & 1], src);
        const float x1 = __shfl_sync(kFull, oacc[4 + e][h & 1], src);
        const float y0 = __shfl_sync(kFull, oacc[e][2 + (h & 1)], src);
        const float y1 = __shfl_sync(kFull, oacc[4 + e][2 + (h & 1)], src);
        o[h][e] = par == 0 ? make_float2((odd ? x1 : x0) * os, (odd ? y1 : y0) * os) : make_float2(0.f, 0.f);
      }
    }
    float lr[2] = {l2[0], l2[1]};
#pragma unroll
    for (int k = 0; k < 2; ++k)
#pragma unroll
      for (int o2 = 4; o2 < 32; o2 <<= 1) lr[k] += __shfl_xor_sync(kFull, lr[k], o2);
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      const float mh0 = __shfl_sync(kFull, m2[0], h >> 1), mh1 = __shfl_sync(kFull, m2[1], h >> 1);
      const float lh0 = __shfl_sync(kFull, lr[0], h >> 1), lh1 = __shfl_sync(kFull, lr[1], h >> 1);
      m[h] = (h & 1) ? mh1 : mh0;
      lfin[h] = (h & 1) ? lh1 : lh0;
    }
  };

  auto flush_segment = [&]() {
    frag_to_common();
#pragma unroll
    for (int h = 0; h < GH; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        o[h][e].x += __shfl_xor_sync(kFull, o[h][e].x, 16);
        o[h][e].y += __shfl_xor_sync(kFull, o[h][e].y, 16);
      }
    float l[GH];
#pragma unroll
    for (int h = 0; h < GH; ++h) l[h] = lfin[h];
    const int npages = (cur_nvis + kPage - 1) / kPage;
    const bool whole = cur_item_start >= u_begin && cur_item_start + npages <= u_begin + chunk;
    constexpr int HPL = GH >= 2 ? GH / 2 : 1;  // heads written per lane
    const bool writer = GH >= 2 || par == 0;
    auto pick = [&](int h, int e) {
      float2 v = o[0][e];
#pragma unroll
      for (int x = 0; x < GH; ++x)
        if (x == h) v = o[x][e];
      return v;
    };
    // shared-prefix fold for the whole-item write (all lanes take part)
    PrefixFold<GH> pf;
    float self_w[GH], Lf[GH];
    // the writes below run on the writer lanes only (all 32, or lanes 0-15
    // when GH == 1); chunk weights come from lanes < chunks <= 16
    const unsigned pf_mask = GH >= 2 ? 0xffffffffu : 0x0000ffffu;
    if (whole && p.np > 0) {
      float M[GH];
#pragma unroll
      for (int x = 0; x < GH; ++x) M[x] = m[x];
      pf.load(p, lane, cur_row, cur_h0);
      pf.max_into(M);
#pragma unroll
      for (int x = 0; x < GH; ++x) {
        self_w[x] = ex2(m[x] - M[x]);
        Lf[x] = self_w[x] * l[x];
      }
      pf.weigh(M, Lf);
    }
    if (whole) {
      if (writer) {
#pragma unroll
        for (int hh = 0; hh < HPL; ++hh) {
          const int h = (GH >= 2 ? par * HPL : 0) + hh;
          float lh = l[0], mh = m[0];
#pragma unroll
          for (int x = 0; x < GH; ++x)
            if (x == h) {
              lh = l[x];
              mh = m[x];
            }
          float2 v[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) v[e] = pick(h, e);
          if (p.np > 0) {  // fold in the shared-prefix records of this head
            float ws = 1.f;
#pragma unroll
            for (int x = 0; x < GH; ++x)
              if (x == h) {
                ws = self_w[x];
                lh = Lf[x];
              }
#pragma unroll
            for (int e = 0; e < 4; ++e) v[e] = make_float2(v[e].x * ws, v[e].y * ws);
#pragma unroll 4
            for (int c = 0; c < p.chunks; ++c) {
              // lane c holds chunk c's weights of every head; take head h's
              float sc = 0.f;
#pragma unroll
              for (int x = 0; x < GH; ++x) {
                const float sx = __shfl_sync(pf_mask, pf.w[x], c);
                if (x == h) sc = sx;
              }
              const float* rec = prefix_rec(p, cur_row, cur_h0 + h, c);
              const float4 a = __ldcg(reinterpret_cast<const float4*>(rec + dc * 8));
              const float4 b2 = __ldcg(reinterpret_cast<const float4*>(rec + dc * 8 + 4));
              v[0].x += sc * a.x;
              v[0].y += sc * a.y;
              v[1].x += sc * a.z;
              v[1].y += sc * a.w;
              v[2].x += sc * b2.x;
              v[2].y += sc * b2.y;
              v[3].x += sc * b2.z;
              v[3].y += sc * b2.w;
            }
          }
          const float inv = 1.f / lh;
          uint32_t pk[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) pk[e] = pack_bf16x2(v[e].x * inv, v[e].y * inv);
          *reinterpret_cast<uint4*>(p.out + (size_t(cur_row) * p.Hq + cur_h0 + h) * kHeadDim + dc * 8) =
              make_uint4(pk[0], pk[1], pk[2], pk[3]);
        }
      }
      return;
    }
    const int slot = 2 * w + (cur_seg_start == u_begin ? 0 : 1);
    float* base = p.partials + size_t(slot) * partial_floats(GH);
    if (lane == 0) {
#pragma unroll
      for (int h = 0; h < GH; ++h) {
        base[h] = m[h];
        base[4 + h] = l[h];
      }
    }
    if (writer) {
#pragma unroll
      for (int hh = 0; hh < HPL; ++hh) {
        const int h = (GH >= 2 ? par * HPL : 0) + hh;
        float4* dst = reinterpret_cast<float4*>(base + kPartialHeader + h * kHeadDim + dc * 8);
        const float2 v0 = pick(h, 0), v1 = pick(h, 1), v2 = pick(h, 2), v3 = pick(h, 3);
        dst[0] = make_float4(v0.x, v0.y, v1.x, v1.y);
        dst[1] = make_float4(v2.x, v2.y, v3.x, v3.y);
      }
    }
    __syncwarp();
    // arrival: the last warp of this (row, head group) merges all partials
    int last = 0;
    if (lane == 0) {
      const int w0 = cur_item_start / chunk, w1 = (cur_item_start + npages - 1) / chunk;
      const int nparts = w1 - w0 + 1;
      const int before = arrive_stamped(p.counters + size_t(cur_row) * per_row + cur_item, p.epoch);
      if (before < 0) flag_status(p.status, PKV_STATUS_TIMEOUT);  // no merge: the row stays unwritten
      last = before + 1 == nparts;
    }
    last = __shfl_sync(kFull, last, 0);
    if (last) {
      __syncwarp();  // the lanes read the partials after lane 0's acquire
      merge_item<GH>(p, lane, cur_row, cur_h0, cur_item_start, npages, chunk);
    }
  };

  bool timed_out = false;
  int it = 0;
  for (; it < n_units; ++it) {
    const int stage = it % NS;
    const uint32_t parity = (it / NS) & 1;
    // the warp leaves together (the loop body is warp-collective), even if
    // the lanes' clocks disagree about the limit
    if (!__all_sync(kFull, mbar_wait(&M.bar[stage], parity))) {
      timed_out = true;
      break;
    }
    const StageDesc d = M.desc[stage];
    const int u = u_begin + it;
    if (d.row != cur_row || d.item != cur_item) {
      if (cur_row >= 0) flush_segment();
      start_segment(d, u);
    }
    const int j = u - d.item_start;
    const int nvalid = min(kPage, d.nvis - j * kPage);
    if constexpr (F8) {
      // ---- operands of this lane out of the swizzled stage ----
      const uint8_t* Kp = R.kv[stage][0];
      const uint8_t* Vp = R.kv[stage][1];
      // K rows gq and gq+8, codes of dims 32tq..32tq+31 (chunks 2tq, 2tq+1)
      const uint4 ka0 = swz(Kp, gq, 2 * tq), ka1 = swz(Kp, gq, 2 * tq + 1);
      const uint4 kb0 = swz(Kp, gq + 8, 2 * tq), kb1 = swz(Kp, gq + 8, 2 * tq + 1);
      // V rows 2tq, 2tq+1, 2tq+8, 2tq+9, codes of dims 16gq..16gq+15 (chunk gq)
      uint4 va = swz(Vp, 2 * tq, gq), vb = swz(Vp, 2 * tq + 1, gq);
      uint4 vc = swz(Vp, 2 * tq + 8, gq), vd = swz(Vp, 2 * tq + 9, gq);
      const uint4 ksc = M.sc[stage][0], vsc = M.sc[stage][1];
      // The page now lives in registers: hand the stage back to the copy engine.
      __syncwarp();
      if (it + NS < n_units) {
        issue(stage);
        if (it + NS + 1 < n_units) cursor_advance(pc, p, sq, per_row);
      }

      // ---- S^T = K . Q^T: 8 k-steps of 16 (permuted) dims ----
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
      {
        // two accumulator chains (even / odd k-steps) halve the MMA latency chain
        float sodd[4] = {0.f, 0.f, 0.f, 0.f};
        const uint32_t wa[8] = {ka0.x, ka0.y, ka0.z, ka0.w, ka1.x, ka1.y, ka1.z, ka1.w};
        const uint32_t wb[8] = {kb0.x, kb0.y, kb0.z, kb0.w, kb1.x, kb1.y, kb1.z, kb1.w};
#pragma unroll
        for (int st = 0; st < 8; ++st) {
          uint32_t a0, a1, a2, a3;
          e4m3x4_to_f16x2(wa[st], a0, a2);
          e4m3x4_to_f16x2(wb[st], a1, a3);
          mma_f16((st & 1) ? sodd : sacc, a0, a1, a2, a3, qb[st][0], qb[st][1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[e] += sodd[e];
      }
      // scores (log2 domain) of tokens gq, gq+8 for heads 2tq, 2tq+1
      const bool t0 = gq < nvalid, t1 = gq + 8 < nvalid;
      const bool h0 = 2 * tq < 2 * GH, h1r = 2 * tq + 1 < 2 * GH;
      uint32_t kb_0, kb_1, vb_0, vb_1;
      bytes_t_t8(ksc, gq, kb_0, kb_1);
      bytes_t_t8(vsc, gq, vb_0, vb_1);
      const float f0 = qmul * scale_of(kb_0), f1 = qmul * scale_of(kb_1);
      float sv[4];
      sv[0] = t0 && h0 ? sacc[0] * f0 : -INFINITY;
      sv[1] = t0 && h1r ? sacc[1] * f0 : -INFINITY;
      sv[2] = t1 && h0 ? sacc[2] * f1 : -INFINITY;
      sv[3] = t1 && h1r ? sacc[3] * f1 : -INFINITY;

      // largest V scale byte among the page's valid rows
      uint32_t vmax;
      {
        uint32_t w4[4] = {vsc.x, vsc.y, vsc.z, vsc.w};
        if (nvalid < kPage) {
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int keep = min(4, max(0, nvalid - 4 * q4));  // valid bytes in this word
            w4[q4] &= keep >= 4 ? 0xFFFFFFFFu : ((1u << (8 * keep)) - 1u);
          }
        }
        const uint32_t x = __vmaxu4(__vmaxu4(w4[0], w4[1]), __vmaxu4(w4[2], w4[3]));
        const uint32_t y = __vmaxu4(x, x >> 16);
        vmax = max(y & 0xFFu, (y >> 8) & 0xFFu);
      }

      // ---- lazy running maximum (and the V-scale reference) ----
      bool exceed = sv[0] > m2[0] + kTau || sv[2] > m2[0] + kTau || sv[1] > m2[1] + kTau ||
                    sv[3] > m2[1] + kTau;
      const bool grow = int(vmax) > eref;  // warp-uniform
      if (__any_sync(kFull, exceed) || grow) {
        float full0 = fmaxf(sv[0], sv[2]), full1 = fmaxf(sv[1], sv[3]);
#pragma unroll
        for (int o2 = 4; o2 < 32; o2 <<= 1) {
          full0 = fmaxf(full0, __shfl_xor_sync(kFull, full0, o2));
          full1 = fmaxf(full1, __shfl_xor_sync(kFull, full1, o2));
        }
        const float mn0 = fmaxf(m2[0], full0), mn1 = fmaxf(m2[1], full1);
        float a0 = m2[0] == -INFINITY ? 0.f : ex2(m2[0] - mn0);
        float a1 = m2[1] == -INFINITY ? 0.f : ex2(m2[1] - mn1);
        m2[0] = mn0;
        m2[1] = mn1;
        l2[0] *= a0;
        l2[1] *= a1;
        if (grow) {
          // O was weighted relative to 2^(eref-127); move it to the new reference
          const int dlt = eref - int(vmax) + 127;
          const float b = dlt >= 1 ? scale_of(uint32_t(dlt)) : 0.f;
          a0 *= b;
          a1 *= b;
          eref = int(vmax);
        }
#pragma unroll
        for (int mb = 0; mb < 8; ++mb) {
          oacc[mb][0] *= a0;
          oacc[mb][1] *= a1;
          oacc[mb][2] *= a0;
          oacc[mb][3] *= a1;
        }
      }

      // ---- probabilities, weighted by 2^(V scale - reference) for the PV product ----
      const float r0 = m2[0] == -INFINITY ? 0.f : m2[0], r1 = m2[1] == -INFINITY ? 0.f : m2[1];
      const float p0 = ex2(sv[0] - r0), p1 = ex2(sv[1] - r1), p2 = ex2(sv[2] - r0), p3 = ex2(sv[3] - r1);
      l2[0] += p0 + p2;
      l2[1] += p1 + p3;
      float w0 = 0.f, w1 = 0.f;
      if (t0) {
        const int dl = int(vb_0) - eref + 127;
        w0 = dl >= 1 ? scale_of(uint32_t(dl)) : 0.f;
      }
      if (t1) {
        const int dl = int(vb_1) - eref + 127;
        w1 = dl >= 1 ? scale_of(uint32_t(dl)) : 0.f;
      }
      // this lane's P for its even column (2tq) and odd column (2tq+1): tokens
      // gq, gq+8; a remainder column takes what the f16 rounding dropped
      const float pw0 = p0 * w0, pw2 = p2 * w1, pw1 = p1 * w0, pw3 = p3 * w1;
      uint32_t pe = pack_f16x2(pw0, pw2), po = pack_f16x2(pw1, pw3);
      if (2 * tq >= GH) pe = f16_remainder(pe, pw0, pw2);
      if (2 * tq + 1 >= GH) po = f16_remainder(po, pw1, pw3);
      // P^T operand: column gq, tokens 2tq, 2tq+1 (b0) and 2tq+8, 2tq+9 (b1),
      // gathered from the lanes that hold those tokens for column pair gq/2
      const int src0 = 8 * tq + (gq >> 1), src1 = src0 + 4;
      const uint32_t x0 = __shfl_sync(kFull, pe, src0), x1 = __shfl_sync(kFull, po, src0);
      const uint32_t y0 = __shfl_sync(kFull, pe, src1), y1 = __shfl_sync(kFull, po, src1);
      const uint32_t X = (gq & 1) ? x1 : x0, Y = (gq & 1) ? y1 : y0;
      uint32_t pb0 = __byte_perm(X, Y, 0x5410), pb1 = __byte_perm(X, Y, 0x7632);
      if (gq >= 2 * GH) pb0 = pb1 = 0u;

      // ---- O^T += V^T . P^T: 8 M-blocks of 16 (permuted) dims ----
      if (nvalid < kPage) {  // rows past the sequence may hold anything (NaN)
        const uint4 z = make_uint4(0, 0, 0, 0);
        if (2 * tq >= nvalid) va = z;
        if (2 * tq + 1 >= nvalid) vb = z;
        if (2 * tq + 8 >= nvalid) vc = z;
        if (2 * tq + 9 >= nvalid) vd = z;
      }
      const uint32_t A4[4] = {va.x, va.y, va.z, va.w}, B4[4] = {vb.x, vb.y, vb.z, vb.w};
      const uint32_t C4[4] = {vc.x, vc.y, vc.z, vc.w}, D4[4] = {vd.x, vd.y, vd.z, vd.w};
#pragma unroll
      for (int mb = 0; mb < 8; ++mb) {
        const uint32_t sel = (mb & 1) ? 0x7362u : 0x5140u;
        uint32_t a0, a1, a2, a3;
        e4m3x4_to_f16x2(__byte_perm(A4[mb >> 1], B4[mb >> 1], sel), a0, a1);
        e4m3x4_to_f16x2(__byte_perm(C4[mb >> 1], D4[mb >> 1], sel), a2, a3);
        mma_f16(oacc[mb], a0, a1, a2, a3, pb0, pb1);
      }
    } else {
      // ---- bf16 pages on MMA fragments (same lane roles as FP8) ----
      const uint8_t* Kp = R.kv[stage][0];  // 32 swizzled units: token r = units 2r, 2r+1
      const uint8_t* Vp = R.kv[stage][1];
      // K rows gq, gq+8: dims 32tq..32tq+31 = unit half tq/2, chunks 4(tq%2)..+3
      uint4 ka[4], kb[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        ka[c] = swz(Kp, 2 * gq + (tq >> 1), 4 * (tq & 1) + c);
        kb[c] = swz(Kp, 2 * (gq + 8) + (tq >> 1), 4 * (tq & 1) + c);
      }
      // ---- S^T = K . Q^T ----
      float sacc[4] = {0.f, 0.f, 0.f, 0.f};
      {
        float sodd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int st = 0; st < 8; ++st) {
          const uint4& A = ka[st >> 1];
          const uint4& B = kb[st >> 1];
          const uint32_t a0 = (st & 1) ? A.z : A.x, a2 = (st & 1) ? A.w : A.y;
          const uint32_t a1 = (st & 1) ? B.z : B.x, a3 = (st & 1) ? B.w : B.y;
          mma_bf16((st & 1) ? sodd : sacc, a0, a1, a2, a3, qb[st][0], qb[st][1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) sacc[e] += sodd[e];
      }
      // V rows tq, tq+4, tq+8, tq+12: dims 8gq..8gq+7 (chunk gq of the first
      // unit) and 64+8gq..64+8gq+7 (chunk gq of the second).  Read after the
      // S products, so that K's and V's fragments are never live together.
      uint4 vr[4][2];
#pragma unroll
      for (int c = 0; c < 2; ++c) {
#pragma unroll
        for (int x = 0; x < 4; ++x) vr[x][c] = swz(Vp, 2 * (tq + 4 * x) + c, gq);
      }
      __syncwarp();
      if (it + NS < n_units) {
        issue(stage);
        if (it + NS + 1 < n_units) cursor_advance(pc, p, sq, per_row);
      }
      const bool t0 = gq < nvalid, t1 = gq + 8 < nvalid;
      const bool h0 = 2 * tq < 2 * GH, h1r = 2 * tq + 1 < 2 * GH;
      float sv[4];
      sv[0] = t0 && h0 ? sacc[0] * qmul : -INFINITY;
      sv[1] = t0 && h1r ? sacc[1] * qmul : -INFINITY;
      sv[2] = t1 && h0 ? sacc[2] * qmul : -INFINITY;
      sv[3] = t1 && h1r ? sacc[3] * qmul : -INFINITY;
      const bool exceed = sv[0] > m2[0] + kTau || sv[2] > m2[0] + kTau || sv[1] > m2[1] + kTau ||
                          sv[3] > m2[1] + kTau;
      if (__any_sync(kFull, exceed)) {
        float full0 = fmaxf(sv[0], sv[2]), full1 = fmaxf(sv[1], sv[3]);
#pragma unroll
        for (int o2 = 4; o2 < 32; o2 <<= 1) {
          full0 = fmaxf(full0, __shfl_xor_sync(kFull, full0, o2));
          full1 = fmaxf(full1, __shfl_xor_sync(kFull, full1, o2));
        }
        const float mn0 = fmaxf(m2[0], full0), mn1 = fmaxf(m2[1], full1);
        const float a0 = m2[0] == -INFINITY ? 0.f : ex2(m2[0] - mn0);
        const float a1 = m2[1] == -INFINITY ? 0.f : ex2(m2[1] - mn1);
        m2[0] = mn0;
        m2[1] = mn1;
        l2[0] *= a0;
        l2[1] *= a1;
#pragma unroll
        for (int mb = 0; mb < 8; ++mb) {
          oacc[mb][0] *= a0;
          oacc[mb][1] *= a1;
          oacc[mb][2] *= a0;
          oacc[mb][3] *= a1;
        }
      }
      const float r0 = m2[0] == -INFINITY ? 0.f : m2[0], r1 = m2[1] == -INFINITY ? 0.f : m2[1];
      const float p0 = ex2(sv[0] - r0), p1 = ex2(sv[1] - r1), p2 = ex2(sv[2] - r0), p3 = ex2(sv[3] - r1);
      l2[0] += p0 + p2;
      l2[1] += p1 + p3;
      uint32_t pe = pack_bf16x2(p0, p2), po = pack_bf16x2(p1, p3);
      // remainder columns: p - bf16(p) (exact in fp32), rounded to bf16
      if (2 * tq >= GH) pe = pack_bf16x2(p0 - bf_lo(pe), p2 - bf_hi(pe));
      if (2 * tq + 1 >= GH) po = pack_bf16x2(p1 - bf_lo(po), p3 - bf_hi(po));
      // P^T operand: column gq, tokens tq, tq+4 (b0) and tq+8, tq+12 (b1)
      const int src0 = 4 * tq + (gq >> 1), src1 = src0 + 16;
      const uint32_t x0 = __shfl_sync(kFull, pe, src0), x1 = __shfl_sync(kFull, po, src0);
      const uint32_t y0 = __shfl_sync(kFull, pe, src1), y1 = __shfl_sync(kFull, po, src1);
      const uint32_t X = (gq & 1) ? x1 : x0, Y = (gq & 1) ? y1 : y0;
      uint32_t pb0 = __byte_perm(X, Y, 0x5410), pb1 = __byte_perm(X, Y, 0x7632);
      if (gq >= 2 * GH) pb0 = pb1 = 0u;

      // ---- O^T += V^T . P^T (rows past the sequence may hold anything) ----
      if (nvalid < kPage) {
        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int x = 0; x < 4; ++x)
          if (tq + 4 * x >= nvalid) vr[x][0] = vr[x][1] = z;
      }
#pragma unroll
      for (int mb = 0; mb < 8; ++mb) {
        // word mb % 4 of chunk mb / 4: dims 64(mb/4) + 8gq + 2(mb%4), +1
        const int k = mb & 3, hv = mb >> 2;
        auto word = [&](const uint4& x) { return k == 0 ? x.x : (k == 1 ? x.y : (k == 2 ? x.z : x.w)); };
        const uint32_t A = word(vr[0][hv]), B = word(vr[1][hv]), Cw = word(vr[2][hv]), Dw = word(vr[3][hv]);
        mma_bf16(oacc[mb], __byte_perm(A, B, 0x5410), __byte_perm(A, B, 0x7632), __byte_perm(Cw, Dw, 0x5410),
                 __byte_perm(Cw, Dw, 0x7632), pb0, pb1);
      }
    }
  }

  if (timed_out) {
    if (lane == 0) flag_status(p.status, PKV_STATUS_TIMEOUT);
    // let copies still in flight land before the CTA's shared memory is released
    for (int k = it; k < min(n_units, it + NS); ++k)
      mbar_wait(&M.bar[k % NS], (k / NS) & 1, kDrainLimitNs);
    if (!p.wait_prev) griddep_wait();
    return;
  }
  if (cur_row >= 0) flush_segment();
  if (!p.wait_prev) griddep_wait();  // beside the prefill pass: end after it
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static int group_per_item(int G) { return G >= 4 ? 4 : G; }
static int variant_of(int gh) { return gh == 4 ? 2 : gh - 1; }

// Rings, then the plan's per-sequence arrays: unit prefix and query_start_loc
// ([B+1] each) and seq_lens ([B]).
template <bool F8>
static size_t decode_smem_bytes(int num_seqs) {
  return 1024 + (sizeof(DecRing<F8>) + sizeof(DecMeta<F8>)) * (F8 ? kDecWarpsF8 : kDecWarps) +
         sizeof(int) * (3 * size_t(num_seqs) + 2);
}

template <int GH, bool F8>
static int occupancy_for() {
  auto fn = pkv_decode_kernel<GH, F8>;
  const size_t smem = decode_smem_bytes<F8>(kMaxSeqs);
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem)) != cudaSuccess) {
    cudaGetLastError();  // not sticky; leave no error behind for later launches
    return 0;
  }
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, fn, (F8 ? kDecWarpsF8 : kDecWarps) * 32, smem) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return blocks;
}

int decode_ctas_per_sm(int variant, bool fp8) {
  switch (variant) {
    case 0: return fp8 ? occupancy_for<1, true>() : occupancy_for<1, false>();
    case 1: return fp8 ? occupancy_for<2, true>() : occupancy_for<2, false>();
    default: return fp8 ? occupancy_for<4, true>() : occupancy_for<4, false>();
  }
}

// Split-KV units (one page of one kv head, K and V) the whole GPU streams
// while one SM runs one K/V tile step of the prefill pass: bf16 pages about
// 3.1 us per step (two Q tiles, P as two terms) against 6.5 TB/s / 8 KiB per
// unit.  Sizes the SM share the split-KV kernel leaves the pass when the
// pass runs behind it; 0 puts the pass first instead.  Measured on the
// 96-row mixed step (two 512-token chunks; 2,880 steps against 188,544
// units): bf16 1900 / 2300 / 2600 / 3000 -> 298 / 270 / 271 / 271 us.  FP8
// pages (the pass widens codes with three warps per operand, about 4 us a
// step, and split-KV is bound by issue, so the SMs are split in
// proportion): 4000 / 5000 / 6500 -> 275 / 255 / 275 us (pass first: 340
// us).
static int prefill_step_units(bool fp8) {
  static int v[2] = {-1, -1};
  int& x = v[fp8 ? 1 : 0];
  if (x < 0) {
    const char* e = getenv(fp8 ? "PKV_PREFILL_STEP_UNITS_FP8" : "PKV_PREFILL_STEP_UNITS");
    x = e ? atoi(e) : (fp8 ? 5000 : 2400);
  }
  return x;
}

// SMs at which the split-KV kernel's page stream saturates HBM.  bf16 pages:
// on the mixed step it took 262-268 us on 122 SMs against 254 us on 152,
// which puts saturation near 126.  FP8 pages: never (bound by issue).
static int split_kv_saturating_sms(bool fp8) { return fp8 ? 0 : 126; }

// Sequences with more query rows than this go to the tensor-core prefill
// kernel (when it is built in); the rest go through split-KV.
static int simt_max_q() {
  static int v = [] {
    const char* e = getenv("PKV_SPLITKV_MAX_QLEN");
    return e ? atoi(e) : PKV_SPLITKV_MAX_QLEN;
  }();
  return v;
}

static unsigned long long next_epoch() {
  static std::atomic<unsigned long long> ctr{
      (static_cast<unsigned long long>(
           std::chrono::steady_clock::now().time_since_epoch().count()) *
       0x9E3779B97F4A7C15ull) >> 20};
  for (;;) {
    const unsigned long long e = (ctr.fetch_add(1) + 1) & ((1ull << 48) - 1);
    if (e) return e;
  }
}

static size_t prefix_records(const pkv_desc& d, int32_t num_tokens, int32_t prefix_pages) {
  int ct = 0;
  const int chunks = prefix_chunks(d, num_tokens, prefix_pages, &ct);
  return size_t(num_tokens) * d.num_q_heads * size_t(chunks);
}

size_t attend_workspace_bytes(const DeviceInfo& dev, const pkv_desc& d, int32_t num_seqs,
                              int32_t num_tokens, int32_t shared_prefix_pages, bool fp8) {
  const int G = d.num_q_heads / d.num_kv_heads;
  const int gh = group_per_item(G);
  const int nw = fp8 ? dev.dec_warps_f8[variant_of(gh)] : dev.dec_warps[variant_of(gh)];
  return workspace_layout(num_tokens, d.num_kv_heads * (G / gh), nw, gh,
                          prefill_max_tiles(d, num_seqs, num_tokens),
                          prefix_records(d, num_tokens, shared_prefix_pages))
      .total;
}

template <int GH, bool F8>
static int launch_decode(const LaunchCtx& ctx, const DecodeParams& dp, const CUtensorMap& tk,
                         const CUtensorMap& tv) {
  cudaLaunchConfig_t cfg = {};
  constexpr int NW = F8 ? kDecWarpsF8 : kDecWarps;
  cfg.gridDim = dim3(dp.nwarps / NW);
  cfg.blockDim = dim3(NW * 32);
  cfg.dynamicSmemBytes = decode_smem_bytes<F8>(dp.B);
  cfg.stream = ctx.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  TraceScope ts(ctx.stream, PKV_K_DECODE);
  cudaLaunchKernelEx(&cfg, pkv_decode_kernel<GH, F8>, dp, tk, tv);
  return ts.done();
}

int launch_attend(const LaunchCtx& ctx, const AttendArgs& a) {
  const pkv_desc& d = a.desc;
  const int G = d.num_q_heads / d.num_kv_heads;
  const int GH = group_per_item(G);
  const int nsub = G / GH;
  const int nwarps = a.fp8 ? ctx.dev->dec_warps_f8[variant_of(GH)] : ctx.dev->dec_warps[variant_of(GH)];
  if (nwarps <= 0) return PKV_ERR_LAUNCH;
  if (a.num_seqs > kMaxSeqs) return PKV_ERR_RANGE;
  // unit indices are int32 on the device
  if (int64_t(a.num_tokens) * d.max_blocks_per_seq * d.num_kv_heads * nsub >= (int64_t(1) << 31))
    return PKV_ERR_RANGE;
  const int max_tiles = prefill_max_tiles(d, a.num_seqs, a.num_tokens);
  if (a.shared_prefix_pages < 0 || a.shared_prefix_pages > d.max_blocks_per_seq) return PKV_ERR_RANGE;
  int chunk_tiles = 0;
  const int chunks = prefix_chunks(d, a.num_tokens, a.shared_prefix_pages, &chunk_tiles);
  const WorkspaceLayout L =
      workspace_layout(a.num_tokens, d.num_kv_heads * nsub, nwarps, GH, max_tiles,
                       prefix_records(d, a.num_tokens, a.shared_prefix_pages));
  if (a.workspace_bytes < L.total) return PKV_ERR_WORKSPACE;
  if (a.num_tokens == 0 || a.num_seqs == 0) return PKV_OK;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  // Long query chunks go to the tensor-core kernel (bf16 or FP8 pages) unless
  // the caller's bound says there are none; then split-KV takes every row.
  const bool prefill = max_tiles > 0 && a.num_tokens > simt_max_q() &&
                       (a.max_query_len <= 0 || a.max_query_len > simt_max_q());
  const int split_max_q = prefill ? simt_max_q() : INT_MAX;
  // Without a shared prefix: split-KV first, on the SMs its plan keeps, and
  // the prefill pass behind it on the rest.  Otherwise the pass first and
  // split-KV beside it on the SMs it leaves free.
  const int pf_cost = prefill_step_units(a.fp8);
  // (the pass counts its CTAs' exits on a 16-bit count: fewer than 32768)
  const bool lead = prefill && a.shared_prefix_pages == 0 && pf_cost > 0 &&
                    int64_t(d.num_kv_heads) * prefill_groups(d, a.num_seqs, a.num_tokens, max_tiles) < 0x8000;
  const unsigned long long epoch = next_epoch();
  unsigned long long* join = reinterpret_cast<unsigned long long*>(ws + L.tiles);
  if (prefill && !lead) {
    if (int e = launch_prefill(ctx, a, split_max_q, max_tiles, nullptr, 0)) return e;
  }
  if (a.shared_prefix_pages > 0) {
    if (int e = launch_prefix(ctx, a, reinterpret_cast<float*>(ws + L.prefix), chunks, chunk_tiles))
      return e;
  }

  DecodeParams dp{};
  dp.q = a.q;
  dp.k_cache = static_cast<const uint8_t*>(a.k_cache);
  dp.v_cache = static_cast<const uint8_t*>(a.v_cache);
  dp.k_scale = a.k_scale;
  dp.v_scale = a.v_scale;
  dp.block_tables = a.block_tables;
  dp.seq_lens = a.seq_lens;
  dp.qsl = a.query_start_loc;
  dp.out = a.out;
  dp.partials = reinterpret_cast<float*>(ws + L.partials);
  dp.counters = reinterpret_cast<unsigned long long*>(ws + L.counters);
  dp.status = ctx.status;
  dp.B = a.num_seqs;
  dp.T = a.num_tokens;
  dp.num_blocks = d.num_blocks;
  dp.Hkv = d.num_kv_heads;
  dp.Hq = d.num_q_heads;
  dp.G = G;
  dp.nsub = nsub;
  dp.max_blocks = d.max_blocks_per_seq;
  dp.simt_max_q = split_max_q;
  dp.nwarps = nwarps;
  dp.qscale = a.scale * 1.4426950408889634f;
  dp.epoch = epoch;
  dp.wait_prev = (prefill && !lead && a.shared_prefix_pages == 0) ? 0 : 1;
  dp.lead = lead ? 1 : 0;
  dp.pf_cost = pf_cost;
  dp.lead_sat = split_kv_saturating_sms(a.fp8);
  dp.join = lead ? join : nullptr;
  dp.np = a.shared_prefix_pages;
  dp.chunks = chunks;
  dp.prefix_part = reinterpret_cast<const float*>(ws + L.prefix);

  // the pools as [units][128 bytes], one box of a whole (page, kv head): 16
  // units of E4M3 codes, or 32 units (two per token) of bf16
  CUtensorMap tk{}, tv{};
  {
    const int upp = (a.fp8 ? kPageBytesF8 : kPageBytes) / 128;  // units per page
    const cuuint64_t units = cuuint64_t(d.num_blocks) * d.num_kv_heads * upp;
    if (units > cuuint64_t(INT_MAX)) return PKV_ERR_RANGE;  // TMA coordinates are int32
    const cuuint64_t dims[2] = {cuuint64_t(a.fp8 ? 128 : 64), units};
    const cuuint64_t strides[1] = {128};
    const cuuint32_t box[2] = {cuuint32_t(a.fp8 ? 128 : 64), cuuint32_t(upp)};
    const CUtensorMapDataType dt = a.fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (!encode_tensor_map(&tk, dt, a.k_cache, 2, dims, strides, box) ||
        !encode_tensor_map(&tv, dt, a.v_cache, 2, dims, strides, box))
      return PKV_ERR_LAUNCH;
  }
  int e;
  if (a.fp8) {
    switch (GH) {
      case 1: e = launch_decode<1, true>(ctx, dp, tk, tv); break;
      case 2: e = launch_decode<2, true>(ctx, dp, tk, tv); break;
      default: e = launch_decode<4, true>(ctx, dp, tk, tv); break;
    }
  } else {
    switch (GH) {
      case 1: e = launch_decode<1, false>(ctx, dp, tk, tv); break;
      case 2: e = launch_decode<2, false>(ctx, dp, tk, tv); break;
      default: e = launch_decode<4, false>(ctx, dp, tk, tv); break;
    }
  }
  if (e || !lead) return e;
  return launch_prefill(ctx, a, split_max_q, max_tiles, join, epoch);
}

}  // namespace pkv
