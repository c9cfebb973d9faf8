// pkv_decode.cu -- split-KV paged attention on CUDA cores (decode rows), the
// device-side work plan, and the log-sum-exp merge of split partials.
//
// What is computed (llm-d blog post "What does production-grade LLM inference
// look like?", introduction: paged attention over a paged KV cache, decode
// being memory-bandwidth bound): for every query row r of the batch and every
// query head h, softmax(scale * q_r,h . K^T) V over the row's visible keys,
// with K/V read page by page through the sequence's block table.
//
// Design (GB300):
//  * Work unit = one (query row, group of GH query heads sharing a kv head,
//    page).  A unit moves exactly one 4 KiB K page and one 4 KiB V page of
//    one kv head (pool layout [NB, Hkv, 16, 128] makes each a single
//    contiguous block), and the GH query heads reuse that read (GQA).
//  * The plan kernel numbers all units row-major and gives every decode warp
//    an equal contiguous range ("chunk") of them, so a 16-token sequence and
//    a 32768-token one are balanced to within one page.
//  * Every warp is an independent worker with its own 3-stage ring of pages:
//    lane 0 issues cp.async.bulk copies (one per 4 KiB page, L2 evict-first)
//    that complete on an mbarrier; all 32 lanes compute.  No CTA-wide
//    barrier sits on the page loop.
//  * QK^T: lane (c = lane%8, g = lane/8) owns dims {8c..8c+7, 64+8c..64+8c+7}
//    of tokens g, g+4, g+8, g+12; partial dots are reduced over the 8 lanes
//    of a token with a transposing butterfly (each step halves the values a
//    lane holds), so 16 dot products cost 14 shuffles.
//  * Online softmax in the log2 domain (q pre-scaled by scale*log2 e).  The
//    running maximum is only raised when a score exceeds it by more than
//    kTau (a warp vote), so most pages skip the max reduction and rescale.
//  * PV: lane (dc = lane%16, parity = lane/16) owns dims 8dc..8dc+7 of
//    even/odd tokens; probabilities are broadcast through shared memory.
//  * A warp that sees a whole (row, head group) writes bf16 output directly;
//    a split one writes (m, l, o) to one of two partial slots of the warp,
//    merged afterwards by pkv_merge_kernel.
#include <climits>
#include <cmath>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

// ---------------------------------------------------------------------------
// plan
// ---------------------------------------------------------------------------
constexpr int kPlanThreads = 1024;
constexpr int kPlanMaxSeqs = 4096;

struct PlanParams {
  const int32_t* seq_lens;
  const int32_t* qsl;
  int32_t B, T, Hkv, nsub, nwarps, max_blocks;
  int32_t simt_max_q;   // sequences with q_len <= this go through split-KV
  int32_t tile_tokens;  // query tokens per tensor-core prefill tile
  int32_t max_tiles;
  PlanHeader* hdr;
  int32_t* row_unit_start;  // [T+1]
  int32_t* row_seq;         // [T]
  int32_t* row_nvis;        // [T]
  int32_t* warp_first_row;  // [nwarps]
  int32_t* tiles;           // [max_tiles][2] = (seq, first query row of the tile)
  unsigned* status;
};

__global__ void __launch_bounds__(kPlanThreads) pkv_plan_kernel(PlanParams p) {
  __shared__ int32_t s_qsl[kPlanMaxSeqs + 1];
  __shared__ int32_t s_len[kPlanMaxSeqs];
  __shared__ uint8_t s_bad[kPlanMaxSeqs];
  __shared__ int32_t s_warp[32];
  __shared__ int32_t s_ntiles;
  const int tid = threadIdx.x;
  if (tid == 0) s_ntiles = 0;
  for (int b = tid; b <= p.B; b += kPlanThreads) s_qsl[b] = p.qsl[b];
  for (int b = tid; b < p.B; b += kPlanThreads) s_len[b] = p.seq_lens[b];
  __syncthreads();

  // 1. validate sequences; queue tensor-core tiles of long query chunks
  for (int b = tid; b < p.B; b += kPlanThreads) {
    const int q0 = s_qsl[b], q1 = s_qsl[b + 1], L = s_len[b], n = q1 - q0;
    const bool bad = q0 < 0 || n < 0 || q1 > p.T || n > L || L < 0 ||
                     (L + kPage - 1) / kPage > p.max_blocks || (b == 0 && q0 != 0);
    s_bad[b] = bad;
    if (bad) {
      flag_status(p.status, PKV_STATUS_BAD_QUERY);
      continue;
    }
    if (n > p.simt_max_q) {
      const int nt = (n + p.tile_tokens - 1) / p.tile_tokens;
      const int at = atomicAdd(&s_ntiles, nt);
      for (int i = 0; i < nt && at + i < p.max_tiles; ++i) {
        p.tiles[2 * (at + i)] = b;
        p.tiles[2 * (at + i) + 1] = q0 + i * p.tile_tokens;
      }
    }
  }
  __syncthreads();

  // 2. per query row: owning sequence (binary search), visible keys, units
  const int per_page = p.Hkv * p.nsub;
  for (int r = tid; r < p.T; r += kPlanThreads) {
    int lo = 0, hi = p.B;  // last b with qsl[b] <= r
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_qsl[mid] <= r) lo = mid; else hi = mid;
    }
    int seq = -1, nvis = 0, units = 0;
    if (p.B > 0 && !s_bad[lo] && s_qsl[lo] <= r && r < s_qsl[lo + 1]) {
      const int n = s_qsl[lo + 1] - s_qsl[lo];
      nvis = s_len[lo] - n + (r - s_qsl[lo]) + 1;
      if (n <= p.simt_max_q) {
        seq = lo;
        units = (nvis + kPage - 1) / kPage * per_page;
      }
    }
    p.row_seq[r] = seq;
    p.row_nvis[r] = nvis;
    p.row_unit_start[r] = units;  // counts; scanned in place below
  }
  __syncthreads();

  // 3. exclusive scan of the unit counts (each thread a contiguous run)
  const int per = (p.T + kPlanThreads - 1) / kPlanThreads;
  const int r0 = min(p.T, tid * per), r1 = min(p.T, r0 + per);
  int local = 0;
  for (int r = r0; r < r1; ++r) local += p.row_unit_start[r];
  const int lane = tid & 31, wid = tid >> 5;
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_warp[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int v = s_warp[lane], x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    s_warp[lane] = x - v;  // exclusive warp offsets
  }
  __syncthreads();
  int run = s_warp[wid] + incl - local;
  for (int r = r0; r < r1; ++r) {
    const int c = p.row_unit_start[r];
    p.row_unit_start[r] = run;
    run += c;
  }
  if (tid == kPlanThreads - 1) {
    const int total = s_warp[31] + incl;  // last thread's inclusive sum = total
    p.row_unit_start[p.T] = total;
    const int chunk = max(1, (total + p.nwarps - 1) / p.nwarps);
    p.hdr->units = total;
    p.hdr->chunk = chunk;
    p.hdr->nwarps = p.nwarps;
    p.hdr->prefill_tiles = min(s_ntiles, p.max_tiles);
  }
  __syncthreads();

  // 4. first row of every decode warp's range
  const int total = p.row_unit_start[p.T];
  const int chunk = max(1, (total + p.nwarps - 1) / p.nwarps);
  for (int r = tid; r < p.T; r += kPlanThreads) {
    const int st = p.row_unit_start[r], en = p.row_unit_start[r + 1];
    if (en <= st) continue;
    const int w_lo = (st + chunk - 1) / chunk, w_hi = min(p.nwarps - 1, (en - 1) / chunk);
    for (int w = w_lo; w <= w_hi; ++w) p.warp_first_row[w] = r;
  }
}

// ---------------------------------------------------------------------------
// split-KV decode
// ---------------------------------------------------------------------------
struct DecodeParams {
  const uint16_t* q;
  const uint16_t* k_cache;
  const uint16_t* v_cache;
  const int32_t* block_tables;
  uint16_t* out;
  const PlanHeader* hdr;
  const int32_t* row_unit_start;
  const int32_t* row_seq;
  const int32_t* row_nvis;
  const int32_t* warp_first_row;
  float* partials;
  unsigned* status;
  int32_t num_blocks, Hkv, Hq, G, nsub, max_blocks;
  float qscale;  // scale * log2(e)
};

struct StageDesc {
  int32_t row, item, item_start, nvis;
};

struct __align__(128) DecWarpSmem {
  uint4 kv[kDecStages][2][kPageBytes / 16];  // [stage][K|V][16 rows x 16 vec]
  float ps[kPage * kMaxGroupPerItem];         // probabilities [token][head]
  StageDesc desc[kDecStages];
  uint64_t bar[kDecStages];
};

constexpr float kTau = 8.0f;  // log2-domain slack before the running max moves
constexpr unsigned kFull = 0xffffffffu;

// Producer cursor over the warp's units (all lanes hold identical copies).
struct Cursor {
  int row, item, j, us, npages, nvis, seq, item_start, bid;
};

__device__ __forceinline__ void cursor_load_row(Cursor& c, const DecodeParams& p, int r) {
  c.row = r;
  c.seq = __ldg(p.row_seq + r);
  c.nvis = __ldg(p.row_nvis + r);
  c.us = __ldg(p.row_unit_start + r);
  c.npages = (c.nvis + kPage - 1) / kPage;
}

__device__ __forceinline__ void cursor_load_bid(Cursor& c, const DecodeParams& p) {
  int bid = __ldg(p.block_tables + int64_t(c.seq) * p.max_blocks + c.j);
  if (bid < 0 || bid >= p.num_blocks) {
    flag_status(p.status, PKV_STATUS_BAD_BLOCK);
    bid = 0;
  }
  c.bid = bid;
}

__device__ __forceinline__ void cursor_advance(Cursor& c, const DecodeParams& p) {
  if (++c.j == c.npages) {
    c.j = 0;
    c.item_start += c.npages;
    if (++c.item == p.Hkv * p.nsub) {
      c.item = 0;
      int r = c.row + 1;
      while (__ldg(p.row_unit_start + r + 1) == __ldg(p.row_unit_start + r)) ++r;
      cursor_load_row(c, p, r);
      c.item_start = c.us;
    }
  }
  cursor_load_bid(c, p);
}

template <int GH>
__global__ void __launch_bounds__(kDecWarps * 32, 2) pkv_decode_kernel(DecodeParams p) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  const int lane = threadIdx.x & 31;
  const int wib = threadIdx.x >> 5;
  DecWarpSmem& S = reinterpret_cast<DecWarpSmem*>(smem_raw)[wib];
  const int w = blockIdx.x * kDecWarps + wib;
  const int U = p.hdr->units;
  const int chunk = p.hdr->chunk;
  const int u_begin = w * chunk;  // < 2^31: host checks the unit count
  if (w >= p.hdr->nwarps || u_begin >= U) return;
  const int n_units = min(U - u_begin, chunk);

  if (lane == 0) {
    for (int s = 0; s < kDecStages; ++s) mbar_init(&S.bar[s], 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint64_t policy = l2_evict_first_policy();

  // ---- producer -----------------------------------------------------------
  Cursor pc;
  {
    const int r = __ldg(p.warp_first_row + w);
    cursor_load_row(pc, p, r);
    const int local = u_begin - pc.us;
    pc.item = local / pc.npages;
    pc.j = local - pc.item * pc.npages;
    pc.item_start = pc.us + pc.item * pc.npages;
    cursor_load_bid(pc, p);
  }
  auto issue = [&](int stage) {
    if (lane == 0) {
      const int g = pc.item / p.nsub;
      const size_t off = (size_t(pc.bid) * p.Hkv + g) * (kPageBytes / 2);
      S.desc[stage] = StageDesc{pc.row, pc.item, pc.item_start, pc.nvis};
      mbar_arrive_expect_tx(&S.bar[stage], 2 * kPageBytes);
      bulk_g2s(&S.kv[stage][0][0], p.k_cache + off, kPageBytes, &S.bar[stage], policy);
      bulk_g2s(&S.kv[stage][1][0], p.v_cache + off, kPageBytes, &S.bar[stage], policy);
    }
  };
  const int prologue = min(kDecStages, n_units);
  for (int s = 0; s < prologue; ++s) {
    issue(s);
    if (s + 1 < n_units) cursor_advance(pc, p);
  }

  // ---- consumer state -------------------------------------------------------
  constexpr int NVL = GH == 4 ? 2 : 1;  // scores a lane holds after the butterfly
  const int c8 = lane & 7, grp = lane >> 3;
  const int h1 = (lane >> 2) & 1, h2 = (lane >> 1) & 1, h3 = lane & 1;
  const int my_tok = grp + 4 * (2 * h1 + h2);
  const int dc = lane & 15, par = lane >> 4;
  auto head_of = [&](int k) { return GH == 4 ? 2 * h3 + k : (GH == 2 ? h3 : 0); };

  float qf[GH][16];
  float o[GH][8];
  float m[GH];
  float lsum[NVL];
  int cur_row = -1, cur_item = -1, cur_item_start = 0, cur_seg_start = 0, cur_nvis = 0;

  auto start_segment = [&](const StageDesc& d, int u) {
    cur_row = d.row;
    cur_item = d.item;
    cur_item_start = d.item_start;
    cur_nvis = d.nvis;
    cur_seg_start = u;
    const int g = d.item / p.nsub, sub = d.item - g * p.nsub;
    const int h0 = g * p.G + sub * GH;
    const uint4* qrow = reinterpret_cast<const uint4*>(p.q + (size_t(d.row) * p.Hq + h0) * kHeadDim);
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      const uint4 a = __ldg(qrow + h * 16 + c8);
      const uint4 b = __ldg(qrow + h * 16 + 8 + c8);
      const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        qf[h][2 * e] = bf_lo(wa[e]) * p.qscale;
        qf[h][2 * e + 1] = bf_hi(wa[e]) * p.qscale;
        qf[h][8 + 2 * e] = bf_lo(wb[e]) * p.qscale;
        qf[h][8 + 2 * e + 1] = bf_hi(wb[e]) * p.qscale;
      }
      m[h] = -INFINITY;
#pragma unroll
      for (int k = 0; k < 8; ++k) o[h][k] = 0.f;
    }
#pragma unroll
    for (int k = 0; k < NVL; ++k) lsum[k] = 0.f;
  };

  auto flush_segment = [&]() {
#pragma unroll
    for (int h = 0; h < GH; ++h)
#pragma unroll
      for (int k = 0; k < 8; ++k) o[h][k] += __shfl_xor_sync(kFull, o[h][k], 16);
    float lpart[NVL];
#pragma unroll
    for (int k = 0; k < NVL; ++k) {
      float x = lsum[k];
      x += __shfl_xor_sync(kFull, x, 2);
      x += __shfl_xor_sync(kFull, x, 4);
      x += __shfl_xor_sync(kFull, x, 8);
      x += __shfl_xor_sync(kFull, x, 16);
      lpart[k] = x;
    }
    float l[GH];
    if constexpr (GH == 4) {
      const float x0 = __shfl_xor_sync(kFull, lpart[0], 1), x1 = __shfl_xor_sync(kFull, lpart[1], 1);
      l[0] = h3 ? x0 : lpart[0];
      l[1] = h3 ? x1 : lpart[1];
      l[2] = h3 ? lpart[0] : x0;
      l[3] = h3 ? lpart[1] : x1;
    } else if constexpr (GH == 2) {
      const float x0 = __shfl_xor_sync(kFull, lpart[0], 1);
      l[0] = h3 ? x0 : lpart[0];
      l[1] = h3 ? lpart[0] : x0;
    } else {
      l[0] = lpart[0];
    }
    const int npages = (cur_nvis + kPage - 1) / kPage;
    const bool whole = cur_item_start >= u_begin && cur_item_start + npages <= u_begin + chunk;
    const int g = cur_item / p.nsub, sub = cur_item - g * p.nsub;
    const int h0 = g * p.G + sub * GH;
    constexpr int HPL = GH >= 2 ? GH / 2 : 1;  // heads written per lane
    const bool writer = GH >= 2 || par == 0;
    if (whole) {
      if (writer) {
#pragma unroll
        for (int hh = 0; hh < HPL; ++hh) {
          const int h = (GH >= 2 ? par * HPL : 0) + hh;
          float vals[8];
          float lh = l[0];
#pragma unroll
          for (int x = 0; x < GH; ++x)
            if (x == h) lh = l[x];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float ov = o[0][k];
#pragma unroll
            for (int x = 0; x < GH; ++x)
              if (x == h) ov = o[x][k];
            vals[k] = ov / lh;
          }
          uint4 pk;
          pk.x = pack_bf16x2(vals[0], vals[1]);
          pk.y = pack_bf16x2(vals[2], vals[3]);
          pk.z = pack_bf16x2(vals[4], vals[5]);
          pk.w = pack_bf16x2(vals[6], vals[7]);
          *reinterpret_cast<uint4*>(p.out + (size_t(cur_row) * p.Hq + h0 + h) * kHeadDim + dc * 8) = pk;
        }
      }
    } else {
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
          float vals[8];
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            float ov = o[0][k];
#pragma unroll
            for (int x = 0; x < GH; ++x)
              if (x == h) ov = o[x][k];
            vals[k] = ov;
          }
          float4* dst = reinterpret_cast<float4*>(base + kPartialHeader + h * kHeadDim + dc * 8);
          dst[0] = make_float4(vals[0], vals[1], vals[2], vals[3]);
          dst[1] = make_float4(vals[4], vals[5], vals[6], vals[7]);
        }
      }
    }
  };

  bool timed_out = false;
  int it = 0;
  for (; it < n_units; ++it) {
    const int stage = it % kDecStages;
    const uint32_t parity = (it / kDecStages) & 1;
    if (!mbar_wait(&S.bar[stage], parity)) {
      timed_out = true;
      break;
    }
    const StageDesc d = S.desc[stage];
    const int u = u_begin + it;
    if (d.row != cur_row || d.item != cur_item) {
      if (cur_row >= 0) flush_segment();
      start_segment(d, u);
    }
    const int j = u - d.item_start;
    const int nvalid = min(kPage, d.nvis - j * kPage);
    const uint4* Ks = S.kv[stage][0];
    const uint4* Vs = S.kv[stage][1];

    // ---- scores: 4 tokens x GH heads per lane, partial over 16 dims ----
    float v[4 * GH];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int t = grp + 4 * i;
      const uint4 a = Ks[t * 16 + c8];
      const uint4 b = Ks[t * 16 + 8 + c8];
      const uint32_t wa[4] = {a.x, a.y, a.z, a.w}, wb[4] = {b.x, b.y, b.z, b.w};
      float kf[16];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        kf[2 * e] = bf_lo(wa[e]);
        kf[2 * e + 1] = bf_hi(wa[e]);
        kf[8 + 2 * e] = bf_lo(wb[e]);
        kf[8 + 2 * e + 1] = bf_hi(wb[e]);
      }
#pragma unroll
      for (int h = 0; h < GH; ++h) {
        float acc = 0.f;
#pragma unroll
        for (int d2 = 0; d2 < 16; ++d2) acc = fmaf(qf[h][d2], kf[d2], acc);
        v[i * GH + h] = acc;
      }
    }
    // transposing butterfly over lanes xor 4, 2, 1
    {
      constexpr int N0 = 4 * GH;
#pragma unroll
      for (int i = 0; i < N0 / 2; ++i) {
        const float a = v[i], b = v[i + N0 / 2];
        const float send = h1 ? a : b, keep = h1 ? b : a;
        v[i] = keep + __shfl_xor_sync(kFull, send, 4);
      }
      constexpr int N1 = N0 / 2;
#pragma unroll
      for (int i = 0; i < N1 / 2; ++i) {
        const float a = v[i], b = v[i + N1 / 2];
        const float send = h2 ? a : b, keep = h2 ? b : a;
        v[i] = keep + __shfl_xor_sync(kFull, send, 2);
      }
      constexpr int N2 = N1 / 2;
      if constexpr (N2 >= 2) {
#pragma unroll
        for (int i = 0; i < N2 / 2; ++i) {
          const float a = v[i], b = v[i + N2 / 2];
          const float send = h3 ? a : b, keep = h3 ? b : a;
          v[i] = keep + __shfl_xor_sync(kFull, send, 1);
        }
      } else {
        v[0] += __shfl_xor_sync(kFull, v[0], 1);
      }
    }
    float s[NVL];
#pragma unroll
    for (int k = 0; k < NVL; ++k) s[k] = my_tok < nvalid ? v[k] : -INFINITY;

    // ---- online softmax (log2 domain) ----
    float mine[NVL];
#pragma unroll
    for (int k = 0; k < NVL; ++k) {
      float mm = m[0];
#pragma unroll
      for (int x = 0; x < GH; ++x)
        if (x == head_of(k)) mm = m[x];
      mine[k] = mm;
    }
    bool exceed = false;
#pragma unroll
    for (int k = 0; k < NVL; ++k) exceed |= s[k] > mine[k] + kTau;
    if (__any_sync(kFull, exceed)) {
      float pm[NVL];
#pragma unroll
      for (int k = 0; k < NVL; ++k) {
        float x = s[k];
        x = fmaxf(x, __shfl_xor_sync(kFull, x, 2));
        x = fmaxf(x, __shfl_xor_sync(kFull, x, 4));
        x = fmaxf(x, __shfl_xor_sync(kFull, x, 8));
        x = fmaxf(x, __shfl_xor_sync(kFull, x, 16));
        pm[k] = x;
      }
      float full[GH];
      if constexpr (GH == 4) {
        const float x0 = __shfl_xor_sync(kFull, pm[0], 1), x1 = __shfl_xor_sync(kFull, pm[1], 1);
        full[0] = h3 ? x0 : pm[0];
        full[1] = h3 ? x1 : pm[1];
        full[2] = h3 ? pm[0] : x0;
        full[3] = h3 ? pm[1] : x1;
      } else if constexpr (GH == 2) {
        const float x0 = __shfl_xor_sync(kFull, pm[0], 1);
        full[0] = h3 ? x0 : pm[0];
        full[1] = h3 ? pm[0] : x0;
      } else {
        full[0] = pm[0];
      }
      float alpha[GH];
#pragma unroll
      for (int h = 0; h < GH; ++h) {
        const float mn = fmaxf(m[h], full[h]);
        alpha[h] = m[h] == -INFINITY ? 0.f : ex2(m[h] - mn);
        m[h] = mn;
#pragma unroll
        for (int k = 0; k < 8; ++k) o[h][k] *= alpha[h];
      }
#pragma unroll
      for (int k = 0; k < NVL; ++k) {
        float a = alpha[0], mm = m[0];
#pragma unroll
        for (int x = 0; x < GH; ++x)
          if (x == head_of(k)) {
            a = alpha[x];
            mm = m[x];
          }
        lsum[k] *= a;
        mine[k] = mm;
      }
    }
    float pr[NVL];
#pragma unroll
    for (int k = 0; k < NVL; ++k) {
      pr[k] = ex2(s[k] - mine[k]);
      lsum[k] += pr[k];
    }
    if constexpr (GH == 4) {
      *reinterpret_cast<float2*>(&S.ps[my_tok * 4 + 2 * h3]) = make_float2(pr[0], pr[1]);
    } else if constexpr (GH == 2) {
      S.ps[my_tok * 2 + h3] = pr[0];
    } else {
      S.ps[my_tok] = pr[0];
    }
    __syncwarp();

    // ---- PV: even/odd tokens x 8 dims per lane ----
#pragma unroll
    for (int i = 0; i < kPage / 2; ++i) {
      const int t = par + 2 * i;
      if (t < nvalid) {
        const uint4 vv = Vs[t * 16 + dc];
        const uint32_t wv[4] = {vv.x, vv.y, vv.z, vv.w};
        float vf[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          vf[2 * e] = bf_lo(wv[e]);
          vf[2 * e + 1] = bf_hi(wv[e]);
        }
        float pv[GH];
        if constexpr (GH == 4) {
          const float4 x = *reinterpret_cast<const float4*>(&S.ps[t * 4]);
          pv[0] = x.x; pv[1] = x.y; pv[2] = x.z; pv[3] = x.w;
        } else if constexpr (GH == 2) {
          const float2 x = *reinterpret_cast<const float2*>(&S.ps[t * 2]);
          pv[0] = x.x; pv[1] = x.y;
        } else {
          pv[0] = S.ps[t];
        }
#pragma unroll
        for (int h = 0; h < GH; ++h)
#pragma unroll
          for (int k = 0; k < 8; ++k) o[h][k] = fmaf(pv[h], vf[k], o[h][k]);
      }
    }
    __syncwarp();

    // ---- refill this stage with the unit kDecStages ahead ----
    if (it + kDecStages < n_units) {
      issue(stage);
      if (it + kDecStages + 1 < n_units) cursor_advance(pc, p);
    }
  }

  if (timed_out) {
    if (lane == 0) flag_status(p.status, PKV_STATUS_TIMEOUT);
    // let copies still in flight land before the CTA's shared memory is released
    for (int k = it; k < min(n_units, it + kDecStages); ++k)
      mbar_wait(&S.bar[k % kDecStages], (k / kDecStages) & 1, 1u << 16);
    return;
  }
  if (cur_row >= 0) flush_segment();
}

// ---------------------------------------------------------------------------
// merge of split partials (log-sum-exp)
// ---------------------------------------------------------------------------
struct MergeParams {
  const PlanHeader* hdr;
  const int32_t* row_unit_start;
  const int32_t* row_seq;
  const int32_t* row_nvis;
  const float* partials;
  uint16_t* out;
  int32_t T, Hkv, Hq, G, nsub;
};

constexpr int kMergeWarps = 8;

template <int GH>
__global__ void __launch_bounds__(kMergeWarps * 32) pkv_merge_kernel(MergeParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t gi = int64_t(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
  const int items_per_row = p.Hkv * p.nsub;
  const int64_t row64 = gi / items_per_row;
  if (row64 >= p.T) return;
  const int row = int(row64), item = int(gi - row64 * items_per_row);
  if (__ldg(p.row_seq + row) < 0) return;
  const int chunk = p.hdr->chunk;
  const int npages = (__ldg(p.row_nvis + row) + kPage - 1) / kPage;
  const int item_start = __ldg(p.row_unit_start + row) + item * npages;
  const int item_end = item_start + npages;
  const int w0 = item_start / chunk, w1 = (item_end - 1) / chunk;
  if (w0 == w1) return;  // whole item seen by one warp, output already written
  float M[GH], L[GH];
#pragma unroll
  for (int h = 0; h < GH; ++h) {
    M[h] = -INFINITY;
    L[h] = 0.f;
  }
  auto slot_of = [&](int w) { return 2 * w + (item_start <= w * chunk ? 0 : 1); };
  for (int w = w0; w <= w1; ++w) {
    const float* base = p.partials + size_t(slot_of(w)) * partial_floats(GH);
#pragma unroll
    for (int h = 0; h < GH; ++h) M[h] = fmaxf(M[h], base[h]);
  }
  float4 acc[GH];
#pragma unroll
  for (int h = 0; h < GH; ++h) acc[h] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int w = w0; w <= w1; ++w) {
    const float* base = p.partials + size_t(slot_of(w)) * partial_floats(GH);
#pragma unroll
    for (int h = 0; h < GH; ++h) {
      const float sc = ex2(base[h] - M[h]);
      L[h] += sc * base[4 + h];
      const float4 x = reinterpret_cast<const float4*>(base + kPartialHeader + h * kHeadDim)[lane];
      acc[h].x += sc * x.x;
      acc[h].y += sc * x.y;
      acc[h].z += sc * x.z;
      acc[h].w += sc * x.w;
    }
  }
  const int g = item / p.nsub, sub = item - g * p.nsub;
  const int h0 = g * p.G + sub * GH;
#pragma unroll
  for (int h = 0; h < GH; ++h) {
    const float inv = 1.f / L[h];
    uint2 pk;
    pk.x = pack_bf16x2(acc[h].x * inv, acc[h].y * inv);
    pk.y = pack_bf16x2(acc[h].z * inv, acc[h].w * inv);
    *reinterpret_cast<uint2*>(p.out + (size_t(row) * p.Hq + h0 + h) * kHeadDim + lane * 4) = pk;
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static int group_per_item(int G) { return G >= 4 ? 4 : G; }

static size_t decode_smem_bytes() { return sizeof(DecWarpSmem) * kDecWarps; }

template <int GH>
static int occupancy_for() {
  auto fn = pkv_decode_kernel<GH>;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(decode_smem_bytes())) != cudaSuccess)
    return 0;
  int blocks = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, fn, kDecWarps * 32,
                                                    decode_smem_bytes()) != cudaSuccess)
    return 0;
  return blocks;
}

int decode_ctas_per_sm(int gh) {
  switch (gh) {
    case 1: return occupancy_for<1>();
    case 2: return occupancy_for<2>();
    default: return occupancy_for<4>();
  }
}

// Sequences with q_len above this go to the tensor-core prefill kernel.
static int simt_max_q() {
  static int v = [] {
    const char* e = getenv("PKV_SPLITKV_MAX_QLEN");
    return e ? atoi(e) : 8;
  }();
  return v;
}

size_t attend_workspace_bytes(const DeviceInfo& dev, const pkv_desc& d, int32_t num_seqs,
                              int32_t num_tokens) {
  const int G = d.num_q_heads / d.num_kv_heads;
  return workspace_layout(num_seqs, num_tokens, dev.dec_warps_total, group_per_item(G),
                          prefill_max_tiles(d, num_seqs, num_tokens))
      .total;
}

template <int GH>
static int launch_decode_and_merge(const LaunchCtx& ctx, const DecodeParams& dp,
                                   const MergeParams& mp, int nwarps) {
  {
    TraceScope ts(ctx.stream, PKV_K_DECODE);
    pkv_decode_kernel<GH><<<nwarps / kDecWarps, kDecWarps * 32, decode_smem_bytes(), ctx.stream>>>(dp);
    if (int e = ts.done()) return e;
  }
  const int64_t items = int64_t(mp.T) * mp.Hkv * mp.nsub;
  const int64_t blocks = (items + kMergeWarps - 1) / kMergeWarps;
  if (blocks == 0) return PKV_OK;
  TraceScope ts(ctx.stream, PKV_K_MERGE);
  pkv_merge_kernel<GH><<<unsigned(blocks), kMergeWarps * 32, 0, ctx.stream>>>(mp);
  return ts.done();
}

int launch_attend(const LaunchCtx& ctx, const AttendArgs& a) {
  const pkv_desc& d = a.desc;
  const int G = d.num_q_heads / d.num_kv_heads;
  const int GH = group_per_item(G);
  const int nsub = G / GH;
  const int nwarps = ctx.dev->dec_warps_total;
  if (a.num_seqs > kPlanMaxSeqs) return PKV_ERR_RANGE;
  // unit indices are int32 on the device
  if (int64_t(a.num_tokens) * d.max_blocks_per_seq * d.num_kv_heads * nsub >= (int64_t(1) << 31))
    return PKV_ERR_RANGE;
  const int max_tiles = prefill_max_tiles(d, a.num_seqs, a.num_tokens);
  const WorkspaceLayout L = workspace_layout(a.num_seqs, a.num_tokens, nwarps, GH, max_tiles);
  if (a.workspace_bytes < L.total) return PKV_ERR_WORKSPACE;
  if (a.num_tokens == 0 || a.num_seqs == 0) return PKV_OK;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);

  PlanParams pp{};
  pp.seq_lens = a.seq_lens;
  pp.qsl = a.query_start_loc;
  pp.B = a.num_seqs;
  pp.T = a.num_tokens;
  pp.Hkv = d.num_kv_heads;
  pp.nsub = nsub;
  pp.nwarps = nwarps;
  pp.max_blocks = d.max_blocks_per_seq;
  pp.simt_max_q = max_tiles > 0 ? simt_max_q() : INT_MAX;
  pp.tile_tokens = max_tiles > 0 ? 128 / G : 1;
  pp.max_tiles = max_tiles;
  pp.hdr = reinterpret_cast<PlanHeader*>(ws + L.header);
  pp.row_unit_start = reinterpret_cast<int32_t*>(ws + L.row_unit_start);
  pp.row_seq = reinterpret_cast<int32_t*>(ws + L.row_seq);
  pp.row_nvis = reinterpret_cast<int32_t*>(ws + L.row_nvis);
  pp.warp_first_row = reinterpret_cast<int32_t*>(ws + L.warp_first_row);
  pp.tiles = reinterpret_cast<int32_t*>(ws + L.tiles);
  pp.status = ctx.status;
  {
    TraceScope ts(ctx.stream, PKV_K_PLAN);
    pkv_plan_kernel<<<1, kPlanThreads, 0, ctx.stream>>>(pp);
    if (int e = ts.done()) return e;
  }

  if (max_tiles > 0) {
    if (int e = launch_prefill(ctx, a, pp.tiles, pp.hdr, max_tiles)) return e;
  }

  DecodeParams dp{};
  dp.q = a.q;
  dp.k_cache = a.k_cache;
  dp.v_cache = a.v_cache;
  dp.block_tables = a.block_tables;
  dp.out = a.out;
  dp.hdr = pp.hdr;
  dp.row_unit_start = pp.row_unit_start;
  dp.row_seq = pp.row_seq;
  dp.row_nvis = pp.row_nvis;
  dp.warp_first_row = pp.warp_first_row;
  dp.partials = reinterpret_cast<float*>(ws + L.partials);
  dp.status = ctx.status;
  dp.num_blocks = d.num_blocks;
  dp.Hkv = d.num_kv_heads;
  dp.Hq = d.num_q_heads;
  dp.G = G;
  dp.nsub = nsub;
  dp.max_blocks = d.max_blocks_per_seq;
  dp.qscale = a.scale * 1.4426950408889634f;

  MergeParams mp{};
  mp.hdr = pp.hdr;
  mp.row_unit_start = pp.row_unit_start;
  mp.row_seq = pp.row_seq;
  mp.row_nvis = pp.row_nvis;
  mp.partials = dp.partials;
  mp.out = a.out;
  mp.T = a.num_tokens;
  mp.Hkv = d.num_kv_heads;
  mp.Hq = d.num_q_heads;
  mp.G = G;
  mp.nsub = nsub;

  switch (GH) {
    case 1: return launch_decode_and_merge<1>(ctx, dp, mp, nwarps);
    case 2: return launch_decode_and_merge<2>(ctx, dp, mp, nwarps);
    default: return launch_decode_and_merge<4>(ctx, dp, mp, nwarps);
  }
}

}  // namespace pkv
