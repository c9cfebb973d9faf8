// pkv_write.cu -- KV write step: scatter each new token's K and V rows into
// the page pool through the slot mapping (llm-d blog post "What does
// production-grade LLM inference look like?", introduction: the engine keeps
// the KV cache in pages; vLLM notes "EngineCoreClient ...", "Flujo de datos":
// a pool of num_gpu_blocks blocks of block_size tokens).
//
// Token t with slot s >= 0 goes to page s / 16, row s % 16 of every kv head;
// pool layout [num_blocks, Hkv, 16, 128] bf16.  A pure bit copy.
//
// One thread moves one 16-byte vector; 16 consecutive threads move one
// 256-byte (token, head) row, so both the read of k_new/v_new and the write
// into the page are fully coalesced 16-byte accesses.  The kernel is tiny
// (T * Hkv * 512 bytes) and launch bound; it uses a grid-stride loop over
// a grid sized to the work.
#include <cuda_fp8.h>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

__global__ void __launch_bounds__(256) pkv_write_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int64_t* __restrict__ slot_mapping, int64_t num_tokens, uint4* __restrict__ k_cache,
    uint4* __restrict__ v_cache, int32_t num_blocks, int32_t num_kv_heads,
    unsigned* __restrict__ status) {
  // Let a dependent attention kernel start its set-up now; it waits for this
  // grid's writes before it reads the pool.
  asm volatile("griddepcontrol.launch_dependents;");
  constexpr int kVecPerRow = kHeadDim * 2 / 16;  // 16 vectors of 16 B per row
  const int64_t rows = num_tokens * num_kv_heads;
  const int64_t total = rows * 2 * kVecPerRow;   // K and V
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int vec = int(i % kVecPerRow);
    const int64_t rest = i / kVecPerRow;
    const int which = int(rest % 2);  // 0: K, 1: V
    const int64_t row = rest / 2;     // token * Hkv + head
    const int64_t t = row / num_kv_heads;
    const int h = int(row % num_kv_heads);
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;
    const int64_t page = slot / kPage;
    const int r = int(slot % kPage);
    if (page >= num_blocks) {
      if (vec == 0 && which == 0) flag_status(status, PKV_STATUS_BAD_SLOT);
      continue;
    }
    const uint4* src = (which ? v_new : k_new) + row * kVecPerRow + vec;
    uint4* dst = (which ? v_cache : k_cache) +
                 ((page * num_kv_heads + h) * kPage + r) * kVecPerRow + vec;
    *dst = __ldg(src);
  }
}

int launch_write(const LaunchCtx& ctx, const uint16_t* k_new, const uint16_t* v_new,
                 const int64_t* slot_mapping, int64_t num_tokens, uint16_t* k_cache,
                 uint16_t* v_cache, int32_t num_blocks, int32_t num_kv_heads) {
  const int64_t total = num_tokens * num_kv_heads * 2 * (kHeadDim * 2 / 16);
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = int64_t(ctx.dev->sm_count) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  TraceScope ts(ctx.stream, PKV_K_WRITE);
  pkv_write_kernel<<<unsigned(blocks), threads, 0, ctx.stream>>>(
      reinterpret_cast<const uint4*>(k_new), reinterpret_cast<const uint4*>(v_new), slot_mapping,
      num_tokens, reinterpret_cast<uint4*>(k_cache), reinterpret_cast<uint4*>(v_cache),
      num_blocks, num_kv_heads, ctx.status);
  return ts.done();
}

// ---------------------------------------------------------------------------
// FP8 pages: the same scatter, with each (token, kv head) row of K and of V
// encoded as E4M3 codes (OCP 8-bit Floating Point Specification) under a
// power-of-two row scale 2^e, e the smallest integer with max|x| <= 448 * 2^e
// (clamped to [-126, 127]); the byte e + 127 goes to the row's slot of the
// scale array [NB][Hkv][16].  x * 2^-e is exact, so the only rounding is the
// E4M3 one (to nearest, ties to even, sign kept).
//
// Half a warp handles one row: lane v holds dims 8v..8v+7 (one 16-byte load),
// the row maximum is a 4-step shuffle reduction over the 16 lanes, and the
// codes go out as one coalesced 128-byte row (8 bytes per lane).
// ---------------------------------------------------------------------------

// Scale exponent of a row from the bit pattern of its largest magnitude (a
// finite bf16 without its sign): amax = (1 + m/128) * 2^E needs e = E - 8,
// one more when the mantissa exceeds 448's 1.75 (m > 96); zero and subnormal
// maxima take the lowest exponent.
__device__ __forceinline__ int row_exponent(uint32_t amax_bits) {
  if (amax_bits < 0x0080u) return -126;
  const int E = int(amax_bits >> 7) - 127;
  const int e = E - 8 + ((amax_bits & 0x7Fu) > 96u ? 1 : 0);
  return e < -126 ? -126 : (e > 127 ? 127 : e);
}

__global__ void __launch_bounds__(256) pkv_write_fp8_kernel(
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
    const int64_t* __restrict__ slot_mapping, int64_t num_tokens, uint2* __restrict__ k_cache,
    uint2* __restrict__ v_cache, uint8_t* __restrict__ k_scale, uint8_t* __restrict__ v_scale,
    int32_t num_blocks, int32_t num_kv_heads, unsigned* __restrict__ status) {
  asm volatile("griddepcontrol.launch_dependents;");
  constexpr int kVecPerRow = kHeadDim * 2 / 16;  // 16 lanes x 8 dims
  const int lane16 = threadIdx.x & 15;
  const int64_t rows = num_tokens * num_kv_heads * 2;  // K and V rows
  // The loop runs per warp (two rows per step) so that every lane of a warp
  // takes part in the shuffles of every step.
  const int64_t warp0 = (blockIdx.x * int64_t(blockDim.x) + threadIdx.x) >> 5;
  const int64_t nwarps = (int64_t(gridDim.x) * blockDim.x) >> 5;
  for (int64_t base = 2 * warp0; base < rows; base += 2 * nwarps) {
    const int64_t rr = base + ((threadIdx.x >> 4) & 1);
    const bool live = rr < rows;
    const int which = int(rr % 2);
    const int64_t row = rr / 2;  // token * Hkv + head
    const int64_t t = row / num_kv_heads;
    const int h = int(row % num_kv_heads);
    int64_t slot = -1;
    if (live) slot = __ldg(slot_mapping + t);
    uint4 x = make_uint4(0, 0, 0, 0);
    if (live && slot >= 0) x = __ldg((which ? v_new : k_new) + row * kVecPerRow + lane16);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t amax = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) amax = max(amax, max(w[e] & 0x7FFFu, (w[e] >> 16) & 0x7FFFu));
    // maximum over the 16 lanes of this half warp
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (!live) continue;
    if (slot < 0) continue;
    const int64_t page = slot / kPage;
    const int r = int(slot % kPage);
    if (page >= num_blocks) {
      if (lane16 == 0 && which == 0) flag_status(status, PKV_STATUS_BAD_SLOT);
      continue;
    }
    const int ex = row_exponent(amax);
    const float inv = __uint_as_float(uint32_t(127 - ex) << 23);  // 2^-e, a normal float
    uint32_t code[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float2 lo = make_float2(bf_lo(w[2 * e]) * inv, bf_hi(w[2 * e]) * inv);
      const float2 hi = make_float2(bf_lo(w[2 * e + 1]) * inv, bf_hi(w[2 * e + 1]) * inv);
      const uint32_t a = __nv_cvt_float2_to_fp8x2(lo, __NV_SATFINITE, __NV_E4M3);
      const uint32_t b = __nv_cvt_float2_to_fp8x2(hi, __NV_SATFINITE, __NV_E4M3);
      code[e] = (a & 0xFFFFu) | (b << 16);
    }
    const int64_t ph = page * num_kv_heads + h;
    (which ? v_cache : k_cache)[(ph * kPage + r) * kVecPerRow + lane16] = make_uint2(code[0], code[1]);
    if (lane16 == 0) (which ? v_scale : k_scale)[ph * kPage + r] = uint8_t(ex + 127);
  }
}

int launch_write_fp8(const LaunchCtx& ctx, const uint16_t* k_new, const uint16_t* v_new,
                     const int64_t* slot_mapping, int64_t num_tokens, uint8_t* k_cache,
                     uint8_t* v_cache, uint8_t* k_scale, uint8_t* v_scale, int32_t num_blocks,
                     int32_t num_kv_heads) {
  const int64_t rows = num_tokens * num_kv_heads * 2;
  const int threads = 256;  // 16 rows per block
  int64_t blocks = (rows * 16 + threads - 1) / threads;
  const int64_t cap = int64_t(ctx.dev->sm_count) * 16;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  TraceScope ts(ctx.stream, PKV_K_WRITE);
  pkv_write_fp8_kernel<<<unsigned(blocks), threads, 0, ctx.stream>>>(
      reinterpret_cast<const uint4*>(k_new), reinterpret_cast<const uint4*>(v_new), slot_mapping,
      num_tokens, reinterpret_cast<uint2*>(k_cache), reinterpret_cast<uint2*>(v_cache), k_scale,
      v_scale, num_blocks, num_kv_heads, ctx.status);
  return ts.done();
}

}  // namespace pkv
