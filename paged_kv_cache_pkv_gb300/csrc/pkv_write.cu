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

}  // namespace pkv
