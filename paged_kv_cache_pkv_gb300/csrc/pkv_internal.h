// pkv_internal.h -- host-side plumbing shared by the translation units of the
// library: per-device facts, the launch context, launch tracing.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/pkv.h"

namespace pkv {

struct DeviceInfo {
  int device = -1;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  // Decode warps of one persistent launch, per kernel variant: index 0, 1, 2
  // for 1, 2, 4 query heads sharing a page read.
  int dec_warps[3] = {0, 0, 0};
  int dec_warps_f8[3] = {0, 0, 0};  // FP8-page variant (its own CTA shape)
  size_t smem_optin = 0;
};

// Facts about the current device (cached; filled on first use per device).
// Returns nullptr and sets *err when the device is unusable.
const DeviceInfo* current_device(int* err);

// Device address of the current device's status word.
unsigned* status_word(int device);

struct LaunchCtx {
  cudaStream_t stream;
  const DeviceInfo* dev;
  unsigned* status;  // device address of this device's status word
};

// Records a trace event pair around one launch when a trace is attached to
// the calling thread, and counts the launch.
class TraceScope {
 public:
  TraceScope(cudaStream_t s, int kernel_id);
  // Call right after the launch: returns PKV_OK or PKV_ERR_LAUNCH.
  int done();

 private:
  cudaStream_t stream_;
  int kernel_;
  int slot_;
};

int launch_write(const LaunchCtx& ctx, const uint16_t* k_new, const uint16_t* v_new,
                 const int64_t* slot_mapping, int64_t num_tokens, uint16_t* k_cache,
                 uint16_t* v_cache, int32_t num_blocks, int32_t num_kv_heads);
int launch_write_fp8(const LaunchCtx& ctx, const uint16_t* k_new, const uint16_t* v_new,
                     const int64_t* slot_mapping, int64_t num_tokens, uint8_t* k_cache,
                     uint8_t* v_cache, uint8_t* k_scale, uint8_t* v_scale, int32_t num_blocks,
                     int32_t num_kv_heads);

struct AttendArgs {
  const uint16_t* q;
  const void* k_cache;  // bf16 pages, or E4M3 codes when fp8
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* query_start_loc;
  int32_t num_seqs, num_tokens, max_query_len, shared_prefix_pages;
  float scale;
  uint16_t* out;
  void* workspace;
  size_t workspace_bytes;
  pkv_desc desc;
  bool fp8 = false;                 // E4M3 pages with per-row scale bytes
  const uint8_t* k_scale = nullptr;  // [NB][Hkv][16], fp8 only
  const uint8_t* v_scale = nullptr;
};

// Workspace bytes for a batch on the current device.
size_t attend_workspace_bytes(const DeviceInfo& dev, const pkv_desc& d, int32_t num_seqs,
                              int32_t num_tokens, int32_t shared_prefix_pages, bool fp8 = false);
int launch_attend(const LaunchCtx& ctx, const AttendArgs& a);

// Resident CTAs per SM of the decode kernel variant (occupancy query).
int decode_ctas_per_sm(int variant, bool fp8);

// Tensor-core chunked-prefill path (pkv_prefill.cu).
int prefill_max_tiles(const pkv_desc& d, int32_t num_seqs, int32_t num_tokens);
// CTAs per kv head of the prefill launch.
int prefill_groups(const pkv_desc& d, int32_t num_seqs, int32_t num_tokens, int max_tiles);
// Launches the prefill kernel for sequences with more than split_max_q query
// rows.  join == null: it runs first (normal launch).  Otherwise it is
// launched behind this call's split-KV kernel, which stamped `join` (an
// 8-byte workspace word) with `epoch`.
int launch_prefill(const LaunchCtx& ctx, const AttendArgs& a, int split_max_q, int max_tiles,
                   unsigned long long* join, unsigned long long epoch);
// Shared-prefix pass: key chunks of the prefix and tiles per chunk.
// A tiled TMA descriptor with 128-byte swizzle (rank <= 3; strides in bytes
// for dims 1..rank-1).  Returns false when the driver entry point is missing
// or the driver rejects the description.
bool encode_tensor_map(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, int rank,
                       const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box);

int prefix_chunks(const pkv_desc& d, int32_t num_tokens, int32_t prefix_pages, int* chunk_tiles);
// Every query row against the shared prefix pages -> partial records.
int launch_prefix(const LaunchCtx& ctx, const AttendArgs& a, float* records, int chunks,
                  int chunk_tiles);

}  // namespace pkv
