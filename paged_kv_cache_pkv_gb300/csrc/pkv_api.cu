// pkv_api.cu -- the extern "C" boundary of the library: argument checks,
// per-device facts, the device status word, launch tracing.
//
// Ownership and error rules follow the native-runtime contract of TensorRT
// Edge-LLM "HTTP Inference Server Architecture" ("Request Lifecycle",
// "Extension Rules": the native side owns retained pages and keeps a single
// writer; unsupported options are rejected up front) and the tensor-lifetime
// rule of the vLLM notes "EngineCoreClient ..." ("Flujo de datos": buffers
// stay alive until the asynchronous consumer is done with them).
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {

// One status word per device (each device that loads the library gets its
// own copy of this variable).
__device__ unsigned g_status_word;

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
DeviceInfo g_dev[kMaxDevices];
unsigned* g_status_addr[kMaxDevices];
std::atomic<uint64_t> g_launches{0};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_desc(const pkv_desc* d) {
  if (!d) return PKV_ERR_NULL;
  if (d->head_dim != kHeadDim || d->page_size != kPage) return PKV_ERR_SHAPE;
  if (d->num_kv_heads <= 0 || d->num_q_heads <= 0 || d->num_q_heads % d->num_kv_heads)
    return PKV_ERR_SHAPE;
  const int G = d->num_q_heads / d->num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) return PKV_ERR_SHAPE;
  if (d->num_blocks <= 0 || d->max_blocks_per_seq <= 0) return PKV_ERR_RANGE;
  // page byte offsets are computed in 64 bits; bound the pool to int32 pages
  return PKV_OK;
}

}  // namespace

const DeviceInfo* current_device(int* err) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *err = PKV_ERR_DEVICE;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceInfo& info = g_dev[dev];
  if (info.device == dev) return &info;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) {
    *err = PKV_ERR_DEVICE;
    return nullptr;
  }
  if (prop.major != 10 || prop.minor != 3) {  // built for sm_103a only
    *err = PKV_ERR_DEVICE;
    return nullptr;
  }
  DeviceInfo fresh;
  fresh.device = dev;
  fresh.sm_count = prop.multiProcessorCount;
  fresh.cc_major = prop.major;
  fresh.cc_minor = prop.minor;
  fresh.smem_optin = prop.sharedMemPerBlockOptin;
  // A variant that cannot be resident gets 0 warps; pkv_attend then rejects
  // the head ratios that need it instead of failing here.
  for (int v = 0; v < 3; ++v) {
    fresh.dec_warps[v] = fresh.sm_count * decode_ctas_per_sm(v, false) * kDecWarps;
    fresh.dec_warps_f8[v] = fresh.sm_count * decode_ctas_per_sm(v, true) * kDecWarpsF8;
  }
  void* addr = nullptr;
  if (cudaGetSymbolAddress(&addr, g_status_word) != cudaSuccess) {
    *err = PKV_ERR_LAUNCH;
    return nullptr;
  }
  g_status_addr[dev] = static_cast<unsigned*>(addr);
  info = fresh;
  return &info;
}

unsigned* status_word(int device) {
  return device >= 0 && device < kMaxDevices ? g_status_addr[device] : nullptr;
}

static int make_ctx(pkv_stream_t stream, LaunchCtx* ctx) {
  int err = PKV_OK;
  const DeviceInfo* dev = current_device(&err);
  if (!dev) return err != PKV_OK ? err : PKV_ERR_DEVICE;
  ctx->stream = reinterpret_cast<cudaStream_t>(stream);
  ctx->dev = dev;
  ctx->status = g_status_addr[dev->device];
  return PKV_OK;
}

// ---------------------------------------------------------------------------
// tracing
// ---------------------------------------------------------------------------
}  // namespace pkv

struct pkv_trace {
  int device = -1;
  int capacity = 0;
  std::vector<cudaEvent_t> events;  // 2 per record
  std::vector<int> kernel;          // kernel id per record
  int used = 0;
  int64_t untimed[PKV_K_COUNT] = {};
};

namespace pkv {
namespace {
thread_local pkv_trace* t_trace = nullptr;
}

TraceScope::TraceScope(cudaStream_t s, int kernel_id) : stream_(s), kernel_(kernel_id), slot_(-1) {
  pkv_trace* tr = t_trace;
  if (tr) {
    if (tr->used < tr->capacity) {
      slot_ = tr->used++;
      tr->kernel[slot_] = kernel_id;
      cudaEventRecord(tr->events[2 * slot_], s);
    } else {
      tr->untimed[kernel_id]++;
    }
  }
}

int TraceScope::done() {
  const cudaError_t e = cudaGetLastError();
  g_launches.fetch_add(1, std::memory_order_relaxed);
  if (slot_ >= 0 && t_trace) cudaEventRecord(t_trace->events[2 * slot_ + 1], stream_);
  return e == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}

}  // namespace pkv

using namespace pkv;

static_assert(kMaxSeqs == PKV_MAX_SEQS, "the plan's shared-memory arrays hold PKV_MAX_SEQS sequences");

extern "C" {

int pkv_write(const pkv_bf16* k_new, const pkv_bf16* v_new, const int64_t* slot_mapping,
              int64_t num_tokens, pkv_bf16* k_cache, pkv_bf16* v_cache, const pkv_desc* desc,
              pkv_stream_t stream) {
  if (int e = check_desc(desc)) return e;
  if (num_tokens < 0) return PKV_ERR_RANGE;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_NULL;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(slot_mapping, 8))
    return PKV_ERR_ALIGN;
  LaunchCtx ctx{};
  if (int e = make_ctx(stream, &ctx)) return e;
  return launch_write(ctx, k_new, v_new, slot_mapping, num_tokens, k_cache, v_cache,
                      desc->num_blocks, desc->num_kv_heads);
}

int pkv_attend_workspace_size(const pkv_desc* desc, int32_t num_seqs, int32_t num_tokens,
                              int32_t shared_prefix_pages, size_t* bytes) {
  if (int e = check_desc(desc)) return e;
  if (!bytes) return PKV_ERR_NULL;
  if (num_seqs < 0 || num_seqs > PKV_MAX_SEQS || num_tokens < 0 || shared_prefix_pages < 0 ||
      shared_prefix_pages > desc->max_blocks_per_seq)
    return PKV_ERR_RANGE;
  int err = PKV_OK;
  const DeviceInfo* dev = current_device(&err);
  if (!dev) return err;
  *bytes = attend_workspace_bytes(*dev, *desc, num_seqs, num_tokens, shared_prefix_pages);
  return PKV_OK;
}

int pkv_attend_fp8_workspace_size(const pkv_desc* desc, int32_t num_seqs, int32_t num_tokens,
                                  int32_t shared_prefix_pages, size_t* bytes) {
  if (int e = check_desc(desc)) return e;
  if (!bytes) return PKV_ERR_NULL;
  if (num_seqs < 0 || num_seqs > PKV_MAX_SEQS || num_tokens < 0 || shared_prefix_pages < 0 ||
      shared_prefix_pages > desc->max_blocks_per_seq)
    return PKV_ERR_RANGE;
  int err = PKV_OK;
  const DeviceInfo* dev = current_device(&err);
  if (!dev) return err;
  *bytes = attend_workspace_bytes(*dev, *desc, num_seqs, num_tokens, shared_prefix_pages, true);
  return PKV_OK;
}

int pkv_attend(const pkv_bf16* q, const pkv_bf16* k_cache, const pkv_bf16* v_cache,
               const int32_t* block_tables, const int32_t* seq_lens,
               const int32_t* query_start_loc, int32_t num_seqs, int32_t num_tokens,
               int32_t max_query_len, int32_t shared_prefix_pages, float scale, pkv_bf16* out,
               void* workspace, size_t workspace_bytes, const pkv_desc* desc,
               pkv_stream_t stream) {
  if (int e = check_desc(desc)) return e;
  if (num_seqs < 0 || num_seqs > PKV_MAX_SEQS || num_tokens < 0 || shared_prefix_pages < 0 ||
      shared_prefix_pages > desc->max_blocks_per_seq)
    return PKV_ERR_RANGE;
  if (num_seqs == 0 || num_tokens == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !query_start_loc || !out ||
      !workspace)
    return PKV_ERR_NULL;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(block_tables, 4) || !aligned(seq_lens, 4) || !aligned(query_start_loc, 4) ||
      !aligned(workspace, 256))
    return PKV_ERR_ALIGN;
  LaunchCtx ctx{};
  if (int e = make_ctx(stream, &ctx)) return e;
  AttendArgs a{q,          k_cache,    v_cache,    block_tables,  seq_lens,
               query_start_loc, num_seqs, num_tokens, max_query_len, shared_prefix_pages,
               scale,      out,        workspace,  workspace_bytes, *desc};
  return launch_attend(ctx, a);
}

int pkv_write_fp8(const pkv_bf16* k_new, const pkv_bf16* v_new, const int64_t* slot_mapping,
                  int64_t num_tokens, pkv_fp8* k_cache, pkv_fp8* v_cache, uint8_t* k_scale,
                  uint8_t* v_scale, const pkv_desc* desc, pkv_stream_t stream) {
  if (int e = check_desc(desc)) return e;
  if (num_tokens < 0) return PKV_ERR_RANGE;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping || !k_cache || !v_cache || !k_scale || !v_scale)
    return PKV_ERR_NULL;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(slot_mapping, 8))
    return PKV_ERR_ALIGN;
  LaunchCtx ctx{};
  if (int e = make_ctx(stream, &ctx)) return e;
  return launch_write_fp8(ctx, k_new, v_new, slot_mapping, num_tokens, k_cache, v_cache, k_scale,
                          v_scale, desc->num_blocks, desc->num_kv_heads);
}

int pkv_attend_fp8(const pkv_bf16* q, const pkv_fp8* k_cache, const pkv_fp8* v_cache,
                   const uint8_t* k_scale, const uint8_t* v_scale, const int32_t* block_tables,
                   const int32_t* seq_lens, const int32_t* query_start_loc, int32_t num_seqs,
                   int32_t num_tokens, int32_t max_query_len, int32_t shared_prefix_pages,
                   float scale, pkv_bf16* out,
                   void* workspace, size_t workspace_bytes, const pkv_desc* desc,
                   pkv_stream_t stream) {
  if (int e = check_desc(desc)) return e;
  if (num_seqs < 0 || num_seqs > PKV_MAX_SEQS || num_tokens < 0 || shared_prefix_pages < 0 ||
      shared_prefix_pages > desc->max_blocks_per_seq)
    return PKV_ERR_RANGE;
  if (num_seqs == 0 || num_tokens == 0) return PKV_OK;
  if (!q || !k_cache || !v_cache || !k_scale || !v_scale || !block_tables || !seq_lens ||
      !query_start_loc || !out || !workspace)
    return PKV_ERR_NULL;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_scale, 16) ||
      !aligned(v_scale, 16) || !aligned(out, 16) || !aligned(block_tables, 4) ||
      !aligned(seq_lens, 4) || !aligned(query_start_loc, 4) || !aligned(workspace, 256))
    return PKV_ERR_ALIGN;
  LaunchCtx ctx{};
  if (int e = make_ctx(stream, &ctx)) return e;
  AttendArgs a{q,     k_cache, v_cache,   block_tables,    seq_lens, query_start_loc,
               num_seqs, num_tokens, max_query_len, shared_prefix_pages, scale, out, workspace,
               workspace_bytes, *desc};
  a.fp8 = true;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  return launch_attend(ctx, a);
}

int pkv_get_last_error(pkv_stream_t stream, uint32_t* flags) {
  if (!flags) return PKV_ERR_NULL;
  LaunchCtx ctx{};
  if (int e = make_ctx(stream, &ctx)) return e;
  unsigned host = 0;
  if (cudaMemcpyAsync(&host, ctx.status, sizeof(unsigned), cudaMemcpyDeviceToHost, ctx.stream) !=
          cudaSuccess ||
      cudaMemsetAsync(ctx.status, 0, sizeof(unsigned), ctx.stream) != cudaSuccess ||
      cudaStreamSynchronize(ctx.stream) != cudaSuccess)
    return PKV_ERR_LAUNCH;
  *flags = host;
  return PKV_OK;
}

const char* pkv_strerror(int code) {
  switch (code) {
    case PKV_OK: return "ok";
    case PKV_ERR_NULL: return "a required pointer is NULL";
    case PKV_ERR_ALIGN: return "a pointer is not aligned as required (16 B tensors, 256 B workspace)";
    case PKV_ERR_SHAPE: return "unsupported geometry (head_dim 128, page_size 16, Hq/Hkv in {1,2,4,8,16})";
    case PKV_ERR_RANGE: return "a count or size is out of range";
    case PKV_ERR_WORKSPACE: return "workspace smaller than pkv_attend_workspace_size";
    case PKV_ERR_LAUNCH: return "a CUDA launch or runtime call failed";
    case PKV_ERR_DEVICE: return "the current device is not an sm_103 (GB300) GPU";
    case PKV_ERR_STATE: return "trace API misuse";
    case PKV_ERR_SCRATCH: return "batch needs more scratch than PKV_STATIC_SCRATCH_BYTES (use pkv_attend with a workspace)";
    case PKV_ERR_NOSPACE: return "page pool: not enough free pages";
    default: return "unknown error";
  }
}

uint64_t pkv_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

int pkv_trace_create(int32_t capacity, pkv_trace** out) {
  if (!out) return PKV_ERR_NULL;
  if (capacity <= 0) return PKV_ERR_RANGE;
  auto* tr = new pkv_trace();
  cudaGetDevice(&tr->device);
  tr->capacity = capacity;
  tr->events.resize(2 * size_t(capacity));
  tr->kernel.assign(capacity, -1);
  for (auto& e : tr->events) {
    if (cudaEventCreate(&e) != cudaSuccess) {
      e = nullptr;
      pkv_trace_destroy(tr);
      return PKV_ERR_LAUNCH;
    }
  }
  *out = tr;
  return PKV_OK;
}

int pkv_trace_attach(pkv_trace* tr) {
  if (!tr) return PKV_ERR_NULL;
  if (t_trace) return PKV_ERR_STATE;
  t_trace = tr;
  return PKV_OK;
}

int pkv_trace_detach(void) {
  if (!t_trace) return PKV_ERR_STATE;
  t_trace = nullptr;
  return PKV_OK;
}

int pkv_trace_read(pkv_trace* tr, int32_t kernel_id, double* total_ms, int64_t* launches) {
  if (!tr || !total_ms || !launches) return PKV_ERR_NULL;
  if (kernel_id < 0 || kernel_id >= PKV_K_COUNT) return PKV_ERR_RANGE;
  double ms = 0;
  int64_t n = 0;
  for (int i = 0; i < tr->used; ++i) {
    if (tr->kernel[i] != kernel_id) continue;
    if (cudaEventSynchronize(tr->events[2 * i + 1]) != cudaSuccess) return PKV_ERR_LAUNCH;
    float x = 0;
    if (cudaEventElapsedTime(&x, tr->events[2 * i], tr->events[2 * i + 1]) != cudaSuccess)
      return PKV_ERR_LAUNCH;
    ms += x;
    ++n;
  }
  *total_ms = ms;
  *launches = n + tr->untimed[kernel_id];
  return PKV_OK;
}

int pkv_trace_reset(pkv_trace* tr) {
  if (!tr) return PKV_ERR_NULL;
  tr->used = 0;
  for (auto& u : tr->untimed) u = 0;
  return PKV_OK;
}

int pkv_trace_destroy(pkv_trace* tr) {
  if (!tr) return PKV_ERR_NULL;
  if (t_trace == tr) t_trace = nullptr;
  for (auto e : tr->events)
    if (e) cudaEventDestroy(e);
  delete tr;
  return PKV_OK;
}

}  // extern "C"
