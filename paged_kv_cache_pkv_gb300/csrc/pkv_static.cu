// pkv_static.cu -- pkv_attend_static: paged attention whose scratch memory is
// a fixed array inside the library, for callers that cannot allocate device
// memory (a host program that owns all device memory and forbids allocation
// after start-up, or a C caller that only holds pointers handed to it).
//
// The scratch array below exists once per GPU that loads the library and
// lives until the process exits.  Host code must not pass the array's name
// to a kernel: on the host that name is only a stand-in, not a device
// address.  The device address is looked up once per device, with that
// device current, and cached.
#include <mutex>

#include "pkv_common.cuh"
#include "pkv_internal.h"

namespace pkv {
namespace {

static __device__ __align__(256) uint8_t g_static_scratch[PKV_STATIC_SCRATCH_BYTES];

constexpr int kMaxStaticDevices = 64;
std::mutex g_static_mu;
void* g_static_addr[kMaxStaticDevices];

// Device address of this device's scratch array (looked up on first use).
int static_scratch(int device, void** out) {
  if (device < 0 || device >= kMaxStaticDevices) return PKV_ERR_DEVICE;
  std::lock_guard<std::mutex> lk(g_static_mu);
  if (!g_static_addr[device]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess || !ptr)
      return PKV_ERR_LAUNCH;
    g_static_addr[device] = ptr;
  }
  *out = g_static_addr[device];
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" PKV_API int pkv_attend_static(const pkv_bf16* q, const pkv_bf16* k_cache,
                                         const pkv_bf16* v_cache, const int32_t* block_tables,
                                         const int32_t* seq_lens, const int32_t* query_start_loc,
                                         int32_t num_seqs, int32_t num_tokens,
                                         int32_t max_query_len, int32_t shared_prefix_pages,
                                         float scale, pkv_bf16* out, const pkv_desc* desc,
                                         pkv_stream_t stream) {
  using namespace pkv;
  size_t need = 0;
  if (int e = pkv_attend_workspace_size(desc, num_seqs, num_tokens, shared_prefix_pages, &need))
    return e;
  if (need > PKV_STATIC_SCRATCH_BYTES) return PKV_ERR_SCRATCH;
  int device = -1;
  if (cudaGetDevice(&device) != cudaSuccess) return PKV_ERR_DEVICE;
  void* scratch = nullptr;
  if (int e = static_scratch(device, &scratch)) return e;
  return pkv_attend(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, num_seqs,
                    num_tokens, max_query_len, shared_prefix_pages, scale, out, scratch,
                    PKV_STATIC_SCRATCH_BYTES, desc, stream);
}
