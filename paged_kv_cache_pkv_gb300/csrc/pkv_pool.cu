// pkv_pool.cu -- host-side page pool: allocation, reference counts for pages
// shared through a common prefix, copy-on-write of a shared page, and the
// usage gauge.
//
// The pages this follows: the engine reserves num_gpu_blocks pages of
// block_size tokens (vLLM notes "EngineCoreClient ...", "Flujo de datos");
// the native coordinator owns the retained pages and keeps a single writer
// (TensorRT Edge-LLM "HTTP Inference Server Architecture", "Request
// Lifecycle", "Extension Rules"); prefix KV is reused by later requests and
// serving stacks export a KV-cache usage gauge (llm-d blog, routing factors,
// prefix producers and the vllm:kv_cache_usage_perc metric snippet).
//
// Design: a LIFO free list (recently freed pages are reused first, so they
// are more likely still in L2) and a 32-bit reference count per page, under
// one mutex.  A page is writable by exactly one sequence when its count is 1;
// pkv_pool_make_writable gives a sequence a private copy of a shared page
// (the rows already written, for every kv head, K and V) before it appends.
#include <algorithm>
#include <mutex>
#include <vector>

#include "pkv_common.cuh"
#include "pkv_internal.h"

struct pkv_pool {
  std::mutex mu;
  std::vector<int32_t> refs;  // per page; 0 = free
  std::vector<int32_t> free_list;
  int64_t allocs = 0, frees = 0;
};

namespace pkv {

// Copy rows [0, rows) of (page src, every kv head) to page dst, K and V.
__global__ void __launch_bounds__(256) pkv_copy_page_kernel(uint4* __restrict__ k_cache,
                                                            uint4* __restrict__ v_cache,
                                                            int32_t src, int32_t dst, int32_t rows,
                                                            int32_t num_kv_heads) {
  constexpr int kVecPerRow = kHeadDim * 2 / 16;
  const int per_head = rows * kVecPerRow;
  const int total = 2 * num_kv_heads * per_head;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int which = i / (num_kv_heads * per_head);
    const int rest = i - which * num_kv_heads * per_head;
    const int h = rest / per_head, v = rest - h * per_head;
    uint4* cache = which ? v_cache : k_cache;
    const size_t page_vecs = size_t(kPage) * kVecPerRow;
    cache[(size_t(dst) * num_kv_heads + h) * page_vecs + v] =
        cache[(size_t(src) * num_kv_heads + h) * page_vecs + v];
  }
}

// Page transfer: buffer layout [n][2 (K, V)][Hkv][16][128] bf16, i.e. the
// listed pages back to back, each as its K rows then its V rows.  One thread
// moves 16 bytes; consecutive threads move consecutive bytes of one 4 KiB
// (page, head) block on both sides.
template <bool EXPORT>
__global__ void __launch_bounds__(256) pkv_transfer_kernel(uint4* __restrict__ k_cache,
                                                           uint4* __restrict__ v_cache,
                                                           uint4* __restrict__ buf,
                                                           const int32_t* __restrict__ pages,
                                                           int32_t n, int32_t num_kv_heads,
                                                           int32_t num_blocks,
                                                           unsigned* __restrict__ status) {
  constexpr int kVec = kPageBytes / 16;  // 256 vectors per (page, head)
  const int64_t total = int64_t(n) * 2 * num_kv_heads * kVec;
  for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < total;
       i += int64_t(gridDim.x) * blockDim.x) {
    const int v = int(i % kVec);
    const int64_t blk = i / kVec;  // (page index, K/V, head) in buffer order
    const int h = int(blk % num_kv_heads);
    const int which = int((blk / num_kv_heads) % 2);
    const int64_t k = blk / (2 * num_kv_heads);
    const int32_t page = __ldg(pages + k);
    if (page < 0 || page >= num_blocks) {
      if (v == 0 && which == 0 && h == 0) flag_status(status, PKV_STATUS_BAD_BLOCK);
      continue;
    }
    uint4* cache = which ? v_cache : k_cache;
    uint4* slot = cache + (int64_t(page) * num_kv_heads + h) * kVec + v;
    if (EXPORT) buf[i] = *slot;
    else *slot = buf[i];
  }
}

static int transfer(bool export_dir, pkv_bf16* k_cache, pkv_bf16* v_cache, pkv_bf16* buf,
                    const int32_t* pages, int32_t n, const pkv_desc* d, pkv_stream_t stream) {
  if (!d) return PKV_ERR_NULL;
  if (d->head_dim != kHeadDim || d->page_size != kPage || d->num_kv_heads <= 0) return PKV_ERR_SHAPE;
  if (n < 0 || d->num_blocks <= 0) return PKV_ERR_RANGE;
  if (n == 0) return PKV_OK;
  if (!k_cache || !v_cache || !buf || !pages) return PKV_ERR_NULL;
  auto mis = [](const void* x) { return reinterpret_cast<uintptr_t>(x) % 16 != 0; };
  if (mis(k_cache) || mis(v_cache) || mis(buf) || reinterpret_cast<uintptr_t>(pages) % 4)
    return PKV_ERR_ALIGN;
  int err = PKV_OK;
  const DeviceInfo* dev = current_device(&err);
  if (!dev) return err;
  void* status = status_word(dev->device);
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int64_t total = int64_t(n) * 2 * d->num_kv_heads * (kPageBytes / 16);
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, int64_t(dev->sm_count) * 8);
  TraceScope ts(s, PKV_K_WRITE);
  if (export_dir)
    pkv_transfer_kernel<true><<<unsigned(blocks), 256, 0, s>>>(
        reinterpret_cast<uint4*>(k_cache), reinterpret_cast<uint4*>(v_cache),
        reinterpret_cast<uint4*>(buf), pages, n, d->num_kv_heads, d->num_blocks,
        static_cast<unsigned*>(status));
  else
    pkv_transfer_kernel<false><<<unsigned(blocks), 256, 0, s>>>(
        reinterpret_cast<uint4*>(k_cache), reinterpret_cast<uint4*>(v_cache),
        reinterpret_cast<uint4*>(buf), pages, n, d->num_kv_heads, d->num_blocks,
        static_cast<unsigned*>(status));
  return ts.done();
}

}  // namespace pkv

using namespace pkv;

extern "C" {

PKV_API int pkv_pool_create(int32_t num_blocks, pkv_pool** out) {
  if (!out) return PKV_ERR_NULL;
  if (num_blocks <= 0) return PKV_ERR_RANGE;
  auto* p = new pkv_pool();
  p->refs.assign(size_t(num_blocks), 0);
  p->free_list.reserve(size_t(num_blocks));
  for (int32_t b = num_blocks - 1; b >= 0; --b) p->free_list.push_back(b);  // page 0 first
  *out = p;
  return PKV_OK;
}

PKV_API int pkv_pool_destroy(pkv_pool* p) {
  if (!p) return PKV_ERR_NULL;
  delete p;
  return PKV_OK;
}

PKV_API int pkv_pool_alloc(pkv_pool* p, int32_t n, int32_t* pages) {
  if (!p || (n > 0 && !pages)) return PKV_ERR_NULL;
  if (n < 0) return PKV_ERR_RANGE;
  std::lock_guard<std::mutex> lk(p->mu);
  if (size_t(n) > p->free_list.size()) return PKV_ERR_NOSPACE;  // all or nothing
  for (int32_t i = 0; i < n; ++i) {
    const int32_t b = p->free_list.back();
    p->free_list.pop_back();
    p->refs[size_t(b)] = 1;
    pages[i] = b;
  }
  p->allocs += n;
  return PKV_OK;
}

// Checks every page first, so a bad list changes nothing.
static int check_live(const pkv_pool* p, const int32_t* pages, int32_t n) {
  for (int32_t i = 0; i < n; ++i) {
    const int32_t b = pages[i];
    if (b < 0 || size_t(b) >= p->refs.size()) return PKV_ERR_RANGE;
    if (p->refs[size_t(b)] <= 0) return PKV_ERR_STATE;
  }
  return PKV_OK;
}

PKV_API int pkv_pool_retain(pkv_pool* p, const int32_t* pages, int32_t n) {
  if (!p || (n > 0 && !pages)) return PKV_ERR_NULL;
  if (n < 0) return PKV_ERR_RANGE;
  std::lock_guard<std::mutex> lk(p->mu);
  if (int e = check_live(p, pages, n)) return e;
  for (int32_t i = 0; i < n; ++i) ++p->refs[size_t(pages[i])];
  return PKV_OK;
}

PKV_API int pkv_pool_release(pkv_pool* p, const int32_t* pages, int32_t n) {
  if (!p || (n > 0 && !pages)) return PKV_ERR_NULL;
  if (n < 0) return PKV_ERR_RANGE;
  std::lock_guard<std::mutex> lk(p->mu);
  if (int e = check_live(p, pages, n)) return e;
  // a page listed twice must hold two references
  for (int32_t i = 0; i < n; ++i) {
    int32_t times = 0;
    for (int32_t j = 0; j < n; ++j) times += pages[j] == pages[i];
    if (times > p->refs[size_t(pages[i])]) return PKV_ERR_STATE;
  }
  for (int32_t i = 0; i < n; ++i) {
    int32_t& r = p->refs[size_t(pages[i])];
    if (--r == 0) {
      p->free_list.push_back(pages[i]);
      ++p->frees;
    }
  }
  return PKV_OK;
}

PKV_API int pkv_pool_refcount(pkv_pool* p, int32_t page, int32_t* count) {
  if (!p || !count) return PKV_ERR_NULL;
  std::lock_guard<std::mutex> lk(p->mu);
  if (page < 0 || size_t(page) >= p->refs.size()) return PKV_ERR_RANGE;
  *count = p->refs[size_t(page)];
  return PKV_OK;
}

PKV_API int pkv_pool_usage(pkv_pool* p, int32_t* used, int32_t* total) {
  if (!p || !used || !total) return PKV_ERR_NULL;
  std::lock_guard<std::mutex> lk(p->mu);
  *total = int32_t(p->refs.size());
  *used = *total - int32_t(p->free_list.size());
  return PKV_OK;
}

PKV_API int pkv_pool_make_writable(pkv_pool* p, int32_t page, int32_t rows, pkv_bf16* k_cache,
                                   pkv_bf16* v_cache, const pkv_desc* desc, pkv_stream_t stream,
                                   int32_t* new_page) {
  if (!p || !new_page || !desc) return PKV_ERR_NULL;
  if (desc->head_dim != kHeadDim || desc->page_size != kPage || desc->num_kv_heads <= 0)
    return PKV_ERR_SHAPE;
  if (rows < 0 || rows > kPage || size_t(desc->num_blocks) != p->refs.size()) return PKV_ERR_RANGE;
  int32_t fresh = -1;
  {
    std::lock_guard<std::mutex> lk(p->mu);
    if (page < 0 || size_t(page) >= p->refs.size()) return PKV_ERR_RANGE;
    if (p->refs[size_t(page)] <= 0) return PKV_ERR_STATE;
    if (p->refs[size_t(page)] == 1) {  // already private
      *new_page = page;
      return PKV_OK;
    }
    if (p->free_list.empty()) return PKV_ERR_NOSPACE;
    fresh = p->free_list.back();
    p->free_list.pop_back();
    p->refs[size_t(fresh)] = 1;
    --p->refs[size_t(page)];  // still >= 1: the other sharers keep it
    ++p->allocs;
  }
  *new_page = fresh;
  if (rows == 0) return PKV_OK;
  if (!k_cache || !v_cache) return PKV_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(k_cache) % 16 || reinterpret_cast<uintptr_t>(v_cache) % 16)
    return PKV_ERR_ALIGN;
  int err = PKV_OK;
  if (!current_device(&err)) return err;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int total = 2 * desc->num_kv_heads * rows * (kHeadDim * 2 / 16);
  TraceScope ts(s, PKV_K_WRITE);
  pkv_copy_page_kernel<<<(total + 255) / 256, 256, 0, s>>>(
      reinterpret_cast<uint4*>(k_cache), reinterpret_cast<uint4*>(v_cache), page, fresh, rows,
      desc->num_kv_heads);
  return ts.done();
}

PKV_API int pkv_export_pages(const pkv_bf16* k_cache, const pkv_bf16* v_cache,
                             const int32_t* pages, int32_t n, pkv_bf16* dst,
                             const pkv_desc* desc, pkv_stream_t stream) {
  return transfer(true, const_cast<pkv_bf16*>(k_cache), const_cast<pkv_bf16*>(v_cache), dst, pages,
                  n, desc, stream);
}

PKV_API int pkv_import_pages(const pkv_bf16* src, const int32_t* pages, int32_t n,
                             pkv_bf16* k_cache, pkv_bf16* v_cache, const pkv_desc* desc,
                             pkv_stream_t stream) {
  return transfer(false, k_cache, v_cache, const_cast<pkv_bf16*>(src), pages, n, desc, stream);
}

}  // extern "C"
