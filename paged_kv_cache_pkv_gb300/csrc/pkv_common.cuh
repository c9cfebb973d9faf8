// pkv_common.cuh -- constants, workspace layout and PTX helpers shared by the
// paged-KV-cache kernels (sm_103a).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "../../include/pkv.h"

namespace pkv {

// Geometry this library is specialised for (checked on every call).
constexpr int kHeadDim = 128;   // D
constexpr int kPage = 16;       // tokens per page
constexpr int kPageBytes = kPage * kHeadDim * 2;  // one (page, kv head): 4 KiB
constexpr int kPageBytesF8 = kPage * kHeadDim;    // the same in E4M3 codes: 2 KiB
constexpr int kScaleBytes = kPage;                // FP8 row scales of one (page, kv head)

// Split-KV decode kernel shape.
#ifndef PKV_DEC_WARPS
#define PKV_DEC_WARPS 12
#endif
#ifndef PKV_DEC_STAGES
#define PKV_DEC_STAGES 2
#endif
#ifndef PKV_DEC_MIN_CTAS
#define PKV_DEC_MIN_CTAS 1
#endif
constexpr int kDecWarps = PKV_DEC_WARPS;    // warps per CTA
constexpr int kDecStages = PKV_DEC_STAGES;  // pages (K+V) in flight per warp
#ifndef PKV_DEC_STAGES_F8
#define PKV_DEC_STAGES_F8 3
#endif
#ifndef PKV_DEC_WARPS_F8
#define PKV_DEC_WARPS_F8 12
#endif
// FP8 pages are half the bytes: the same 12 warps keep 3 of them in flight.
constexpr int kDecStagesF8 = PKV_DEC_STAGES_F8;
constexpr int kDecWarpsF8 = PKV_DEC_WARPS_F8;
constexpr int kMaxGroupPerItem = 4;  // query heads sharing one page read

// A decode partial state of one warp: m[4], l[4], then o[heads][128] (fp32).
constexpr int kPartialHeader = 8;
__host__ __device__ constexpr int partial_floats(int heads) {
  return kPartialHeader + heads * kHeadDim;
}

// Bounded waits: a kernel gives up on an mbarrier or a counter after this
// many nanoseconds of polling, flags PKV_STATUS_TIMEOUT and returns (after
// letting its own copies and MMAs in flight land, within kDrainLimitNs).
// The limit is a build option so that a test build can make waits run out.
#ifndef PKV_WAIT_LIMIT_NS
#define PKV_WAIT_LIMIT_NS 200000000ull  // 200 ms
#endif
constexpr uint64_t kWaitLimitNs = PKV_WAIT_LIMIT_NS;
constexpr uint64_t kDrainLimitNs = 2ull * 1000 * 1000;   // 2 ms for the clean-up path
// Waits whose only purpose is to let a CTA's own copies or MMAs land before
// it releases shared memory or TMEM: never shorter than the drain limit.
constexpr uint64_t kLandLimitNs = kWaitLimitNs > kDrainLimitNs ? kWaitLimitNs : kDrainLimitNs;

// Shared-prefix partial record: o[128] unnormalised, then m (log2 domain)
// and l; padded to a 16-byte multiple.
constexpr int kPrefixRec = 132;

// Tensor-core prefill tiles: a Q tile is kPfRows query rows (kPfRows / G
// tokens x the G heads of one kv head), a K/V tile kPfKeys keys (8 pages).
constexpr int kPfRows = 128;
constexpr int kPfKeys = 128;

// Most sequences one pkv_attend call may carry (the per-sequence unit prefix
// of the split-KV plan lives in shared memory).
constexpr int kMaxSeqs = 2048;

// Workspace carve-up; every piece starts 256-byte aligned.
struct WorkspaceLayout {
  size_t counters, partials, tiles, prefix, total;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// counters_per_row: arrival counters per query row (items x warps per ring);
// heads_per_warp sizes one partial slot; every decode warp owns two slots.
inline WorkspaceLayout workspace_layout(int num_tokens, int counters_per_row, int nwarps,
                                        int heads_per_warp, int max_tiles,
                                        size_t prefix_records = 0) {
  WorkspaceLayout w{};
  size_t off = 0;
  auto take = [&](size_t bytes) { size_t at = off; off = align_up(off + bytes, 256); return at; };
  w.counters = take(sizeof(unsigned long long) * size_t(num_tokens) * size_t(counters_per_row));
  w.partials = take(sizeof(float) * size_t(partial_floats(heads_per_warp)) * 2 * size_t(nwarps));
  w.tiles = take(sizeof(int32_t) * 4 * size_t(max_tiles));
  w.prefix = take(sizeof(float) * size_t(kPrefixRec) * prefix_records);
  w.total = off;
  return w;
}

// A test build (PKV_TEST_DROP_FIRST_COPY) arms the barrier of a warp's first
// page (split-KV) and of a CTA's Q tiles (prefill) but issues no copy into
// it: the waits on those barriers run out, which exercises every timeout
// path.  Never defined in the library's normal build.
#ifdef PKV_TEST_DROP_FIRST_COPY
constexpr bool kDropFirstCopy = true;
#else
constexpr bool kDropFirstCopy = false;
#endif

// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Atomic add with acquire-release semantics at GPU scope: publishes what the
// caller wrote before it and, for the last arrival of a count, makes what the
// other arrivals wrote visible.
__device__ __forceinline__ unsigned long long atom_add_acq_rel(unsigned long long* p, unsigned long long v) {
  unsigned long long old;
  asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], %2;" : "=l"(old) : "l"(p), "l"(v) : "memory");
  return old;
}

__device__ __forceinline__ unsigned long long ld_acquire_gpu(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

// Arrival on a counter word that holds a 48-bit launch epoch over a 16-bit
// count.  The launch stamps (epoch, 0) into the word before any arrival can
// happen, but the stamp may not be visible yet, and an add that reaches the
// word before it is overwritten by it.  So: one add (the usual case, the
// stamp is there); if the word still held an older epoch, plain loads wait
// for the stamp (bounded) and the add is made again.  No arrival adds twice
// into an older epoch's word, so with fewer than 32768 arrivals per launch
// that word's count never carries into its epoch field.  Returns the count
// before this arrival, or -1 when the stamp did not appear in time.
__device__ __forceinline__ int arrive_stamped(unsigned long long* ctr, unsigned long long epoch) {
  unsigned long long v = atom_add_acq_rel(ctr, 1ull);
  if ((v >> 16) != epoch) {
    const uint64_t t0 = global_ns();
    while ((ld_acquire_gpu(ctr) >> 16) != epoch)
      if (global_ns() - t0 > kWaitLimitNs) return -1;
    v = atom_add_acq_rel(ctr, 1ull);
  }
  return int(v & 0xFFFFull);
}

// Programmatic dependent launch: wait until the grids this one depends on
// have completed and their writes are visible (returns at once without one).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Let the grid launched after this one start once every CTA has executed
// this or exited.
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Wait for the phase with the given parity; false once limit_ns have passed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity))
    if (global_ns() - t0 > limit_ns) return false;
  return true;
}

// mbar_wait that sleeps `sleep_ns` between tests once the first test failed:
// for warps whose wait is long and off the critical path, so that they leave
// their sub-partition's issue slots to a warp doing arithmetic.
__device__ __forceinline__ bool mbar_wait_backoff(uint64_t* bar, uint32_t parity, uint32_t sleep_ns,
                                                  uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    __nanosleep(sleep_ns);
    if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}


// L2 policy for data read exactly once (KV pages of a decode step).
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Hint: bring `bytes` (a multiple of 16, 16-byte aligned) at `src` into L2.
// L2 is the GPU's point of coherence, so a prefetch can never expose stale data
// to a later read.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// Bulk (non-tensor) async copy global -> shared, completing on an mbarrier.
// dst/src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// bf16x2 (packed in a 32-bit word, element 0 in the low half) -> two floats.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);  // .x = a (low half), .y = b
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ void flag_status(unsigned* status, unsigned bits) {
  if (status) atomicOr(status, bits);
}

}  // namespace pkv
