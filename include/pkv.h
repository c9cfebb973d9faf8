/*
 * pkv.h -- C ABI of the paged-KV-cache hot path for one GB300 (sm_103a).
 *
 * Two calls do the per-step work of a continuous batch:
 *   pkv_write   scatters this step's new K/V rows into fixed-size pages of a
 *               pool through a slot mapping;
 *   pkv_attend  runs grouped-query attention for every query row of the
 *               batch (decode rows and chunked-prefill rows alike), reading
 *               K/V through each sequence's block table.
 *
 * What the method is (sources: the pages this library is built from):
 *   - llm-d blog post "What does production-grade LLM inference look like?",
 *     introduction: serving engines keep a KV cache and raise throughput with
 *     paged attention and continuous batching; decode is memory-bandwidth
 *     bound, prefill compute bound.  Its routing-factor and prefix-producer
 *     paragraphs: a prompt whose prefix KV is already cached skips that
 *     prefill, i.e. cached pages are reused by later requests.
 *   - vLLM notes "EngineCoreClient: dos caminos de cliente, en proceso y
 *     multiproceso", "Flujo de datos": the engine reports num_gpu_blocks and
 *     the aligned block_size it reserved -> a pool of fixed-size pages.
 *   - TensorRT Edge-LLM "HTTP Inference Server Architecture", "Request
 *     Lifecycle" and "Extension Rules": the native runtime owns retained
 *     pages under a single-writer contract.
 * The pages give no layout, formula or kernel; the readings below are this
 * library's (pool layout, bottom-right causal alignment, kv head h/(Hq/Hkv)).
 *
 * Conventions for every call
 *   - All tensor pointers are DEVICE pointers on the current CUDA device,
 *     contiguous, row-major, 16-byte aligned; the caller owns them and keeps
 *     them alive until the stream has passed the call (the calls are
 *     stream-ordered and never synchronise or copy device->host).
 *   - The library allocates no device memory.  pkv_attend takes a
 *     caller-provided workspace sized by pkv_attend_workspace_size.
 *   - bf16 data are passed as raw 16-bit patterns (pkv_bf16).
 *   - Return value: PKV_OK (0) or a negative PKV_ERR_* code.  On an argument
 *     error nothing is launched.  Problems only the device can see (a page id
 *     outside the pool, a query count above its sequence length, a bounded
 *     wait that ran out) set bits of a per-device status word that
 *     pkv_get_last_error reads; results of such a call are undefined, but
 *     no out-of-bounds access is made and no kernel hangs.
 *   - The caller is the single writer of the pool: a slot written by
 *     pkv_write must lie in a page that belongs to one sequence only (pages
 *     shared through a common prefix are read-only), and no two tokens of
 *     one call may name the same slot.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t pkv_bf16;                 /* raw bfloat16 bits             */
typedef uint8_t pkv_fp8;                   /* E4M3 code (see FP8 pages)     */
typedef struct CUstream_st* pkv_stream_t;  /* same handle as cudaStream_t   */
typedef struct CUevent_st* pkv_event_t;    /* same handle as cudaEvent_t    */

/* ---- return codes --------------------------------------------------------- */
#define PKV_OK              0
#define PKV_ERR_NULL       (-1)  /* a required pointer is NULL                   */
#define PKV_ERR_ALIGN      (-2)  /* a pointer is not aligned as required         */
#define PKV_ERR_SHAPE      (-3)  /* unsupported head_dim / page_size / heads     */
#define PKV_ERR_RANGE      (-4)  /* a count or size is out of range              */
#define PKV_ERR_WORKSPACE  (-5)  /* workspace smaller than required              */
#define PKV_ERR_LAUNCH     (-6)  /* a CUDA launch or runtime call failed         */
#define PKV_ERR_DEVICE     (-7)  /* current device is not an sm_103 GPU          */
#define PKV_ERR_STATE      (-8)  /* misuse of the trace API                      */
#define PKV_ERR_SCRATCH    (-9)  /* batch too large for pkv_attend_static        */
#define PKV_ERR_NOSPACE   (-10)  /* page pool: not enough free pages             */

/* ---- device status bits (pkv_get_last_error) ------------------------------- */
#define PKV_STATUS_BAD_SLOT   0x1u  /* slot_mapping entry beyond the pool: skipped */
#define PKV_STATUS_BAD_BLOCK  0x2u  /* block_tables entry outside [0,num_blocks)  */
#define PKV_STATUS_BAD_QUERY  0x4u  /* query_start_loc/seq_lens inconsistent      */
#define PKV_STATUS_TIMEOUT    0x8u  /* a bounded wait in a kernel ran out         */

/* Page-pool and head geometry, checked on every call.
 *   k_cache and v_cache are each [num_blocks, num_kv_heads, page_size, head_dim]
 *   bf16: one (page, kv head) is page_size*head_dim contiguous values (4 KiB
 *   for 16 x 128), so a page of one head is a single contiguous copy.
 *   block_tables is [num_seqs, max_blocks_per_seq] int32.
 * Supported: head_dim == 128, page_size == 16, num_q_heads a multiple of
 * num_kv_heads with num_q_heads/num_kv_heads in {1, 2, 4, 8, 16}. */
typedef struct {
  int32_t num_blocks;          /* pages in the pool (vLLM's num_gpu_blocks)   */
  int32_t page_size;           /* tokens per page (vLLM's block_size)         */
  int32_t num_kv_heads;        /* Hkv                                         */
  int32_t num_q_heads;         /* Hq                                          */
  int32_t head_dim;            /* D                                           */
  int32_t max_blocks_per_seq;  /* row stride of block_tables                  */
} pkv_desc;

/* pkv_write -- scatter new K/V rows into the pool (KV write step).
 *   k_new, v_new   [num_tokens, num_kv_heads, head_dim] bf16, device.
 *   slot_mapping   [num_tokens] int64, device.  Token t goes to page
 *                  slot/page_size, row slot%page_size, for every kv head.
 *                  slot < 0: token skipped (padding).  A slot at or beyond
 *                  num_blocks*page_size is skipped and flags
 *                  PKV_STATUS_BAD_SLOT.
 *   k_cache, v_cache  pools, device, updated in place.
 *   num_tokens     >= 0; 0 launches nothing.
 * The copy is bit-exact. */
PKV_API int pkv_write(const pkv_bf16* k_new, const pkv_bf16* v_new,
              const int64_t* slot_mapping, int64_t num_tokens,
              pkv_bf16* k_cache, pkv_bf16* v_cache,
              const pkv_desc* desc, pkv_stream_t stream);

/* Most sequences a single pkv_attend call accepts (PKV_ERR_RANGE above). */
#define PKV_MAX_SEQS 2048
/* Sequences with more query rows than this use the tensor-core prefill
 * kernel (the environment variable PKV_SPLITKV_MAX_QLEN overrides it). */
#define PKV_SPLITKV_MAX_QLEN 8

/* Workspace bytes pkv_attend needs on the CURRENT device for a batch of up
 * to num_seqs sequences and num_tokens query rows (and shared_prefix_pages as
 * passed to pkv_attend).  Writes *bytes. */
PKV_API int pkv_attend_workspace_size(const pkv_desc* desc, int32_t num_seqs,
                              int32_t num_tokens, int32_t shared_prefix_pages,
                              size_t* bytes);

/* pkv_attend -- paged grouped-query attention of one continuous batch.
 *   q             [num_tokens, num_q_heads, head_dim] bf16, device.
 *   k_cache, v_cache  pools as in pkv_desc (already holding this step's rows).
 *   block_tables  [num_seqs, max_blocks_per_seq] int32: logical token j of
 *                 sequence b is in page block_tables[b][j/page_size], row
 *                 j%page_size.  Entries past a sequence's last page are never
 *                 read.  Several rows may name the same page (shared prefix).
 *   seq_lens      [num_seqs] int32: L_b, cached tokens including this step's.
 *   query_start_loc [num_seqs+1] int32, non-decreasing, [0] == 0,
 *                 [num_seqs] <= num_tokens: sequence b owns query rows
 *                 query_start_loc[b] .. query_start_loc[b+1]-1 (n_b rows,
 *                 n_b <= L_b).  Row j of b is at position L_b-n_b+j and sees
 *                 keys 0..L_b-n_b+j (bottom-right causal; n_b == 1 is
 *                 decode over all L_b keys).
 *   max_query_len host-side upper bound on n_b over the batch, or <= 0 if
 *                 unknown.  It only selects kernels: sequences with more
 *                 than PKV_SPLITKV_MAX_QLEN query rows run on the tensor-core
 *                 prefill kernel, the rest on split-KV; when the bound is at
 *                 most that threshold the prefill kernel is not launched and
 *                 split-KV takes every row, so a wrong bound never changes
 *                 results.
 *   shared_prefix_pages  0, or P > 0 when the first P entries of EVERY
 *                 block_tables row name the same pages: a prefix all the
 *                 sequences share (read-only; llm-d blog, prefix-cache
 *                 paragraphs).  Every query row is then attended to those
 *                 pages once, on the tensor cores, and split-KV reads only
 *                 each sequence's own pages after them, merging both parts
 *                 (cascade).  Rows of sequences on the split-KV path must have
 *                 at least one visible key past the prefix (else their
 *                 sequence is skipped and PKV_STATUS_BAD_QUERY is set); the
 *                 prefix is read through row 0 of block_tables.
 *   scale         softmax scale applied to q.k (e.g. 1/sqrt(head_dim)).
 *   out           [num_tokens, num_q_heads, head_dim] bf16, device; rows at
 *                 or beyond query_start_loc[num_seqs] are not written.
 *   workspace     device scratch of >= pkv_attend_workspace_size bytes,
 *                 256-byte aligned; contents need no initialisation.
 * Query head h reads kv head h / (num_q_heads/num_kv_heads).
 * Stream order: when pkv_attend directly follows pkv_write on a stream, its
 * set-up (reading seq_lens, query_start_loc and block_tables, and L2
 * prefetch hints for the first pages) overlaps the write kernel through
 * programmatic dependent launch; the pools are read only after the write has
 * finished.  Those three arrays must therefore not be
 * written by the pkv_write call right before it (pkv_write never does).
 * A call with query chunks longer than PKV_SPLITKV_MAX_QLEN runs its split-KV
 * kernel and its tensor-core prefill kernel at the same time on disjoint
 * SMs; work enqueued on the stream after the call still starts only once
 * both have finished.  The SM share follows the two kernels' work; it is
 * scaled by the environment variables PKV_PREFILL_STEP_UNITS (bf16 pages,
 * default 1900) and PKV_PREFILL_STEP_UNITS_FP8 (default 10000), read once
 * per process; 0 runs the prefill kernel first instead, with split-KV beside
 * it on the SMs it leaves free.  With shared_prefix_pages > 0 the prefill kernel always runs
 * first. */
PKV_API int pkv_attend(const pkv_bf16* q, const pkv_bf16* k_cache,
               const pkv_bf16* v_cache, const int32_t* block_tables,
               const int32_t* seq_lens, const int32_t* query_start_loc,
               int32_t num_seqs, int32_t num_tokens, int32_t max_query_len,
               int32_t shared_prefix_pages, float scale, pkv_bf16* out,
               void* workspace, size_t workspace_bytes, const pkv_desc* desc,
               pkv_stream_t stream);

/* pkv_attend_static -- pkv_attend for callers that cannot allocate device
 * memory.  The pages this library follows have no counterpart for this call;
 * it exists for users, not for the method.
 *
 * Who needs it: code that runs inside a host program which owns every byte
 * of device memory and forbids allocation once it has started (fixed memory
 * budgets decided at start-up), or a caller that reaches this library
 * through a plain C interface and only ever holds pointers handed to it,
 * with no device allocator of its own to size and create a workspace.
 *
 * Same arguments and results as pkv_attend, minus the workspace: the scratch
 * memory lives in a fixed array of PKV_STATIC_SCRATCH_BYTES bytes inside the
 * library, one per GPU that loads it, held until the process exits.  The
 * call allocates nothing, on the device or through any library.
 *   - Batches whose pkv_attend_workspace_size exceeds PKV_STATIC_SCRATCH_BYTES
 *     are rejected with PKV_ERR_SCRATCH before anything is launched.
 *   - The first call on each device looks up that device's copy of the array
 *     (with the device current); make that first call before any stream
 *     capture on the device.
 *   - All calls on a device share the one array and it keeps what the last
 *     call left there; the kernels need none of it cleared first.  Calls
 *     whose work overlaps on the GPU (different streams, no ordering between
 *     them) race on the array and give undefined results: serialise them. */
#define PKV_STATIC_SCRATCH_BYTES (16u << 20)
PKV_API int pkv_attend_static(const pkv_bf16* q, const pkv_bf16* k_cache,
                              const pkv_bf16* v_cache, const int32_t* block_tables,
                              const int32_t* seq_lens, const int32_t* query_start_loc,
                              int32_t num_seqs, int32_t num_tokens,
                              int32_t max_query_len, int32_t shared_prefix_pages,
                              float scale, pkv_bf16* out, const pkv_desc* desc,
                              pkv_stream_t stream);

/* ---- FP8 pages ------------------------------------------------------------ */
/* KV pages of 8-bit E4M3 codes (OCP 8-bit Floating Point Specification: sign,
 * 4 exponent bits with bias 7, 3 mantissa bits; largest magnitude 448) with
 * one power-of-two scale per row, halving the bytes decode reads.  The pages
 * this library follows do not describe 8-bit pages; the format is the OCP one
 * and the scaling is this library's:
 *   k_cache, v_cache  [num_blocks, num_kv_heads, 16, 128] E4M3 codes (2 KiB
 *                     per page and head); k_scale, v_scale [num_blocks,
 *                     num_kv_heads, 16] bytes: row (page, head, r) holds the
 *                     values code * 2^(scale - 127).
 * A single scale per page would have to be fixed before the page's later
 * tokens are known (a page fills one token per decode step), so each row of
 * a page carries its own.  All four arrays 16-byte aligned, device. */

/* pkv_write_fp8 -- pkv_write into FP8 pages.  Each new (token, kv head) row
 * of K and of V (bf16) gets e = the smallest integer with max|x| <= 448 * 2^e,
 * clamped to [-126, 127]; its codes are x * 2^-e rounded to the nearest E4M3
 * value (ties to even, sign kept, so -0 and negative values that round to 0
 * give 0x80) and its scale byte is e + 127.  Inputs must be finite.  Slots,
 * skipping and PKV_STATUS_BAD_SLOT as in pkv_write.  Deterministic: the same
 * row always gives the same bytes. */
PKV_API int pkv_write_fp8(const pkv_bf16* k_new, const pkv_bf16* v_new,
                          const int64_t* slot_mapping, int64_t num_tokens,
                          pkv_fp8* k_cache, pkv_fp8* v_cache, uint8_t* k_scale,
                          uint8_t* v_scale, const pkv_desc* desc, pkv_stream_t stream);

/* Workspace bytes pkv_attend_fp8 needs on the CURRENT device (its kernel
 * runs a different number of warps than pkv_attend's), for num_seqs
 * sequences, num_tokens query rows and shared_prefix_pages as passed to
 * pkv_attend_fp8.  Writes *bytes. */
PKV_API int pkv_attend_fp8_workspace_size(const pkv_desc* desc, int32_t num_seqs,
                                          int32_t num_tokens, int32_t shared_prefix_pages,
                                          size_t* bytes);

/* pkv_attend_fp8 -- pkv_attend over FP8 pages: the same result with K and V
 * the exact values code * 2^(scale - 127).  Query chunks longer than
 * PKV_SPLITKV_MAX_QLEN run on the tensor-core prefill kernel (the pages
 * widened exactly to bf16 in shared memory), the rest on split-KV, as in
 * pkv_attend; max_query_len and shared_prefix_pages (the cascade over a
 * prefix every sequence shares) have pkv_attend's meaning.  workspace: at
 * least pkv_attend_fp8_workspace_size(desc, num_seqs, num_tokens,
 * shared_prefix_pages) bytes, 256-byte aligned, no initialisation needed.  Scale bytes of rows a query sees must
 * lie in [1, 254] (pkv_write_fp8 writes nothing else); rows it does not see
 * are never used, whatever they hold. */
PKV_API int pkv_attend_fp8(const pkv_bf16* q, const pkv_fp8* k_cache,
                           const pkv_fp8* v_cache, const uint8_t* k_scale,
                           const uint8_t* v_scale, const int32_t* block_tables,
                           const int32_t* seq_lens, const int32_t* query_start_loc,
                           int32_t num_seqs, int32_t num_tokens, int32_t max_query_len,
                           int32_t shared_prefix_pages, float scale,
                           pkv_bf16* out, void* workspace, size_t workspace_bytes,
                           const pkv_desc* desc, pkv_stream_t stream);

/* ---- page pool (host side) ------------------------------------------------ */
/* The engine reserves num_gpu_blocks pages of block_size tokens (vLLM notes
 * "EngineCoreClient ...", "Flujo de datos"); the native coordinator owns the
 * retained pages with a single writer (TensorRT Edge-LLM "HTTP Inference
 * Server Architecture", "Request Lifecycle"); cached prefix pages are reused
 * by later requests and the usage fraction is exported as a gauge (llm-d
 * blog, prefix producers; vllm:kv_cache_usage_perc).  pkv_pool hands out
 * page ids for block tables, counts references to pages shared by several
 * sequences, and gives a sequence a private copy of a shared page before it
 * writes into it.  Calls are serialised by an internal mutex.  Page ids are
 * indices into the pools of pkv_desc (num_blocks must match). */
typedef struct pkv_pool pkv_pool;
PKV_API int pkv_pool_create(int32_t num_blocks, pkv_pool** out);
PKV_API int pkv_pool_destroy(pkv_pool* pool);
/* n fresh pages (reference count 1) into pages[0..n); all or nothing:
 * PKV_ERR_NOSPACE when fewer than n are free.  Recently freed pages first. */
PKV_API int pkv_pool_alloc(pkv_pool* pool, int32_t n, int32_t* pages);
/* One more reference to each listed page (a sequence reusing a prefix). */
PKV_API int pkv_pool_retain(pkv_pool* pool, const int32_t* pages, int32_t n);
/* Drop one reference per listed page; a page is freed at zero.  Releasing a
 * free page (or more references than held) is PKV_ERR_STATE and changes
 * nothing. */
PKV_API int pkv_pool_release(pkv_pool* pool, const int32_t* pages, int32_t n);
PKV_API int pkv_pool_refcount(pkv_pool* pool, int32_t page, int32_t* count);
/* Pages in use and in the pool; usage = used / total. */
PKV_API int pkv_pool_usage(pkv_pool* pool, int32_t* used, int32_t* total);
/* Copy-on-write: if `page` has one reference it is already private and is
 * returned in *new_page.  Otherwise a fresh page is taken, rows [0, rows) of
 * every kv head of `page` are copied into it (K and V, device, on `stream`),
 * the caller's reference moves to the fresh page and *new_page names it.
 * The caller then points its block table at *new_page. */
PKV_API int pkv_pool_make_writable(pkv_pool* pool, int32_t page, int32_t rows,
                                   pkv_bf16* k_cache, pkv_bf16* v_cache,
                                   const pkv_desc* desc, pkv_stream_t stream,
                                   int32_t* new_page);

/* ---- page transfer -------------------------------------------------------- */
/* Disaggregated serving moves a request's KV pages from the prefill engine to
 * the decode engine (llm-d blog, P/D disaggregation paragraphs; there over
 * RDMA).  These calls are its single-GPU part: copy whole pages between the
 * pools and a contiguous buffer laid out [n][2 (K, V)][num_kv_heads][16][128]
 * bf16, i.e. each listed page's K rows then its V rows.  The buffer may be
 * device memory or pinned host memory the GPU can reach (on GB300 pinned
 * host memory is read and written directly over NVLink-C2C).
 *   pages [n] int32, device (readable by the device): page ids; an id
 *   outside [0, num_blocks) is skipped and flags PKV_STATUS_BAD_BLOCK.
 * Stream-ordered; bit-exact. */
PKV_API int pkv_export_pages(const pkv_bf16* k_cache, const pkv_bf16* v_cache,
                             const int32_t* pages, int32_t n, pkv_bf16* dst,
                             const pkv_desc* desc, pkv_stream_t stream);
PKV_API int pkv_import_pages(const pkv_bf16* src, const int32_t* pages, int32_t n,
                             pkv_bf16* k_cache, pkv_bf16* v_cache,
                             const pkv_desc* desc, pkv_stream_t stream);

/* Wait for `stream`, then read and clear the current device's status word
 * (PKV_STATUS_* bits) into *flags. */
PKV_API int pkv_get_last_error(pkv_stream_t stream, uint32_t* flags);

/* Human-readable text for a PKV_ERR_* code. */
PKV_API const char* pkv_strerror(int code);

/* Total kernel launches this process has made through the library. */
PKV_API uint64_t pkv_launch_count(void);

/* ---- tracing: per-kernel device time, recorded with CUDA events ----------- */
/* Kernel ids used by the trace. */
#define PKV_K_WRITE    0
#define PKV_K_PLAN     1
#define PKV_K_DECODE   2
#define PKV_K_MERGE    3
#define PKV_K_PREFILL  4
#define PKV_K_COUNT    5

typedef struct pkv_trace pkv_trace;
/* Create a trace with room for `capacity` launches (creates 2*capacity CUDA
 * events on the current device; not meant for the hot path). */
PKV_API int pkv_trace_create(int32_t capacity, pkv_trace** out);
/* While a trace is attached to the calling thread, every launch the library
 * makes on that thread records an event before and after it. */
PKV_API int pkv_trace_attach(pkv_trace* tr);
PKV_API int pkv_trace_detach(void);
/* Wait for the recorded events and sum per kernel id: total milliseconds and
 * number of launches.  Launches beyond the capacity are counted, not timed. */
PKV_API int pkv_trace_read(pkv_trace* tr, int32_t kernel_id, double* total_ms,
                   int64_t* launches);
PKV_API int pkv_trace_reset(pkv_trace* tr);
PKV_API int pkv_trace_destroy(pkv_trace* tr);

#ifdef __cplusplus
}
#endif
#endif /* PKV_H */
