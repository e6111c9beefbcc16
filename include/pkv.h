/*
 * pkv.h -- C ABI of the GB300 paged-KV attention step (libpkv.so).
 *
 * One step of a unified prefill/decode scheduler: every request in the step advances
 * by q_len tokens (1 for a decode, a causal chunk for a chunked prefill) on top of the
 * context_len tokens it already has in a paged KV cache.  This is the problem as
 * niuwancheng.cn "11. chunked prefill and unified scheduling" states it (section "token
 * budget per step": each request records how many tokens are computed and how many it
 * advances this step), with 16-token pages addressed through a block table
 * (lshu.cn/news/11576 §2.2 "written by page index", §2.3 "16 tokens per block").
 *
 * Call order within a step (hotelren.com/news/6181127 §3.1: append the new K/V, then
 * score against all S+t cached keys): pkv_kv_append, then pkv_paged_attention_step.
 *
 * Conventions for every entry point
 *  - Pointers named d_* or documented "device" are CUDA device pointers; all other
 *    pointers are host pointers.  The caller owns every buffer; the library allocates
 *    nothing and keeps no per-call state.
 *  - Pinned host memory (cudaHostAlloc / cudaMallocHost) is mapped into the device's
 *    address space at the same address (unified addressing).  q, k_new, v_new, out,
 *    slot_mapping_out and the step description's four arrays may point there: the kernels
 *    read and write them with plain loads and stores, which reach host memory over the
 *    CPU-GPU link (NVLink-C2C on GB300), so a step moves its inputs and output with no
 *    separate copy.  Exceptions: a step with max_q_len >= 16 (requests with 16 or more
 *    new tokens run on the tensor-core prefill kernel) reads q with tensor-memory-
 *    accelerator copies, which need device memory -- a host q is refused there with
 *    PKV_ERR_INVALID_ARG; the pools, the scales, the workspace and the error flag are
 *    device memory always.
 *  - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *    Work is enqueued asynchronously; only pkv_read_device_error synchronises.
 *  - Return value: PKV_OK (0) or a negative pkv_status.  On an error detected on the
 *    host nothing is launched.  Inconsistent device data (a page id outside the pool, a
 *    position past the block-table row, q_offsets that disagree with total_q_tokens)
 *    never traps: the kernel ORs a bit into *dev_err_flag (when non-NULL), skips the
 *    offending token / tile and completes; read the flag with pkv_read_device_error.
 *
 * Tensor layouts (row-major, innermost last)
 *   q, out      [total_q_tokens][num_q_heads][head_dim]      dtype
 *   k_new,v_new [total_q_tokens][num_kv_heads][head_dim]     dtype
 *   k_cache,
 *   v_cache     [num_pages][num_kv_heads][16][head_dim]      dtype
 *               (one contiguous 16 x head_dim block per page and KV head)
 *   block_table [num_reqs][max_pages_per_req] int32 physical page ids
 *   Token t of the step belongs to request r when q_offsets[r] <= t < q_offsets[r+1];
 *   its position is context_lens[r] + (t - q_offsets[r]); it lives in page
 *   block_table[r][pos / 16], slot pos % 16 (global slot id page * 16 + pos % 16).
 *   Query head h reads KV head h / (num_q_heads / num_kv_heads).
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PKV_PAGE_SIZE 16

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

typedef enum { PKV_BF16 = 0, PKV_FP16 = 1 } pkv_dtype;

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = -1,     /* null pointer, negative size, page_size != 16, ... */
    PKV_ERR_UNSUPPORTED = -2,     /* head_dim not 64/128, Hq % Hkv != 0, group > 8, dtype,
                                     a pool of 2^31 or more (page, KV head, token) rows */
    PKV_ERR_CAPACITY = -3,        /* max_context_len + max_q_len beyond the block table */
    PKV_ERR_WORKSPACE = -4,       /* workspace NULL or smaller than required */
    PKV_ERR_CUDA = -5,            /* a CUDA runtime call or launch failed */
    PKV_ERR_DEVICE = -6,          /* pkv_read_device_error found a non-zero flag */
    PKV_ERR_NO_PAGES = -7         /* the scheduler's page pool cannot cover the step */
} pkv_status;

/* Bits OR-ed into *dev_err_flag by the kernels. */
#define PKV_DEVERR_PAGE_RANGE 1   /* page id outside [0, num_pages) */
#define PKV_DEVERR_TABLE_RANGE 2  /* position past max_pages_per_req * 16 */
#define PKV_DEVERR_TOKENS 4       /* q_offsets[num_reqs] != total_q_tokens, or lengths
                                     above the host-declared maxima */
#define PKV_DEVERR_TIMEOUT 8      /* a bounded wait on an asynchronous copy gave up */

/*
 * Description of one step.  Host integers size the launches; the four arrays are device
 * pointers the kernels read.  The host integers must bound the device data:
 *   total_q_tokens == q_offsets[num_reqs], max_q_len >= every q_lens[r],
 *   max_context_len >= every context_lens[r],
 *   ceil((max_context_len + max_q_len) / 16) <= max_pages_per_req is NOT required
 *   (tables may be sized per request) but every request's own
 *   ceil((context_lens[r] + q_lens[r]) / 16) must fit in max_pages_per_req.
 */
typedef struct {
    int32_t num_reqs;            /* requests in the step (>= 0) */
    int32_t num_q_heads;         /* Hq */
    int32_t num_kv_heads;        /* Hkv, Hq % Hkv == 0, Hq / Hkv in {1, 2, 4, 8} */
    int32_t head_dim;            /* D in {64, 128} */
    int32_t page_size;           /* must be 16 */
    int32_t num_pages;           /* pages in each pool; num_pages * Hkv * 16 < 2^31 */
    int32_t max_pages_per_req;   /* block_table row stride */
    int32_t total_q_tokens;      /* T = sum of q_lens */
    int32_t max_q_len;
    int32_t max_context_len;
    int32_t dtype;               /* pkv_dtype; one dtype for q, k, v, out */
    const int32_t* q_lens;       /* device [num_reqs] */
    const int32_t* q_offsets;    /* device [num_reqs + 1], exclusive prefix sum of q_lens */
    const int32_t* context_lens; /* device [num_reqs], tokens cached BEFORE this step */
    const int32_t* block_table;  /* device [num_reqs * max_pages_per_req] */
} pkv_step_desc;

/*
 * pkv_kv_append -- write this step's new K/V rows into their pages.
 * Defined by lshu.cn/news/11576 §2.2 (K/V written by page index into a pre-allocated
 * pool of fixed pages) and hotelren.com/news/6181127 §3.1 (the new K and V are appended,
 * the cache grows from S+t-1 to S+t).
 *   k_new, v_new       device [T][Hkv][D]
 *   k_cache, v_cache   device [num_pages][Hkv][16][D], updated in place (only the
 *                      slots of this step's tokens are written; bit-exact copies)
 *   slot_mapping_out   device int64 [T] or NULL: receives page * 16 + pos % 16
 *   dev_err_flag       device int32 or NULL (see PKV_DEVERR_*)
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA.  T == 0 is a no-op returning PKV_OK.
 */
PKV_API int pkv_kv_append(const pkv_step_desc* desc, const void* k_new, const void* v_new,
                  void* k_cache, void* v_cache, int64_t* slot_mapping_out,
                  int32_t* dev_err_flag, void* stream);

/*
 * pkv_advance_context -- context_lens[r] += q_lens[r] for every request of *desc, on the
 * device.  After a step the tokens it appended are cached, so the next step of the same
 * batch starts from the grown lengths (niuwancheng.cn "11. Chunked prefill and unified
 * scheduling": each request records the tokens computed so far).  With it, consecutive
 * steps of one batch need no host upload between them and can be captured in one CUDA
 * graph; the block table must already hold the pages the later steps reach.
 *   context_lens   device int32 [num_reqs], updated in place (normally desc->context_lens)
 * Errors: INVALID_ARG, CUDA.  num_reqs == 0 is a no-op returning PKV_OK.  The kernel waits
 * for earlier kernels on the stream that read the lengths before it writes them.
 */
PKV_API int pkv_advance_context(const pkv_step_desc* desc, int32_t* context_lens, void* stream);

/*
 * pkv_attention_workspace_bytes -- device workspace the attention step needs for this
 * description (split-KV partial results and the device-built work list).  Depends only
 * on the host integers of *desc and on the current device's SM count.  Returns 0 for
 * an invalid description.
 */
PKV_API size_t pkv_attention_workspace_bytes(const pkv_step_desc* desc);

/*
 * pkv_paged_attention_step -- causal softmax attention of every new query row over all
 * keys of its request up to and including its own position, K/V read from the pages.
 * Defined by hotelren.com/news/6181127 §1.1 (position i depends on 0..i), §2.1 (scores
 * masked to -inf above the diagonal, row softmax, times V), §3.1 (a decode row scores
 * all S+t cached keys), §5.1 skeleton softmax(q K^T) V with the scale made explicit;
 * niuwancheng.cn "11. chunked prefill..." (a chunk reads the earlier chunks' K/V like a
 * decode, same result as one-shot).
 *   q             device [T][Hq][D]
 *   k_cache,
 *   v_cache       device pools (after this step's pkv_kv_append)
 *   out           device [T][Hq][D], written in full (fp32 accumulation, rounded to
 *                 nearest-even at the end)
 *   scale         multiplies q.k before the softmax (1/sqrt(D) for standard attention)
 *   workspace     device, >= pkv_attention_workspace_bytes(desc) bytes, 256-byte aligned;
 *                 contents need no initialisation and are clobbered
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE, CUDA.
 */
PKV_API int pkv_paged_attention_step(const pkv_step_desc* desc, const void* q, const void* k_cache,
                             const void* v_cache, void* out, float scale, void* workspace,
                             size_t workspace_bytes, int32_t* dev_err_flag, void* stream);

/*
 * pkv_append_attention -- pkv_kv_append followed by pkv_paged_attention_step, in one call
 * (16-bit pools): arguments, results, slot ids and errors are those of the two calls.  When
 * every request advances by at most one token (a decode step) and there are at most 256
 * requests, a single decode grid does both: the warp that streams a (request, KV head)'s
 * last page first writes the request's new K and V rows into it (hotelren.com/news/6181127
 * §3.1: append, then attend over all S+t keys), so no separate append launch or dependency
 * hop sits in the step.  Other steps run the append kernel, then the attention step.  On
 * inconsistent lengths (PKV_DEVERR_TOKENS) such a decode step appends nothing.
 */
PKV_API int pkv_append_attention(const pkv_step_desc* desc, const void* k_new, const void* v_new,
                                 void* k_cache, void* v_cache, int64_t* slot_mapping_out,
                                 const void* q, void* out, float scale, void* workspace,
                                 size_t workspace_bytes, int32_t* dev_err_flag, void* stream);

/*
 * pkv_append_attention_int8 -- pkv_kv_append_int8 followed by pkv_paged_attention_step_int8,
 * in one call (INT8 pools; the arguments of those two calls).  Decode steps of at most 256
 * requests run as one decode grid, as in pkv_append_attention: the warp that streams a
 * (request, KV head)'s last page quantises the request's new K and V rows with the same
 * arithmetic as pkv_kv_append_int8 (so the pool bytes and slot ids are identical) and writes
 * them into that page before reading it.  Other steps run the two calls' kernels.
 */
PKV_API int pkv_append_attention_int8(const pkv_step_desc* desc, const void* k_new,
                                      const void* v_new, const float* k_scale,
                                      const float* v_scale, int8_t* k_cache, int8_t* v_cache,
                                      int64_t* slot_mapping_out, const void* q, void* out,
                                      float scale, void* workspace, size_t workspace_bytes,
                                      int32_t* dev_err_flag, void* stream);

/*
 * pkv_plan_attention, pkv_paged_attention_run -- the attention step in two halves, so that
 * one plan serves every layer of a model step.  The step's work list (decode rows, split-KV
 * items, prefill tiles) depends only on the lengths and the block table, which every layer
 * of a step shares (niuwancheng.cn "11. Chunked prefill and unified scheduling": the step's
 * token budget is divided among requests once per step); the K/V pools, Q and the output
 * are per layer.  pkv_paged_attention_step(...) is exactly pkv_plan_attention followed by
 * pkv_paged_attention_run on the same stream.
 *   pkv_plan_attention   validates the lengths on the device (as the full step does) and
 *                        writes the work list into `workspace`; q, pools and output are not
 *                        touched.
 *   pkv_paged_attention_run(_int8)   the attention kernels over the plan in `workspace`:
 *                        same arguments and results as pkv_paged_attention_step(_int8).
 *                        The plan must come from pkv_plan_attention (or a full step) with the
 *                        same host integers and unchanged device arrays, enqueued earlier on
 *                        the same stream into the same workspace, with no other plan into it
 *                        since; any number of runs may follow one plan.  The plan is the same
 *                        for 16-bit and INT8 pools.
 * Errors: those of pkv_paged_attention_step (the plan call does not check q, pools, out).
 */
PKV_API int pkv_plan_attention(const pkv_step_desc* desc, void* workspace,
                               size_t workspace_bytes, int32_t* dev_err_flag, void* stream);
PKV_API int pkv_paged_attention_run(const pkv_step_desc* desc, const void* q,
                                    const void* k_cache, const void* v_cache, void* out,
                                    float scale, void* workspace, size_t workspace_bytes,
                                    int32_t* dev_err_flag, void* stream);

/*
 * pkv_paged_attention_step_static_ws -- the same attention step as
 * pkv_paged_attention_step, for callers that cannot allocate device memory when they call
 * it.  Examples are code that runs from a plugin or callback that must not synchronise the
 * device (cudaMalloc and cudaFree can synchronise it), and runtimes that hand out all
 * device memory once at start-up and allow no allocation afterwards.  This entry point
 * allocates nothing: its scratch (the work list and split-KV partial results) lives in a
 * fixed array compiled into the library, PKV_STATIC_WORKSPACE_BYTES (32 MiB) on every GPU
 * that loads the library, held until the process exits.  The pages have no counterpart to
 * this call; it only changes where the scratch memory comes from.
 *   Arguments and results are those of pkv_paged_attention_step without the workspace.
 *   A step whose pkv_attention_workspace_bytes exceeds PKV_STATIC_WORKSPACE_BYTES is
 *   rejected with PKV_ERR_WORKSPACE before anything is launched.
 *   The first call on each device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call before any
 *   stream capture.  Later calls on the device reuse the address.
 *   Every call on a device shares the one array, which keeps the previous call's
 *   contents (the step initialises what it needs, nothing has to start at zero).  Calls
 *   that overlap on the GPU -- on different streams, or from several host threads without
 *   ordering -- race on the array: issue them in order on one stream.
 */
#define PKV_STATIC_WORKSPACE_BYTES (32u << 20)
PKV_API int pkv_paged_attention_step_static_ws(const pkv_step_desc* desc, const void* q,
                                               const void* k_cache, const void* v_cache,
                                               void* out, float scale, int32_t* dev_err_flag,
                                               void* stream);

/*
 * INT8 KV cache (wmrh.cn/news/64708 §4.3: the cache held in INT8 instead of FP16 halves its
 * bytes; §5.4: quantising the cache is the lever for long contexts).  The pages have the
 * layout above with one signed byte per element; each KV head and channel has a fixed
 * fp32 scale (per-channel, calibrated before the pool is filled):
 *   code  = clamp(round_half_even(x / scale[h][c]), -127, 127)   (IEEE fp32 quotient)
 *   value = code * scale[h][c]
 * The attention step reads the codes and attends over the values they stand for.  Its
 * scores and weighted sums run on the tensor cores with fp16 operands: the codes exactly,
 * q times the key scales (scaled by a power of two into fp16 range) and the softmax weights
 * rounded to fp16, with fp32 accumulation and softmax; the value scales are applied to the
 * fp32 sums.  Decode rows stream through the split-KV kernel and prefill chunks run as
 * 128-row tiles, as for 16-bit pages.
 *   k_scale, v_scale   device fp32 [num_kv_heads][head_dim], 16-byte aligned, > 0
 *   k_cache            device int8 [num_pages][num_kv_heads][16][head_dim]
 *   v_cache            device int8 [num_pages][num_kv_heads][head_dim][16]: within a page
 *                      block the 16 tokens of one dim are contiguous (the order the
 *                      tensor-core value fragments read)
 * Other arguments, errors and the device error flag are those of the 16-bit calls;
 * k_new, v_new, q and out keep desc->dtype.
 */
PKV_API int pkv_kv_append_int8(const pkv_step_desc* desc, const void* k_new, const void* v_new,
                               const float* k_scale, const float* v_scale, int8_t* k_cache,
                               int8_t* v_cache, int64_t* slot_mapping_out,
                               int32_t* dev_err_flag, void* stream);
PKV_API size_t pkv_attention_workspace_bytes_int8(const pkv_step_desc* desc);
/* the run half over INT8 pools (see pkv_plan_attention) */
PKV_API int pkv_paged_attention_run_int8(const pkv_step_desc* desc, const void* q,
                                         const int8_t* k_cache, const int8_t* v_cache,
                                         const float* k_scale, const float* v_scale,
                                         void* out, float scale, void* workspace,
                                         size_t workspace_bytes, int32_t* dev_err_flag,
                                         void* stream);
PKV_API int pkv_paged_attention_step_int8(const pkv_step_desc* desc, const void* q,
                                          const int8_t* k_cache, const int8_t* v_cache,
                                          const float* k_scale, const float* v_scale,
                                          void* out, float scale, void* workspace,
                                          size_t workspace_bytes, int32_t* dev_err_flag,
                                          void* stream);

/*
 * pkv_copy_pages -- copy whole pages, K and V, from src_pages[i] to dst_pages[i] for
 * i < num_copies: every KV head's 16 slots, bit for bit.  This is the copy-on-write of a
 * page several requests share (include/pkv_sched.h, pkv_sched_fork) before one of them
 * appends into it; enqueue it before that step's pkv_kv_append.  hotelren.com/news/6181127
 * §4.3: cached K/V reused across requests, memory managed by page.
 *   desc             only num_kv_heads, head_dim, page_size, num_pages and dtype are read
 *   src_pages,
 *   dst_pages        device int32 [num_copies]; a destination must not be a source or
 *                    appear twice
 *   k_cache, v_cache the pools: 16-bit (kv_int8 = 0) or INT8 (kv_int8 = 1); a page is the
 *                    same contiguous block of every pool either way
 * A page id outside the pool sets PKV_DEVERR_PAGE_RANGE and that copy is skipped.
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA.  num_copies == 0 is a no-op returning PKV_OK.
 */
PKV_API int pkv_copy_pages(const pkv_step_desc* desc, const int32_t* src_pages,
                           const int32_t* dst_pages, int32_t num_copies, void* k_cache,
                           void* v_cache, int kv_int8, int32_t* dev_err_flag, void* stream);

/*
 * pkv_read_device_error -- synchronise `stream`, copy *dev_err_flag (device) to
 * *host_value and return PKV_OK when it is zero, PKV_ERR_DEVICE when not, PKV_ERR_CUDA
 * when the copy fails.  The only synchronising entry point.
 */
PKV_API int pkv_read_device_error(const int32_t* dev_err_flag, int32_t* host_value, void* stream);

/*
 * pkv_set_kernel_events -- optional timing hook for benchmarks.  While set, each
 * pkv_paged_attention_step call on this host thread records `start` on its stream just
 * before the main kernel of the chosen path and `stop` just after it (which = 0: the
 * decode-stream kernel, which = 1: the tensor-core prefill kernel); a path that does not
 * launch in a call records nothing.  Events are cudaEvent_t passed as void*; NULL clears.
 * Returns PKV_OK, or PKV_ERR_INVALID_ARG for an unknown `which`.
 */
PKV_API int pkv_set_kernel_events(int which, void* start, void* stop);

/* Human-readable name of a pkv_status value (static storage). */
PKV_API const char* pkv_status_string(int status);

/* Library version as major * 10000 + minor * 100 + patch. */
PKV_API int pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
