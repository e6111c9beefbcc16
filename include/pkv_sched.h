/*
 * pkv_sched.h -- C ABI of the host-side step planner and page allocator (libpkv.so).
 *
 * The planner of a unified prefill/decode scheduler, as niuwancheng.cn "11. Chunked
 * prefill and unified scheduling" describes it (section "token budget per step"):
 *  - every request records the tokens already computed (cached) and the tokens it needs;
 *  - each step gives every decoding request 1 token first, then prefilling requests take
 *    min(remaining input, remaining budget) (optionally capped per chunk) in request order;
 *  - a step never exceeds the token budget.
 * Pages hold 16 tokens (lshu.cn/news/11576 §2.3) and come from a free list as a request's
 * cached length crosses a page boundary (§2.2: K/V written by page index).  A plan is
 * written straight into the arrays pkv_kv_append and pkv_paged_attention_step consume.
 *
 * Host code only: no CUDA call, safe to use without a GPU.  A scheduler handle is not
 * thread-safe; use one per thread or lock around it.  Every call that plans a step either
 * succeeds completely or leaves the scheduler exactly as it was.
 */
#ifndef PKV_SCHED_H_
#define PKV_SCHED_H_

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_scheduler pkv_scheduler;  /* opaque */

/*
 * One planned step, written into caller-owned host arrays.
 *   in:  max_reqs            capacity of rids, q_lens, context_lens (q_offsets: +1)
 *        max_pages_per_req   row stride of block_table (pass it as the step
 *                            description's max_pages_per_req)
 *        rids .. block_table host arrays of those capacities
 *        max_copies          capacity of copy_src, copy_dst (may be 0 with NULL arrays
 *                            when no request is ever forked)
 *   out: num_reqs            requests in the step, in launch order
 *        total_q_tokens      sum of q_lens
 *        max_q_len, max_context_len
 *        pages_used          longest block-table row of the step (<= max_pages_per_req)
 *        num_copies          page copies the step needs before its kv_append (copy-on-write
 *                            of pages shared after pkv_sched_fork): copy page copy_src[i]
 *                            to copy_dst[i] with pkv_copy_pages; the block table already
 *                            names the copies
 * block_table row i holds request i's physical pages, -1 past its last page.
 */
typedef struct {
    int32_t max_reqs;
    int32_t max_pages_per_req;
    int32_t* rids;
    int32_t* q_lens;
    int32_t* context_lens;
    int32_t* q_offsets;
    int32_t* block_table;
    int32_t num_reqs;
    int32_t total_q_tokens;
    int32_t max_q_len;
    int32_t max_context_len;
    int32_t pages_used;
    int32_t max_copies;
    int32_t* copy_src;
    int32_t* copy_dst;
    int32_t num_copies;
} pkv_plan;

/*
 * pkv_sched_create -- a planner over a pool of num_pages pages, handed out in
 * page_order[0..num_pages) (NULL: 0, 1, 2, ...), with a per-step token budget (> 0) and
 * an optional per-request chunk cap (0: none).  Returns NULL on bad arguments or when
 * memory runs out.
 */
PKV_API pkv_scheduler* pkv_sched_create(int32_t num_pages, const int32_t* page_order,
                                        int32_t budget, int32_t chunk_cap);
PKV_API void pkv_sched_destroy(pkv_scheduler* s);

/*
 * pkv_sched_add_request -- append a request: `history` tokens already cached elsewhere
 * (loaded by pkv_sched_history_plan), then `prompt` input tokens to prefill, then
 * `decodes` generated tokens.  rid must be new.  Errors: INVALID_ARG.
 */
PKV_API int pkv_sched_add_request(pkv_scheduler* s, int32_t rid, int32_t history,
                                  int32_t prompt, int32_t decodes);

/*
 * pkv_sched_sort_by_length -- order the requests whose prompt has not started by prompt
 * length, shortest first (equal lengths keep their arrival order), after every request
 * that has started (those keep their order).  lshu.cn/news/11576 §2.2: sorting the batch by
 * prompt length before prefill keeps requests of similar length adjacent, so their pages
 * are allocated together rather than short requests' pages landing in the gaps between
 * long ones; later steps plan and launch requests in the new order.  The length is the
 * prompt tokens still to compute (less any reused prefix); a request has started once a
 * step has computed some of its prompt (a history load or a reused prefix does not count).
 * Errors: INVALID_ARG (NULL handle), CAPACITY (out of memory; the order is unchanged).
 */
PKV_API int pkv_sched_sort_by_length(pkv_scheduler* s);

/*
 * pkv_sched_history_plan -- the append that loads every request's cached history
 * (q_len = history, context_len = 0), pages taken request by request, or round-robin one
 * page at a time across requests when `interleave` is non-zero.  Marks the history
 * computed.  Returns 1 with *out filled, 0 when no request has history, or INVALID_ARG,
 * CAPACITY (out arrays too small), NO_PAGES.
 */
PKV_API int pkv_sched_history_plan(pkv_scheduler* s, int interleave, pkv_plan* out);

/*
 * pkv_sched_next_step -- plan the next step (decodes first, then prefill chunks within the
 * budget), take the pages it reaches and advance the requests as if it ran.  Returns 1 with
 * *out filled, 0 when every request is done, or INVALID_ARG, CAPACITY, NO_PAGES.
 */
PKV_API int pkv_sched_next_step(pkv_scheduler* s, pkv_plan* out);

/*
 * pkv_sched_release -- return a finished request's pages to the end of the free list (its
 * shared prefix blocks: its references to them) and forget the request.
 * Errors: INVALID_ARG (unknown rid or request not finished).
 */
PKV_API int pkv_sched_release(pkv_scheduler* s, int32_t rid);

/* Pages currently on the free list (-1 for a NULL handle). */
PKV_API int32_t pkv_sched_free_pages(const pkv_scheduler* s);

/*
 * Prefix caching (hotelren.com/news/6181127 §4.3): the K/V of prompt tokens already
 * computed for one request are reused by later requests whose prompt starts with exactly
 * the same token ids.
 *  - Caching works on full 16-token blocks of prompt tokens.  Once a step covers a block,
 *    the block is registered under its token ids and those of every block before it, and
 *    its page becomes shared.
 *  - A new prompt reuses the longest run of registered blocks that matches its leading
 *    token ids exactly (ids are compared, not only hashed).  At least one prompt token is
 *    always left to compute.  The request starts with context_len = the reused tokens, so
 *    new tokens continue the positions.
 *  - Shared blocks are reference-counted.  A request's release returns its references;
 *    blocks nobody uses stay cached and are evicted least-recently-used first, block by
 *    block, only when the free list is empty.
 *  - Registered blocks are always full, so no step ever writes into one (pages shared by
 *    pkv_sched_fork, which may be partly filled, are copied on write instead).
 */

/*
 * pkv_sched_add_prompt -- append a request whose `n_prompt` prompt token ids are known,
 * followed by `decodes` generated tokens; it takes part in prefix caching.  Returns the
 * number of prompt tokens reused from the cache (a multiple of 16, >= 0), or INVALID_ARG.
 */
PKV_API int pkv_sched_add_prompt(pkv_scheduler* s, int32_t rid, const int32_t* tokens,
                                 int32_t n_prompt, int32_t decodes);

/*
 * pkv_sched_fork -- append request `rid` that continues from everything request
 * `parent_rid` has cached so far (its prompt must be complete) with `decodes` generated
 * tokens of its own: parallel samples or beams of one prompt.  The child shares all of the
 * parent's pages, a partly filled last page included; every shared page counts its holders
 * (hotelren.com/news/6181127 §4.3: reused K/V, memory managed by page).  Copy-on-write: when
 * a step is about to write a request's next token into a page that already holds tokens and
 * that another request also holds, the planner gives the request a fresh page, names it in
 * the block table and lists the copy (old page -> fresh page) in the plan; the last holder
 * of a page writes into it in place.  Releasing a request drops its hold on every page; a
 * page returns to the free list with its last holder.  Errors: INVALID_ARG (unknown parent,
 * parent still prefilling or without cached tokens, rid already used), CAPACITY (out of
 * memory).
 */
PKV_API int pkv_sched_fork(pkv_scheduler* s, int32_t parent_rid, int32_t rid, int32_t decodes);

/* Registered blocks: all of them, and those no request uses (evictable).  -1 for NULL. */
PKV_API int32_t pkv_sched_cached_blocks(const pkv_scheduler* s);
PKV_API int32_t pkv_sched_evictable_blocks(const pkv_scheduler* s);

#ifdef __cplusplus
}
#endif

#endif  /* PKV_SCHED_H_ */
