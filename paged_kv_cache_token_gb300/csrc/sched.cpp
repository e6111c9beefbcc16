// Host-side step planner and page allocator (include/pkv_sched.h).
//
// niuwancheng.cn "11. Chunked prefill and unified scheduling", section "token budget per
// step": each request records the tokens already computed and the tokens it needs; a step
// gives every decoding request one token first, then prefilling requests take
// min(remaining input, remaining budget) in request order, never exceeding the budget.
// lshu.cn/news/11576 §2.2-§2.3: 16-token pages, taken from a pool as a request's cached
// length crosses a page boundary and addressed through a block table.
//
// Every planning call first works out the whole step (requests, lengths, pages it needs)
// without touching the scheduler, checks the caller's arrays and the free list, and only
// then takes pages and advances the requests, so a failed call changes nothing.
#include <algorithm>
#include <cstdint>
#include <deque>
#include <new>
#include <unordered_map>
#include <utility>
#include <vector>

#include "pkv_sched.h"

namespace {

constexpr int64_t kPage = 16;

int64_t pages_for(int64_t tokens) { return (tokens + kPage - 1) / kPage; }

struct Req {
    int32_t rid = 0;
    int64_t history = 0;
    int64_t prompt_end = 0;  // history + prompt: positions below are input, not generated
    int64_t total = 0;       // every position the request will ever hold
    int64_t computed = 0;    // tokens already in the KV cache
    bool history_pending = false;
    std::vector<int32_t> pages;
    bool decoding() const { return computed >= prompt_end && computed < total; }
    bool prefilling() const { return computed < prompt_end; }
    bool done() const { return computed >= total; }
};

// one request of a planned step: index into reqs, tokens it advances, pages it will hold
struct Pick {
    size_t i;
    int64_t n;
    int64_t pages_after;
};

}  // namespace

struct pkv_scheduler {
    std::deque<int32_t> free_list;
    int64_t budget = 0;
    int64_t chunk_cap = 0;  // 0: no cap
    std::vector<Req> reqs;  // in the order they were added
    std::unordered_map<int32_t, size_t> index;

    void reindex() {
        index.clear();
        for (size_t i = 0; i < reqs.size(); ++i) index[reqs[i].rid] = i;
    }

    // Whether the caller's arrays hold the step and the free list covers the pages it
    // still has to take.
    int check(const std::vector<Pick>& picks, const pkv_plan* out) const {
        if (!out || out->max_reqs < 0 || out->max_pages_per_req < 0) return PKV_ERR_INVALID_ARG;
        if (!out->rids || !out->q_lens || !out->context_lens || !out->q_offsets ||
            (!picks.empty() && !out->block_table))
            return PKV_ERR_INVALID_ARG;
        if (static_cast<int64_t>(picks.size()) > out->max_reqs) return PKV_ERR_CAPACITY;
        int64_t need = 0, total_q = 0, max_ctx = 0;
        for (const Pick& p : picks) {
            const Req& r = reqs[p.i];
            if (p.pages_after > out->max_pages_per_req) return PKV_ERR_CAPACITY;
            need += std::max<int64_t>(0, p.pages_after - static_cast<int64_t>(r.pages.size()));
            total_q += p.n;
            max_ctx = std::max(max_ctx, r.computed);
        }
        if (total_q > INT32_MAX || max_ctx > INT32_MAX) return PKV_ERR_CAPACITY;
        if (need > static_cast<int64_t>(free_list.size())) return PKV_ERR_NO_PAGES;
        return PKV_OK;
    }

    // Check, then take the step's pages (in pick order, as the step reaches them one
    // request after another), write the plan and advance the requests.
    int commit(const std::vector<Pick>& picks, bool history, pkv_plan* out) {
        const int rc = check(picks, out);
        if (rc != PKV_OK) return rc;
        int64_t total_q = 0, max_q = 0, max_ctx = 0, pages_used = 0;
        for (const Pick& p : picks) {
            total_q += p.n;
            max_q = std::max(max_q, p.n);
            max_ctx = std::max(max_ctx, history ? int64_t{0} : reqs[p.i].computed);
            pages_used = std::max(pages_used, p.pages_after);
        }
        // nothing can fail from here on
        const int64_t stride = out->max_pages_per_req;
        int32_t off = 0;
        for (size_t k = 0; k < picks.size(); ++k) {
            const Pick& p = picks[k];
            Req& r = reqs[p.i];
            while (static_cast<int64_t>(r.pages.size()) < p.pages_after) {
                r.pages.push_back(free_list.front());
                free_list.pop_front();
            }
            out->rids[k] = r.rid;
            out->q_lens[k] = static_cast<int32_t>(p.n);
            out->context_lens[k] = history ? 0 : static_cast<int32_t>(r.computed);
            out->q_offsets[k] = off;
            off += static_cast<int32_t>(p.n);
            int32_t* row = out->block_table + static_cast<int64_t>(k) * stride;
            for (int64_t c = 0; c < stride; ++c)
                row[c] = c < static_cast<int64_t>(r.pages.size()) ? r.pages[c] : -1;
        }
        out->q_offsets[picks.size()] = off;
        out->num_reqs = static_cast<int32_t>(picks.size());
        out->total_q_tokens = static_cast<int32_t>(total_q);
        out->max_q_len = static_cast<int32_t>(max_q);
        out->max_context_len = static_cast<int32_t>(max_ctx);
        out->pages_used = static_cast<int32_t>(pages_used);
        for (const Pick& p : picks) {
            Req& r = reqs[p.i];
            if (history) {
                r.computed = r.history;
                r.history_pending = false;
            } else {
                r.computed += p.n;
            }
        }
        return 1;
    }
};

extern "C" {

pkv_scheduler* pkv_sched_create(int32_t num_pages, const int32_t* page_order, int32_t budget,
                                int32_t chunk_cap) {
    if (num_pages < 0 || budget <= 0 || chunk_cap < 0) return nullptr;
    try {
        pkv_scheduler* s = new pkv_scheduler();
        for (int32_t i = 0; i < num_pages; ++i)
            s->free_list.push_back(page_order ? page_order[i] : i);
        s->budget = budget;
        s->chunk_cap = chunk_cap;
        return s;
    } catch (...) {
        return nullptr;
    }
}

void pkv_sched_destroy(pkv_scheduler* s) { delete s; }

int pkv_sched_add_request(pkv_scheduler* s, int32_t rid, int32_t history, int32_t prompt,
                          int32_t decodes) {
    if (!s || history < 0 || prompt < 0 || decodes < 0) return PKV_ERR_INVALID_ARG;
    if (s->index.count(rid)) return PKV_ERR_INVALID_ARG;
    try {
        Req r;
        r.rid = rid;
        r.history = history;
        r.prompt_end = static_cast<int64_t>(history) + prompt;
        r.total = r.prompt_end + decodes;
        r.history_pending = history > 0;
        s->reqs.push_back(std::move(r));
        s->index[rid] = s->reqs.size() - 1;
        return PKV_OK;
    } catch (...) {
        return PKV_ERR_CAPACITY;
    }
}

int pkv_sched_history_plan(pkv_scheduler* s, int interleave, pkv_plan* out) {
    if (!s) return PKV_ERR_INVALID_ARG;
    try {
        std::vector<Pick> picks;
        for (size_t i = 0; i < s->reqs.size(); ++i)
            if (s->reqs[i].history_pending)
                picks.push_back({i, s->reqs[i].history, pages_for(s->reqs[i].history)});
        if (picks.empty()) return 0;
        if (!interleave) return s->commit(picks, true, out);
        // round-robin: one page at a time across the requests until each has its history
        // pages; the plan is the same, only the order the free list is drained differs
        const int rc = s->check(picks, out);
        if (rc != PKV_OK) return rc;
        for (bool more = true; more;) {
            more = false;
            for (const Pick& p : picks) {
                Req& r = s->reqs[p.i];
                if (static_cast<int64_t>(r.pages.size()) < p.pages_after) {
                    r.pages.push_back(s->free_list.front());
                    s->free_list.pop_front();
                    more = true;
                }
            }
        }
        return s->commit(picks, true, out);  // pages already held: only writes the plan
    } catch (...) {
        return PKV_ERR_CAPACITY;
    }
}

int pkv_sched_next_step(pkv_scheduler* s, pkv_plan* out) {
    if (!s) return PKV_ERR_INVALID_ARG;
    try {
        std::vector<Pick> picks;
        int64_t left = s->budget;
        for (size_t i = 0; i < s->reqs.size(); ++i) {  // decodes first, one token each
            const Req& r = s->reqs[i];
            if (r.decoding() && left > 0) {
                picks.push_back({i, 1, pages_for(r.computed + 1)});
                left -= 1;
            }
        }
        for (size_t i = 0; i < s->reqs.size(); ++i) {  // then prefills take what is left
            const Req& r = s->reqs[i];
            if (r.prefilling() && left > 0) {
                int64_t n = std::min(r.prompt_end - r.computed, left);
                if (s->chunk_cap > 0) n = std::min(n, s->chunk_cap);
                picks.push_back({i, n, pages_for(r.computed + n)});
                left -= n;
            }
        }
        if (picks.empty()) return 0;
        return s->commit(picks, false, out);
    } catch (...) {
        return PKV_ERR_CAPACITY;
    }
}

int pkv_sched_release(pkv_scheduler* s, int32_t rid) {
    if (!s) return PKV_ERR_INVALID_ARG;
    const auto it = s->index.find(rid);
    if (it == s->index.end() || !s->reqs[it->second].done()) return PKV_ERR_INVALID_ARG;
    try {
        Req& r = s->reqs[it->second];
        for (int32_t p : r.pages) s->free_list.push_back(p);
        s->reqs.erase(s->reqs.begin() + static_cast<std::ptrdiff_t>(it->second));
        s->reindex();
        return PKV_OK;
    } catch (...) {
        return PKV_ERR_CAPACITY;
    }
}

int32_t pkv_sched_free_pages(const pkv_scheduler* s) {
    return s ? static_cast<int32_t>(s->free_list.size()) : -1;
}

}  // extern "C"
