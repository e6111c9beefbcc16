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
//
// Prefix caching, hotelren.com/news/6181127 §4.3: K/V of prompt tokens are reused by later
// requests whose prompt starts with exactly the same token ids; memory is managed in
// blocks (pages) and unused blocks are evicted least-recently-used, block by block.
#include <algorithm>
#include <array>
#include <cstdint>
#include <deque>
#include <list>
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
    bool cached = false;              // takes part in prefix caching (prompt ids known)
    std::vector<int32_t> tokens;      // prompt token ids of a cached request
    std::vector<uint64_t> block_of;   // per page: key of the shared block it holds, or 0
    int64_t registered = 0;           // prompt blocks already matched or registered
    uint64_t chain = 0;               // key of the last of them (0: none)
    int64_t history = 0;
    int64_t prompt_end = 0;  // history + prompt: positions below are input, not generated
    int64_t total = 0;       // every position the request will ever hold
    int64_t computed = 0;    // tokens already in the KV cache
    bool history_pending = false;
    bool begun = false;      // a step has computed some of its prompt
    std::vector<int32_t> pages;
    bool decoding() const { return computed >= prompt_end && computed < total; }
    bool prefilling() const { return computed < prompt_end; }
    bool done() const { return computed >= total; }
};

// A shared prompt block: its page, how many requests hold it, the key of the block before
// it and its own token ids (compared on every match, so a key collision cannot alias).
struct Block {
    int32_t page = -1;
    int32_t refs = 0;
    uint64_t parent = 0;
    std::array<int32_t, 16> tokens{};
    std::list<uint64_t>::iterator lru;  // valid while refs == 0
};

// Key of a block from the key of the block before it and its 16 token ids (splitmix64
// steps); 0 is reserved for "no block".
uint64_t block_key(uint64_t parent, const int32_t* t) {
    uint64_t h = parent ^ 0x9e3779b97f4a7c15ull;
    for (int i = 0; i < 16; ++i) {
        h ^= static_cast<uint32_t>(t[i]);
        h += 0x9e3779b97f4a7c15ull;
        h = (h ^ (h >> 30)) * 0xbf58476d1ce4e5b9ull;
        h = (h ^ (h >> 27)) * 0x94d049bb133111ebull;
        h ^= h >> 31;
    }
    return h ? h : 1;
}

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
    std::unordered_map<uint64_t, Block> blocks;  // shared prompt blocks by key
    std::list<uint64_t> lru;                      // unreferenced blocks, least recent first
    // pages outside the block registry held by more than one request (after a fork), with
    // their number of holders; a page absent here has one holder
    std::unordered_map<int32_t, int32_t> holders;

    int32_t holders_of(int32_t page) const {
        const auto it = holders.find(page);
        return it == holders.end() ? 1 : it->second;
    }
    // one holder lets go of a private page: the last one returns it to the free list
    void drop_page(int32_t page) {
        const auto it = holders.find(page);
        if (it == holders.end()) {
            free_list.push_back(page);
        } else if (--it->second <= 1) {
            holders.erase(it);
        }
    }

    int64_t available() const {
        return static_cast<int64_t>(free_list.size()) + static_cast<int64_t>(lru.size());
    }

    // a page from the free list, else the least recently used unreferenced block's
    int32_t take_page() {
        if (!free_list.empty()) {
            const int32_t p = free_list.front();
            free_list.pop_front();
            return p;
        }
        const uint64_t key = lru.front();
        lru.pop_front();
        const auto it = blocks.find(key);
        const int32_t p = it->second.page;
        blocks.erase(it);
        return p;
    }

    // the block matching (parent, tokens) exactly, or nullptr
    Block* find_block(uint64_t key, uint64_t parent, const int32_t* t) {
        const auto it = blocks.find(key);
        if (it == blocks.end() || it->second.parent != parent ||
            !std::equal(t, t + 16, it->second.tokens.begin()))
            return nullptr;
        return &it->second;
    }

    // Register the prompt blocks a step has just completed: each becomes shared unless an
    // identical block is already registered (then this request keeps its page private and
    // stops registering, since later blocks would hang off a page it does not share).
    void register_blocks(Req& r) {
        const int64_t full = std::min(r.computed, r.prompt_end) / kPage;
        while (r.registered < full) {
            const int64_t b = r.registered;
            if (r.block_of[static_cast<size_t>(b)] == 0) {
                const int32_t* t = r.tokens.data() + b * kPage;
                const uint64_t key = block_key(r.chain, t);
                if (blocks.count(key)) {
                    r.registered = INT64_MAX;
                    return;
                }
                Block blk;
                blk.page = r.pages[static_cast<size_t>(b)];
                blk.refs = 1;
                blk.parent = r.chain;
                std::copy(t, t + 16, blk.tokens.begin());
                blocks.emplace(key, blk);
                r.block_of[static_cast<size_t>(b)] = key;
            }
            r.chain = r.block_of[static_cast<size_t>(b)];
            ++r.registered;
        }
    }

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
        const int64_t copies = copy_on_write_pages(picks).size();
        if (copies > 0 && (out->max_copies < copies || !out->copy_src || !out->copy_dst))
            return PKV_ERR_CAPACITY;
        if (need + copies > available()) return PKV_ERR_NO_PAGES;
        return PKV_OK;
    }

    // Copy-on-write: the picks (in order) whose first new token lands in a page that
    // already holds tokens and that another request also holds.  A request about to write
    // into a shared page gets a copy of it first; the holders left keep the original, and
    // the last of them writes into it in place.  Returns, per such pick, its index in
    // `picks` (the holder counts as they will be when the pick is reached).
    std::vector<size_t> copy_on_write_pages(const std::vector<Pick>& picks) const {
        std::vector<size_t> cow;
        std::unordered_map<int32_t, int32_t> left;  // holders still on a page in this step
        for (size_t k = 0; k < picks.size(); ++k) {
            const Pick& p = picks[k];
            const Req& r = reqs[p.i];
            if (p.n <= 0 || r.computed % kPage == 0) continue;  // starts a fresh page
            const int32_t page = r.pages[static_cast<size_t>(r.computed / kPage)];
            auto it = left.find(page);
            if (it == left.end()) it = left.emplace(page, holders_of(page)).first;
            if (it->second > 1) {
                cow.push_back(k);
                --it->second;
            }
        }
        return cow;
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
        const std::vector<size_t> cow = history ? std::vector<size_t>() :
                                                   copy_on_write_pages(picks);
        // nothing can fail from here on
        out->num_copies = 0;
        for (size_t k : cow) {
            Req& r = reqs[picks[k].i];
            int32_t& slot = r.pages[static_cast<size_t>(r.computed / kPage)];
            const int32_t fresh = take_page();
            out->copy_src[out->num_copies] = slot;
            out->copy_dst[out->num_copies] = fresh;
            ++out->num_copies;
            drop_page(slot);  // another request still holds the original
            slot = fresh;
        }
        const int64_t stride = out->max_pages_per_req;
        int32_t off = 0;
        for (size_t k = 0; k < picks.size(); ++k) {
            const Pick& p = picks[k];
            Req& r = reqs[p.i];
            while (static_cast<int64_t>(r.pages.size()) < p.pages_after) {
                r.pages.push_back(take_page());
                r.block_of.push_back(0);
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
                r.begun = true;
            }
            if (r.cached && r.registered != INT64_MAX) register_blocks(r);
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
        try {
            s->index[rid] = s->reqs.size() - 1;
        } catch (...) {
            s->reqs.pop_back();
            throw;
        }
        return PKV_OK;
    } catch (...) {
        return PKV_ERR_CAPACITY;
    }
}

int pkv_sched_sort_by_length(pkv_scheduler* s) {
    if (!s) return PKV_ERR_INVALID_ARG;
    try {
        // key: prompt tokens still to compute; equal keys keep their arrival order
        std::vector<size_t> started, waiting;
        for (size_t i = 0; i < s->reqs.size(); ++i)
            (s->reqs[i].begun ? started : waiting).push_back(i);
        std::stable_sort(waiting.begin(), waiting.end(), [s](size_t a, size_t b) {
            return s->reqs[a].prompt_end - s->reqs[a].computed <
                   s->reqs[b].prompt_end - s->reqs[b].computed;
        });
        std::vector<Req> order;
        order.reserve(s->reqs.size());
        for (size_t i : started) order.push_back(std::move(s->reqs[i]));
        for (size_t i : waiting) order.push_back(std::move(s->reqs[i]));
        s->reqs.swap(order);
        s->reindex();
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
                    r.pages.push_back(s->take_page());
                    r.block_of.push_back(0);
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
        for (size_t i = 0; i < r.pages.size(); ++i) {
            const uint64_t key = i < r.block_of.size() ? r.block_of[i] : 0;
            if (key == 0) {
                s->drop_page(r.pages[i]);
                continue;
            }
            Block& blk = s->blocks.at(key);
            if (--blk.refs == 0) blk.lru = s->lru.insert(s->lru.end(), key);
        }
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

int pkv_sched_add_prompt(pkv_scheduler* s, int32_t rid, const int32_t* tokens,
                         int32_t n_prompt, int32_t decodes) {
    if (!s || n_prompt < 0 || decodes < 0 || (n_prompt > 0 && !tokens))
        return PKV_ERR_INVALID_ARG;
    if (s->index.count(rid)) return PKV_ERR_INVALID_ARG;
    try {
        Req r;
        r.rid = rid;
        r.cached = true;
        r.tokens.assign(tokens, tokens + n_prompt);
        r.prompt_end = n_prompt;
        r.total = static_cast<int64_t>(n_prompt) + decodes;
        // longest run of registered blocks matching the prompt, leaving >= 1 token to run
        const int64_t max_blocks = n_prompt > 0 ? (n_prompt - 1) / kPage : 0;
        std::vector<Block*> hit;
        uint64_t parent = 0;
        for (int64_t b = 0; b < max_blocks; ++b) {
            const int32_t* t = r.tokens.data() + b * kPage;
            const uint64_t key = block_key(parent, t);
            Block* blk = s->find_block(key, parent, t);
            if (!blk) break;
            hit.push_back(blk);
            r.pages.push_back(blk->page);
            r.block_of.push_back(key);
            parent = key;
        }
        r.registered = static_cast<int64_t>(hit.size());
        r.chain = parent;
        r.computed = r.registered * kPage;
        s->reqs.push_back(std::move(r));
        try {
            s->index[rid] = s->reqs.size() - 1;
        } catch (...) {
            s->reqs.pop_back();
            throw;
        }
        for (Block* blk : hit)  // nothing can fail any more: take the references
            if (blk->refs++ == 0) s->lru.erase(blk->lru);
        return static_cast<int>(hit.size() * kPage);
    } catch (...) {
        return PKV_ERR_CAPACITY;
    }
}

int pkv_sched_fork(pkv_scheduler* s, int32_t parent_rid, int32_t rid, int32_t decodes) {
    if (!s || decodes < 0 || s->index.count(rid)) return PKV_ERR_INVALID_ARG;
    const auto it = s->index.find(parent_rid);
    if (it == s->index.end()) return PKV_ERR_INVALID_ARG;
    const Req& parent = s->reqs[it->second];
    if (parent.computed <= 0 || parent.computed < parent.prompt_end ||
        parent.history_pending)
        return PKV_ERR_INVALID_ARG;
    try {
        Req r;
        r.rid = rid;
        r.history = 0;
        r.computed = parent.computed;
        r.prompt_end = parent.computed;
        r.total = parent.computed + decodes;
        r.begun = true;
        r.pages.assign(parent.pages.begin(),
                       parent.pages.begin() + static_cast<std::ptrdiff_t>(pages_for(r.computed)));
        r.block_of.assign(parent.block_of.begin(),
                          parent.block_of.begin() + static_cast<std::ptrdiff_t>(r.pages.size()));
        // reserve every container insertion before the first reference is taken
        s->holders.reserve(s->holders.size() + r.pages.size());
        s->reqs.push_back(std::move(r));
        try {
            s->index[rid] = s->reqs.size() - 1;
        } catch (...) {
            s->reqs.pop_back();
            throw;
        }
        const Req& child = s->reqs.back();  // nothing can fail any more: take references
        for (size_t i = 0; i < child.pages.size(); ++i) {
            const uint64_t key = child.block_of[i];
            if (key != 0) {
                Block& blk = s->blocks.at(key);
                if (blk.refs++ == 0) s->lru.erase(blk.lru);
            } else {
                s->holders[child.pages[i]] = s->holders_of(child.pages[i]) + 1;
            }
        }
        return PKV_OK;
    } catch (...) {
        return PKV_ERR_CAPACITY;
    }
}

int32_t pkv_sched_cached_blocks(const pkv_scheduler* s) {
    return s ? static_cast<int32_t>(s->blocks.size()) : -1;
}

int32_t pkv_sched_evictable_blocks(const pkv_scheduler* s) {
    return s ? static_cast<int32_t>(s->lru.size()) : -1;
}

}  // extern "C"
