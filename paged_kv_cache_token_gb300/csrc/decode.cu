// Decode path of the paged attention step: work planning, the split-KV streaming kernel
// and the split combine.
//
// hotelren.com/news/6181127 §3.1: a decode row scores its query against all S+t cached
// keys, softmax, then a weighted sum of all S+t values; §3.2: this is a stream over the
// cache whose bytes grow linearly with the context, so it is bound by memory bandwidth;
// §6.3: with grouped-query attention several query heads share one KV head (here they are
// processed together, so each K/V byte is read once per KV head, not once per query head).
//
// Work item = (request, row, KV head, split).  A split is a run of pages of one request;
// a CTA of four warps takes one item at a time from a device work queue.  Each warp owns
// every fourth page of the item and a private ring of 3 stages; a page's K block and V
// block (16 x D each, contiguous in the pool) arrive through two 1-D bulk async copies on
// one mbarrier.  Scores stay in base-2 units (q is pre-scaled by scale * log2 e) and an
// online softmax keeps (running max, running sum, un-normalised output) per query head.
// The four warps merge in shared memory; a request split over several items leaves
// partial results that the combine kernel reduces with the same rescaling.
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "launch.h"

namespace pkv {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kDecWarps = 4;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kStages = 3;
constexpr int kMinSplitPages = 8;
constexpr int kItemsPerSm = 8;  // target decode items per SM when choosing the split size

__device__ __forceinline__ int4* ws_req_info(const StepArgs& a) {
    return reinterpret_cast<int4*>(a.ws + a.lay.req_info);
}
__device__ __forceinline__ int4* ws_items(const StepArgs& a) {
    return reinterpret_cast<int4*>(a.ws + a.lay.items);
}
__device__ __forceinline__ int4* ws_tiles(const StepArgs& a) {
    return reinterpret_cast<int4*>(a.ws + a.lay.tiles);
}
__device__ __forceinline__ int32_t* ws_ctrl(const StepArgs& a) {
    return reinterpret_cast<int32_t*>(a.ws + a.lay.ctrl);
}

// Exclusive block-wide scan of one int per thread (blockDim.x == kPlanThreads).
__device__ int block_exclusive_scan(int v, int* total, int* s_warp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(kFull, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int w = s_warp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(kFull, w, o);
            if (lane >= o) w += y;
        }
        s_warp[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const int before = (warp ? s_warp[warp - 1] : 0) + x - v;
    *total = s_warp[31];
    __syncthreads();
    return before;
}

}  // namespace

// ------------------------------------------------------------------------------------
// plan: validate per-request lengths, choose the split size, number the work.
// One CTA.  Requests with q_len == 1 become split items (first, so their partial results
// are indexed by item), rows of requests with 1 < q_len < prefill_min_q become one item
// per (row, KV head), requests with q_len >= prefill_min_q become prefill tiles
// (q tile of 128 rows, query head), longest first.
// ------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kPlanThreads) plan_kernel(StepArgs a) {
    __shared__ unsigned long long s_sum;
    __shared__ int s_max, s_split, s_bad;
    __shared__ int s_warp[32];
    const int tid = threadIdx.x;
    int32_t* ctrl = ws_ctrl(a);
    int4* info = ws_req_info(a);
    if (tid == 0) {
        s_sum = 0;
        s_max = 0;
        s_bad = (a.q_offsets[0] != 0 || a.q_offsets[a.num_reqs] != a.total_q_tokens);
    }
    __syncthreads();
    const int Hkv = a.num_kv_heads;
    unsigned long long my_sum = 0;
    int my_max = 0;
    for (int r = tid; r < a.num_reqs; r += kPlanThreads) {
        const int q = a.q_lens[r], c = a.context_lens[r];
        const bool ok = q >= 0 && c >= 0 && q <= a.max_q_len && c <= a.max_context_len &&
                        a.q_offsets[r + 1] - a.q_offsets[r] == q;
        if (!ok) { atomicOr(&s_bad, 1); continue; }
        const int pages = cdiv(c + q, kPage);
        if (pages > a.max_pages) set_error(a.err, PKV_DEVERR_TABLE_RANGE);
        if (q == 1) {
            my_sum += pages;
            my_max = max(my_max, pages);
        }
    }
    atomicAdd(&s_sum, my_sum);
    atomicMax(&s_max, my_max);
    __syncthreads();
    const bool bad = s_bad != 0;
    if (tid == 0) {
        if (bad) set_error(a.err, PKV_DEVERR_TOKENS);
        const long long target = static_cast<long long>(kItemsPerSm) * a.num_sms;
        long long sp = kMinSplitPages;
        sp = max(sp, static_cast<long long>(cdiv(s_max, a.lay.max_splits)));
        sp = max(sp, static_cast<long long>((s_sum * Hkv + target - 1) / target));
        sp = (sp + kDecWarps - 1) / kDecWarps * kDecWarps;
        s_split = static_cast<int>(min(sp, static_cast<long long>(INT_MAX / 2)));
    }
    __syncthreads();
    const int sp = s_split;

    // three numbering passes: split items, row items, prefill tiles
    int carry_split = 0, carry_items = 0, carry_tiles = 0;
    for (int pass = 0; pass < 3; ++pass) {
        int carry = pass == 2 ? 0 : carry_items;
        for (int base = 0; base < a.num_reqs; base += kPlanThreads) {
            const int r = base + tid;
            int n = 0, q = 0, pages = 0;
            if (r < a.num_reqs && !bad) {
                q = a.q_lens[r];
                const int c = a.context_lens[r];
                const bool ok = q >= 0 && c >= 0 && q <= a.max_q_len && c <= a.max_context_len &&
                                a.q_offsets[r + 1] - a.q_offsets[r] == q;
                if (!ok) q = 0;
                pages = cdiv(c + q, kPage);
                if (pass == 0 && q == 1) n = Hkv * cdiv(pages, sp);
                if (pass == 1 && q > 1 && q < a.prefill_min_q) n = Hkv * q;
                if (pass == 2 && q >= a.prefill_min_q && q > 1)
                    n = cdiv(q, 128) * (a.num_q_heads / a.heads_per_tile);
            }
            int total;
            const int ex = block_exclusive_scan(n, &total, s_warp);
            if (r < a.num_reqs) {
                if (pass == 0) info[r] = make_int4(carry + ex, q == 1 ? cdiv(pages, sp) : 0, q, 0);
                if (pass == 1 && n) info[r].x = carry + ex;
                if (pass == 1 && q > 1) info[r].y = 1;
                if (pass == 2 && n) info[r].w = carry + ex;
            }
            carry += total;
        }
        if (pass == 0) carry_split = carry;
        if (pass < 2) carry_items = carry; else carry_tiles = carry;
    }
    if (carry_items > a.lay.max_items || carry_tiles > a.lay.max_tiles ||
        carry_split > a.lay.max_split_items) {  // cannot happen when the host maxima hold
        if (tid == 0) set_error(a.err, PKV_DEVERR_TOKENS);
        carry_items = carry_tiles = carry_split = 0;
    }
    __syncthreads();

    // fill the item and tile lists: one warp per request, lanes over its items
    const int lane = tid & 31, warp = tid >> 5;
    int4* items = ws_items(a);
    int4* tiles = ws_tiles(a);
    if (carry_items || carry_tiles) {
        for (int r = warp; r < a.num_reqs; r += kPlanThreads / 32) {
            const int4 in = info[r];
            const int q = in.z;
            if (q == 1) {
                const int ns = in.y;
                for (int i = lane; i < Hkv * ns; i += 32)
                    items[in.x + i] = make_int4(r, 0, i / ns, i % ns);
            } else if (q > 1 && q < a.prefill_min_q) {
                for (int i = lane; i < q * Hkv; i += 32)
                    items[in.x + i] = make_int4(r, i / Hkv, i % Hkv, 0);
            } else if (q > 1) {
                const int nt = cdiv(q, 128);
                const int slots = a.num_q_heads / a.heads_per_tile;
                for (int i = lane; i < nt * slots; i += 32)
                    tiles[in.w + i] = make_int4(r, nt - 1 - i / slots, i % slots, 0);
            }
        }
    }
    if (tid == 0) {
        ctrl[0] = 0;
        ctrl[1] = carry_items;
        ctrl[2] = carry_split;
        ctrl[3] = sp;
        ctrl[8] = 0;
        ctrl[9] = carry_tiles;
    }
}

// ------------------------------------------------------------------------------------
// decode: persistent CTAs pull items; see the file comment for the data flow.
// ------------------------------------------------------------------------------------
template <typename T, int D, int G>
struct DecodeSmem {
    static constexpr int kPageBytes = kPage * D * 2;      // one K (or V) page block
    static constexpr int kStageBytes = 2 * kPageBytes;
    static constexpr int kRing = kDecWarps * kStages * kStageBytes;
    static constexpr int kPbuf = kDecWarps * kPage * G * 4;
    static constexpr int kMerge = kDecWarps * G * (D + 2) * 4;
    static constexpr int kBars = kDecWarps * kStages * 8;
    static constexpr int kBytes = kRing + kPbuf + kMerge + kBars + 16;
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(StepArgs a) {
    using S = DecodeSmem<T, D, G>;
    using Cv = F16<T>;
    constexpr int QKD = D / 8;      // dims per lane in q.k (16 or 8)
    constexpr int NCH = QKD / 8;    // 16-byte chunks per lane per key row (2 or 1)
    constexpr int DPL = D / 32;     // dims per lane in p.V (4 or 2)
    constexpr int N0 = 4 * G, N1 = N0 / 2, N2 = N1 / 2 > 0 ? N1 / 2 : 1;
    constexpr int NV = (N2 >= 2) ? N2 / 2 : 1;  // score values a lane holds after reduction

    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* ring = smem + warp * kStages * S::kStageBytes;
    float* pbuf = reinterpret_cast<float*>(smem + S::kRing) + warp * kPage * G;
    float* merge = reinterpret_cast<float*>(smem + S::kRing + S::kPbuf);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kRing + S::kPbuf + S::kMerge) +
                     warp * kStages;
    int* s_item = reinterpret_cast<int*>(smem + S::kRing + S::kPbuf + S::kMerge + S::kBars);

    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
    }
    __syncwarp();

    const int32_t* ctrl = ws_ctrl(a);
    const int num_items = ctrl[1];
    const int sp = ctrl[3];
    const int4* items = ws_items(a);
    const int4* info = ws_req_info(a);
    float2* part_ml = reinterpret_cast<float2*>(a.ws + a.lay.part_ml);
    float* part_o = reinterpret_cast<float*>(a.ws + a.lay.part_o);
    const int Hkv = a.num_kv_heads, Hq = a.num_q_heads;
    const int c8 = lane & 7, tg = lane >> 3;
    const bool b0 = lane & 1, b1 = lane & 2, b2 = lane & 4;
    const int swz = (c8 >> 2) & 1;  // staggered chunk order: conflict-free 16-byte loads
    const int my_tok = tg * 4 + 2 * (b2 ? 1 : 0) + (b1 ? 1 : 0);  // token of my reduced scores

    uint32_t issued = 0, consumed = 0;  // per-warp ring counters (persist across items)
    bool aborted = false;
    if (threadIdx.x == 0) s_item[1] = 0;

    for (;;) {
        if (threadIdx.x == 0) s_item[0] = atomicAdd(const_cast<int32_t*>(ctrl), 1);
        __syncthreads();
        const int item = s_item[0];
        if (item >= num_items || s_item[1]) break;  // s_item[1]: some warp gave up waiting
        const int4 it = items[item];
        const int r = it.x, row = it.y, g = it.z, split = it.w;
        const int4 in = info[r];
        const int nsplit = in.y;
        const int ctx = a.context_lens[r];
        const int t = a.q_offsets[r] + row;
        const int nkv = ctx + row + 1;                // keys 0..pos inclusive
        const int npages = cdiv(nkv, kPage);
        // q_len == 1 requests are cut into splits of sp pages; a row of a longer request
        // is one item over all of its pages
        const int pb = split * sp;
        const int pe = in.z == 1 ? min(npages, pb + sp) : npages;
        const int n_mine = pe - pb > warp ? cdiv(pe - pb - warp, kDecWarps) : 0;
        const int32_t* bt_row = a.block_table + static_cast<int64_t>(r) * a.max_pages;

        // query heads g*G .. g*G+G-1, my q.k dims, pre-scaled into base-2 units
        float qf[G][QKD];
        {
            const uint16_t* qbase = static_cast<const uint16_t*>(a.q) +
                                    (static_cast<int64_t>(t) * Hq + g * G) * D + c8 * QKD;
#pragma unroll
            for (int j = 0; j < G; ++j) {
#pragma unroll
                for (int ci = 0; ci < NCH; ++ci) {
                    const uint4 w = __ldg(reinterpret_cast<const uint4*>(qbase + j * D) + (ci ^ (NCH == 2 ? swz : 0)));
                    const uint32_t ws4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = Cv::unpack(ws4[e]);
                        qf[j][ci * 8 + 2 * e] = f.x * a.scale_log2;
                        qf[j][ci * 8 + 2 * e + 1] = f.y * a.scale_log2;
                    }
                }
            }
        }

        // physical page ids of my first 32 pages (lane i holds page i of this warp)
        auto load_window = [&](int first) -> int {
            const int i = first + lane;
            int phys = 0;
            if (i < n_mine) {
                const int lp = pb + warp + i * kDecWarps;
                if (lp < a.max_pages) {
                    phys = __ldg(bt_row + lp);
                    if (phys < 0 || phys >= a.num_pages) {
                        set_error(a.err, PKV_DEVERR_PAGE_RANGE);
                        phys = 0;
                    }
                } else {
                    set_error(a.err, PKV_DEVERR_TABLE_RANGE);
                }
            }
            return phys;
        };
        int window = load_window(0);
        int window_base = 0;
        const uint16_t* kc = static_cast<const uint16_t*>(a.k_cache);
        const uint16_t* vc = static_cast<const uint16_t*>(a.v_cache);
        auto issue = [&](int i) {  // whole warp calls; lane 0 issues
            if (i >= window_base + 32) {
                window_base += 32;
                window = load_window(window_base);
            }
            const int phys = __shfl_sync(kFull, window, i - window_base);
            if (lane == 0) {
                const int stage = issued % kStages;
                uint8_t* dst = ring + stage * S::kStageBytes;
                const int64_t off = (static_cast<int64_t>(phys) * Hkv + g) * (kPage * D);
                mbar_arrive_expect_tx(&bars[stage], 2 * S::kPageBytes);
                bulk_g2s(dst, kc + off, S::kPageBytes, &bars[stage]);
                bulk_g2s(dst + S::kPageBytes, vc + off, S::kPageBytes, &bars[stage]);
            }
            ++issued;
        };

        float m[G], o[G][DPL], lsum[NV];
#pragma unroll
        for (int j = 0; j < G; ++j) {
            m[j] = -1e30f;
#pragma unroll
            for (int e = 0; e < DPL; ++e) o[j][e] = 0.f;
        }
#pragma unroll
        for (int i = 0; i < NV; ++i) lsum[i] = 0.f;

        const int prologue = min(kStages, n_mine);
        for (int i = 0; i < prologue; ++i) issue(i);

        for (int i = 0; i < n_mine; ++i) {
            const int stage = consumed % kStages;
            const uint32_t parity = (consumed / kStages) & 1;
            if (!mbar_wait(&bars[stage], parity)) {
                if (lane == 0) set_error(a.err, PKV_DEVERR_TIMEOUT);
                aborted = true;
                break;
            }
            ++consumed;
            const uint8_t* sK = ring + stage * S::kStageBytes;
            const uint8_t* sV = sK + S::kPageBytes;
            const int lp = pb + warp + i * kDecWarps;
            const int nvalid = min(kPage, nkv - lp * kPage);

            // ---- scores: lane (tg, c8) does tokens tg*4..tg*4+3 over dims c8*QKD..+QKD
            float v[N0];
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                float acc[G];
#pragma unroll
                for (int j = 0; j < G; ++j) acc[j] = 0.f;
                const uint4* krow = reinterpret_cast<const uint4*>(sK + (tg * 4 + kk) * D * 2) +
                                    c8 * NCH;
#pragma unroll
                for (int ci = 0; ci < NCH; ++ci) {
                    const uint4 w = krow[ci ^ (NCH == 2 ? swz : 0)];
                    const uint32_t ws4[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = Cv::unpack(ws4[e]);
#pragma unroll
                        for (int j = 0; j < G; ++j) {
                            acc[j] = fmaf(qf[j][ci * 8 + 2 * e], f.x, acc[j]);
                            acc[j] = fmaf(qf[j][ci * 8 + 2 * e + 1], f.y, acc[j]);
                        }
                    }
                }
#pragma unroll
                for (int j = 0; j < G; ++j) v[kk * G + j] = acc[j];
            }
            // ---- reduce over the 8 lanes of a token group by recursive halving
#pragma unroll
            for (int i2 = 0; i2 < N1; ++i2) {
                const float send = b2 ? v[i2] : v[i2 + N1];
                const float keep = b2 ? v[i2 + N1] : v[i2];
                v[i2] = keep + __shfl_xor_sync(kFull, send, 4);
            }
            if constexpr (N1 >= 2) {
#pragma unroll
                for (int i2 = 0; i2 < N2; ++i2) {
                    const float send = b1 ? v[i2] : v[i2 + N2];
                    const float keep = b1 ? v[i2 + N2] : v[i2];
                    v[i2] = keep + __shfl_xor_sync(kFull, send, 2);
                }
            }
            if constexpr (N2 >= 2) {
#pragma unroll
                for (int i2 = 0; i2 < NV; ++i2) {
                    const float send = b0 ? v[i2] : v[i2 + NV];
                    const float keep = b0 ? v[i2 + NV] : v[i2];
                    v[i2] = keep + __shfl_xor_sync(kFull, send, 1);
                }
            } else {
                v[0] += __shfl_xor_sync(kFull, v[0], 1);
            }
            // now v[i] = score of token my_tok for head (G>=2 ? b0*NV + i : 0)
            const bool valid = my_tok < nvalid;
            float s[NV], pmx[NV];
#pragma unroll
            for (int i2 = 0; i2 < NV; ++i2) {
                s[i2] = valid ? v[i2] : -INFINITY;
                float x = s[i2];
                x = fmaxf(x, __shfl_xor_sync(kFull, x, 2));
                x = fmaxf(x, __shfl_xor_sync(kFull, x, 4));
                x = fmaxf(x, __shfl_xor_sync(kFull, x, 8));
                x = fmaxf(x, __shfl_xor_sync(kFull, x, 16));
                pmx[i2] = x;
            }
            float pm[G];
            if constexpr (G == 1) {
                pm[0] = pmx[0];
            } else {
#pragma unroll
                for (int i2 = 0; i2 < NV; ++i2) {
                    const float other = __shfl_xor_sync(kFull, pmx[i2], 1);
                    pm[i2] = b0 ? other : pmx[i2];
                    pm[NV + i2] = b0 ? pmx[i2] : other;
                }
            }
            float alpha[G];
            bool rescale = false;
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const float mn = fmaxf(m[j], pm[j]);
                alpha[j] = fast_exp2(m[j] - mn);
                rescale |= mn != m[j];
                m[j] = mn;
            }
#pragma unroll
            for (int i2 = 0; i2 < NV; ++i2) {
                const float mh = (G == 1) ? m[0] : (b0 ? m[NV + i2] : m[i2]);
                const float ah = (G == 1) ? alpha[0] : (b0 ? alpha[NV + i2] : alpha[i2]);
                const float p = fast_exp2(s[i2] - mh);
                lsum[i2] = fmaf(lsum[i2], ah, p);
                if (G > 1 || !b0) pbuf[my_tok * G + ((G == 1) ? 0 : (b0 ? NV : 0) + i2)] = p;
            }
            __syncwarp();

            // ---- o[j][:] = o[j][:] * alpha[j] + sum_tok p[tok][j] * V[tok][:]
            if (rescale) {
#pragma unroll
                for (int j = 0; j < G; ++j)
#pragma unroll
                    for (int e = 0; e < DPL; ++e) o[j][e] *= alpha[j];
            }
            auto pv_token = [&](int tok) {
                float vf[DPL];
                if constexpr (DPL == 4) {
                    const uint2 w = *reinterpret_cast<const uint2*>(sV + tok * D * 2 + lane * 8);
                    const float2 f0 = Cv::unpack(w.x), f1 = Cv::unpack(w.y);
                    vf[0] = f0.x; vf[1] = f0.y; vf[2] = f1.x; vf[3] = f1.y;
                } else {
                    const uint32_t w = *reinterpret_cast<const uint32_t*>(sV + tok * D * 2 + lane * 4);
                    const float2 f0 = Cv::unpack(w);
                    vf[0] = f0.x; vf[1] = f0.y;
                }
                const float* pr = pbuf + tok * G;
#pragma unroll
                for (int j = 0; j < G; ++j) {
                    const float pj = pr[j];
#pragma unroll
                    for (int e = 0; e < DPL; ++e) o[j][e] = fmaf(pj, vf[e], o[j][e]);
                }
            };
            if (nvalid == kPage) {
#pragma unroll
                for (int tok = 0; tok < kPage; ++tok) pv_token(tok);
            } else {
                for (int tok = 0; tok < nvalid; ++tok) pv_token(tok);
            }
            __syncwarp();
            if (i + kStages < n_mine) issue(i + kStages);
        }
        if (aborted) {  // drain what this warp still has in flight, bounded
            if (lane == 0) s_item[1] = 1;
            while (consumed < issued) {
                const int stage = consumed % kStages;
                mbar_wait(&bars[stage], (consumed / kStages) & 1);
                ++consumed;
            }
        }

        // ---- warp totals: sum lsum over the token lanes, gather every head
        float lh[G];
#pragma unroll
        for (int i2 = 0; i2 < NV; ++i2) {
            float x = lsum[i2];
            x += __shfl_xor_sync(kFull, x, 2);
            x += __shfl_xor_sync(kFull, x, 4);
            x += __shfl_xor_sync(kFull, x, 8);
            x += __shfl_xor_sync(kFull, x, 16);
            if constexpr (G == 1) {
                lh[0] = x;
            } else {
                const float other = __shfl_xor_sync(kFull, x, 1);
                lh[i2] = b0 ? other : x;
                lh[NV + i2] = b0 ? x : other;
            }
        }
        float* mw = merge + warp * G * (D + 2);
#pragma unroll
        for (int j = 0; j < G; ++j) {
#pragma unroll
            for (int e = 0; e < DPL; ++e) mw[j * (D + 2) + lane * DPL + e] = o[j][e];
            if (lane == 0) {
                mw[j * (D + 2) + D] = m[j];
                mw[j * (D + 2) + D + 1] = lh[j];
            }
        }
        __syncthreads();

        // ---- merge the four warps; finish the row or leave a partial for the combine
        for (int idx = threadIdx.x; idx < G * D; idx += kDecThreads) {
            const int j = idx / D, d = idx % D;
            float M = -1e30f;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) M = fmaxf(M, merge[(w * G + j) * (D + 2) + D]);
            float L = 0.f, O = 0.f;
#pragma unroll
            for (int w = 0; w < kDecWarps; ++w) {
                const float* mr = merge + (w * G + j) * (D + 2);
                const float sc = fast_exp2(mr[D] - M);
                L = fmaf(mr[D + 1], sc, L);
                O = fmaf(mr[d], sc, O);
            }
            if (nsplit <= 1) {
                const float res = O / L;
                uint16_t* op = static_cast<uint16_t*>(a.out) +
                               (static_cast<int64_t>(t) * Hq + g * G + j) * D + d;
                const uint32_t packed = Cv::pack(res, 0.f);
                *op = static_cast<uint16_t>(packed & 0xffffu);
            } else {
                part_o[(static_cast<int64_t>(item) * G + j) * D + d] = O;
                if (d == 0) part_ml[static_cast<int64_t>(item) * G + j] = make_float2(M, L);
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------------------------
// combine: out = sum_s 2^(m_s - M) o_s / sum_s 2^(m_s - M) l_s for split requests.
// One CTA per (request, KV head); requests with a single split were finished in place.
// ------------------------------------------------------------------------------------
template <typename T, int D, int G>
__global__ void __launch_bounds__(128) combine_kernel(StepArgs a) {
    using Cv = F16<T>;
    constexpr int kMaxSplitsSmem = 64;
    __shared__ float s_w[G][kMaxSplitsSmem];
    __shared__ float s_inv_l[G];
    const int r = blockIdx.x / a.num_kv_heads, g = blockIdx.x % a.num_kv_heads;
    const int4 in = ws_req_info(a)[r];
    if (in.z != 1 || in.y <= 1) return;
    const int ns = min(in.y, kMaxSplitsSmem);
    const int item0 = in.x + g * in.y;
    if (item0 + ns > ws_ctrl(a)[2]) return;  // the plan dropped the work (bad device data)
    const float2* part_ml = reinterpret_cast<const float2*>(a.ws + a.lay.part_ml);
    const float* part_o = reinterpret_cast<const float*>(a.ws + a.lay.part_o);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int j = warp; j < G; j += 4) {
        float M = -1e30f;
        for (int s = lane; s < ns; s += 32) M = fmaxf(M, part_ml[(int64_t)(item0 + s) * G + j].x);
#pragma unroll
        for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
        float L = 0.f;
        for (int s = lane; s < ns; s += 32) {
            const float2 ml = part_ml[(int64_t)(item0 + s) * G + j];
            const float w = fast_exp2(ml.x - M);
            s_w[j][s] = w;
            L = fmaf(ml.y, w, L);
        }
#pragma unroll
        for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(kFull, L, o);
        if (lane == 0) s_inv_l[j] = 1.f / L;
    }
    __syncthreads();
    const int t = a.q_offsets[r];
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
        const int j = idx / D, d = idx % D;
        float O = 0.f;
        for (int s = 0; s < ns; ++s)
            O = fmaf(part_o[((int64_t)(item0 + s) * G + j) * D + d], s_w[j][s], O);
        const float res = O * s_inv_l[j];
        uint16_t* op = static_cast<uint16_t*>(a.out) +
                       (static_cast<int64_t>(t) * a.num_q_heads + g * G + j) * D + d;
        *op = static_cast<uint16_t>(Cv::pack(res, 0.f) & 0xffffu);
    }
}

// ------------------------------------------------------------------------------------
// host launchers
// ------------------------------------------------------------------------------------
WorkspaceLayout workspace_layout(int num_reqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int total_q_tokens, int max_q_len, int num_sms,
                                 int prefill_min_q) {
    WorkspaceLayout L{};
    const int G = num_q_heads / num_kv_heads;
    const int pairs = std::max(1, num_reqs * num_kv_heads);
    int max_splits = cdiv(2 * kItemsPerSm * num_sms, pairs);
    max_splits = std::min(64, std::max(4, max_splits));
    L.max_splits = max_splits;
    L.max_split_items = num_reqs * num_kv_heads * max_splits;
    L.max_items = L.max_split_items + total_q_tokens * num_kv_heads;
    // prefill tiles: none unless some request can reach prefill_min_q tokens; then at most
    // T/128 full tiles plus one partial tile per prefilling request
    const int prefill_reqs = max_q_len >= prefill_min_q
                                 ? std::min(num_reqs, total_q_tokens / std::max(1, prefill_min_q))
                                 : 0;
    L.max_tiles = prefill_reqs ? (total_q_tokens / 128 + prefill_reqs) *
                                     (num_q_heads / prefill_heads_per_tile(num_q_heads, num_kv_heads))
                               : 0;
    auto up = [](size_t x) { return (x + 255) / 256 * 256; };
    size_t off = 0;
    L.ctrl = off; off = up(off + 64 * sizeof(int32_t));
    L.req_info = off; off = up(off + static_cast<size_t>(num_reqs) * 16);
    L.items = off; off = up(off + static_cast<size_t>(L.max_items) * 16);
    L.tiles = off; off = up(off + static_cast<size_t>(L.max_tiles) * 16);
    L.part_ml = off; off = up(off + static_cast<size_t>(L.max_split_items) * G * 8);
    L.part_o = off; off = up(off + static_cast<size_t>(L.max_split_items) * G * head_dim * 4);
    L.total = off;
    return L;
}

int launch_plan(const StepArgs& a, cudaStream_t stream) {
    plan_kernel<<<1, kPlanThreads, 0, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

template <typename T, int D, int G>
static int launch_decode_t(const StepArgs& a, cudaStream_t stream, cudaEvent_t ev0,
                           cudaEvent_t ev1) {
    using S = DecodeSmem<T, D, G>;
    static int blocks_per_sm = 0;  // benign race: every thread computes the same value
    if (blocks_per_sm == 0) {
        if (cudaFuncSetAttribute(decode_kernel<T, D, G>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 S::kBytes) != cudaSuccess)
            return PKV_ERR_CUDA;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<T, D, G>,
                                                          kDecThreads, S::kBytes) != cudaSuccess)
            return PKV_ERR_CUDA;
        blocks_per_sm = std::max(1, n);
    }
    const int grid = blocks_per_sm * a.num_sms;
    if (ev0 && cudaEventRecord(ev0, stream) != cudaSuccess) return PKV_ERR_CUDA;
    decode_kernel<T, D, G><<<grid, kDecThreads, S::kBytes, stream>>>(a);
    if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
    if (ev1 && cudaEventRecord(ev1, stream) != cudaSuccess) return PKV_ERR_CUDA;
    combine_kernel<T, D, G><<<std::max(1, a.num_reqs * a.num_kv_heads), 128, 0, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

template <typename T, int D>
static int dispatch_group(const StepArgs& a, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
    switch (a.num_q_heads / a.num_kv_heads) {
        case 1: return launch_decode_t<T, D, 1>(a, s, e0, e1);
        case 2: return launch_decode_t<T, D, 2>(a, s, e0, e1);
        case 4: return launch_decode_t<T, D, 4>(a, s, e0, e1);
        case 8: return launch_decode_t<T, D, 8>(a, s, e0, e1);
        default: return PKV_ERR_UNSUPPORTED;
    }
}

int launch_decode(const StepArgs& a, cudaStream_t stream, cudaEvent_t e0, cudaEvent_t e1) {
    if (a.dtype == PKV_BF16)
        return a.head_dim == 128 ? dispatch_group<__nv_bfloat16, 128>(a, stream, e0, e1)
                                 : dispatch_group<__nv_bfloat16, 64>(a, stream, e0, e1);
    return a.head_dim == 128 ? dispatch_group<__half, 128>(a, stream, e0, e1)
                             : dispatch_group<__half, 64>(a, stream, e0, e1);
}

}  // namespace pkv
