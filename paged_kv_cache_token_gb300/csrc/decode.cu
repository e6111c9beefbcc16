// Decode path of the paged attention step: work planning, the split-KV streaming kernel
// and the split combine.
//
// hotelren.com/news/6181127 §3.1: a decode row scores its query against all S+t cached
// keys, softmax, then a weighted sum of all S+t values; §3.2: this is a stream over the
// cache whose bytes grow linearly with the context, so it is bound by memory bandwidth;
// §6.3: with grouped-query attention several query heads share one KV head (here they are
// processed together, so each K/V byte is read once per KV head, not once per query head).
//
// Rows of requests that advance by fewer than `prefill_min_q` tokens are decode rows; each
// row i of such a request attends keys 0..ctx+i.  Work item = (decode row, KV head, split),
// a split being an even share of the row's pages.  Every warp is an independent worker:
// it takes items from a device queue, streams each page's K block and V block (16 x D
// each, contiguous in the pool) through a private shared-memory ring with 1-D bulk async
// copies, and starts the next item's first pages while finishing the current one so the
// copy pipeline never drains.  A page's scores for the item's G query heads are one set of
// mma.sync tensor-core contractions (16 tokens x 8 head columns); an online softmax in base-2
// units keeps (running max, running sum, un-normalised output) per query head; the weighted
// sum over the page's values runs on the FP32 pipes for 16-bit pages (FFMA2 over V rows)
// and on the tensor cores for INT8 pages.  A row with one split is normalised and written
// directly; otherwise each split leaves its partial (m, l, O) in a fixed slot and the
// combine kernel reduces them: m* = max m_s, l* = sum l_s 2^(m_s - m*),
// O = sum O_s 2^(m_s - m*) / l* (in two passes over 64-split chunks for long rows).
//
// The plan kernel builds the step's work lists on the device: the split size from the
// total decode pages, row records by one warp per request, item records one per thread
// over the whole grid (a single long row has thousands), prefill tile records longest
// first.
#include <algorithm>
#include <climits>
#include <type_traits>

#include "common.cuh"
#include "launch.h"

namespace pkv {

namespace {

constexpr int kPlanThreads = 1024;
constexpr int kPlanBlocks = 32;   // CTAs sharing the record writes
constexpr int kDecWarps = 4;
constexpr int kDecThreads = kDecWarps * 32;
constexpr int kStages = 3;
constexpr int kMinSplitPages = 4;
constexpr int kItemsPerWarp = 6;  // target decode items per resident warp
constexpr int kManySplits = 64;   // rows that may have more splits get a grouped combine
constexpr int kChunkedCtas = 4096;  // largest grid of the two-pass combine
constexpr int kDecMaxCtasPerSm = 3;  // decode CTAs an SM can hold (INT8 pages)
constexpr int kMinChunkPages = 4;    // smallest dynamic chunk of a self-planned step
constexpr int kStaticOnlyPagesPerWarp = 32;  // below this per warp: no 3/4 static split
constexpr int kSlotsPerWarp = 6;     // partial slots a self-planned step may use per warp

template <typename T>
__device__ __forceinline__ T* ws_at(const StepArgs& a, size_t off) {
    return reinterpret_cast<T*>(a.ws + off);
}

// A request is valid for this step when its lengths agree with q_offsets (o0 = q_offsets[r],
// o1 = q_offsets[r + 1]) and the host maxima.
__device__ __forceinline__ bool request_ok(const StepArgs& a, int q, int c, int o0, int o1) {
    return q >= 0 && c >= 0 && q <= a.max_q_len && c <= a.max_context_len && o1 - o0 == q;
}

// sum_{x=a}^{b} ceil(x / B) for 1 <= a, in closed form: with S(n) = sum_{y=0}^{n} floor(y/B)
// = B m (m-1) / 2 + m (r+1) for n = B m + r, the sum is S(b + B - 1) - S(a + B - 2).  A decode
// row over x keys holds ceil(x / 16) pages and, with splits of sp pages, ceil(x / (16 sp))
// items (ceil(ceil(x/16)/sp) = ceil(x/(16 sp))), so a request's totals need no loop over
// its rows.
__device__ __forceinline__ long long sum_ceil(long long a, long long b, long long B) {
    auto S = [B](long long n) {
        const long long m = n / B, r = n - B * m;
        return B * m * (m - 1) / 2 + m * (r + 1);
    };
    return b < a ? 0 : S(b + B - 1) - S(a + B - 2);
}

// Lengths of request r, all four loads issued together (no dependent round trip).
struct ReqLens { int q, c, t0; bool ok; };
// Read before the kernel's dependency wait (the lengths are final before the step starts).
// context_lens is the one step input a library kernel updates in place (advance_context,
// between the steps of a device-side loop): it fences its write before letting this grid
// launch, and the read goes to L2, past any line an SM's L1 kept from an earlier step.
__device__ __forceinline__ ReqLens load_request(const StepArgs& a, int r) {
    const int q = a.q_lens[r], c = __ldcg(a.context_lens + r);
    const int o0 = a.q_offsets[r], o1 = a.q_offsets[r + 1];
    return ReqLens{q, c, o0, request_ok(a, q, c, o0, o1)};
}

}  // namespace

// ------------------------------------------------------------------------------------
// plan: validate lengths, choose the split size, number decode rows, decode items and
// prefill tiles.  kPlanBlocks CTAs each compute the same counts, split size and scans
// (per-request values of a chunk of 1024 requests live in shared memory); the record
// writes are dealt out across all of them, because one SM alone drains stores slowly
// enough to dominate the step's planning time.
// ------------------------------------------------------------------------------------
namespace {
// exclusive block-wide scan of three ints per thread at once
struct Int3 { int x, y, z; };
__device__ Int3 block_exclusive_scan3(Int3 v, Int3* total, Int3* s_warp) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    Int3 x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int yx = __shfl_up_sync(kFull, x.x, o), yy = __shfl_up_sync(kFull, x.y, o),
                  yz = __shfl_up_sync(kFull, x.z, o);
        if (lane >= o) { x.x += yx; x.y += yy; x.z += yz; }
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        Int3 w = s_warp[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int yx = __shfl_up_sync(kFull, w.x, o), yy = __shfl_up_sync(kFull, w.y, o),
                      yz = __shfl_up_sync(kFull, w.z, o);
            if (lane >= o) { w.x += yx; w.y += yy; w.z += yz; }
        }
        s_warp[lane] = w;
    }
    __syncthreads();
    const Int3 before = warp ? s_warp[warp - 1] : Int3{0, 0, 0};
    *total = s_warp[31];
    __syncthreads();
    return Int3{before.x + x.x - v.x, before.y + x.y - v.y, before.z + x.z - v.z};
}
}  // namespace

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(StepArgs a) {
    __shared__ unsigned long long s_sum;
    __shared__ int s_bad, s_split, s_npf;
    __shared__ int s_pf[kPlanThreads];  // chunk positions of the prefill requests
    __shared__ Int3 s_warp3[32];
    __shared__ int s_q[kPlanThreads], s_c[kPlanThreads], s_t0[kPlanThreads];
    __shared__ int s_row0[kPlanThreads], s_item0[kPlanThreads], s_tile0[kPlanThreads];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int32_t* ctrl = ws_at<int32_t>(a, a.lay.ctrl);
    int4* rows = ws_at<int4>(a, a.lay.rows);
    int4* items = ws_at<int4>(a, a.lay.items);
    int4* tiles = ws_at<int4>(a, a.lay.tiles);
    const int Hkv = a.num_kv_heads;
    const int slots = a.num_q_heads / a.heads_per_tile;
    // prefill tiles of a request: one per 128-row query tile and head pair (an even KV
    // group), or one per pair of 128-row query tiles and query head (one head per KV head)
    auto tile_units = [&](int q) {
        return a.heads_per_tile == 2 ? cdiv(q, 128) : cdiv(cdiv(q, 128), 2);
    };
    if (tid == 0) {
        s_sum = 0;
        s_bad = 0;
    }
    if (a.plan_wait_first) pdl_wait();
    __syncthreads();

    // ---- pass A: validity and the decode page total (sets the split size).  The lengths of
    //      this thread's request in the first chunk stay in registers for the fill.
    unsigned long long my_sum = 0;
    ReqLens first{0, 0, 0, false};
    if (tid == 0 && (a.q_offsets[0] != 0 || a.q_offsets[a.num_reqs] != a.total_q_tokens))
        atomicOr(&s_bad, 1);
    for (int r = tid; r < a.num_reqs; r += kPlanThreads) {
        const ReqLens L = load_request(a, r);
        if (r == tid) first = L;
        if (!L.ok) { atomicOr(&s_bad, 1); continue; }
        if (cdiv(L.c + L.q, kPage) > a.max_pages) set_error(a.err, PKV_DEVERR_TABLE_RANGE);
        if (L.q >= 1 && L.q < a.prefill_min_q) my_sum += sum_ceil(L.c + 1, L.c + L.q, kPage);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) my_sum += __shfl_xor_sync(kFull, my_sum, o);
    if (lane == 0 && my_sum) atomicAdd(&s_sum, my_sum);
    __syncthreads();
    const bool bad = s_bad != 0;
    if (tid == 0) {
        if (bad && blockIdx.x == 0) set_error(a.err, PKV_DEVERR_TOKENS);
        const unsigned long long heads = s_sum * static_cast<unsigned long long>(Hkv);
        const unsigned long long tgt = static_cast<unsigned long long>(a.lay.target_items);
        const unsigned long long sp = (heads + tgt - 1) / tgt;
        s_split = static_cast<int>(max(sp, static_cast<unsigned long long>(kMinSplitPages)));
    }
    __syncthreads();
    const int sp = s_split;

    // ---- per chunk: count, scan, then fill rows / items / tiles (warp per request)
    Int3 carry{0, 0, 0};
    bool overflow = false;
    for (int base = 0; base < a.num_reqs; base += kPlanThreads) {
        const int r = base + tid;
        int q = 0, c = 0, t0 = 0;
        Int3 n{0, 0, 0};  // decode rows, decode items, prefill tiles of request r
        if (r < a.num_reqs && !bad) {
            const ReqLens L = base == 0 ? first : load_request(a, r);
            q = L.ok ? L.q : 0;
            c = L.c;
            t0 = L.t0;
            if (q >= 1 && q < a.prefill_min_q) {
                n.x = q;
                // clamped past the bound, which still trips the overflow check below
                const long long items = Hkv * sum_ceil(c + 1, c + q, kPage * sp);
                n.y = static_cast<int>(min(items, static_cast<long long>(a.lay.max_items) + 1));
            }
            if (q > 1 && q >= a.prefill_min_q) n.z = tile_units(q) * slots;
        }
        if (tid == 0) s_npf = 0;  // read after the scan's barriers
        Int3 tot;
        const Int3 ex = block_exclusive_scan3(n, &tot, s_warp3);
        overflow = overflow || carry.x + tot.x > a.lay.max_rows ||
                   carry.y + tot.y > a.lay.max_items || carry.z + tot.z > a.lay.max_tiles;
        if (r < a.num_reqs) {
            s_q[tid] = q;
            s_c[tid] = c;
            s_t0[tid] = t0;
            s_row0[tid] = carry.x + ex.x;
            s_item0[tid] = carry.y + ex.y;
            s_tile0[tid] = carry.z + ex.z;
            if (n.z > 0) s_pf[atomicAdd(&s_npf, 1)] = tid;
        }
        __syncthreads();
        const int nreq = min(kPlanThreads, a.num_reqs - base);
        // request k of the chunk belongs to warp (k / grid) of CTA (k % grid); the tiles of a
        // prefill request are spread over every warp of every CTA
        const int gwarp = blockIdx.x * (kPlanThreads / 32) + warp;
        const int nwarps = gridDim.x * (kPlanThreads / 32);
        for (int f = 0; !overflow && f < s_npf; ++f) {
            const int k = s_pf[f], qk = s_q[k];
            {
                const int nt = tile_units(qk), rq = base + k;
                for (int i = gwarp * 32 + lane; i < nt * slots; i += nwarps * 32)
                    tiles[s_tile0[k] + i] = make_int4(rq, nt - 1 - i / slots, i % slots, 0);
            }
        }
        for (int k = blockIdx.x + gridDim.x * warp; !overflow && k < nreq;
             k += gridDim.x * (kPlanThreads / 32)) {
            const int qk = s_q[k], ck = s_c[k];
            if (qk >= 1 && qk < a.prefill_min_q) {
                // rows of this request, 32 at a time: lane i = row r0 + i; warp scan of item
                // counts, carried from one group of rows to the next
                int item0 = s_item0[k];
                for (int r0 = 0; r0 < qk; r0 += 32) {
                    const int row = r0 + lane;
                    const int ns = row < qk ? cdiv(ck + row + 1, kPage * sp) : 0;
                    int incl = Hkv * ns;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int y = __shfl_up_sync(kFull, incl, o);
                        if (lane >= o) incl += y;
                    }
                    const int first = item0 + incl - Hkv * ns;
                    if (row < qk)
                        rows[s_row0[k] + row] = make_int4(s_t0[k] + row, first, ck + row + 1, ns);
                    item0 += __shfl_sync(kFull, incl, 31);
                }
            }
        }
        // item records, one item per thread over the whole grid (a long row has thousands):
        // the request by binary search over the chunk's first-item offsets (requests without
        // items share their successor's offset, so the last offset <= e is the owner), then
        // the row by walking the request's < prefill_min_q rows.  Record 0 = {token,
        // head | split << 16, first page, pages}, record 1 = {keys, splits, request, slot of
        // split 0}; the first `rem` splits of a row get one page more than `per`.
        const int nitems = overflow ? 0 : tot.y;
        for (int i = blockIdx.x * kPlanThreads + tid; i < nitems; i += gridDim.x * kPlanThreads) {
            const int e = carry.y + i;
            int lo = 0, hi = nreq - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (s_item0[mid] <= e) lo = mid; else hi = mid - 1;
            }
            const int k = lo, ck = s_c[k];
            int local = e - s_item0[k], row = 0, first = s_item0[k], ns = 1;
            for (;; ++row) {
                ns = cdiv(ck + row + 1, kPage * sp);
                if (local < Hkv * ns || row + 1 >= s_q[k]) break;
                local -= Hkv * ns;
                first += Hkv * ns;
            }
            const int g = local / ns, sidx = local - g * ns;
            const int nkv = ck + row + 1, pages = cdiv(nkv, kPage);
            const int per = pages / ns, rem = pages - per * ns;
            int4* dst = items + 2 * static_cast<int64_t>(e);
            dst[0] = make_int4(s_t0[k] + row, g | (sidx << 16), sidx * per + min(sidx, rem),
                               per + (sidx < rem ? 1 : 0));
            dst[1] = make_int4(nkv, ns, base + k, first + g * ns);
        }
        carry = Int3{carry.x + tot.x, carry.y + tot.y, carry.z + tot.z};
        __syncthreads();
    }
    // the plan ran alongside this step's kv_append; finish only after it (so a kernel that
    // waits for the plan also sees the appended K/V), then let the attention kernels start.
    // A plan launched on its own does not let the next kernel start early: a run over it
    // reads the work list before its own wait, so the list must be complete when that
    // kernel launches.
    pdl_wait();
    if (!a.plan_wait_first) pdl_trigger();
    if (tid == 0 && blockIdx.x == 0) {
        if (overflow) set_error(a.err, PKV_DEVERR_TOKENS);  // host maxima were wrong
        ctrl[0] = 0;
        ctrl[1] = overflow ? 0 : carry.y;
        ctrl[2] = overflow ? 0 : carry.x;
        ctrl[3] = sp;
        ctrl[8] = 0;
        ctrl[9] = overflow ? 0 : carry.z;
    }
}

// ------------------------------------------------------------------------------------
// decode: independent warps pull items; see the file comment for the data flow.
// ------------------------------------------------------------------------------------
// Q8: the pools hold INT8 codes (half the bytes per page; the scores need no shared-memory
// staging).  Four stages of half-size pages let three CTAs share an SM: more warps to hide
// the latency of the per-page dependency chain, with as many bytes in flight as before.
template <typename T, int D, int G, bool Q8>
struct DecodeSmem {
    static constexpr int kNst = Q8 ? 4 : kStages;
    static constexpr int kPageBytes = kPage * D * (Q8 ? 1 : 2);  // one K (or V) page block
    static constexpr int kStageBytes = 2 * kPageBytes;
    static constexpr int kRing = kDecWarps * kNst * kStageBytes;
    static constexpr int kPbuf = Q8 ? 0 : kDecWarps * kPage * G * 8;  // (p, p) per token, head
    static constexpr int kBars = kDecWarps * kNst * 8;
    static constexpr int kBytes = kRing + kPbuf + kBars;
};

// ---- INT8 pages on the tensor cores (mma.sync m16n8k16, fp16 operands, fp32 accumulate).
// A code c of byte u = c + 128 (sign bit flipped) becomes the fp16 number 1024 + u exactly
// when u is the low byte under an exponent byte 0x64.  Keys enter the score MMA in that
// form: every key dim then carries an extra 1152 (= 1024 + 128), which adds
// 1152 * sum_d q'_d to every score of a query head -- the same for every token, so the
// softmax is unchanged.  Values get the 1152 subtracted (exact in fp16) because they are
// summed with weights.
__device__ __forceinline__ uint32_t codes_lo_h2(uint32_t x) {  // bytes 0, 1 -> 1024 + u
    return __byte_perm(x, 0x6464u, 0x4140);
}
__device__ __forceinline__ uint32_t codes_hi_h2(uint32_t x) {  // bytes 2, 3 -> 1024 + u
    return __byte_perm(x, 0x6464u, 0x4342);
}
__device__ __forceinline__ uint32_t minus_1152_h2(uint32_t h) {
    const uint32_t c = 0x64806480u;   // fp16 1152 in both halves
    const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&h),
                              *reinterpret_cast<const __half2*>(&c));
    return *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}
// d += A (16x16, row-major fragments a0..a3) * B (16x8, col-major fragments b0, b1)
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// 2^x in one MUFU operation (results below 2^-126 flush to zero: softmax weights that small
// vanish against the row's maximum weight of 1)
__device__ __forceinline__ float ex2_ftz(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// the same for 16-bit T operands (bf16 or fp16), exact products, fp32 accumulation
template <typename T>
__device__ __forceinline__ void mma_16816_t(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                            uint32_t a3, uint32_t b0, uint32_t b1) {
    if constexpr (std::is_same<T, __half>::value) {
        mma_16816(d, a0, a1, a2, a3, b0, b1);
    } else {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
            "{%8,%9}, {%0,%1,%2,%3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}
// transpose of an 8x8 16-bit matrix held one row-pair register per thread
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// Units of a self-planned step: nw static units of `static_pages` pages (the fraction
// num / den of the total, rounded down), then chunks of `chunk_pages` pages.  Every unit has
// two partial slots, so the chunks are no smaller than the workspace's slots allow.
// Measured on the decode batches (A/B in one process): 16-bit pages do best with 3/4 static
// and chunks of at least 4 pages (the warps' streaming rates differ by about +-8%, and the
// chunks even out the tail); INT8 pages with everything static (a piece's setup -- q times
// the key scales -- costs too much for small chunks), the remainder only in chunks.
struct SelfPlanUnits { int static_pages, chunk_pages, chunks; };
__device__ __forceinline__ SelfPlanUnits self_plan_units(int total, int nw, int slots, int num,
                                                         int den) {
    SelfPlanUnits u;
    u.static_pages = static_cast<int>(static_cast<int64_t>(total) * num /
                                      (static_cast<int64_t>(den) * nw));
    const int dyn = total - nw * u.static_pages;
    const int max_chunks = max(1, slots / 2 - nw);
    u.chunk_pages = max(kMinChunkPages, cdiv(dyn, max_chunks));
    u.chunks = cdiv(dyn, u.chunk_pages);
    return u;
}

// The chunk counter of a self-planned step is one 64-bit word: the call's epoch (40 bits,
// from the host, never 0) above a 24-bit count, so the workspace needs no initialisation.
// Every CTA tries once, in its prologue, to move the word from an earlier call's epoch (or
// 0, where the combine parks it) to this call's with a zero count; claims, long after, are
// then single atomic adds.
__device__ __forceinline__ void install_epoch(unsigned long long* ctr, unsigned long long epoch) {
    const unsigned long long cur = atomicAdd(ctr, 0ull);
    if ((cur >> 24) != epoch) atomicCAS(ctr, cur, epoch << 24);
}
// The chunk a claim got: `old` is the word an atomic add of 1 returned.  A claim that still
// found another epoch (no CTA's install had landed) moves the word itself, taking chunk 0,
// or claims again once another thread has; bounded: after kWaitLimit failed swaps it gives
// up (no more chunks) and sets PKV_DEVERR_TIMEOUT.
__device__ __forceinline__ int claimed_chunk(unsigned long long* ctr, unsigned long long old,
                                             unsigned long long epoch, int32_t* err) {
    for (uint32_t i = 0; i < kWaitLimit; ++i) {
        if ((old >> 24) == epoch) return static_cast<int>(old & 0xffffffull);
        const unsigned long long expected = old + 1;  // the word after this thread's add
        const unsigned long long prev = atomicCAS(ctr, expected, (epoch << 24) | 1ull);
        if (prev == expected) return 0;
        // another thread moved or bumped the word: claim again on its current value
        old = (prev >> 24) == epoch ? atomicAdd(ctr, 1ull) : prev - 1;
    }
    set_error(err, PKV_DEVERR_TIMEOUT);
    return INT_MAX;
}

struct UnitMap {
    int64_t S, C, D0;
    int nw;
    __device__ int64_t unit(int64_t p) const { return p < D0 ? p / S : nw + (p - D0) / C; }
    __device__ int64_t start(int64_t u) const { return u < nw ? u * S : D0 + (u - nw) * C; }
};
__device__ __forceinline__ UnitMap unit_map(const int32_t* ctrl) {
    UnitMap m;
    m.nw = ctrl[4];
    m.S = ctrl[5];
    m.C = ctrl[6];
    m.D0 = static_cast<int64_t>(m.nw) * m.S;
    return m;
}

// Segments of more than kLongPieces pieces -- e.g. one long row spread over the whole grid --
// are folded by the combine in chunks of kPieceChunk pieces on different CTAs.  A chunk's
// state replaces its first piece (a thread reads and writes only its own elements of a
// slot).  The CTA whose chunk arrives last at the segment's counter (zeroed by the decode
// kernel) merges the chunk states in chunk order: nothing waits, and the result does not
// depend on which CTA merges.  Up to kMaxLong such pairs are listed, in pair order, by the
// decode kernel (the rest are folded whole by one CTA).
constexpr int kPieceChunk = 32;
constexpr int kLongPieces = 96;
constexpr int kMaxLong = 512;
// Lists the pairs with more than kLongPieces pieces: l_rh[k] the k-th in pair order,
// l_off[k] its first chunk in the sequence of all listed pairs' chunks; hdr = {listed pairs,
// their chunks}.  The whole CTA of NT threads calls it; lsum is 2 x NT / 32 ints of shared
// memory.
template <int NT, typename CountFn>
__device__ __forceinline__ void list_long_pairs(CountFn count_of, int npairs, int32_t* l_rh,
                                                int32_t* l_off, int32_t* hdr,
                                                int (*lsum)[NT / 32]) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = cdiv(npairs, NT);
    const int p0 = min(npairs, tid * per), p1 = min(npairs, p0 + per);
    int nb = 0, nc = 0;
    for (int rh = p0; rh < p1; ++rh) {
        const int cnt = count_of(rh);
        if (cnt > kLongPieces) {
            ++nb;
            nc += cdiv(cnt, kPieceChunk);
        }
    }
    int ib = nb, ic = nc;  // inclusive scans over the warp, then over the warps
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int yb = __shfl_up_sync(kFull, ib, o), yc = __shfl_up_sync(kFull, ic, o);
        if (lane >= o) {
            ib += yb;
            ic += yc;
        }
    }
    if (lane == 31) {
        lsum[0][warp] = ib;
        lsum[1][warp] = ic;
    }
    __syncthreads();
    int eb = ib - nb, ec = ic - nc, tb = 0, tc = 0;
    for (int w = 0; w < NT / 32; ++w) {
        if (w < warp) {
            eb += lsum[0][w];
            ec += lsum[1][w];
        }
        tb += lsum[0][w];
        tc += lsum[1][w];
    }
    for (int rh = p0; rh < p1 && nb > 0 && eb <= kMaxLong; ++rh) {
        const int cnt = count_of(rh);
        if (cnt > kLongPieces) {
            if (eb < kMaxLong) {
                l_rh[eb] = rh;
                l_off[eb] = ec;
            } else {
                hdr[1] = ec;  // where the listed pairs' chunks end
            }
            ++eb;
            ec += cdiv(cnt, kPieceChunk);
        }
    }
    if (tid == 0) {
        hdr[0] = min(tb, kMaxLong);
        if (tb <= kMaxLong) hdr[1] = tc;
    }
}

// One work item as a warp sees it.
struct DecItem {
    int idx;        // queue position; >= count when none
    int t, g, s, pb, np;   // token of the row in the step, KV head, split, first page, pages
    int nkv, ns, r, base;  // keys of the row, splits of the row, request, slot of split 0
};

template <typename T, int D, int G, bool Q8>
__global__ void __launch_bounds__(kDecThreads) decode_kernel(StepArgs a) {
    using S = DecodeSmem<T, D, G, Q8>;
    constexpr int kNst = S::kNst;   // ring stages per warp
    using Cv = F16<T>;
    constexpr int DPL = D / 32;     // dims per lane in the 16-bit p.V (4 or 2)
    constexpr int DP2 = DPL / 2;    // ... as float2 pairs
    // Lane (qg, t4) = (lane / 4, lane % 4) in the MMA fragment layouts.  The score MMA is
    // S^T = K q^T (rows = tokens, k = dims, n = query heads, padded to 8).  A lane's k-slots
    // of step kk are 4 dims: INT8 pages -- t4 * D/4 + 4 kk .. + 3, so its key bytes are D/4
    // contiguous ones per row; 16-bit pages -- chunk kk / 2 of 8 dims at t4 * 8 + 32 (kk / 2),
    // so one 16-byte load per row serves two k-steps and the four lanes of a row group read
    // four different bank groups.
    constexpr int KW = D / 16;      // MMA k-steps over the dims
    constexpr int NQ = D / 32;      // 16-byte q chunks a lane holds

    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* ring = smem + warp * kNst * S::kStageBytes;
    float2* pbuf = reinterpret_cast<float2*>(smem + S::kRing) + warp * kPage * G;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kRing + S::kPbuf) + warp * kNst;

    if (lane == 0) {
        for (int s = 0; s < kNst; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
    }
    __syncwarp();
    const int nwarps = static_cast<int>(gridDim.x) * kDecWarps;  // workers in the grid
    const int gw = static_cast<int>(blockIdx.x) * kDecWarps + warp;
    const int Hkv = a.num_kv_heads, Hq = a.num_q_heads;

    // ---- self-planned steps (every request advances by at most one token, few requests):
    //      the CTA plans the step itself from the lengths, before its dependency wait (they
    //      were final before this step's kv_append started).  The work is the sequence of
    //      (request, KV head) segments of the requests' pages, in request order -- request
    //      r's head g covers pages [seg0[r] + g P_r, seg0[r] + (g + 1) P_r) with P_r its
    //      pages.  A share of the T pages is cut into nw equal static units, one per warp;
    //      the rest into small chunks that warps take from a counter once their own unit is
    //      done, which evens out the warps' different streaming rates (self_plan_units).
    //      A warp's pieces are the segments a unit meets; a piece that is not a whole
    //      segment leaves a partial in slot 2u (the unit's first piece) or 2u + 1 (its
    //      last).  No work records and no separate plan launch.
    __shared__ int s_seg0[kSelfPlanMaxReqs + 1];
    __shared__ int s_tok[kSelfPlanMaxReqs];
    __shared__ int s_keys[kSelfPlanMaxReqs];
    __shared__ int s_wsum[kDecWarps];
    __shared__ int s_bad;
    __shared__ int s_lsum[2][kDecWarps];
    int sp_total = 0, sp_nw = 0, sp_static = 0, sp_chunk = 1, sp_chunks = 0, sp_unit = -1;
    int range_start = 0, range_end = 0;  // the unit this warp works through (T < 2^30)
    if (a.self_plan) {
        const int tid = threadIdx.x;
        if (tid == 0)
            s_bad = (a.q_offsets[0] != 0 || a.q_offsets[a.num_reqs] != a.total_q_tokens) ? 1 : 0;
        __syncthreads();
        // request tid + 128 k of the first / second half: its segments' total pages
        int pages[2] = {0, 0};
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int r = tid + k * kDecThreads;
            if (r < a.num_reqs) {
                const ReqLens L = load_request(a, r);
                if (!L.ok) atomicOr(&s_bad, 1);
                s_tok[r] = L.t0;
                s_keys[r] = L.c + 1;
                pages[k] = (L.ok && L.q == 1) ? cdiv(L.c + 1, kPage) * Hkv : 0;
            }
        }
        // exclusive scan over requests 0..255 in order: the first half, then the second
        int run = 0;
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            int incl = pages[k];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(kFull, incl, o);
                if (lane >= o) incl += y;
            }
            if (lane == 31) s_wsum[warp] = incl;
            __syncthreads();
            int before = run;
            for (int w = 0; w < warp; ++w) before += s_wsum[w];
            int half = 0;
            for (int w = 0; w < kDecWarps; ++w) half += s_wsum[w];
            const int r = tid + k * kDecThreads;
            if (r < a.num_reqs) s_seg0[r] = before + incl - pages[k];
            run += half;
            __syncthreads();
        }
        if (tid == 0) s_seg0[a.num_reqs] = run;
        __syncthreads();
        if (tid == 0)
            install_epoch(reinterpret_cast<unsigned long long*>(
                              ws_at<int32_t>(a, a.lay.ctrl) + 10), a.epoch);
        sp_total = s_bad ? 0 : run;
        // two partial slots per working warp, within the workspace's slots (a third of them
        // at most; the rest serve the chunks)
        sp_nw = min(min(nwarps, sp_total), a.lay.max_items / kSlotsPerWarp);
        if (sp_nw > 0) {
            // small steps (few pages per warp) are all static, as INT8 steps are: there a
            // piece's setup outweighs what the chunks even out
            const bool all_static = Q8 || sp_total < kStaticOnlyPagesPerWarp * sp_nw;
            const SelfPlanUnits u = self_plan_units(sp_total, sp_nw, a.lay.max_items,
                                                    all_static ? 1 : 3, all_static ? 1 : 4);
            sp_static = u.static_pages;
            sp_chunk = u.chunk_pages;
            sp_chunks = u.chunks;
            if (gw < sp_nw) {
                range_start = gw * sp_static;
                range_end = range_start + sp_static;
                sp_unit = gw;
            }
        }
    }
    // The plan must be complete before the work list is read, and this step's kv_append
    // before the pages are.  Behind a prefill grid both completed before any prefill CTA
    // passed its own wait, and this grid launched only after every prefill CTA had started.
    // Over a plan made by an earlier call the plan completed before this step's kv_append
    // started, so only the pages wait (below).  Otherwise the plan is this grid's
    // predecessor and completes after the kv_append.
    if (!a.overlap && !a.plan_ready && !a.self_plan) pdl_wait();

    int32_t* ctrl = ws_at<int32_t>(a, a.lay.ctrl);
    const int num_items = a.self_plan ? 0 : ctrl[1];
    const int4* items = ws_at<const int4>(a, a.lay.items);
    float2* part_ml = ws_at<float2>(a, a.lay.part_ml);
    float* part_o = ws_at<float>(a, a.lay.part_o);
    const uint8_t* kc = static_cast<const uint8_t*>(a.k_cache);
    const uint8_t* vc = static_cast<const uint8_t*>(a.v_cache);
    // K/V pages are read once per step: evict them first so the split partials written
    // meanwhile stay in L2 for the combine
    const uint64_t kv_policy = l2_policy_evict_first();
    const int qg = lane >> 2, t4 = lane & 3;
    // Score rows: MMA row qg is token 4 (qg / 2) + qg % 2 and row qg + 8 the token two after
    // it.  INT8 pages need this order: after the transpose of P a lane's PV k-slots (2 t4,
    // 2 t4 + 1, 2 t4 + 8, 2 t4 + 9) are tokens 4 t4 .. 4 t4 + 3, one 32-bit word of a value
    // row.  16-bit pages share it (any order serves their pbuf hand-off).
    const int kr0 = 4 * (qg >> 1) + (qg & 1), kr1 = kr0 + 2;

    // ---- item metadata moves through a pipeline so no dependent load sits on the critical
    //      path: queue index claimed 3 items ahead, record loaded 2 ahead, page ids and q 1
    //      ahead; each load is consumed one item switch after it was issued.
    auto resolve = [&](int idx, const int4& ra, const int4& rb) {
        DecItem it;
        it.idx = idx;
        it.t = ra.x; it.g = ra.y & 0xffff; it.s = ra.y >> 16; it.pb = ra.z; it.np = ra.w;
        it.nkv = rb.x; it.ns = rb.y; it.r = rb.z; it.base = rb.w;
        if (idx >= num_items) it.np = 0;
        return it;
    };
    auto load_record = [&](int idx, int4& ra, int4& rb) {
        if (idx < num_items) {
            ra = items[2 * idx];
            rb = items[2 * idx + 1];
        } else {
            ra = make_int4(0, 0, 0, 0);
            rb = make_int4(0, 1, 0, 0);
        }
    };
    // lane l: physical id of page pb + w + l (-1 when it is not a valid page: flagged, and
    // page 0 is copied in its place)
    auto load_window = [&](const DecItem& it, int w) {
        int phys = 0;
        const int i = w + lane;
        if (i < it.np) {
            const int lp = it.pb + i;
            if (lp < a.max_pages) {
                phys = __ldg(a.block_table + static_cast<int64_t>(it.r) * a.max_pages + lp);
                if (phys < 0 || phys >= a.num_pages) {
                    set_error(a.err, PKV_DEVERR_PAGE_RANGE);
                    phys = -1;
                }
            } else {
                set_error(a.err, PKV_DEVERR_TABLE_RANGE);
                phys = -1;
            }
        }
        return phys;
    };
    // raw q of an item: query head qg (zero for qg >= G).  INT8 pages: dims t4 * D/4 ..
    // + D/4 - 1; 16-bit pages: chunks of 8 dims t4 * 8 + 32 m (m = 0 .. D/32 - 1)
    auto load_q = [&](const DecItem& it, uint4 (&qr)[NQ]) {
        if (it.np == 0) return;
        if (qg < G) {
            const uint16_t* qh = static_cast<const uint16_t*>(a.q) +
                                 (static_cast<int64_t>(it.t) * Hq + it.g * G + qg) * D;
#pragma unroll
            for (int u = 0; u < NQ; ++u)
                qr[u] = __ldg(reinterpret_cast<const uint4*>(qh + (Q8 ? t4 * (D / 4) + 8 * u
                                                                      : t4 * 8 + 32 * u)));
        } else {
#pragma unroll
            for (int u = 0; u < NQ; ++u) qr[u] = make_uint4(0, 0, 0, 0);
        }
    };
    auto claim = [&]() {  // lane 0 holds the claimed index; read it with __shfl_sync later
        int idx = 0;
        if (lane == 0) idx = atomicAdd(&ctrl[0], 1) + 2 * nwarps;
        return idx;
    };
    // self-planned steps: the piece of this warp's range that starts at flattened page `pos`
    auto make_piece = [&](int pos) {
        DecItem it{};
        it.ns = 1;
        if (pos >= range_end) return it;  // np = 0: none
        const int p = pos;
        int lo = 0, hi = a.num_reqs - 1;  // last request whose segments start at or before p
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_seg0[mid] <= p) lo = mid; else hi = mid - 1;
        }
        const int r = lo, per = cdiv(s_keys[r], kPage);
        const int g = (p - s_seg0[r]) / per;
        const int seg = s_seg0[r] + g * per;
        const int end = min(seg + per, range_end);
        it.t = s_tok[r];
        it.g = g;
        it.pb = p - seg;
        it.np = end - p;
        it.nkv = s_keys[r];
        it.r = r;
        it.ns = (p == seg && end == seg + per) ? 1 : 2;  // a whole segment writes its row
        it.base = 2 * sp_unit + (pos == range_start ? 0 : 1);  // unit's first / last piece
        it.s = 0;
        return it;
    };
    // fused append (self-planned 16-bit steps): the warp whose piece holds a segment's last
    // page loads the request's new K and V rows of that KV head when it makes the piece (16
    // bytes per lane, keys on the low lanes, values above) and, once that page has landed in
    // shared memory, writes the row into the page's slot there and into the pool.  No proxy
    // fence sits before the copies: the copy reads the pool slot before the row is written,
    // and the row reaches the computation through shared memory.
    constexpr int kAppLanes = D * 2 / 16;  // 16-byte chunks of one K (or V) row
    auto load_append = [&](const DecItem& it) {
        uint4 r = make_uint4(0, 0, 0, 0);
        if constexpr (!Q8) {
            if (lane < 2 * kAppLanes) {
                const bool is_v = lane >= kAppLanes;
                const int chunk = is_v ? lane - kAppLanes : lane;
                const uint16_t* sp = static_cast<const uint16_t*>(is_v ? a.v_new : a.k_new) +
                                     (static_cast<int64_t>(it.t) * Hkv + it.g) * D;
                r = __ldg(reinterpret_cast<const uint4*>(sp) + chunk);
            }
        }
        return r;
    };
    uint4 app_cur = make_uint4(0, 0, 0, 0), app_nxt = app_cur;
    // whether a piece holds its segment's last page
    auto holds_last = [&](const DecItem& it) {
        return it.np > 0 && it.pb + it.np == cdiv(it.nkv, kPage);
    };
    bool waited = false;           // the dependency wait has returned
    int sp_pos = range_start;  // self-planned: where the warp's next piece starts
    unsigned long long* chunk_ctr = reinterpret_cast<unsigned long long*>(ctrl + 10);
    // a chunk claim is issued when a unit's last piece is made and read one piece later, so
    // the atomic's round trip overlaps the streaming (lane 0 holds the returned word)
    unsigned long long claim_word = 0;
    bool claim_pending = false;
    auto issue_claim = [&]() {
        if (lane == 0) claim_word = atomicAdd(chunk_ctr, 1ull);
        claim_pending = true;
    };
    auto next_piece = [&]() {
        if (sp_pos >= range_end && sp_unit >= 0) {
            // this unit is done: take the chunk claimed for it (lane 0, the warp follows)
            if (!claim_pending) issue_claim();
            int k = 0;
            if (lane == 0) k = claimed_chunk(chunk_ctr, claim_word, a.epoch, a.err);
            k = __shfl_sync(kFull, k, 0);
            claim_pending = false;
            if (k < sp_chunks) {
                sp_unit = sp_nw + k;
                range_start = sp_nw * sp_static + k * sp_chunk;
                range_end = min(range_start + sp_chunk, sp_total);
                sp_pos = range_start;
            } else {
                sp_unit = -1;
                range_end = range_start = sp_pos;
            }
        }
        const DecItem it = make_piece(sp_pos);
        sp_pos += it.np;
        if (it.np > 0 && sp_pos >= range_end && !claim_pending) issue_claim();
        if (a.fused_append && waited && holds_last(it)) app_nxt = load_append(it);
        return it;
    };

    // prime the pipeline: a warp's first two items are fixed by its index (no queue round
    // trip before the first copy); later ones come from the queue, numbered after them
    const int i0 = gw;
    const int i1 = i0 + nwarps;
    int4 ra, rb;
    DecItem cur, nxt;
    if (a.self_plan) {
        cur = next_piece();
        nxt = next_piece();
    } else {
        load_record(i0, ra, rb);
        cur = resolve(i0, ra, rb);
        load_record(i1, ra, rb);
        nxt = resolve(i1, ra, rb);
    }
    int cur_win = load_window(cur, 0), cur_win_base = 0;
    // the window after cur_win, loaded 32 pages ahead of its use: the block table can be a
    // round trip away (L2, or host memory over the CPU-GPU link)
    int cur_pf = cur.np > 32 ? load_window(cur, 32) : 0;
    int nxt_win = load_window(nxt, 0);
    // Over an earlier plan only the work list (written by a plan that completed before this
    // grid launched) and the block table were read so far.  The preceding kernel may still
    // be writing anything else -- the pages of this step's kv_append, or, when it is the
    // previous layer's combine, the queue counter it rewinds -- so the queue and q wait.
    if (!a.overlap && (a.plan_ready || a.self_plan)) pdl_wait();
    waited = true;
    if (a.fused_append) {  // rows of the two pieces made before the wait
        if (holds_last(cur)) app_cur = load_append(cur);
        if (holds_last(nxt)) app_nxt = load_append(nxt);
    }
    pdl_trigger();  // the combine may be scheduled; it waits for this grid to finish
    if (a.self_plan && blockIdx.x == 0) {
        // what the combine needs: per request {token, first segment page, keys, pages per
        // head}, the totals, zeroed arrival counts (every earlier kernel has completed: the
        // workspace is free)
        int4* rec = ws_at<int4>(a, a.lay.req_info);
        for (int r = threadIdx.x; r < a.num_reqs; r += kDecThreads)
            rec[r] = make_int4(s_tok[r], s_seg0[r], s_keys[r],
                               (s_seg0[r + 1] - s_seg0[r]) / Hkv);
        int32_t* pair_ctr = ws_at<int32_t>(a, a.lay.pair_ctr);  // the combine's arrivals
        for (int i = threadIdx.x; i < a.num_reqs * Hkv; i += kDecThreads) pair_ctr[i] = 0;
        // the long pairs, for the combine
        const UnitMap um{sp_static, sp_chunk, static_cast<int64_t>(sp_nw) * sp_static, sp_nw};
        auto count_of = [&](int rh) {
            const int r = rh / Hkv, g = rh % Hkv;
            const int per = (s_seg0[r + 1] - s_seg0[r]) / Hkv;
            if (per == 0) return 0;
            const int64_t b = static_cast<int64_t>(s_seg0[r]) + static_cast<int64_t>(g) * per;
            return static_cast<int>(um.unit(b + per - 1) - um.unit(b) + 1);
        };
        int32_t* l_rh = pair_ctr + a.num_reqs * Hkv;
        list_long_pairs<kDecThreads>(count_of, (s_bad || sp_nw == 0) ? 0 : a.num_reqs * Hkv,
                                     l_rh, l_rh + kMaxLong, ctrl + 12, s_lsum);
        if (threadIdx.x == 0) {
            if (s_bad) set_error(a.err, PKV_DEVERR_TOKENS);
            ctrl[1] = sp_total;
            ctrl[2] = s_bad ? 0 : a.num_reqs;
            ctrl[4] = sp_nw;
            ctrl[5] = sp_static;
            ctrl[6] = sp_chunk;
        }
    }
    // the next item's q is prefetched when the registers allow (not for 8 x 128-dim heads)
    constexpr bool kPrefetchQ = NQ <= 8;
    uint4 q_cur[NQ], q_nxt[kPrefetchQ ? NQ : 1];
    load_q(cur, q_cur);
    if constexpr (kPrefetchQ) load_q(nxt, q_nxt);
    int p2_idx = 0, p3_lane0 = 0;
    int4 p2a, p2b;
    if (!a.self_plan) {
        p2_idx = __shfl_sync(kFull, claim(), 0);
        load_record(p2_idx, p2a, p2b);
        p3_lane0 = claim();
    }
    uint32_t issued = 0, consumed = 0;  // ring counters
    bool aborted = false;
    int ic = 0;          // pages of `cur` issued so far
    int in_nxt = 0;      // pages of `nxt` issued ahead (at most its first window)
    // issue one page into the ring: `cur` first, then the head of `nxt` (whole warp)
    auto issue_one = [&]() {
        int win, lidx, g;
        if (ic < cur.np) {
            if (ic >= cur_win_base + 32) {
                cur_win_base += 32;
                cur_win = cur_pf;
                cur_pf = cur.np > cur_win_base + 32 ? load_window(cur, cur_win_base + 32) : 0;
            }
            win = cur_win;
            lidx = ic - cur_win_base;
            g = cur.g;
            ++ic;
        } else if (in_nxt < nxt.np && in_nxt < 32) {
            win = nxt_win;
            lidx = in_nxt;
            g = nxt.g;
            ++in_nxt;
        } else {
            return;
        }
        const int phys = max(0, __shfl_sync(kFull, win, lidx));
        if (lane == 0) {
            const int stage = issued % kNst;
            uint8_t* dst = ring + stage * S::kStageBytes;
            const int64_t off = (static_cast<int64_t>(phys) * Hkv + g) * S::kPageBytes;
            mbar_arrive_expect_tx(&bars[stage], 2 * S::kPageBytes);
            bulk_g2s_hint(dst, kc + off, S::kPageBytes, &bars[stage], kv_policy);
            bulk_g2s_hint(dst + S::kPageBytes, vc + off, S::kPageBytes, &bars[stage], kv_policy);
        }
        ++issued;
    };
    for (int k = 0; k < kNst; ++k) issue_one();

    // output row of (token t, KV head g): lanes write DPL dims of each of the G heads
    auto store_row = [&](int t, int g, int j, const float (&res)[DPL]) {
        uint16_t* out_row = static_cast<uint16_t*>(a.out) +
                            (static_cast<int64_t>(t) * Hq + g * G + j) * D + lane * DPL;
        if constexpr (DPL == 4) {
            *reinterpret_cast<uint2*>(out_row) =
                make_uint2(Cv::pack(res[0], res[1]), Cv::pack(res[2], res[3]));
        } else {
            *reinterpret_cast<uint32_t*>(out_row) = Cv::pack(res[0], res[1]);
        }
    };

    // ---- INT8 pages: one item on the tensor cores.  q' = q * k_scale * scale * log2(e) is
    //      scaled by a power of two f so its largest element lies in [2^13, 2^14) (inside fp16
    //      range at full precision); scores come back times f and are scaled by 1/f exactly.
    //      O^T = V^T P^T accumulates in o: m-tile i rows qg, qg + 8 are dims 16 i + qg and
    //      16 i + 8 + qg, columns 2 t4, 2 t4 + 1 query heads.  Returns false on a timeout.
    auto run_item_q8 = [&]() -> bool {
        if constexpr (Q8) {
            float qv[D / 4];
            {
                const float4* ks = reinterpret_cast<const float4*>(a.k_scale + cur.g * D +
                                                                   t4 * (D / 4));
#pragma unroll
                for (int u = 0; u < NQ; ++u) {
                    const uint32_t w4[4] = {q_cur[u].x, q_cur[u].y, q_cur[u].z, q_cur[u].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = Cv::unpack(w4[e]);
                        const int d = u * 8 + 2 * e;
                        const float4 k4 = __ldg(ks + d / 4);
                        const float ka = (d & 2) ? k4.z : k4.x, kb = (d & 2) ? k4.w : k4.y;
                        qv[d] = f.x * ka * a.scale_log2;
                        qv[d + 1] = f.y * kb * a.scale_log2;
                    }
                }
            }
            float amax = 0.f;
#pragma unroll
            for (int d = 0; d < D / 4; ++d) amax = fmaxf(amax, fabsf(qv[d]));
#pragma unroll
            for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
            const int e_amax = static_cast<int>(__float_as_uint(amax) >> 23) - 127;
            const int ex = min(100, max(-100, 13 - e_amax));
            const float fq = __uint_as_float(static_cast<uint32_t>(127 + ex) << 23);
            const float inv_f = __uint_as_float(static_cast<uint32_t>(127 - ex) << 23);
            uint32_t qb[KW][2];
#pragma unroll
            for (int kk = 0; kk < KW; ++kk) {
                qb[kk][0] = pack_h2(qv[4 * kk] * fq, qv[4 * kk + 1] * fq);
                qb[kk][1] = pack_h2(qv[4 * kk + 2] * fq, qv[4 * kk + 3] * fq);
            }
            float o[KW][4];
#pragma unroll
            for (int i = 0; i < KW; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
            float m0 = -1e30f, m1 = -1e30f, l0 = 0.f, l1 = 0.f;  // heads 2 t4, 2 t4 + 1

            for (int i = 0; i < cur.np; ++i) {
                const int stage = consumed % kNst;
                if (!mbar_wait_warp(&bars[stage], (consumed / kNst) & 1)) {
                    if (lane == 0) set_error(a.err, PKV_DEVERR_TIMEOUT);
                    return false;
                }
                ++consumed;
                const uint8_t* sK = ring + stage * S::kStageBytes;   // [16 tokens][D] codes
                const uint8_t* sV = sK + S::kPageBytes;               // [D][16 tokens] codes
                const int nvalid = min(kPage, cur.nkv - (cur.pb + i) * kPage);
                const bool patch = a.fused_append && i == cur.np - 1 && holds_last(cur);
                if (patch) {
                    // this step's row of the segment's last page, quantised as the INT8
                    // append does: lane l's channels l DPL .. into the staged page (K: row
                    // `slot`; V: column `slot` of the [D][16] block) and into the pool
                    constexpr int DPL = D / 32;
                    const int phys = __shfl_sync(kFull, cur_win, i - cur_win_base);
                    const int slot = (cur.nkv - 1) % kPage;
                    if (phys >= 0) {
                        const int64_t src =
                            (static_cast<int64_t>(cur.t) * Hkv + cur.g) * D + lane * DPL;
                        const int chan = cur.g * D + lane * DPL;
                        const uint16_t* ks = static_cast<const uint16_t*>(a.k_new) + src;
                        const uint16_t* vs = static_cast<const uint16_t*>(a.v_new) + src;
                        uint32_t kword = 0, vq[DPL];
#pragma unroll
                        for (int e = 0; e < DPL; e += 2) {
                            const float2 kf =
                                Cv::unpack(__ldg(reinterpret_cast<const uint32_t*>(ks + e)));
                            const float2 vf =
                                Cv::unpack(__ldg(reinterpret_cast<const uint32_t*>(vs + e)));
                            kword |= int8_code(kf.x, __ldg(a.k_scale + chan + e)) << (8 * e);
                            kword |= int8_code(kf.y, __ldg(a.k_scale + chan + e + 1))
                                     << (8 * (e + 1));
                            vq[e] = int8_code(vf.x, __ldg(a.v_scale + chan + e));
                            vq[e + 1] = int8_code(vf.y, __ldg(a.v_scale + chan + e + 1));
                        }
                        const int64_t block =
                            (static_cast<int64_t>(phys) * Hkv + cur.g) * kPage * D;
                        uint8_t* kst = const_cast<uint8_t*>(sK) + slot * D + lane * DPL;
                        uint8_t* kpo = static_cast<uint8_t*>(const_cast<void*>(a.k_cache)) +
                                       block + slot * D + lane * DPL;
                        if constexpr (DPL == 4) {
                            *reinterpret_cast<uint32_t*>(kst) = kword;
                            *reinterpret_cast<uint32_t*>(kpo) = kword;
                        } else {
                            *reinterpret_cast<uint16_t*>(kst) = static_cast<uint16_t>(kword);
                            *reinterpret_cast<uint16_t*>(kpo) = static_cast<uint16_t>(kword);
                        }
                        uint8_t* vst = const_cast<uint8_t*>(sV) + slot;
                        uint8_t* vpo = static_cast<uint8_t*>(const_cast<void*>(a.v_cache)) +
                                       block + slot;
#pragma unroll
                        for (int e = 0; e < DPL; ++e) {
                            vst[(lane * DPL + e) * kPage] = static_cast<uint8_t>(vq[e]);
                            vpo[(lane * DPL + e) * kPage] = static_cast<uint8_t>(vq[e]);
                        }
                    }
                    if (phys >= 0 && lane == 0 && cur.g == 0 && a.slot_mapping)
                        a.slot_mapping[cur.t] = static_cast<int64_t>(phys) * kPage + slot;
                    __syncwarp();
                }
                // key words of rows kr0, kr1 (D/4 bytes each; rows kr0 of lanes qg = 2p and
                // 2p + 1 share banks, a 2-way conflict the shared-memory pipe absorbs)
                uint32_t k0[KW], k1[KW];
#pragma unroll
                for (int h = 0; h < KW / 4; ++h) {
                    const uint4 w0 = *reinterpret_cast<const uint4*>(sK + kr0 * D + t4 * (D / 4) +
                                                                     16 * h);
                    const uint4 w1 = *reinterpret_cast<const uint4*>(sK + kr1 * D + t4 * (D / 4) +
                                                                     16 * h);
                    k0[4 * h] = w0.x; k0[4 * h + 1] = w0.y;
                    k0[4 * h + 2] = w0.z; k0[4 * h + 3] = w0.w;
                    k1[4 * h] = w1.x; k1[4 * h + 1] = w1.y;
                    k1[4 * h + 2] = w1.z; k1[4 * h + 3] = w1.w;
                }
                // two accumulators (even and odd k-steps) halve the dependent MMA chain
                float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int kk = 0; kk < KW; ++kk) {
                    const uint32_t x0 = k0[kk] ^ 0x80808080u, x1 = k1[kk] ^ 0x80808080u;
                    mma_16816((kk & 1) ? sd : sc, codes_lo_h2(x0), codes_lo_h2(x1),
                              codes_hi_h2(x0), codes_hi_h2(x1), qb[kk][0], qb[kk][1]);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[e] += sd[e];
                // sc: (token kr0: heads 2 t4, 2 t4 + 1), (token kr1: same heads)
                const float s0 = kr0 < nvalid ? sc[0] * inv_f : -INFINITY;
                const float s1 = kr0 < nvalid ? sc[1] * inv_f : -INFINITY;
                const float s2 = kr1 < nvalid ? sc[2] * inv_f : -INFINITY;
                const float s3 = kr1 < nvalid ? sc[3] * inv_f : -INFINITY;
                float pm0 = fmaxf(s0, s2), pm1 = fmaxf(s1, s3);
#pragma unroll
                for (int x = 4; x < 32; x <<= 1) {
                    pm0 = fmaxf(pm0, __shfl_xor_sync(kFull, pm0, x));
                    pm1 = fmaxf(pm1, __shfl_xor_sync(kFull, pm1, x));
                }
                const float mn0 = fmaxf(m0, pm0), mn1 = fmaxf(m1, pm1);
                const float al0 = ex2_ftz(m0 - mn0), al1 = ex2_ftz(m1 - mn1);
                const bool rescale = mn0 != m0 || mn1 != m1;
                m0 = mn0;
                m1 = mn1;
                const float p0 = ex2_ftz(s0 - mn0), p1 = ex2_ftz(s1 - mn1);
                const float p2 = ex2_ftz(s2 - mn0), p3 = ex2_ftz(s3 - mn1);
                l0 = fmaf(l0, al0, p0 + p2);
                l1 = fmaf(l1, al1, p1 + p3);
                // P^T fragments: k-slots (2 t4, 2 t4 + 1) and (2 t4 + 8, 2 t4 + 9), query head qg
                const uint32_t pb0 = movmatrix_t(pack_h2(p0, p1));
                const uint32_t pb1 = movmatrix_t(pack_h2(p2, p3));
                if (__any_sync(kFull, rescale)) {  // warp-uniform: no divergent paths
#pragma unroll
                    for (int ii = 0; ii < KW; ++ii) {
                        o[ii][0] *= al0; o[ii][1] *= al1; o[ii][2] *= al0; o[ii][3] *= al1;
                    }
                }
#pragma unroll
                for (int ii = 0; ii < KW; ++ii) {
                    const int d0 = 16 * ii + qg;
                    const uint32_t* vrow = reinterpret_cast<const uint32_t*>(sV + d0 * kPage) + t4;
                    const uint32_t x0 = vrow[0] ^ 0x80808080u;           // dim d0
                    const uint32_t x1 = vrow[2 * kPage] ^ 0x80808080u;   // dim d0 + 8
                    mma_16816(o[ii], minus_1152_h2(codes_lo_h2(x0)),
                              minus_1152_h2(codes_lo_h2(x1)), minus_1152_h2(codes_hi_h2(x0)),
                              minus_1152_h2(codes_hi_h2(x1)), pb0, pb1);
                }
                if (patch) fence_proxy_async_smem();  // the patched stage is refilled by a copy
                __syncwarp();
                issue_one();  // refill the stage just freed
            }
            // row sums over the 16 token rows of every page (lanes with equal t4)
#pragma unroll
            for (int x = 4; x < 32; x <<= 1) {
                l0 += __shfl_xor_sync(kFull, l0, x);
                l1 += __shfl_xor_sync(kFull, l1, x);
            }
            const float* vs = a.v_scale + cur.g * D;
            const int j0 = 2 * t4, j1 = 2 * t4 + 1;
            const bool w0 = j0 < G, w1 = j1 < G;
            if (cur.ns == 1) {
                const float i0 = 1.f / l0, i1 = 1.f / l1;
                uint16_t* out0 = static_cast<uint16_t*>(a.out) +
                                 (static_cast<int64_t>(cur.t) * Hq + cur.g * G + j0) * D;
#pragma unroll
                for (int ii = 0; ii < KW; ++ii) {
#pragma unroll
                    for (int hr = 0; hr < 2; ++hr) {
                        const int d = 16 * ii + 8 * hr + qg;
                        const float sv = __ldg(vs + d);
                        const uint32_t pk = Cv::pack(o[ii][2 * hr] * sv * i0,
                                                     o[ii][2 * hr + 1] * sv * i1);
                        if (w0) out0[d] = static_cast<uint16_t>(pk & 0xffffu);
                        if (w1) out0[D + d] = static_cast<uint16_t>(pk >> 16);
                    }
                }
            } else {
                const int64_t slot = static_cast<int64_t>(cur.base) + cur.s;
                float* po = part_o + (slot * G + j0) * D;
#pragma unroll
                for (int ii = 0; ii < KW; ++ii) {
#pragma unroll
                    for (int hr = 0; hr < 2; ++hr) {
                        const int d = 16 * ii + 8 * hr + qg;
                        const float sv = __ldg(vs + d);
                        if (w0) po[d] = o[ii][2 * hr] * sv;
                        if (w1) po[D + d] = o[ii][2 * hr + 1] * sv;
                    }
                }
                if (qg == 0) {
                    if (w0) part_ml[slot * G + j0] = make_float2(m0, l0);
                    if (w1) part_ml[slot * G + j1] = make_float2(m1, l1);
                }
            }
        }
        return true;
    };

    // ---- 16-bit pages: scores on the tensor cores (S^T = K q^T as in the INT8 path, exact
    //      16-bit products), weighted sums on the FP32 pipes (FFMA2 over V rows, with the
    //      weights shared through pbuf).  Returns false on a timeout.
    auto run_item_16 = [&]() -> bool {
        uint32_t qb[KW][2];
#pragma unroll
        for (int kk = 0; kk < KW; ++kk) {
            const uint4 w = q_cur[kk >> 1];
            qb[kk][0] = (kk & 1) ? w.z : w.x;
            qb[kk][1] = (kk & 1) ? w.w : w.y;
        }
        float m[G];              // running max per query head (same in every lane)
        float ma = -1e30f, mb = -1e30f, la = 0.f, lb = 0.f;  // my heads 2 t4, 2 t4 + 1
        float2 o[G][DP2];  // dims (2e, 2e+1) of my DPL output dims, per head
#pragma unroll
        for (int j = 0; j < G; ++j) {
            m[j] = -1e30f;
#pragma unroll
            for (int e = 0; e < DP2; ++e) o[j][e] = make_float2(0.f, 0.f);
        }
        const int ja = 2 * t4, jb = 2 * t4 + 1;
        for (int i = 0; i < cur.np; ++i) {
            const int stage = consumed % kNst;
            if (!mbar_wait_warp(&bars[stage], (consumed / kNst) & 1)) {
                if (lane == 0) set_error(a.err, PKV_DEVERR_TIMEOUT);
                return false;
            }
            ++consumed;
            const uint8_t* sK = ring + stage * S::kStageBytes;
            const uint8_t* sV = sK + S::kPageBytes;
            const int nvalid = min(kPage, cur.nkv - (cur.pb + i) * kPage);
            const bool patch = a.fused_append && i == cur.np - 1 && holds_last(cur);
            if (patch) {
                // this step's row of the segment's last page: into the staged page (its pool
                // slot was copied before the row was written) and into the pool
                const int phys = __shfl_sync(kFull, cur_win, i - cur_win_base);
                const int slot = (cur.nkv - 1) % kPage;
                if (phys >= 0 && lane < 2 * kAppLanes) {
                    const bool is_v = lane >= kAppLanes;
                    const int chunk = is_v ? lane - kAppLanes : lane;
                    reinterpret_cast<uint4*>(const_cast<uint8_t*>(is_v ? sV : sK) +
                                             slot * D * 2)[chunk] = app_cur;
                    const int64_t dst =
                        ((static_cast<int64_t>(phys) * Hkv + cur.g) * kPage + slot) * D;
                    uint16_t* dp = static_cast<uint16_t*>(const_cast<void*>(
                                       is_v ? a.v_cache : a.k_cache)) + dst;
                    reinterpret_cast<uint4*>(dp)[chunk] = app_cur;
                }
                if (phys >= 0 && lane == 0 && cur.g == 0 && a.slot_mapping)
                    a.slot_mapping[cur.t] = static_cast<int64_t>(phys) * kPage + slot;
                __syncwarp();
            }
            // ---- scores: rows kr0, kr1, chunk m of 8 dims = k-steps 2m, 2m + 1
            float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int mm = 0; mm < NQ; ++mm) {
                const int col = (t4 * 8 + 32 * mm) * 2;   // byte offset of the chunk in a row
                const uint4 w0 = *reinterpret_cast<const uint4*>(sK + kr0 * D * 2 + col);
                const uint4 w1 = *reinterpret_cast<const uint4*>(sK + kr1 * D * 2 + col);
                mma_16816_t<T>(sc, w0.x, w1.x, w0.y, w1.y, qb[2 * mm][0], qb[2 * mm][1]);
                mma_16816_t<T>(sd, w0.z, w1.z, w0.w, w1.w, qb[2 * mm + 1][0], qb[2 * mm + 1][1]);
            }
            const float sl = a.scale_log2;
            const float s0 = kr0 < nvalid ? (sc[0] + sd[0]) * sl : -INFINITY;
            const float s1 = kr0 < nvalid ? (sc[1] + sd[1]) * sl : -INFINITY;
            const float s2 = kr1 < nvalid ? (sc[2] + sd[2]) * sl : -INFINITY;
            const float s3 = kr1 < nvalid ? (sc[3] + sd[3]) * sl : -INFINITY;
            float pa = fmaxf(s0, s2), pb = fmaxf(s1, s3);
#pragma unroll
            for (int x = 4; x < 32; x <<= 1) {
                pa = fmaxf(pa, __shfl_xor_sync(kFull, pa, x));
                pb = fmaxf(pb, __shfl_xor_sync(kFull, pb, x));
            }
            // every head's page max in every lane (heads 2u, 2u + 1 live in lanes t4 = u)
            float alpha[G];
            bool rescale = false;
#pragma unroll
            for (int j = 0; j < G; ++j) {
                const float pj = __shfl_sync(kFull, (j & 1) ? pb : pa, j >> 1);
                const float mn = fmaxf(m[j], pj);
                alpha[j] = fast_exp2(m[j] - mn);
                rescale |= mn != m[j];
                m[j] = mn;
            }
            const float mna = fmaxf(ma, pa), mnb = fmaxf(mb, pb);
            const float ala = fast_exp2(ma - mna), alb = fast_exp2(mb - mnb);
            ma = mna;
            mb = mnb;
            const float p0 = fast_exp2(s0 - mna), p1 = fast_exp2(s1 - mnb);
            const float p2 = fast_exp2(s2 - mna), p3 = fast_exp2(s3 - mnb);
            la = fmaf(la, ala, p0 + p2);
            lb = fmaf(lb, alb, p1 + p3);
            if (ja < G) {
                pbuf[kr0 * G + ja] = make_float2(p0, p0);
                pbuf[kr1 * G + ja] = make_float2(p2, p2);
            }
            if (jb < G) {
                pbuf[kr0 * G + jb] = make_float2(p1, p1);
                pbuf[kr1 * G + jb] = make_float2(p3, p3);
            }
            __syncwarp();

            // ---- o[j][:] = o[j][:] * alpha[j] + sum_tok p[tok][j] * V[tok][:]
            if (rescale) {
#pragma unroll
                for (int j = 0; j < G; ++j) {
                    const float2 a2 = make_float2(alpha[j], alpha[j]);
#pragma unroll
                    for (int e = 0; e < DP2; ++e) o[j][e] = __fmul2_rn(o[j][e], a2);
                }
            }
            auto pv_token = [&](int tok) {
                float2 vf[DP2];
                if constexpr (DPL == 4) {
                    const uint2 w = *reinterpret_cast<const uint2*>(sV + tok * D * 2 + lane * 8);
                    vf[0] = Cv::unpack(w.x);
                    vf[DP2 - 1] = Cv::unpack(w.y);
                } else {
                    vf[0] = Cv::unpack(
                        *reinterpret_cast<const uint32_t*>(sV + tok * D * 2 + lane * 4));
                }
                const float2* pr = pbuf + tok * G;
#pragma unroll
                for (int j = 0; j < G; ++j) {
                    const float2 pj = pr[j];
#pragma unroll
                    for (int e = 0; e < DP2; ++e) o[j][e] = __ffma2_rn(pj, vf[e], o[j][e]);
                }
            };
            if (nvalid == kPage) {
#pragma unroll
                for (int tok = 0; tok < kPage; ++tok) pv_token(tok);
            } else {
                for (int tok = 0; tok < nvalid; ++tok) pv_token(tok);
            }
            if (patch) fence_proxy_async_smem();  // the patched stage is refilled by a copy
            __syncwarp();
            issue_one();  // refill the stage just freed
        }

        // ---- totals of this split: row sums over the 16 token rows, every head's in every lane
#pragma unroll
        for (int x = 4; x < 32; x <<= 1) {
            la += __shfl_xor_sync(kFull, la, x);
            lb += __shfl_xor_sync(kFull, lb, x);
        }
        float lh[G];
#pragma unroll
        for (int j = 0; j < G; ++j) lh[j] = __shfl_sync(kFull, (j & 1) ? lb : la, j >> 1);
        if (cur.ns == 1) {
#pragma unroll
            for (int j = 0; j < G; ++j) {
                float res[DPL];
                const float inv = 1.f / lh[j];
#pragma unroll
                for (int e = 0; e < DP2; ++e) {
                    res[2 * e] = o[j][e].x * inv;
                    res[2 * e + 1] = o[j][e].y * inv;
                }
                store_row(cur.t, cur.g, j, res);
            }
        } else {
            // leave this split's partial for the combine kernel (plain stores: the next
            // launch on the stream sees them)
            const int64_t slot = static_cast<int64_t>(cur.base) + cur.s;
#pragma unroll
            for (int j = 0; j < G; ++j) {
                float2* po = reinterpret_cast<float2*>(part_o + (slot * G + j) * D + lane * DPL);
#pragma unroll
                for (int e = 0; e < DP2; ++e) po[e] = o[j][e];
                if (lane == 0) part_ml[slot * G + j] = make_float2(m[j], lh[j]);
            }
        }
        return true;
    };

    while (cur.np > 0 && !aborted) {
        bool ok;
        if constexpr (Q8) ok = run_item_q8();
        else ok = run_item_16();
        if (!ok) {
            aborted = true;
            break;
        }

        // ---- advance the metadata pipeline; `nxt`'s first pages are already in flight
        cur = nxt;
        app_cur = app_nxt;
        cur_win = nxt_win;
        cur_win_base = 0;
        cur_pf = cur.np > 32 ? load_window(cur, 32) : 0;
        if constexpr (kPrefetchQ) {
#pragma unroll
            for (int u = 0; u < NQ; ++u) q_cur[u] = q_nxt[u];
        } else {
            load_q(cur, q_cur);
        }
        ic = in_nxt;
        in_nxt = 0;
        if (a.self_plan) {
            nxt = next_piece();
        } else {
            nxt = resolve(p2_idx, p2a, p2b);
        }
        nxt_win = load_window(nxt, 0);
        if constexpr (kPrefetchQ) load_q(nxt, q_nxt);
        if (!a.self_plan) {
            p2_idx = __shfl_sync(kFull, p3_lane0, 0);
            load_record(p2_idx, p2a, p2b);
            p3_lane0 = claim();
        }
        while (issued - consumed < static_cast<uint32_t>(kNst)) {
            const uint32_t before = issued;
            issue_one();
            if (issued == before) break;
        }
    }
    // drain copies still in flight (only after an abort), bounded
    while (consumed < issued) {
        mbar_wait_warp(&bars[consumed % kNst], (consumed / kNst) & 1);
        ++consumed;
    }
    // behind a prefill grid: finish only after it, so the combine and the next step still
    // follow the whole step
    if (a.overlap) pdl_wait();
}

// ------------------------------------------------------------------------------------
// combine.  A row's splits are merged by NG groups of one thread per (query head, 4 dims):
// group k folds splits first + (k + NG i) stride into a running (M, L, acc) -- the loads of
// a batch of splits are independent, so they overlap -- and the groups' states are then
// merged through shared memory:
//   m* = max_s m_s,  l* = sum_s l_s 2^(m_s - m*),  acc* = sum_s O_s 2^(m_s - m*)
// (m in log2 units, O unnormalised).  A (row, KV head) pair is one CTA's unit of work; the
// grids are capped near a full wave (the host only knows a bound on the rows) and each CTA
// walks the step's actual pairs with a grid stride.  The launch shapes:
//   kCombineRow     a pair per CTA turn: NG = 1 when no row can have more than
//                   kManySplits splits; NG groups when rows can be long but there are too
//                   many of them for the chunked form.
//   kCombineChunks  turn (pair, c) merges splits [64c, 64c + 64) into the slot of split
//                   64c -- the merged state has the same (m, l, O) form as a split -- or, for
//                   a row with at most 64 splits, writes the row's output.
//   kCombineParts   a pair with more than 64 splits per CTA turn: merges its chunk states
//                   (stride 64) into the output.
// The chunked pair serves a long context on few rows, where one CTA per (row, KV head)
// would read megabytes of partials at a single SM's bandwidth.
// ------------------------------------------------------------------------------------
enum : int { kCombineRow = 0, kCombineChunks = 1, kCombineParts = 2 };
constexpr int kCombineChunk = 64;

// Slots of a (row, KV head)'s splits: base + first + i * stride.
struct SlotRun {
    int64_t base;
    int first, stride;
    __device__ int64_t operator()(int i) const {
        return base + first + static_cast<int64_t>(i) * stride;
    }
};
// Slots of a self-planned segment's pieces (see combine_pieces_kernel): slot0 for the
// first, then consecutive slots from next.
struct SlotPieces {
    int64_t slot0, next, stride;
    __device__ int64_t operator()(int i) const {
        return i == 0 ? slot0 : next + (i - 1) * stride;
    }
};

// kL2: load through L2 only (states other CTAs of the same grid wrote)
template <typename T, int D, int G, int NG, bool kL2 = false, typename SlotFn>
__device__ __forceinline__ void combine_fold(const StepArgs& a, SlotFn slot_of, int count,
                                             bool to_out, int t, int g,
                                             float2 (*s_ml)[G * D / 4],
                                             float4 (*s_acc)[G * D / 4]) {
    using Cv = F16<T>;
    constexpr int TPG = G * D / 4;              // threads per group
    // splits in flight per thread: 4 when a CTA of 1,024 threads leaves 64 registers each
    constexpr int kBatch = (NG > 1 && TPG * NG >= 1024) ? 4 : 8;
    float2* part_ml = ws_at<float2>(a, a.lay.part_ml);
    float* part_o = ws_at<float>(a, a.lay.part_o);
    const int grp = threadIdx.x / TPG, tin = threadIdx.x % TPG;
    const int j = tin / (D / 4), dim = (tin % (D / 4)) * 4;
    // one pass with a running maximum: acc, L rescaled when a split raises it
    float M = -1e30f, L = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int i0 = grp; i0 < count; i0 += NG * kBatch) {
        float2 ml[kBatch];
        float4 o[kBatch];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int i = i0 + u * NG;
            if (i < count) {
                const int64_t slot = slot_of(i);
                const float4* op = reinterpret_cast<const float4*>(part_o + (slot * G + j) * D + dim);
                if constexpr (kL2) {
                    ml[u] = __ldcg(part_ml + slot * G + j);
                    o[u] = __ldcg(op);
                } else {
                    ml[u] = part_ml[slot * G + j];
                    o[u] = *op;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            if (i0 + u * NG < count) {
                const float mn = fmaxf(M, ml[u].x);
                const float c = fast_exp2(M - mn), w = fast_exp2(ml[u].x - mn);
                M = mn;
                L = fmaf(L, c, ml[u].y * w);
                acc.x = fmaf(acc.x, c, o[u].x * w);
                acc.y = fmaf(acc.y, c, o[u].y * w);
                acc.z = fmaf(acc.z, c, o[u].z * w);
                acc.w = fmaf(acc.w, c, o[u].w * w);
            }
        }
    }
    if constexpr (NG > 1) {
        s_ml[grp][tin] = make_float2(M, L);
        s_acc[grp][tin] = acc;
        __syncthreads();
        if (grp == 0) {
            float Ms = M;
#pragma unroll
            for (int k = 1; k < NG; ++k) Ms = fmaxf(Ms, s_ml[k][tin].x);
            L = 0.f;
            acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int k = 0; k < NG; ++k) {
                const float2 mlk = s_ml[k][tin];
                const float4 ak = s_acc[k][tin];
                const float w = fast_exp2(mlk.x - Ms);  // 0 for a group without splits
                L = fmaf(mlk.y, w, L);
                acc.x = fmaf(ak.x, w, acc.x);
                acc.y = fmaf(ak.y, w, acc.y);
                acc.z = fmaf(ak.z, w, acc.z);
                acc.w = fmaf(ak.w, w, acc.w);
            }
            M = Ms;
        }
        __syncthreads();  // shared state read before a next fold overwrites it
        if (grp != 0) return;
    }
    if (to_out) {
        const float inv = 1.f / L;
        uint16_t* out = static_cast<uint16_t*>(a.out) +
                        (static_cast<int64_t>(t) * a.num_q_heads + g * G + j) * D + dim;
        *reinterpret_cast<uint2*>(out) = make_uint2(Cv::pack(acc.x * inv, acc.y * inv),
                                                    Cv::pack(acc.z * inv, acc.w * inv));
    } else {
        // the chunk's state replaces its first split's: every read of that slot happened
        // before the barrier above
        const int64_t slot = slot_of(0);
        part_ml[slot * G + j] = make_float2(M, L);
        *reinterpret_cast<float4*>(part_o + (slot * G + j) * D + dim) = acc;
    }
}

template <typename T, int D, int G, int NG, int Stage>
__global__ void __launch_bounds__(G * D / 4 * NG) combine_kernel(StepArgs a) {
    constexpr int TPG = G * D / 4;
    __shared__ float2 s_ml[NG > 1 ? NG : 1][TPG];
    __shared__ float4 s_acc[NG > 1 ? NG : 1][TPG];
    const int Hkv = a.num_kv_heads;
    int32_t* ctrl = ws_at<int32_t>(a, a.lay.ctrl);
    const int4* rows = ws_at<const int4>(a, a.lay.rows);  // {token, first slot, keys, splits}
    pdl_wait();  // the previous grid (decode kernel or chunk pass) has finished its writes
    // the next kernel on the stream may be scheduled now; it waits for this grid to finish
    // before it touches memory
    pdl_trigger();
    // the decode grid has completed, so nothing claims work items any more: rewind the queue
    // so the next attention call over the same plan (another layer) starts from item 0
    if (Stage != kCombineParts && blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0)
        ctrl[0] = 0;
    // the grid is capped from host bounds; CTAs walk the step's actual (row, KV head) pairs
    const int nrh = ctrl[2] * Hkv;
    for (int rh = blockIdx.x; rh < nrh; rh += gridDim.x) {  // uniform over the CTA
        const int d = rh / Hkv, g = rh % Hkv;
        const int4 row = rows[d];
        const int ns = row.w;
        if (ns <= 1) continue;  // finished in place by the decode kernel
        const int64_t base = row.y + static_cast<int64_t>(g) * ns;
        if constexpr (Stage == kCombineRow) {
            combine_fold<T, D, G, NG>(a, SlotRun{base, 0, 1}, ns, true, row.x, g, s_ml, s_acc);
        } else if constexpr (Stage == kCombineChunks) {
            // the in-place chunk write relies on the barrier between the groups' reads and it
            static_assert(NG > 1, "the chunk pass needs more than one thread group");
            const int nch = cdiv(ns, kCombineChunk);
            for (int c = blockIdx.y; c < nch; c += gridDim.y) {  // uniform over the CTA
                const int first = c * kCombineChunk;
                combine_fold<T, D, G, NG>(a, SlotRun{base, first, 1},
                                          min(kCombineChunk, ns - first), nch == 1, row.x, g,
                                          s_ml, s_acc);
            }
        } else {
            if (ns <= kCombineChunk) continue;  // written by the chunk pass
            combine_fold<T, D, G, NG>(a, SlotRun{base, 0, kCombineChunk},
                                      cdiv(ns, kCombineChunk), true, row.x, g, s_ml, s_acc);
        }
    }
}

// Combine of a self-planned step.  Segment (request r, KV head g) covers flattened pages
// [b, e) with b = seg0[r] + g P_r, e = b + P_r.  Unit u starts at u S (u < nw, S static
// pages per warp) or nw S + (u - nw) C (chunks of C pages), so the segment meets units
// u1 = unit(b) .. u2 = unit(e - 1).  One unit (u1 == u2) wrote the row itself.  Otherwise
// the pieces are u1's first piece (slot 2 u1) when the unit starts exactly at b, else its
// last (slot 2 u1 + 1), then the first piece of each later unit (slot 2 u).
struct PairPieces {
    int count;        // pieces (<= 1: the decode kernel wrote the row)
    int token, g;
    SlotPieces slots;
};
__device__ __forceinline__ PairPieces pair_pieces(const int4* rec, const UnitMap& m, int Hkv,
                                                  int rh) {
    PairPieces pp{0, 0, 0, {0, 0, 0}};
    const int r = rh / Hkv, g = rh % Hkv;
    const int4 rr = rec[r];
    const int per = rr.w;
    if (per == 0) return pp;
    const int64_t b = static_cast<int64_t>(rr.y) + static_cast<int64_t>(g) * per;
    const int64_t u1 = m.unit(b), u2 = m.unit(b + per - 1);
    pp.count = static_cast<int>(u2 - u1 + 1);
    pp.token = rr.x;
    pp.g = g;
    pp.slots = SlotPieces{2 * u1 + (m.start(u1) == b ? 0 : 1), 2 * (u1 + 1), 2};
    return pp;
}

struct SlotShift {   // pieces first, first + 1, ...
    SlotPieces p;
    int first;
    __device__ int64_t operator()(int i) const { return p(first + i); }
};
struct SlotChunks {  // the first piece of every chunk
    SlotPieces p;
    __device__ int64_t operator()(int i) const { return p(i * kPieceChunk); }
};
struct LongPairs {          // the decode kernel's list, in shared memory
    int rh[kMaxLong];       // listed long pairs, ascending
    int off[kMaxLong];      // their first chunk in the grid's chunk sequence
    int n, chunks, last;
};
// Copies the list (n > 0 entries) to shared memory; the whole CTA calls it.
__device__ __forceinline__ void load_long_pairs(const StepArgs& a, const int32_t* ctrl,
                                                LongPairs& L) {
    const int32_t* l_rh = ws_at<const int32_t>(a, a.lay.pair_ctr) + a.num_reqs * a.num_kv_heads;
    const int n = ctrl[12];
    for (int k = threadIdx.x; k < n; k += blockDim.x) {
        L.rh[k] = l_rh[k];
        L.off[k] = l_rh[kMaxLong + k];
    }
    if (threadIdx.x == 0) {
        L.n = n;
        L.chunks = ctrl[13];
    }
    __syncthreads();
}
// whether pair rh is a listed long pair (folded by fold_long_pairs)
__device__ __forceinline__ bool is_listed(const LongPairs& L, int rh) {
    int lo = 0, hi = L.n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (L.rh[mid] < rh) lo = mid + 1;
        else hi = mid;
    }
    return lo < L.n && L.rh[lo] == rh;
}
// The CTA's first pair: chunk task k of the long pairs runs on CTA k mod grid, and the pairs
// continue the sequence, so that they land on other CTAs while there are enough.
__device__ __forceinline__ int first_after_chunks(bool any_long, const LongPairs& L) {
    if (!any_long) return blockIdx.x;
    const int b = static_cast<int>(blockIdx.x) - L.chunks % static_cast<int>(gridDim.x);
    return b < 0 ? b + static_cast<int>(gridDim.x) : b;
}
template <typename T, int D, int G, int NG>
__device__ __forceinline__ void fold_long_pairs(const StepArgs& a, const int4* rec,
                                                const UnitMap& m, LongPairs& L,
                                                float2 (*s_ml)[G * D / 4],
                                                float4 (*s_acc)[G * D / 4]) {
    const int Hkv = a.num_kv_heads;
    int32_t* ctr = ws_at<int32_t>(a, a.lay.pair_ctr);
    for (int v = blockIdx.x; v < L.chunks; v += gridDim.x) {  // uniform over the CTA
        int lo = 0, hi = L.n - 1;  // the entry k with off[k] <= v < off[k + 1]
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (L.off[mid] <= v) lo = mid;
            else hi = mid - 1;
        }
        const int rh = L.rh[lo], c = v - L.off[lo];
        const PairPieces pp = pair_pieces(rec, m, Hkv, rh);
        const int nch = cdiv(pp.count, kPieceChunk), first = c * kPieceChunk;
        combine_fold<T, D, G, NG>(a, SlotShift{pp.slots, first},
                                  min(kPieceChunk, pp.count - first), false, pp.token, pp.g,
                                  s_ml, s_acc);
        __threadfence();  // the chunk state, before the arrival that publishes it
        __syncthreads();
        if (threadIdx.x == 0) L.last = atomicAdd(ctr + rh, 1) == nch - 1 ? 1 : 0;
        __syncthreads();
        if (L.last) {
            __threadfence();
            combine_fold<T, D, G, NG, true>(a, SlotChunks{pp.slots}, nch, true, pp.token, pp.g,
                                            s_ml, s_acc);
        }
        __syncthreads();  // L.last and the shared fold state, before the next chunk
    }
}

// The combine of a self-planned step with 16-bit pages, whose chunked tail gives many pairs
// dozens of pieces: NG thread groups of a CTA share a pair's pieces (measured faster than
// the per-group form below for them), long pairs are spread over the grid.
template <typename T, int D, int G, int NG>
__global__ void __launch_bounds__(G * D / 4 * NG) combine_pieces_kernel(StepArgs a) {
    constexpr int TPG = G * D / 4;
    __shared__ float2 s_ml[NG > 1 ? NG : 1][TPG];
    __shared__ float4 s_acc[NG > 1 ? NG : 1][TPG];
    __shared__ LongPairs s_long;
    const int Hkv = a.num_kv_heads;
    int32_t* ctrl = ws_at<int32_t>(a, a.lay.ctrl);
    const int4* rec = ws_at<const int4>(a, a.lay.req_info);  // {token, seg0, keys, pages}
    pdl_wait();  // the decode grid has completed
    // park the chunk counter at epoch 0, which no call uses, so the next call starts afresh;
    // before the next kernel may launch, since a decode kernel can claim before its wait
    if (blockIdx.x == 0 && threadIdx.x == 0)
        atomicExch(reinterpret_cast<unsigned long long*>(ctrl + 10), 0ull);
    __syncthreads();
    pdl_trigger();
    const int npairs = ctrl[2] * Hkv;
    const UnitMap m = unit_map(ctrl);
    const bool any_long = ctrl[12] > 0;
    if (any_long) {
        load_long_pairs(a, ctrl, s_long);
        fold_long_pairs<T, D, G, NG>(a, rec, m, s_long, s_ml, s_acc);
    }
    // the pairs, on the CTAs after those that took the long pairs' chunks
    for (int rh = first_after_chunks(any_long, s_long); rh < npairs; rh += gridDim.x) {
        const PairPieces pp = pair_pieces(rec, m, Hkv, rh);  // uniform over the CTA
        if (pp.count <= 1 || (any_long && pp.count > kLongPieces && is_listed(s_long, rh)))
            continue;
        combine_fold<T, D, G, NG>(a, pp.slots, pp.count, true, pp.token, pp.g, s_ml, s_acc);
    }
}

// The same combine for steps whose pairs mostly have few pieces (INT8 pages, whose units are
// static but for a remainder): the CTA's NG thread groups take NG pairs at a time (pairs
// blockIdx.x + k gridDim.x, so pairs of neighbouring requests land in different CTAs); a
// group folds a pair of at most kSmallPieces pieces on its own, in one round of loads; the
// pairs with more are then folded by all groups together, and the long ones are spread over
// the grid.
constexpr int kSmallPieces = 8;
template <typename T, int D, int G, int NG>
__global__ void __launch_bounds__(G * D / 4 * NG) combine_pieces_solo_kernel(StepArgs a) {
    using Cv = F16<T>;
    constexpr int TPG = G * D / 4;
    __shared__ float2 s_ml[NG > 1 ? NG : 1][TPG];
    __shared__ float4 s_acc[NG > 1 ? NG : 1][TPG];
    __shared__ int s_big[NG], s_nbig;
    __shared__ LongPairs s_long;
    const int Hkv = a.num_kv_heads;
    int32_t* ctrl = ws_at<int32_t>(a, a.lay.ctrl);
    const int4* rec = ws_at<const int4>(a, a.lay.req_info);  // {token, seg0, keys, pages}
    const float2* part_ml = ws_at<const float2>(a, a.lay.part_ml);
    const float* part_o = ws_at<const float>(a, a.lay.part_o);
    pdl_wait();  // the decode grid has completed
    // park the chunk counter at epoch 0, which no call uses, so the next call starts afresh;
    // before the next kernel may launch, since a decode kernel can claim before its wait
    if (blockIdx.x == 0 && threadIdx.x == 0)
        atomicExch(reinterpret_cast<unsigned long long*>(ctrl + 10), 0ull);
    __syncthreads();
    pdl_trigger();
    const int npairs = ctrl[2] * Hkv;
    const UnitMap m = unit_map(ctrl);
    const bool any_long = ctrl[12] > 0;
    if (any_long) {
        load_long_pairs(a, ctrl, s_long);
        fold_long_pairs<T, D, G, NG>(a, rec, m, s_long, s_ml, s_acc);
    }
    const int grp = threadIdx.x / TPG, tin = threadIdx.x % TPG;
    const int j = tin / (D / 4), dim = (tin % (D / 4)) * 4;
    const int first = first_after_chunks(any_long, s_long);
    for (int round = 0; static_cast<int64_t>(round) * gridDim.x * NG < npairs; ++round) {
        if (threadIdx.x == 0) s_nbig = 0;
        __syncthreads();
        const int rh = first + (round * NG + grp) * gridDim.x;
        if (rh < npairs) {
            const PairPieces pp = pair_pieces(rec, m, Hkv, rh);
            if (pp.count > kSmallPieces) {
                if (tin == 0 && !(any_long && pp.count > kLongPieces && is_listed(s_long, rh)))
                    s_big[atomicAdd(&s_nbig, 1)] = rh;
            } else if (pp.count > 1) {
                // this group alone: every piece's loads in flight together
                float2 ml[kSmallPieces];
                float4 o[kSmallPieces];
#pragma unroll
                for (int u = 0; u < kSmallPieces; ++u) {
                    if (u < pp.count) {
                        const int64_t slot = pp.slots(u);
                        ml[u] = part_ml[slot * G + j];
                        o[u] = *reinterpret_cast<const float4*>(part_o + (slot * G + j) * D + dim);
                    }
                }
                float M = -1e30f, L = 0.f;
                float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int u = 0; u < kSmallPieces; ++u) {
                    if (u < pp.count) {
                        const float mn = fmaxf(M, ml[u].x);
                        const float c = fast_exp2(M - mn), w = fast_exp2(ml[u].x - mn);
                        M = mn;
                        L = fmaf(L, c, ml[u].y * w);
                        acc.x = fmaf(acc.x, c, o[u].x * w);
                        acc.y = fmaf(acc.y, c, o[u].y * w);
                        acc.z = fmaf(acc.z, c, o[u].z * w);
                        acc.w = fmaf(acc.w, c, o[u].w * w);
                    }
                }
                const float inv = 1.f / L;
                uint16_t* out = static_cast<uint16_t*>(a.out) +
                                (static_cast<int64_t>(pp.token) * a.num_q_heads + pp.g * G + j) *
                                    D + dim;
                *reinterpret_cast<uint2*>(out) = make_uint2(Cv::pack(acc.x * inv, acc.y * inv),
                                                            Cv::pack(acc.z * inv, acc.w * inv));
            }
        }
        __syncthreads();
        for (int k = 0; k < s_nbig; ++k) {  // uniform over the CTA
            const PairPieces pp = pair_pieces(rec, m, Hkv, s_big[k]);
            combine_fold<T, D, G, NG>(a, pp.slots, pp.count, true, pp.token, pp.g, s_ml, s_acc);
        }
    }
}

// ------------------------------------------------------------------------------------
// host launchers
// ------------------------------------------------------------------------------------
WorkspaceLayout workspace_layout(int num_reqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int total_q_tokens, int max_q_len, int max_context_len,
                                 int num_sms, int prefill_min_q) {
    WorkspaceLayout L{};
    const int G = num_q_heads / num_kv_heads;
    // decode rows: every row of a request below the prefill threshold.  No request can have
    // fewer than T - (B - 1) * max_q_len new tokens; when even that reaches the threshold
    // (one request, say) there are no decode rows and the decode kernels are not launched
    L.max_rows = static_cast<int>(std::min<long long>(
        total_q_tokens,
        static_cast<long long>(num_reqs) * std::max(0, std::min(max_q_len, prefill_min_q - 1))));
    const long long min_q = static_cast<long long>(total_q_tokens) -
                            static_cast<long long>(std::max(0, num_reqs - 1)) * max_q_len;
    if (min_q >= prefill_min_q) L.max_rows = 0;
    L.target_items = 2 * kDecWarps * kItemsPerWarp * num_sms;  // 2 CTAs per SM
    // pages per split >= total / target, so items <= target + one per (row, KV head);
    // pages per split >= kMinSplitPages bounds them by the longest row as well
    const long long row_pages = cdiv(max_context_len + max_q_len, kPage);
    const long long by_len = static_cast<long long>(L.max_rows) * num_kv_heads *
                             ((row_pages + kMinSplitPages - 1) / kMinSplitPages);
    const long long by_target = L.target_items + static_cast<long long>(L.max_rows) * num_kv_heads;
    L.max_items = L.max_rows ? static_cast<int>(std::min(by_len, by_target)) : 0;
    // every request advances by at most one token and there are few requests: the decode
    // kernel plans the step itself, with two partial slots per warp
    const long long seg_pages = static_cast<long long>(num_reqs) * num_kv_heads *
                                ((static_cast<long long>(max_context_len) + kPage) / kPage);
    L.self_plan = L.max_rows > 0 && max_q_len <= 1 && num_reqs <= kSelfPlanMaxReqs &&
                  seg_pages < INT_MAX / 2;
    if (L.self_plan)
        L.max_items = std::max(L.max_items, kSlotsPerWarp * kDecWarps * kDecMaxCtasPerSm * num_sms);
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
    L.rows = off; off = up(off + static_cast<size_t>(L.max_rows) * 16);
    L.items = off; off = up(off + static_cast<size_t>(L.max_items) * 32);
    L.tiles = off; off = up(off + static_cast<size_t>(L.max_tiles) * 16);
    L.part_ml = off; off = up(off + static_cast<size_t>(L.max_items) * G * 8);
    L.part_o = off; off = up(off + static_cast<size_t>(L.max_items) * G * head_dim * 4);
    L.pair_ctr = off;  // then the long-pair list: kMaxLong pairs, kMaxLong chunk offsets
    off = up(off + (L.self_plan ? (static_cast<size_t>(num_reqs) * num_kv_heads + 2 * kMaxLong) * 4
                                : 0));
    L.total = off;
    return L;
}

int launch_plan(const StepArgs& a, cudaStream_t stream) {
    return launch_pdl(plan_kernel, dim3(kPlanBlocks), dim3(kPlanThreads), 0, stream, a) ==
                   cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

template <typename T, int D, int G, bool Q8>
static int launch_decode_t(const StepArgs& a, cudaStream_t stream, cudaEvent_t ev0,
                           cudaEvent_t ev1) {
    using S = DecodeSmem<T, D, G, Q8>;
    static int blocks_per_sm = 0;  // benign race: every thread computes the same value
    if (blocks_per_sm == 0) {
        if (cudaFuncSetAttribute(decode_kernel<T, D, G, Q8>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 S::kBytes) != cudaSuccess)
            return PKV_ERR_CUDA;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_kernel<T, D, G, Q8>,
                                                          kDecThreads, S::kBytes) != cudaSuccess)
            return PKV_ERR_CUDA;
        blocks_per_sm = std::max(1, n);
    }
    const int grid = blocks_per_sm * a.num_sms;
    if (ev0 && cudaEventRecord(ev0, stream) != cudaSuccess) return PKV_ERR_CUDA;
    if (launch_pdl(decode_kernel<T, D, G, Q8>, dim3(grid), dim3(kDecThreads), S::kBytes, stream,
                   a) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (ev1 && cudaEventRecord(ev1, stream) != cudaSuccess) return PKV_ERR_CUDA;
    // rows can have at most ceil(pages / kMinSplitPages) splits.  Past kManySplits the
    // combine runs in two passes over chunks of splits with NG thread groups per CTA, or --
    // when rows x heads x chunks would launch mostly idle CTAs -- in one pass per (row, KV
    // head) with NG groups
    constexpr int kTpg = G * D / 4, kNg = std::min(8, 1024 / kTpg);
    const int max_splits = cdiv(cdiv(a.max_context_len + a.max_q_len, kPage), kMinSplitPages);
    const int rows_heads = std::max(1, a.lay.max_rows * a.num_kv_heads);
    // grids capped near a full wave: a host bound on rows can be far above the step's rows
    const int cap_small = std::min(rows_heads, 16 * a.num_sms);  // 128-thread CTAs
    const int cap_big = std::min(rows_heads, 2 * a.num_sms);     // up to 1,024 threads
    const int chunks = cdiv(max_splits, kCombineChunk);
    cudaError_t e;
    // self-planned steps: at most four thread groups and 512 threads per CTA, so two CTAs
    // fit an SM
    constexpr int kNg4 = std::max(1, std::min(4, 512 / kTpg));
    // A step with few (request, KV head) pairs spreads every pair over many units, so the
    // grids do not shrink with the pairs: the long pairs' chunks need many CTAs.  (A wider
    // grid than the work needs costs time: a combine CTA fills an SM's registers, so the next
    // step's kernels wait for it to exit.)
    if (a.self_plan && Q8) {
        // CTAs of kNg4 pairs at a time, at most one per SM; at least 64 for the chunks of
        // long pairs (INT8 units are static: few pairs share ~2,000 of them)
        const int pairs = std::max(1, a.num_reqs * a.num_kv_heads);
        e = launch_pdl(combine_pieces_solo_kernel<T, D, G, kNg4>,
                       dim3(std::min(a.num_sms, std::max(cdiv(pairs, kNg4), 64))),
                       dim3(kTpg * kNg4), 0, stream, a);
    } else if (a.self_plan) {
        // one wave: as many CTAs per SM as fit, at most two (a CTA of 512 threads fills an
        // SM's registers, one of 128 threads -- G = 1 -- leaves room for more; measured: a
        // second wave of the big CTAs cost the 64-request step 1.2 us, halving the small
        // ones cost the MHA-skew steps 8-10%)
        static int per_sm = 0;  // benign race: every thread computes the same value
        if (per_sm == 0) {
            int n = 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(
                    &n, combine_pieces_kernel<T, D, G, kNg4>, kTpg * kNg4, 0) != cudaSuccess)
                return PKV_ERR_CUDA;
            per_sm = std::max(1, std::min(2, n));
        }
        e = launch_pdl(combine_pieces_kernel<T, D, G, kNg4>, dim3(per_sm * a.num_sms),
                       dim3(kTpg * kNg4), 0, stream, a);
    } else if (max_splits <= kManySplits) {
        e = launch_pdl(combine_kernel<T, D, G, 1, kCombineRow>, dim3(cap_small), dim3(kTpg), 0,
                       stream, a);
    } else if (static_cast<long long>(rows_heads) * chunks <= kChunkedCtas) {
        e = launch_pdl(combine_kernel<T, D, G, kNg, kCombineChunks>, dim3(cap_big, chunks),
                       dim3(kTpg * kNg), 0, stream, a);
        if (e == cudaSuccess)
            e = launch_pdl(combine_kernel<T, D, G, kNg, kCombineParts>, dim3(cap_big),
                           dim3(kTpg * kNg), 0, stream, a);
    } else {
        e = launch_pdl(combine_kernel<T, D, G, kNg, kCombineRow>, dim3(cap_big),
                       dim3(kTpg * kNg), 0, stream, a);
    }
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

template <typename T, int D>
static int dispatch_group(const StepArgs& a, cudaStream_t s, cudaEvent_t e0, cudaEvent_t e1) {
    const bool q8 = a.kv_int8 != 0;
    switch (a.num_q_heads / a.num_kv_heads) {
        case 1: return q8 ? launch_decode_t<T, D, 1, true>(a, s, e0, e1)
                          : launch_decode_t<T, D, 1, false>(a, s, e0, e1);
        case 2: return q8 ? launch_decode_t<T, D, 2, true>(a, s, e0, e1)
                          : launch_decode_t<T, D, 2, false>(a, s, e0, e1);
        case 4: return q8 ? launch_decode_t<T, D, 4, true>(a, s, e0, e1)
                          : launch_decode_t<T, D, 4, false>(a, s, e0, e1);
        case 8: return q8 ? launch_decode_t<T, D, 8, true>(a, s, e0, e1)
                          : launch_decode_t<T, D, 8, false>(a, s, e0, e1);
        default: return PKV_ERR_UNSUPPORTED;
    }
}

int launch_decode(const StepArgs& a, cudaStream_t stream, cudaEvent_t e0, cudaEvent_t e1) {
    if (a.lay.max_items <= 0) return PKV_OK;  // no request can have decode rows
    if (a.dtype == PKV_BF16)
        return a.head_dim == 128 ? dispatch_group<__nv_bfloat16, 128>(a, stream, e0, e1)
                                 : dispatch_group<__nv_bfloat16, 64>(a, stream, e0, e1);
    return a.head_dim == 128 ? dispatch_group<__half, 128>(a, stream, e0, e1)
                             : dispatch_group<__half, 64>(a, stream, e0, e1);
}

}  // namespace pkv
