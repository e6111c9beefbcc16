// Prefill-chunk attention over INT8 pages on the tensor cores, the cache in INT8 with fixed
// per-channel scales (wmrh.cn/news/64708 §4.3, §5.4).  Each CTA works on two chains of 128
// query rows sharing one KV head's stream (prefill_tile.cuh): two query heads of one KV
// group (hotelren.com/news/6181127 §6.3), or two consecutive query tiles of one head.
//
// Same mathematics and the same pipeline as prefill_pair.cu: causal softmax attention of a
// 128-row query tile against every key of its request, read from the pages; one MMA warp
// alternates the two heads' S = Q K^T and O += P V while two softmax warpgroups work on the
// other head's scores; P goes into tensor memory over its scores.  What differs:
//   * the MMAs take fp16 operands.  An INT8 code is exact in fp16, so K and V enter as
//     their codes, and the scales move out of the contraction: Q' = Q * k_scale (per dim)
//     replaces Q, and the epilogue multiplies O by v_scale (per dim);
//   * Q' is scaled by a power of two f per head so its largest element lies in
//     [2^13, 2^14): full fp16 precision, no overflow for any bf16 input; the softmax
//     divides the scores by f exactly (a power of two folded into the base-2 scale);
//   * the six producer warps read page blocks of codes straight from the pools (2 KiB of
//     K, 2 KiB of V per page and head) and write them as fp16 into the stage buffers in the
//     128-byte-swizzled layout the MMA descriptors describe.  Keys land as rows of K
//     (K-major, like a TMA box would place them); values arrive dim-major from the pool
//     and land as V^T (each dim a row of keys), the K-major B operand of P V;
//   * pages past the end of a request are written as zeros, so every stage slot the MMA
//     reads holds finite numbers.
// Softmax makes two passes over the score row in tensor memory (max, then exponentials).
#include <cuda.h>

#include <climits>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "prefill_tile.cuh"
#include "tc.cuh"

namespace pkv {

namespace {

constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kStagesK = 3;
constexpr int kStagesV = 2;
constexpr int kProducers = 3;      // warps converting K pages; as many again convert V pages
constexpr int kWarpMma = 8;
constexpr int kWarpProd0 = 9;      // warps 9..11 write K (and load Q), 12..14 write V
constexpr int kThreads = 32 * (kWarpProd0 + 2 * kProducers);  // 480
constexpr int kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;
constexpr float kQTop = 13.f;      // largest |Q'| element scaled into [2^13, 2^14)

template <int D>
struct Q8Smem {
    static constexpr int kHalves = D / 64;
    static constexpr int kHalfBytes = kBM * 128;           // Q, K: 128 rows x 64 dims
    static constexpr int kVHalf = D * 128;                 // V^T: D rows x 64 keys
    static constexpr int kQ = kBM * D * 2;                 // one head's Q' tile
    static constexpr int kKV = kBN * D * 2;
    static constexpr int kQOff = 0;                        // head h at kQOff + h * kQ
    static constexpr int kKOff = 2 * kQ;
    static constexpr int kVOff = kKOff + kStagesK * kKV;
    static constexpr int kBarOff = kVOff + kStagesV * kKV;
    static constexpr int kBars = 24;
    static constexpr int kMiscOff = kBarOff + kBars * 8;   // tmem slot, then 8 floats
    static constexpr int kBytes = kMiscOff + 64 + 1024;
    static constexpr int kLaunchBytes = kBytes > 120 * 1024 ? kBytes : 120 * 1024;
    static_assert(kLaunchBytes <= 227 * 1024, "shared memory budget");
};

// 16 INT8 codes (one 16-byte word) -> 16 fp16 values in two 16-byte words.  With the sign
// bit flipped, code c = u - 128 for the byte u, and 0x64 over u is the fp16 1024 + u, i.e.
// c + 1152; Exact subtracts the 1152 (exactly).  Without it every score of a query row
// would carry the same 1152 * sum_d Q'_d, which the softmax cancels, but the kernel with
// exact keys measured faster (its producer loop compiles to less code), so both K and V
// use exact codes.
template <bool Exact>
__device__ __forceinline__ uint32_t q8_pair(uint32_t x, uint32_t sel) {
    const uint32_t h = __byte_perm(x, 0x6464u, sel);
    if constexpr (!Exact) return h;
    const uint32_t c = 0x64806480u;   // fp16 1152 in both halves
    const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&h),
                              *reinterpret_cast<const __half2*>(&c));
    return *reinterpret_cast<const uint32_t*>(&r);
}
template <bool Exact>
__device__ __forceinline__ void q8_codes16(const uint4 w, uint4& lo, uint4& hi) {
    const uint32_t x0 = w.x ^ 0x80808080u, x1 = w.y ^ 0x80808080u;
    const uint32_t x2 = w.z ^ 0x80808080u, x3 = w.w ^ 0x80808080u;
    lo = make_uint4(q8_pair<Exact>(x0, 0x4140), q8_pair<Exact>(x0, 0x4342),
                    q8_pair<Exact>(x1, 0x4140), q8_pair<Exact>(x1, 0x4342));
    hi = make_uint4(q8_pair<Exact>(x2, 0x4140), q8_pair<Exact>(x2, 0x4342),
                    q8_pair<Exact>(x3, 0x4140), q8_pair<Exact>(x3, 0x4342));
}

// byte offset of the 16-byte chunk `chunk` of row `row` in a 128-byte-swizzled region
__device__ __forceinline__ int sw128(int row, int chunk) {
    return row * 128 + ((chunk ^ (row & 7)) << 4);
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_q8_kernel(const StepArgs a, const __grid_constant__ CUtensorMap tm_q) {
    using S = Q8Smem<D>;
    using Cv = F16<T>;          // the step's dtype: Q in, output out
    using Ch = F16<__half>;     // the MMA operands: Q', codes, P
    constexpr uint32_t kIdescS = tc::idesc_f16(0, 0, kBM, kBN);
    constexpr uint32_t kIdescO = tc::idesc_f16(0, 0, kBM, D);   // B = V^T, K-major

    pdl_wait();  // the plan and kv_append (and the decode kernel, if it ran first) completed
    // the next grid (the decode stream of a mixed step, or the next step's first kernel)
    // may launch once every CTA has started; the decode kernel only waits for this grid at
    // its end, any other kernel before it touches memory
    pdl_trigger();
    const int32_t* ctrl = reinterpret_cast<const int32_t*>(a.ws + a.lay.ctrl);
    if (static_cast<int>(blockIdx.x) >= ctrl[9]) return;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
    uint64_t* q_full = bars + 0;    // Q tile landed (TMA)
    uint64_t* k_full = bars + 1;    // [3]
    uint64_t* k_empty = bars + 4;   // [3]
    uint64_t* v_full = bars + 7;    // [2]
    uint64_t* v_empty = bars + 9;   // [2]
    uint64_t* s_full = bars + 11;   // [2] per head
    uint64_t* p_full = bars + 13;   // [2] per head
    uint64_t* o_final = bars + 15;
    uint64_t* drain = bars + 16;
    uint64_t* p_half = bars + 17;   // [2] per head: P of keys 0..63 written
    uint64_t* q_ready = bars + 19;  // Q' of both heads written
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kMiscOff);
    float* red = reinterpret_cast<float*>(smem + S::kMiscOff + 16);  // [2 heads][4 warps]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- two chains of 128 query rows sharing one KV head's key/value stream
    const int4 tile_rec = reinterpret_cast<const int4*>(a.ws + a.lay.tiles)[blockIdx.x];
    const PairTile tile = pair_tile(a, tile_rec, kBM, kBN);
    const int g = tile.g;
    const int kv_len = tile.kv_len, n_kv = tile.n_kv, npages_seq = tile.npages_seq;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_ready, 256);
        for (int s = 0; s < kStagesK; ++s) {
            mbar_init(&k_full[s], kProducers);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < kStagesV; ++s) {
            mbar_init(&v_full[s], kProducers);
            mbar_init(&v_empty[s], 1);
        }
        for (int h = 0; h < 2; ++h) {
            mbar_init(&s_full[h], 1);
            mbar_init(&p_full[h], 128);
            mbar_init(&p_half[h], 128);
        }
        mbar_init(o_final, 1);
        mbar_init(drain, 1);
        fence_barrier_init();
    }
    if (warp == kWarpMma) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    auto tm_s = [&](int h) { return tmem + static_cast<uint32_t>(h * kBN); };     // S_h / P_h
    auto tm_o = [&](int h) { return tmem + static_cast<uint32_t>(2 * kBN + h * 128); };
    auto sQ = [&](int h) { return smem + S::kQOff + h * S::kQ; };
    auto sK = [&](int j) { return smem + S::kKOff + (j % kStagesK) * S::kKV; };
    auto sV = [&](int j) { return smem + S::kVOff + (j % kStagesV) * S::kKV; };

    if (warp >= kWarpProd0) {
        // ================================================================ producers
        const bool is_v = warp >= kWarpProd0 + kProducers;
        const int pi = (warp - kWarpProd0) % kProducers;
        if (!is_v && pi == 0 && lane == 0) {
            tc::prefetch_tmap(&tm_q);
            mbar_arrive_expect_tx(q_full, 2 * S::kQ);
            for (int h = 0; h < 2; ++h)
                for (int c = 0; c < S::kHalves; ++c)
                    tc::tma_load_3d(sQ(h) + c * S::kHalfBytes, &tm_q, c * 64, tile.head[h],
                                    tile.q_row[h], q_full);
        }
        const int32_t* bt = a.block_table + static_cast<int64_t>(tile.r) * a.max_pages;
        const uint8_t* pool = static_cast<const uint8_t*>(is_v ? a.v_cache : a.k_cache);
        int win_base = -1, win = 0;
        auto page_of = [&](int lp) -> int {  // warp-wide
            const int base = lp & ~31;
            if (base != win_base) {
                win_base = base;
                const int l = base + lane;
                win = 0;
                if (l < npages_seq) {
                    if (l < a.max_pages) {
                        win = __ldg(bt + l);
                        if (win < 0 || win >= a.num_pages) {
                            set_error(a.err, PKV_DEVERR_PAGE_RANGE);
                            win = 0;
                        }
                    } else {
                        set_error(a.err, PKV_DEVERR_TABLE_RANGE);
                    }
                }
            }
            return __shfl_sync(kFull, win, lp & 31);
        };
        // A producer owns pages pi, pi + 3, pi + 6 of every tile.  All their code words are
        // loaded first, before the wait for the stage slot, so the loads' latency is paid
        // once per tile and overlaps that wait.  K page: lane = (key l % 16, dims
        // (l / 16) * D/2 .. + D/2 - 1); eight lanes of a store phase hit eight rows, so the
        // swizzled chunks never share banks.  V page (dim-major): lane = dims l, l + 32, ...;
        // one word = the dim's 16 keys.  (One loop for both roles: separately compiled K
        // and V loops measured slower.)
        constexpr int PPW = (kBN / kPage + kProducers - 1) / kProducers;  // pages per warp
        constexpr int W = D / 32;          // 16-byte code words per lane per page
        const int lane_off = is_v ? lane * kPage : (lane & 15) * D + (lane >> 4) * (D / 2);
        const int lane_step = is_v ? 32 * kPage : 16;
        bool ok = true;
        for (int j = 0; ok && j < n_kv; ++j) {
            const int p0 = j * (kBN / kPage);
            const int np = min(kBN / kPage, npages_seq - p0);
            uint4 w[PPW][W];
#pragma unroll
            for (int t = 0; t < PPW; ++t) {
                const int p = pi + kProducers * t;
                if (p < np) {
                    const int phys = page_of(p0 + p);
                    const int64_t block = static_cast<int64_t>(phys) * a.num_kv_heads + g;
                    const uint8_t* src = pool + lane_off + block * (kPage * D);
#pragma unroll
                    for (int u = 0; u < W; ++u)
                        w[t][u] = __ldg(reinterpret_cast<const uint4*>(src + u * lane_step));
                }
            }
            const int nst = is_v ? kStagesV : kStagesK;
            uint64_t* full = is_v ? &v_full[j % kStagesV] : &k_full[j % kStagesK];
            uint64_t* empty = is_v ? &v_empty[j % kStagesV] : &k_empty[j % kStagesK];
            if (j >= nst && lane == 0 && !mbar_wait(empty, ((j / nst) - 1) & 1)) ok = false;
            ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
            if (!ok) break;
            uint8_t* dst = is_v ? sV(j) : sK(j);
#pragma unroll
            for (int t = 0; t < PPW; ++t) {
                const int p = pi + kProducers * t;
                if (p >= kBN / kPage) continue;
#pragma unroll
                for (int u = 0; u < W; ++u) {
                    uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;   // zeros: a page past the end
                    if (p < np) q8_codes16<true>(w[t][u], lo, hi);
                    if (is_v) {
                        uint8_t* half = dst + (p / 4) * S::kVHalf;
                        const int d = lane + 32 * u, ch = (p % 4) * 2;
                        *reinterpret_cast<uint4*>(half + sw128(d, ch)) = lo;
                        *reinterpret_cast<uint4*>(half + sw128(d, ch + 1)) = hi;
                    } else {
                        const int row = p * kPage + (lane & 15);
                        const int d = (lane >> 4) * (D / 2) + 16 * u;   // first dim of the word
                        uint8_t* half = dst + (d / 64) * S::kHalfBytes;
                        const int ch = (d % 64) / 8;
                        *reinterpret_cast<uint4*>(half + sw128(row, ch)) = lo;
                        *reinterpret_cast<uint4*>(half + sw128(row, ch + 1)) = hi;
                    }
                }
            }
            tc::fence_proxy_async_smem();  // generic-proxy writes -> the tensor core's reads
            __syncwarp();
            if (lane == 0) mbar_arrive(full);
        }
        if (!ok && lane == 0) set_error(a.err, PKV_DEVERR_TIMEOUT);
    } else if (warp == kWarpMma) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            bool ok = mbar_wait(q_ready, 0);
            // descriptors of every tile base; a k-step adds its byte offset >> 4 to the
            // 14-bit start-address field (all addresses stay below 256 KiB)
            const uint64_t dq0 = tc::smem_desc_sw128(smem_u32(sQ(0)), 16, 1024);
            const uint64_t dq1 = tc::smem_desc_sw128(smem_u32(sQ(1)), 16, 1024);
            const uint64_t dk0 = tc::smem_desc_sw128(smem_u32(sK(0)), 16, 1024);
            const uint64_t dv0 = tc::smem_desc_sw128(smem_u32(sV(0)), 16, 1024);
            constexpr uint64_t kKStep = (S::kKV) >> 4;          // stage stride in 16 B units
            auto issue_s = [&](int h, int j) {
                const uint64_t dq = h ? dq1 : dq0;
                const uint64_t dk = dk0 + static_cast<uint64_t>(j % kStagesK) * kKStep;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off =
                        static_cast<uint64_t>(((kk >> 2) * S::kHalfBytes + (kk & 3) * 32) >> 4);
                    tc::mma_f16_ss(tm_s(h), dq + off, dk + off, kIdescS, kk > 0 ? 1u : 0u);
                }
                tc::commit(&s_full[h]);
            };
            // half 0: keys 0..63 of the tile, half 1: keys 64..127 (V^T: key halves of
            // D rows x 128 bytes, a k-step of 16 keys is 32 bytes along the row)
            auto issue_pv = [&](int h, int j, int half) {
                const uint64_t dv = dv0 + static_cast<uint64_t>(j % kStagesV) * kKStep;
#pragma unroll
                for (int k4 = 0; k4 < kBN / 32; ++k4) {
                    const int kk = half * (kBN / 32) + k4;
                    const uint64_t off =
                        static_cast<uint64_t>(((kk >> 2) * S::kVHalf + (kk & 3) * 32) >> 4);
                    tc::mma_f16_ts(tm_o(h), tm_s(h) + kk * 8, dv + off, kIdescO,
                                   (j > 0 || kk > 0) ? 1u : 0u);
                }
            };
            auto wait_k = [&](int j) {
                return mbar_wait(&k_full[j % kStagesK], (j / kStagesK) & 1);
            };
            if (ok && n_kv > 0 && (ok = wait_k(0))) {
                tc::fence_after_sync();
                issue_s(0, 0);
                issue_s(1, 0);
                tc::commit(&k_empty[0]);
            }
            for (int j = 0; ok && j < n_kv; ++j) {
                if (!mbar_wait(&v_full[j % kStagesV], (j / kStagesV) & 1) ||
                    !mbar_wait(&p_half[0], j & 1)) { ok = false; break; }
                tc::fence_after_sync();
                issue_pv(0, j, 0);
                if (!mbar_wait(&p_full[0], j & 1)) { ok = false; break; }
                tc::fence_after_sync();
                issue_pv(0, j, 1);
                const bool more = j + 1 < n_kv;
                if (more) {
                    if (!wait_k(j + 1)) { ok = false; break; }
                    tc::fence_after_sync();
                    issue_s(0, j + 1);
                }
                if (!mbar_wait(&p_half[1], j & 1)) { ok = false; break; }
                tc::fence_after_sync();
                issue_pv(1, j, 0);
                if (!mbar_wait(&p_full[1], j & 1)) { ok = false; break; }
                tc::fence_after_sync();
                issue_pv(1, j, 1);
                tc::commit(&v_empty[j % kStagesV]);
                if (more) {
                    issue_s(1, j + 1);
                    tc::commit(&k_empty[(j + 1) % kStagesK]);
                }
            }
            if (!ok) set_error(a.err, PKV_DEVERR_TIMEOUT);
            tc::commit(o_final);
            tc::commit(drain);
            mbar_wait(drain, 0);
        }
    } else {
        // ================================================================ softmax (head h)
        const int h = warp >> 2;
        const int i = threadIdx.x & 127;
        const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t my_s = tm_s(h) + lane_off, my_o = tm_o(h) + lane_off;
        // this warpgroup's chain (selects, not indexing: the tile stays in registers)
        const int first_pos = h ? tile.first_pos[1] : tile.first_pos[0];
        const int rows_valid = h ? tile.rows_valid[1] : tile.rows_valid[0];
        const int q_row = h ? tile.q_row[1] : tile.q_row[0];
        const int q_head = h ? tile.head[1] : tile.head[0];
        const int pos = first_pos + i;
        bool ok = mbar_wait_warp(q_full, 0);
        // ---- Q' = Q * k_scale * f in place, row i of head h.  Physical chunk pc ^ (i & 7)
        //      of the row holds dims 8 pc .. 8 pc + 7 of its half, so every lane reads the
        //      same dims (broadcast scales) and eight rows hit eight different banks.
        const float* ks = a.k_scale + g * D;
        float amax = 0.f;
#pragma unroll 1
        for (int c = 0; c < S::kHalves; ++c) {
#pragma unroll
            for (int pc = 0; pc < 8; ++pc) {
                const uint4 w = *reinterpret_cast<const uint4*>(sQ(h) + c * S::kHalfBytes +
                                                                sw128(i, pc));
                const float4 k0 = __ldg(reinterpret_cast<const float4*>(ks + c * 64 + pc * 8));
                const float4 k1 = __ldg(reinterpret_cast<const float4*>(ks + c * 64 + pc * 8) + 1);
                const float kv[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = Cv::unpack(ww[e]);
                    amax = fmaxf(amax, fmaxf(fabsf(f.x * kv[2 * e]), fabsf(f.y * kv[2 * e + 1])));
                }
            }
        }
        if (i >= rows_valid) amax = 0.f;   // rows past the chunk do not set the scale
#pragma unroll
        for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
        if (lane == 0) red[h * 4 + (warp & 3)] = amax;
        asm volatile("bar.sync %0, 128;" ::"r"(1 + h) : "memory");
        amax = fmaxf(fmaxf(red[h * 4], red[h * 4 + 1]), fmaxf(red[h * 4 + 2], red[h * 4 + 3]));
        const int e_amax = static_cast<int>(__float_as_uint(amax) >> 23) - 127;
        const int ex = min(100, max(-100, static_cast<int>(kQTop) - e_amax));
        const float fq = __uint_as_float(static_cast<uint32_t>(127 + ex) << 23);
        const float inv_f = __uint_as_float(static_cast<uint32_t>(127 - ex) << 23);
#pragma unroll 1
        for (int c = 0; c < S::kHalves; ++c) {
#pragma unroll
            for (int pc = 0; pc < 8; ++pc) {
                uint4* wp = reinterpret_cast<uint4*>(sQ(h) + c * S::kHalfBytes + sw128(i, pc));
                const uint4 w = *wp;
                const float4 k0 = __ldg(reinterpret_cast<const float4*>(ks + c * 64 + pc * 8));
                const float4 k1 = __ldg(reinterpret_cast<const float4*>(ks + c * 64 + pc * 8) + 1);
                const float kv[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
                uint32_t o4[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = Cv::unpack(ww[e]);
                    // rows past the chunk (or a whole chain past it) become zeros: finite
                    // scores whatever the rows held, and a chain without rows has f = 2^100
                    o4[e] = i < rows_valid ? Ch::pack(f.x * kv[2 * e] * fq, f.y * kv[2 * e + 1] * fq)
                                           : 0u;
                }
                *wp = make_uint4(o4[0], o4[1], o4[2], o4[3]);
            }
        }
        tc::fence_proxy_async_smem();
        mbar_arrive(q_ready);
        const float sl2 = a.scale_log2 * inv_f;   // scores come back times f
        float m = -INFINITY, l = 0.f;
        for (int j = 0; ok && j < n_kv; ++j) {
            if (!mbar_wait_warp(&s_full[h], j & 1)) { ok = false; break; }
            tc::fence_after_sync();
            const int kbase = j * kBN;
            // keys at or past `lim` are masked for this row (only on the diagonal tiles)
            const bool diag = kbase + kBN - 1 > first_pos;
            const int lim = diag ? pos + 1 - kbase : kBN;
            uint32_t c0[32], c1[32];
            float mx[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
            auto chunk_max = [&](const uint32_t (&sr)[32], int cb) {
                if (!diag) {
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        mx[e & 7] = fmaxf(mx[e & 7], __uint_as_float(sr[e]));
                } else {
                    const int rem = lim - cb * 32;  // valid keys in this chunk
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        mx[e & 7] = fmaxf(mx[e & 7], e < rem ? __uint_as_float(sr[e]) : -INFINITY);
                }
            };
            tc::tmem_ld32(my_s + 64, c0);
            tc::tmem_ld32(my_s + 96, c1);
            tc::tmem_wait_ld();
            chunk_max(c0, 2);
            chunk_max(c1, 3);
            tc::tmem_ld32(my_s, c0);
            tc::tmem_ld32(my_s + 32, c1);
            tc::tmem_wait_ld();
            chunk_max(c0, 0);
            chunk_max(c1, 1);
            const float tmax =
                fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                      fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl2;
            const float m_new = fmaxf(m, tmax);
            const bool need = (j == 0) || (m_new > m + kRescaleThreshold);
            const float alpha = (j > 0 && need) ? tc::ex2(m - m_new) : 1.f;
            if (need) m = m_new;
            if (j > 0 && __any_sync(kFull, alpha != 1.f)) {
                // O_h is stable: its last P V completed before these scores did
#pragma unroll 1
                for (int cb = 0; cb < D / 32; ++cb) {
                    uint32_t orow[32];
                    tc::tmem_ld32(my_o + cb * 32, orow);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        orow[e] = __float_as_uint(__uint_as_float(orow[e]) * alpha);
                    tc::tmem_st32(my_o + cb * 32, orow);
                }
            }
            // pass 2: P = 2^(s * scale_log2 / f - m) as fp16 pairs over the consumed scores
            float2 ls[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) ls[q] = make_float2(0.f, 0.f);
            const float2 sl2x2 = make_float2(sl2, sl2), nm2 = make_float2(-m, -m);
            auto exps = [&](const uint32_t (&sr)[32], int cb) {
                const int rem = diag ? lim - cb * 32 : 32;
                float p[32];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const float2 x = __ffma2_rn(
                        make_float2(__uint_as_float(sr[2 * u]), __uint_as_float(sr[2 * u + 1])),
                        sl2x2, nm2);
                    p[2 * u] = x.x;
                    p[2 * u + 1] = x.y;
                }
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    p[e] = tc::ex2(p[e]);
                    if (diag) p[e] = e < rem ? p[e] : 0.f;
                }
                uint32_t pk[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    ls[u & 1] = __fadd2_rn(ls[u & 1], make_float2(p[2 * u], p[2 * u + 1]));
                    pk[u] = Ch::pack(p[2 * u], p[2 * u + 1]);
                }
                tc::tmem_st16(my_s + cb * 16, pk);
            };
            exps(c0, 0);
            tc::tmem_ld32(my_s + 64, c0);
            exps(c1, 1);
            tc::tmem_wait_st();  // P of keys 0..63 is in tensor memory
            tc::fence_before_sync();
            mbar_arrive(&p_half[h]);
            tc::tmem_wait_ld();
            tc::tmem_ld32(my_s + 96, c1);
            exps(c0, 2);
            tc::tmem_wait_ld();
            exps(c1, 3);
            tc::tmem_wait_st();
            const float2 lsum = __fadd2_rn(ls[0], ls[1]);
            l = l * alpha + (lsum.x + lsum.y);
            tc::fence_before_sync();
            mbar_arrive(&p_full[h]);
        }
        // ---- epilogue: O / l * v_scale -> the step's dtype, row i of chain h
        if (ok && n_kv > 0 && mbar_wait_warp(o_final, 0)) {
            tc::fence_after_sync();
            const float inv_l = 1.f / l;
            const float* vs = a.v_scale + g * D;
            T* orow = static_cast<T*>(a.out) +
                      (static_cast<int64_t>(q_row + i) * a.num_q_heads + q_head) * D;
#pragma unroll 1
            for (int cb = 0; cb < D / 32; ++cb) {
                uint32_t o32[32];
                tc::tmem_ld32(my_o + cb * 32, o32);
                tc::tmem_wait_ld();
                if (i < rows_valid) {
                    uint4* dst = reinterpret_cast<uint4*>(orow + cb * 32);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float4* vp = reinterpret_cast<const float4*>(vs + cb * 32 + u * 8);
                        const float4 s0 = __ldg(vp), s1 = __ldg(vp + 1);
                        const float sv[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w[e] = Cv::pack(__uint_as_float(o32[u * 8 + 2 * e]) * inv_l * sv[2 * e],
                                            __uint_as_float(o32[u * 8 + 2 * e + 1]) * inv_l *
                                                sv[2 * e + 1]);
                        dst[u] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
                __syncwarp();
            }
        } else if (n_kv > 0) {
            set_error(a.err, PKV_DEVERR_TIMEOUT);
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == kWarpMma) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

template <typename T, int D>
int launch_q8_t(const StepArgs& a, cudaStream_t stream, cudaEvent_t e0, cudaEvent_t e1) {
    using S = Q8Smem<D>;
    static bool configured = false;
    if (!configured) {
        if (cudaFuncSetAttribute(prefill_q8_kernel<T, D>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 S::kLaunchBytes) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured = true;
    }
    alignas(64) CUtensorMap mq;
    if (!make_q_map(a, &mq)) return PKV_ERR_CUDA;
    if (a.lay.max_tiles <= 0) return PKV_OK;
    if (e0 && cudaEventRecord(e0, stream) != cudaSuccess) return PKV_ERR_CUDA;
    if (launch_pdl(prefill_q8_kernel<T, D>, dim3(a.lay.max_tiles), dim3(kThreads),
                   S::kLaunchBytes, stream, a, mq) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (e1 && cudaEventRecord(e1, stream) != cudaSuccess) return PKV_ERR_CUDA;
    return PKV_OK;
}

}  // namespace

int launch_prefill_q8(const StepArgs& a, cudaStream_t stream, cudaEvent_t e0, cudaEvent_t e1) {
    if (a.dtype == PKV_BF16)
        return a.head_dim == 128 ? launch_q8_t<__nv_bfloat16, 128>(a, stream, e0, e1)
                                 : launch_q8_t<__nv_bfloat16, 64>(a, stream, e0, e1);
    return a.head_dim == 128 ? launch_q8_t<__half, 128>(a, stream, e0, e1)
                             : launch_q8_t<__half, 64>(a, stream, e0, e1);
}

}  // namespace pkv
