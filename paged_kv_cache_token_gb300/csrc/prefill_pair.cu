// Prefill-chunk attention on tcgen05 over 16-bit pages.  Each CTA works on two chains of
// 128 query rows that share one KV head's key/value stream (prefill_tile.cuh): two query
// heads of one KV group (grouped-query attention with an even group size,
// hotelren.com/news/6181127 §6.3), or two consecutive query tiles of one head when every
// query head has its own KV head.
//
// Causal softmax attention of each 128-row query tile against every key of its request
// read from the pages (hotelren.com §1.1, §2.1; niuwancheng.cn "11. chunked prefill and
// unified scheduling"), organised so the tensor core stays busy:
//   * both chains consume one K/V stream: each 128-key tile (8 pages) is loaded once for
//     2 x 128 query rows, halving L2->SM traffic per FLOP;
//   * six producer warps issue the page boxes in parallel, three for keys and three for
//     values, each stream on its own ring (a tiled TMA instruction keeps its issuing
//     thread busy for ~190 cycles, so one issuer cannot feed the MMA);
//   * P = 2^(s - m) is written as packed 16-bit pairs into tensor memory over the scores it
//     came from and read from there by the P V MMA, so shared memory holds only Q, K, V;
//   * the MMA warp alternates the chains -- S0, S1, P0 V, S0', P1 V, S1', ... -- while the
//     two softmax warpgroups work on the other chain's scores;
//   * a chain's scores S_j complete only after its previous P V (one thread issues every
//     MMA and tcgen05.commit tracks all of them), so the softmax may rescale O right away.
// Softmax makes two passes over the score row in tensor memory (max, then exponentials) to
// stay within the register budget of 480 threads.
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
constexpr int kProducers = 3;      // warps issuing K boxes; as many again issue V boxes
constexpr int kWarpMma = 8;
constexpr int kWarpProd0 = 9;      // warps 9..11 load K (and Q), 12..14 load V
constexpr int kThreads = 32 * (kWarpProd0 + 2 * kProducers);  // 480
constexpr int kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;

template <int D>
struct PairSmem {
    static constexpr int kHalves = D / 64;
    static constexpr int kHalfBytes = kBM * 128;
    static constexpr int kQ = kBM * D * 2;                 // one head's Q tile
    static constexpr int kKV = kBN * D * 2;
    static constexpr int kQOff = 0;                        // head h at kQOff + h * kQ
    static constexpr int kKOff = 2 * kQ;
    static constexpr int kVOff = kKOff + kStagesK * kKV;
    static constexpr int kBarOff = kVOff + kStagesV * kKV;
    static constexpr int kBars = 24;
    static constexpr int kMiscOff = kBarOff + kBars * 8;
    static constexpr int kBytes = kMiscOff + 64 + 1024;
    static constexpr int kLaunchBytes = kBytes > 120 * 1024 ? kBytes : 120 * 1024;
    static_assert(kLaunchBytes <= 227 * 1024, "shared memory budget");
};

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_pair_kernel(const StepArgs a, const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v) {
    using S = PairSmem<D>;
    using Cv = F16<T>;
    constexpr int kAB = std::is_same<T, __nv_bfloat16>::value ? 1 : 0;
    constexpr uint32_t kIdescS = tc::idesc_f16(kAB, 0, kBM, kBN);
    constexpr uint32_t kIdescO = tc::idesc_f16(kAB, 1, kBM, D);

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
    uint64_t* q_full = bars + 0;
    uint64_t* k_full = bars + 1;    // [3]
    uint64_t* k_empty = bars + 4;   // [3]
    uint64_t* v_full = bars + 7;    // [2]
    uint64_t* v_empty = bars + 9;   // [2]
    uint64_t* s_full = bars + 11;   // [2] per head
    uint64_t* p_full = bars + 13;   // [2] per head
    uint64_t* o_final = bars + 15;
    uint64_t* drain = bars + 16;
    uint64_t* p_half = bars + 17;   // [2] per head: P of keys 0..63 written
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kMiscOff);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- two chains of 128 query rows sharing one KV head's key/value stream
    const int4 tile_rec = reinterpret_cast<const int4*>(a.ws + a.lay.tiles)[blockIdx.x];
    const PairTile tile = pair_tile(a, tile_rec, kBM, kBN);
    const int g = tile.g;
    const int kv_len = tile.kv_len, n_kv = tile.n_kv, npages_seq = tile.npages_seq;

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
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
            tc::prefetch_tmap(&tm_k);
            tc::prefetch_tmap(&tm_v);
            mbar_arrive_expect_tx(q_full, 2 * S::kQ);
            for (int h = 0; h < 2; ++h)
                for (int c = 0; c < S::kHalves; ++c)
                    tc::tma_load_3d(sQ(h) + c * S::kHalfBytes, &tm_q, c * 64, tile.head[h],
                                    tile.q_row[h], q_full);
        }
        const int32_t* bt = a.block_table + static_cast<int64_t>(tile.r) * a.max_pages;
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
        bool ok = true;
        auto issue = [&](int j, bool is_v) {
            const int nst = is_v ? kStagesV : kStagesK;
            uint64_t* full = is_v ? &v_full[j % kStagesV] : &k_full[j % kStagesK];
            uint64_t* empty = is_v ? &v_empty[j % kStagesV] : &k_empty[j % kStagesK];
            if (j >= nst && lane == 0 && !mbar_wait(empty, ((j / nst) - 1) & 1)) ok = false;
            ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
            if (!ok) return;
            const int p0 = j * (kBN / kPage);
            const int np = min(kBN / kPage, npages_seq - p0);
            const int mine = np > pi ? (np - pi + kProducers - 1) / kProducers : 0;
            uint8_t* dst = is_v ? sV(j) : sK(j);
            const void* map = is_v ? static_cast<const void*>(&tm_v) : static_cast<const void*>(&tm_k);
            if (lane == 0) mbar_arrive_expect_tx(full, mine * kPage * D * 2);
            for (int p = 0; p < np; ++p) {
                const int phys = page_of(p0 + p);
                if (lane == 0 && p % kProducers == pi) {
                    const int row0 = (phys * a.num_kv_heads + g) * kPage;
                    for (int c = 0; c < S::kHalves; ++c)
                        tc::tma_load_2d(dst + c * S::kHalfBytes + p * kPage * 128, map, c * 64,
                                        row0, full);
                }
            }
        };
        for (int j = 0; ok && j < n_kv; ++j) issue(j, is_v);
        if (!ok && lane == 0) set_error(a.err, PKV_DEVERR_TIMEOUT);
    } else if (warp == kWarpMma) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            bool ok = mbar_wait(q_full, 0);
            // descriptors of every tile base; a k-step adds its byte offset >> 4 to the
            // 14-bit start-address field (all addresses stay below 256 KiB)
            const uint64_t dq0 = tc::smem_desc_sw128(smem_u32(sQ(0)), 16, 1024);
            const uint64_t dq1 = tc::smem_desc_sw128(smem_u32(sQ(1)), 16, 1024);
            const uint64_t dk0 = tc::smem_desc_sw128(smem_u32(sK(0)), 16, 1024);
            const uint64_t dv0 = tc::smem_desc_sw128(smem_u32(sV(0)), S::kHalfBytes, 1024);
            constexpr uint64_t kKStep = (S::kKV) >> 4;          // stage stride in 16 B units
            auto issue_s = [&](int h, int j) {
                const uint64_t dq = h ? dq1 : dq0;
                const uint64_t dk = dk0 + static_cast<uint64_t>(j % kStagesK) * kKStep;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * S::kHalfBytes + (kk & 3) * 32) >> 4);
                    tc::mma_f16_ss(tm_s(h), dq + off, dk + off, kIdescS, kk > 0 ? 1u : 0u);
                }
                tc::commit(&s_full[h]);
            };
            // half 0: keys 0..63 of the tile, half 1: keys 64..127
            auto issue_pv = [&](int h, int j, int half) {
                const uint64_t dv = dv0 + static_cast<uint64_t>(j % kStagesV) * kKStep;
#pragma unroll
                for (int k4 = 0; k4 < kBN / 32; ++k4) {
                    const int kk = half * (kBN / 32) + k4;
                    tc::mma_f16_ts(tm_o(h), tm_s(h) + kk * 8, dv + static_cast<uint64_t>(kk * 2048 >> 4),
                                   kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
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
            // P V of a head starts on the first half of P while the softmax finishes the
            // second half
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
        const float sl2 = a.scale_log2;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_kv; ++j) {
            if (!mbar_wait_warp(&s_full[h], j & 1)) { ok = false; break; }
            tc::fence_after_sync();
            const int kbase = j * kBN;
            // keys at or past `lim` are masked for this row (only on the diagonal tiles)
            const bool diag = kbase + kBN - 1 > first_pos;
            const int lim = diag ? pos + 1 - kbase : kBN;
            // pass 1: row maximum of the raw scores, two 32-column loads per wait; columns
            // 64..127 first, then 0..63, which stay in registers for pass 2
            uint32_t c0[32], c1[32];
            float mx[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) mx[e] = -INFINITY;
            auto chunk_max = [&](const uint32_t (&sr)[32], int cb) {
                if (!diag) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) mx[e & 7] = fmaxf(mx[e & 7], __uint_as_float(sr[e]));
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
            // pass 2: P = 2^(s * scale_log2 - m), packed pairs written over the scores of
            // columns already consumed (P of chunk cb goes to columns 16 cb .. 16 cb + 15);
            // scale-and-subtract and the row sums run two columns per instruction
            // two independent partial sums, so no add chain waits on each exponential
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
                    pk[u] = Cv::pack(p[2 * u], p[2 * u + 1]);
                }
                tc::tmem_st16(my_s + cb * 16, pk);
            };
            // each reload (S columns 64..127, still intact) goes into the chunk just consumed
            // and lands while the other chunk's exponentials run
            // the two remaining chunks are loaded before the first half of P is released,
            // so their loads do not queue behind the P V reads of tensor memory
            exps(c0, 0);
            tc::tmem_ld32(my_s + 64, c0);
            exps(c1, 1);
            // final tile: V rows past the last key are zeroed (P is 0 there; stale pool
            // data may be NaN and 0 * NaN would poison the product) before any P V of the
            // tile can read them
            if (h == 0 && j == n_kv - 1 && kv_len - kbase < kBN) {
                if (mbar_wait_warp(&v_full[j % kStagesV], (j / kStagesV) & 1) &&
                    kbase + i >= kv_len) {
                    uint8_t* vrow = sV(j);
#pragma unroll
                    for (int c = 0; c < S::kHalves; ++c) {
                        uint4* dst = reinterpret_cast<uint4*>(vrow + c * S::kHalfBytes + i * 128);
#pragma unroll
                        for (int u = 0; u < 8; ++u) dst[u] = make_uint4(0, 0, 0, 0);
                    }
                }
                tc::fence_proxy_async_smem();
            }
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
            const float ls0 = lsum.x, ls1 = lsum.y;
            l = l * alpha + (ls0 + ls1);
            tc::fence_before_sync();
            mbar_arrive(&p_full[h]);
        }
        // ---- epilogue: O / l -> 16-bit, row i of chain h
        if (ok && n_kv > 0 && mbar_wait_warp(o_final, 0)) {
            tc::fence_after_sync();
            const float inv_l = 1.f / l;
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
                        uint32_t w[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e)
                            w[e] = Cv::pack(__uint_as_float(o32[u * 8 + 2 * e]) * inv_l,
                                            __uint_as_float(o32[u * 8 + 2 * e + 1]) * inv_l);
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
int launch_pair_t(const StepArgs& a, cudaStream_t stream, cudaEvent_t e0, cudaEvent_t e1) {
    using S = PairSmem<D>;
    static bool configured = false;
    if (!configured) {
        if (cudaFuncSetAttribute(prefill_pair_kernel<T, D>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 S::kLaunchBytes) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured = true;
    }
    alignas(64) CUtensorMap mq, mk, mv;
    if (!make_prefill_maps(a, &mq, &mk, &mv)) return PKV_ERR_CUDA;
    if (a.lay.max_tiles <= 0) return PKV_OK;
    if (e0 && cudaEventRecord(e0, stream) != cudaSuccess) return PKV_ERR_CUDA;
    if (launch_pdl(prefill_pair_kernel<T, D>, dim3(a.lay.max_tiles), dim3(kThreads),
                   S::kLaunchBytes, stream, a, mq, mk, mv) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (e1 && cudaEventRecord(e1, stream) != cudaSuccess) return PKV_ERR_CUDA;
    return PKV_OK;
}

}  // namespace

int launch_prefill_pair(const StepArgs& a, cudaStream_t stream, cudaEvent_t e0, cudaEvent_t e1) {
    if (a.dtype == PKV_BF16)
        return a.head_dim == 128 ? launch_pair_t<__nv_bfloat16, 128>(a, stream, e0, e1)
                                 : launch_pair_t<__nv_bfloat16, 64>(a, stream, e0, e1);
    return a.head_dim == 128 ? launch_pair_t<__half, 128>(a, stream, e0, e1)
                             : launch_pair_t<__half, 64>(a, stream, e0, e1);
}

}  // namespace pkv
