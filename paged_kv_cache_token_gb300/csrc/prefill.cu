// Prefill-chunk path of the paged attention step on the 5th-generation tensor cores.
//
// Rows of a request that advances by many tokens (a chunked prefill) form a causal block:
// query row i at position ctx + i scores keys 0..ctx+i (hotelren.com/news/6181127 §1.1,
// §2.1: row softmax of the masked score matrix, times V; §2.1 also notes that blocked
// computation avoids materialising the S x S matrix).  A chunk reads the earlier chunks'
// K/V like a decode and writes its own (niuwancheng.cn "11. chunked prefill and unified
// scheduling"), so the keys of every tile come from the pages through the block table.
// Prefill is a dense contraction (wmrh.cn §2.2, hotelren.com §1.2), so QK^T and PV run on
// tcgen05 with fp32 accumulators in tensor memory.
//
// One CTA computes one tile = (request, 128 query rows, query head) against all its keys
// in 128-key tiles (8 pages).  Warp roles:
//   warps 0-3  softmax: thread i owns query row i (TMEM lane i); reads S from TMEM, masks
//              the causal diagonal, keeps a running max (rescaling O only when the max grows
//              by more than 2^8), writes P = 2^(s - m) as 16-bit values into shared memory
//              in the 128-byte-swizzled K-major layout, normalises O at the end;
//   warp 4     producer: TMA loads of the Q tile (3-D map over [T][Hq][D]) and of each
//              page's 16 x D block of K and V (2-D map over the pool rows); K has a 3-stage
//              ring freed as soon as its scores are computed, V a 2-stage ring freed after
//              P V, and keys are requested a tile ahead of values;
//   warp 5     MMA: S_j = Q K_j^T into one of two TMEM buffers, then O += P_{j-1} V_{j-1},
//              so the tensor core computes the next scores while softmax works.
// Keys past the request's last key in the final tile have their V rows zeroed in shared
// memory before the P V product (their P is 0, but stale pool data may be NaN).
#include <cuda.h>
#include <cudaTypedefs.h>

#include <climits>
#include <type_traits>

#include "common.cuh"
#include "launch.h"
#include "tc.cuh"

namespace pkv {

namespace {

constexpr int kBM = 128;          // query rows per tile
constexpr int kBN = 128;          // keys per KV tile (8 pages)
constexpr int kStagesK = 3;       // K ring: released as soon as its S = Q K^T completes
constexpr int kStagesV = 2;       // V ring: released after its O += P V
constexpr int kThreads = 192;     // 4 softmax warps + producer + MMA
constexpr int kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows > 2^8

template <int D>
struct PrefillSmem {
    static constexpr int kHalves = D / 64;               // 128-byte column blocks
    static constexpr int kHalfBytes = kBM * 128;          // 128 rows x 128 bytes
    static constexpr int kQ = kBM * D * 2;
    static constexpr int kKV = kBN * D * 2;               // one K or V tile
    static constexpr int kP = kBM * kBN * 2;
    static constexpr int kQOff = 0;
    static constexpr int kKOff = kQ;                       // K stage s at kKOff + s*kKV
    static constexpr int kVOff = kKOff + kStagesK * kKV;   // V stage s at kVOff + s*kKV
    static constexpr int kPOff = kVOff + kStagesV * kKV;
    static constexpr int kBarOff = kPOff + kP;
    static constexpr int kBars = 16;
    static constexpr int kMiscOff = kBarOff + kBars * 8;
    static constexpr int kBytes = kMiscOff + 64 + 1024;    // + alignment slack
    // keep one CTA per SM so the 512-column TMEM allocation never waits
    static constexpr int kLaunchBytes = kBytes > 120 * 1024 ? kBytes : 120 * 1024;
    static_assert(kLaunchBytes <= 227 * 1024, "shared memory budget");
};

struct TileInfo {
    int r, qt, h, g;
    int ctx, q_off, rows_valid, kv_len, n_kv, npages_seq, first_pos;
};

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
prefill_kernel(const StepArgs a, const __grid_constant__ CUtensorMap tm_q,
               const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
    using S = PrefillSmem<D>;
    using Cv = F16<T>;
    constexpr int kAB = std::is_same<T, __nv_bfloat16>::value ? 1 : 0;
    constexpr uint32_t kIdescS = tc::idesc_f16(kAB, 0, kBM, kBN);
    constexpr uint32_t kIdescO = tc::idesc_f16(kAB, 1, kBM, D);

    pdl_wait();  // plan, kv_append and the decode kernel of this step have completed
    const int32_t* ctrl = reinterpret_cast<const int32_t*>(a.ws + a.lay.ctrl);
    if (static_cast<int>(blockIdx.x) >= ctrl[9]) return;  // fewer tiles than the bound

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S::kBarOff);
    uint64_t* q_full = bars + 0;
    uint64_t* k_full = bars + 1;     // [kStagesK]
    uint64_t* k_empty = bars + 4;    // [kStagesK]
    uint64_t* v_full = bars + 7;     // [kStagesV]
    uint64_t* v_empty = bars + 9;    // [kStagesV]
    uint64_t* s_full = bars + 11;    // [2]
    uint64_t* p_full = bars + 13;
    uint64_t* o_done = bars + 14;
    uint64_t* drain = bars + 15;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::kMiscOff);
    int* abort_flag = reinterpret_cast<int*>(smem + S::kMiscOff + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- tile description (every thread computes the same values)
    TileInfo ti;
    {
        const int4 tl = reinterpret_cast<const int4*>(a.ws + a.lay.tiles)[blockIdx.x];
        ti.r = tl.x;
        ti.qt = tl.y;
        ti.h = tl.z;
        ti.g = ti.h / (a.num_q_heads / a.num_kv_heads);
        ti.ctx = a.context_lens[ti.r];
        ti.q_off = a.q_offsets[ti.r];
        const int qlen = a.q_lens[ti.r];
        ti.rows_valid = min(kBM, qlen - ti.qt * kBM);
        ti.first_pos = ti.ctx + ti.qt * kBM;
        ti.kv_len = ti.first_pos + ti.rows_valid;
        ti.n_kv = cdiv(ti.kv_len, kBN);
        ti.npages_seq = cdiv(ti.kv_len, kPage);
    }

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        for (int s = 0; s < kStagesK; ++s) {
            mbar_init(&k_full[s], 1);
            mbar_init(&k_empty[s], 1);
        }
        for (int s = 0; s < kStagesV; ++s) {
            mbar_init(&v_full[s], 1);
            mbar_init(&v_empty[s], 1);
        }
        mbar_init(&s_full[0], 1);
        mbar_init(&s_full[1], 1);
        mbar_init(p_full, 128);
        mbar_init(o_done, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 5) {
        tc::tmem_alloc(tmem_slot, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    auto tm_s = [&](int j) { return tmem + static_cast<uint32_t>((j & 1) * kBN); };
    const uint32_t tm_o = tmem + 2 * kBN;

    uint8_t* sQ = smem + S::kQOff;
    uint8_t* sP = smem + S::kPOff;
    auto sK = [&](int j) { return smem + S::kKOff + (j % kStagesK) * S::kKV; };  // tile j
    auto sV = [&](int j) { return smem + S::kVOff + (j % kStagesV) * S::kKV; };

    if (warp == 4) {
        // ================================================================ producer
        // whole warp: lanes fetch 32 block-table entries at a time, lane 0 issues TMA.
        // Order K_0, then for every j: K_{j+1}, V_j -- keys run a tile ahead of values.
        if (lane == 0) {
            tc::prefetch_tmap(&tm_q);
            tc::prefetch_tmap(&tm_k);
            tc::prefetch_tmap(&tm_v);
            mbar_arrive_expect_tx(q_full, S::kQ);
            for (int c = 0; c < S::kHalves; ++c)
                tc::tma_load_3d(sQ + c * S::kHalfBytes, &tm_q, c * 64, ti.h,
                                ti.q_off + ti.qt * kBM, q_full);
        }
        const int32_t* bt = a.block_table + static_cast<int64_t>(ti.r) * a.max_pages;
        int win_base = -1, win = 0;
        auto page_of = [&](int lp) -> int {  // warp-wide; physical page of logical page lp
            const int base = lp & ~31;
            if (base != win_base) {
                win_base = base;
                const int l = base + lane;
                win = 0;
                if (l < ti.npages_seq) {
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
            const int np = min(kBN / kPage, ti.npages_seq - p0);
            uint8_t* dst = is_v ? sV(j) : sK(j);
            const void* map = is_v ? static_cast<const void*>(&tm_v) : static_cast<const void*>(&tm_k);
            if (lane == 0) mbar_arrive_expect_tx(full, np * kPage * D * 2);
            for (int p = 0; p < np; ++p) {
                const int phys = page_of(p0 + p);
                if (lane == 0) {
                    const int row0 = (phys * a.num_kv_heads + ti.g) * kPage;
                    for (int c = 0; c < S::kHalves; ++c)
                        tc::tma_load_2d(dst + c * S::kHalfBytes + p * kPage * 128, map, c * 64,
                                        row0, full);
                }
            }
        };
        if (ti.n_kv > 0) issue(0, false);
        for (int j = 0; ok && j < ti.n_kv; ++j) {
            if (j + 1 < ti.n_kv) issue(j + 1, false);
            if (ok) issue(j, true);
        }
        if (!ok && lane == 0) {
            set_error(a.err, PKV_DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
    } else if (warp == 5) {
        // ================================================================ MMA issuer
        if (lane == 0) {
            const uint32_t q_addr = smem_u32(sQ);
            const uint32_t p_addr = smem_u32(sP);
            bool ok = mbar_wait(q_full, 0);
            auto issue_pv = [&](int jj) {  // O (+)= P_jj V_jj
                const uint32_t v_addr = smem_u32(sV(jj));
#pragma unroll
                for (int kk = 0; kk < kBN / 16; ++kk) {
                    const uint64_t ad = tc::smem_desc_sw128(
                        p_addr + (kk >> 2) * S::kHalfBytes + (kk & 3) * 32, 16, 1024);
                    const uint64_t bd = tc::smem_desc_sw128(v_addr + kk * 2048, S::kHalfBytes, 1024);
                    tc::mma_f16_ss(tm_o, ad, bd, kIdescO, (jj > 0 || kk > 0) ? 1u : 0u);
                }
                tc::commit(o_done);
                tc::commit(&v_empty[jj % kStagesV]);
            };
            auto wait_v = [&](int jj) {
                return mbar_wait(&v_full[jj % kStagesV], (jj / kStagesV) & 1);
            };
            for (int j = 0; ok && j < ti.n_kv; ++j) {
                if (!mbar_wait(&k_full[j % kStagesK], (j / kStagesK) & 1)) { ok = false; break; }
                tc::fence_after_sync();
                const uint32_t k_addr = smem_u32(sK(j));
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * S::kHalfBytes + (kk & 3) * 32;
                    const uint64_t ad = tc::smem_desc_sw128(q_addr + off, 16, 1024);
                    const uint64_t bd = tc::smem_desc_sw128(k_addr + off, 16, 1024);
                    tc::mma_f16_ss(tm_s(j), ad, bd, kIdescS, kk > 0 ? 1u : 0u);
                }
                tc::commit(&s_full[j & 1]);
                tc::commit(&k_empty[j % kStagesK]);
                if (j >= 1) {
                    if (!wait_v(j - 1) || !mbar_wait(p_full, (j - 1) & 1)) { ok = false; break; }
                    tc::fence_after_sync();
                    issue_pv(j - 1);
                }
            }
            if (ok && ti.n_kv > 0) {
                if (wait_v(ti.n_kv - 1) && mbar_wait(p_full, (ti.n_kv - 1) & 1)) {
                    tc::fence_after_sync();
                    issue_pv(ti.n_kv - 1);
                } else {
                    ok = false;
                }
            }
            if (!ok) {
                set_error(a.err, PKV_DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
            tc::commit(drain);            // completes when every MMA above has finished
            mbar_wait(drain, 0);
        }
    } else {
        // ================================================================ softmax
        const int i = threadIdx.x;                    // query row in the tile, TMEM lane
        const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
        const int pos = ti.first_pos + i;
        const float sl2 = a.scale_log2;
        float m = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < ti.n_kv; ++j) {
            if (!mbar_wait(&s_full[j & 1], (j >> 1) & 1)) { ok = false; break; }
            __syncwarp();
            tc::fence_after_sync();
            uint32_t sr[4][32];
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) tc::tmem_ld32(tm_s(j) + lane_off + cb * 32, sr[cb]);
            tc::tmem_wait_ld();
            const int kbase = j * kBN;
            const bool need_mask = kbase + kBN - 1 > ti.first_pos;
            float tmax = -INFINITY;
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    float x = __uint_as_float(sr[cb][e]) * sl2;
                    if (need_mask && kbase + cb * 32 + e > pos) x = -INFINITY;
                    sr[cb][e] = __float_as_uint(x);
                    tmax = fmaxf(tmax, x);
                }
            }
            const float m_new = fmaxf(m, tmax);
            const bool need = (j == 0) || (m_new > m + kRescaleThreshold);
            const float alpha = (j > 0 && need) ? tc::ex2(m - m_new) : 1.f;
            if (need) m = m_new;
            // P = 2^(x - m) packed to 16-bit pairs before waiting for the previous P V, so
            // the exponentials overlap with the tensor core
            uint32_t pk[64];
            float lsum = 0.f;
#pragma unroll
            for (int cb = 0; cb < 4; ++cb) {
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const float p0 = tc::ex2(__uint_as_float(sr[cb][2 * u]) - m);
                    const float p1 = tc::ex2(__uint_as_float(sr[cb][2 * u + 1]) - m);
                    lsum += p0 + p1;
                    pk[cb * 16 + u] = Cv::pack(p0, p1);
                }
            }
            l = l * alpha + lsum;
            if (j > 0 && !mbar_wait(o_done, (j - 1) & 1)) { ok = false; break; }
            __syncwarp();
            if (j > 0 && __any_sync(kFull, alpha != 1.f)) {  // rescale my O row
                tc::fence_after_sync();
#pragma unroll
                for (int cb = 0; cb < D / 32; ++cb) {
                    uint32_t orow[32];
                    tc::tmem_ld32(tm_o + lane_off + cb * 32, orow);
                    tc::tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        orow[e] = __float_as_uint(__uint_as_float(orow[e]) * alpha);
                    tc::tmem_st32(tm_o + lane_off + cb * 32, orow);
                }
                tc::tmem_wait_st();
            }
            // row i of the 128-byte-swizzled K-major P tile
#pragma unroll
            for (int chunk = 0; chunk < 16; ++chunk) {      // 16-byte chunks along the keys
                const int half = chunk >> 3, c = chunk & 7;
                uint8_t* dst = sP + half * S::kHalfBytes + i * 128 + ((c ^ (i & 7)) << 4);
                *reinterpret_cast<uint4*>(dst) =
                    make_uint4(pk[chunk * 4], pk[chunk * 4 + 1], pk[chunk * 4 + 2], pk[chunk * 4 + 3]);
            }
            // final tile: V rows past the last key are zeroed (P is 0 there, V may be NaN)
            if (j == ti.n_kv - 1 && kbase + i >= ti.kv_len &&
                mbar_wait(&v_full[j % kStagesV], (j / kStagesV) & 1)) {
                uint8_t* vrow = sV(j);
#pragma unroll
                for (int c = 0; c < S::kHalves; ++c) {
                    uint4* dst = reinterpret_cast<uint4*>(vrow + c * S::kHalfBytes + i * 128);
#pragma unroll
                    for (int u = 0; u < 8; ++u) dst[u] = make_uint4(0, 0, 0, 0);
                }
            }
            tc::fence_proxy_async_smem();
            tc::fence_before_sync();
            mbar_arrive(p_full);
        }
        // ---- epilogue: O / l -> 16-bit, row i
        if (ok && ti.n_kv > 0 && mbar_wait(o_done, (ti.n_kv - 1) & 1)) {
            __syncwarp();
            tc::fence_after_sync();
            const float inv_l = 1.f / l;
            T* orow = static_cast<T*>(a.out) +
                      (static_cast<int64_t>(ti.q_off + ti.qt * kBM + i) * a.num_q_heads + ti.h) * D;
#pragma unroll
            for (int cb = 0; cb < D / 32; ++cb) {
                uint32_t o32[32];
                __syncwarp();
                tc::tmem_ld32(tm_o + lane_off + cb * 32, o32);
                tc::tmem_wait_ld();
                if (i < ti.rows_valid) {
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
            }
        } else if (!ok || ti.n_kv > 0) {
            set_error(a.err, PKV_DEVERR_TIMEOUT);
            *abort_flag = 1;
        }
    }

    tc::fence_before_sync();
    __syncthreads();
    if (warp == 5) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

// ------------------------------------------------------------------------------------
// host side: tensor maps and launch
// ------------------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool make_q_map(const StepArgs& a, CUtensorMap* mq) {
    auto enc = encode_fn();
    if (!enc) return false;
    const CUtensorMapDataType dt =
        a.dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const cuuint64_t D = static_cast<cuuint64_t>(a.head_dim);
    // Q: [T][Hq][D] as a 3-D tensor, box 64 x 1 x 128 rows
    cuuint64_t dims[3] = {D, static_cast<cuuint64_t>(a.num_q_heads),
                          static_cast<cuuint64_t>(a.total_q_tokens)};
    cuuint64_t strides[2] = {D * 2, D * 2 * a.num_q_heads};
    cuuint32_t box[3] = {64, 1, kBM};
    cuuint32_t es[3] = {1, 1, 1};
    return enc(mq, dt, 3, const_cast<void*>(a.q), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
           CUDA_SUCCESS;
}

bool make_prefill_maps(const StepArgs& a, CUtensorMap* mq, CUtensorMap* mk, CUtensorMap* mv) {
    auto enc = encode_fn();
    if (!enc || !make_q_map(a, mq)) return false;
    const CUtensorMapDataType dt =
        a.dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const cuuint64_t D = static_cast<cuuint64_t>(a.head_dim);
    // K, V pools: [num_pages * Hkv * 16 rows][D], box 64 x 16 rows (one page of one head)
    const cuuint64_t rows = static_cast<cuuint64_t>(a.num_pages) * a.num_kv_heads * kPage;
    cuuint64_t dims[2] = {D, rows};
    cuuint64_t strides[1] = {D * 2};
    cuuint32_t box[2] = {64, kPage};
    cuuint32_t es[2] = {1, 1};
    if (enc(mk, dt, 2, const_cast<void*>(a.k_cache), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    if (enc(mv, dt, 2, const_cast<void*>(a.v_cache), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    return true;
}

namespace {

template <typename T, int D>
int launch_t(const StepArgs& a, cudaStream_t stream, cudaEvent_t e0, cudaEvent_t e1) {
    using S = PrefillSmem<D>;
    static bool configured = false;
    if (!configured) {
        if (cudaFuncSetAttribute(prefill_kernel<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 S::kLaunchBytes) != cudaSuccess)
            return PKV_ERR_CUDA;
        configured = true;
    }
    alignas(64) CUtensorMap mq, mk, mv;
    if (!make_prefill_maps(a, &mq, &mk, &mv)) return PKV_ERR_CUDA;
    if (a.lay.max_tiles <= 0) return PKV_OK;
    if (e0 && cudaEventRecord(e0, stream) != cudaSuccess) return PKV_ERR_CUDA;
    if (launch_pdl(prefill_kernel<T, D>, dim3(a.lay.max_tiles), dim3(kThreads), S::kLaunchBytes,
                   stream, a, mq, mk, mv) != cudaSuccess)
        return PKV_ERR_CUDA;
    if (e1 && cudaEventRecord(e1, stream) != cudaSuccess) return PKV_ERR_CUDA;
    return PKV_OK;
}

}  // namespace

int launch_prefill(const StepArgs& a, cudaStream_t stream, cudaEvent_t e0, cudaEvent_t e1) {
    if (a.kv_int8) return launch_prefill_q8(a, stream, e0, e1);
    if (a.heads_per_tile == 2) return launch_prefill_pair(a, stream, e0, e1);
    if (a.dtype == PKV_BF16)
        return a.head_dim == 128 ? launch_t<__nv_bfloat16, 128>(a, stream, e0, e1)
                                 : launch_t<__nv_bfloat16, 64>(a, stream, e0, e1);
    return a.head_dim == 128 ? launch_t<__half, 128>(a, stream, e0, e1)
                             : launch_t<__half, 64>(a, stream, e0, e1);
}

}  // namespace pkv
