// kv_append: scatter this step's new K/V rows into their 16-token pages.
//
// lshu.cn/news/11576 §2.2: K/V are written by page index into a pre-allocated pool of
// fixed-size pages (dense during prefill, scattered during decode); §2.3: 16 tokens per
// page; §4.3: a write kernel must also cover lengths that are exact multiples of the
// page size.  hotelren.com/news/6181127 §3.1: the new K and V are appended to the cache.
//
// One warp copies one (token, KV head): D 16-bit values of K and of V, 16 bytes per lane,
// so a token's K and V rows move as full 128-byte transactions.  The request of a token
// comes from a binary search of q_offsets; the destination from the block table.  Bad
// device data sets a flag bit and skips the copy; nothing traps.
#include "common.cuh"
#include "launch.h"

namespace pkv {

template <int D>
__global__ void __launch_bounds__(256) kv_append_kernel(AppendArgs a) {
    constexpr int kLanesPerRow = D * 2 / 16;  // 16-byte chunks per K (or V) row: 16 or 8
    const int warp_global = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32;
    const int lane = threadIdx.x & 31;
    const int t = warp_global / a.num_kv_heads;
    const int h = warp_global % a.num_kv_heads;
    if (blockIdx.x == 0 && threadIdx.x == 0 && a.q_offsets[a.num_reqs] != a.total_q_tokens)
        set_error(a.err, PKV_DEVERR_TOKENS);
    if (t >= a.total_q_tokens) return;

    // request of token t: last r with q_offsets[r] <= t
    int lo = 0, hi = a.num_reqs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (__ldg(a.q_offsets + mid) <= t) lo = mid; else hi = mid - 1;
    }
    const int r = lo;
    const int start = __ldg(a.q_offsets + r);
    const int qlen = __ldg(a.q_lens + r);
    if (t - start >= qlen) {  // q_offsets and q_lens disagree
        if (lane == 0) set_error(a.err, PKV_DEVERR_TOKENS);
        return;
    }
    const int pos = __ldg(a.context_lens + r) + (t - start);
    const int lp = pos / kPage;
    if (lp >= a.max_pages) {
        if (lane == 0) set_error(a.err, PKV_DEVERR_TABLE_RANGE);
        return;
    }
    const int page = __ldg(a.block_table + static_cast<int64_t>(r) * a.max_pages + lp);
    if (page < 0 || page >= a.num_pages) {
        if (lane == 0) set_error(a.err, PKV_DEVERR_PAGE_RANGE);
        return;
    }
    const int slot = pos % kPage;
    if (h == 0 && lane == 0 && a.slot_mapping)
        a.slot_mapping[t] = static_cast<int64_t>(page) * kPage + slot;

    const int64_t src = (static_cast<int64_t>(t) * a.num_kv_heads + h) * D;
    const int64_t dst = ((static_cast<int64_t>(page) * a.num_kv_heads + h) * kPage + slot) * D;
    if (lane < 2 * kLanesPerRow) {
        const bool is_v = lane >= kLanesPerRow;
        const int chunk = is_v ? lane - kLanesPerRow : lane;
        const uint16_t* s = static_cast<const uint16_t*>(is_v ? a.v_new : a.k_new) + src;
        uint16_t* d = static_cast<uint16_t*>(is_v ? a.v_cache : a.k_cache) + dst;
        const uint4 val = __ldg(reinterpret_cast<const uint4*>(s) + chunk);
        reinterpret_cast<uint4*>(d)[chunk] = val;
    }
}

int launch_kv_append(const AppendArgs& a, cudaStream_t stream) {
    const int64_t warps = static_cast<int64_t>(a.total_q_tokens) * a.num_kv_heads;
    if (warps == 0) return PKV_OK;
    const int threads = 256;
    const int64_t blocks = (warps + 7) / 8;
    if (blocks > 0x7fffffff) return PKV_ERR_INVALID_ARG;
    if (a.head_dim == 128)
        kv_append_kernel<128><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(a);
    else
        kv_append_kernel<64><<<static_cast<unsigned>(blocks), threads, 0, stream>>>(a);
    return cudaGetLastError() == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
