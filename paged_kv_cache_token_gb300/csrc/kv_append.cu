// kv_append: scatter this step's new K/V rows into their 16-token pages.
//
// lshu.cn/news/11576 §2.2: K/V are written by page index into a pre-allocated pool of
// fixed-size pages (dense during prefill, scattered during decode); §2.3: 16 tokens per
// page; §4.3: a write kernel must also cover lengths that are exact multiples of the
// page size.  hotelren.com/news/6181127 §3.1: the new K and V are appended to the cache.
//
// A CTA takes up to 32 tokens of one request (grid.y = request, so no search for the
// request of a token); one warp copies one (token, KV head): D 16-bit values of K and of
// V, 16 bytes per lane, so each row moves as full 128-byte transactions.  The destination
// comes from the block table.  Bad device data sets a flag bit and skips the copy; nothing
// traps.
#include <algorithm>

#include "common.cuh"
#include "launch.h"

namespace pkv {

constexpr int kTokPerBlock = 32;  // tokens of one request per CTA

// grid.y = request, grid.x = chunk of kTokPerBlock tokens of that request
template <int D>
__global__ void __launch_bounds__(256) kv_append_kernel(AppendArgs a) {
    constexpr int kLanesPerRow = D * 2 / 16;  // 16-byte chunks per K (or V) row: 16 or 8
    const int r = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // earlier kernels on the stream (the previous step) may still read the pool: wait for
    // them before writing; then the attention plan, which reads only metadata, may start
    pdl_wait();
    pdl_trigger();
    if (r == 0 && blockIdx.x == 0 && threadIdx.x == 0 &&
        (a.q_offsets[0] != 0 || a.q_offsets[a.num_reqs] != a.total_q_tokens))
        set_error(a.err, PKV_DEVERR_TOKENS);
    const int qlen = __ldg(a.q_lens + r);
    const int start = __ldg(a.q_offsets + r);
    const int ctx = __ldg(a.context_lens + r);
    const int tok0 = blockIdx.x * kTokPerBlock;
    if (tok0 >= qlen) return;
    if (__ldg(a.q_offsets + r + 1) - start != qlen || ctx < 0 || qlen > a.max_q_len ||
        start < 0 || start + qlen > a.total_q_tokens) {
        if (threadIdx.x == 0) set_error(a.err, PKV_DEVERR_TOKENS);
        return;
    }
    const int ntok = min(kTokPerBlock, qlen - tok0);
    const int32_t* bt = a.block_table + static_cast<int64_t>(r) * a.max_pages;
    // one warp per (token, KV head): 16 bytes per lane, K rows on the low lanes, V above
    for (int w = warp; w < ntok * a.num_kv_heads; w += blockDim.x / 32) {
        const int i = tok0 + w / a.num_kv_heads, h = w % a.num_kv_heads;
        const int t = start + i;
        const int pos = ctx + i;
        const int lp = pos / kPage;
        if (lp >= a.max_pages) {
            if (lane == 0) set_error(a.err, PKV_DEVERR_TABLE_RANGE);
            continue;
        }
        const int page = __ldg(bt + lp);
        if (page < 0 || page >= a.num_pages) {
            if (lane == 0) set_error(a.err, PKV_DEVERR_PAGE_RANGE);
            continue;
        }
        const int slot = pos % kPage;
        if (h == 0 && lane == 0 && a.slot_mapping)
            a.slot_mapping[t] = static_cast<int64_t>(page) * kPage + slot;
        const int64_t src = (static_cast<int64_t>(t) * a.num_kv_heads + h) * D;
        const int64_t dst = ((static_cast<int64_t>(page) * a.num_kv_heads + h) * kPage + slot) * D;
        if (lane < 2 * kLanesPerRow) {
            const bool is_v = lane >= kLanesPerRow;
            const int chunk = is_v ? lane - kLanesPerRow : lane;
            const uint16_t* sp = static_cast<const uint16_t*>(is_v ? a.v_new : a.k_new) + src;
            uint16_t* dp = static_cast<uint16_t*>(is_v ? a.v_cache : a.k_cache) + dst;
            reinterpret_cast<uint4*>(dp)[chunk] = __ldg(reinterpret_cast<const uint4*>(sp) + chunk);
        }
    }
}

// INT8 pools (wmrh.cn/news/64708 §4.3: the KV cache in INT8 halves its memory and
// bandwidth; §5.4: calibrated per channel).  Same placement as kv_append_kernel; each value
// x of channel (h, d) is stored as clamp(rint(x / s[h][d]), -127, 127), the quotient in IEEE
// fp32 and rint rounding to nearest even.  A K page block is [16 slots][D] like the 16-bit
// pools; a V page block is stored [D][16 slots] (each dim's 16 tokens contiguous), the
// order in which the attention step's tensor-core fragments read values.  One warp per
// (token, KV head); lane l quantises channels l*DPL .. l*DPL+DPL-1 of K and of V.
template <typename T, int D>
__global__ void __launch_bounds__(256) kv_append_int8_kernel(AppendArgs a) {
    constexpr int DPL = D / 32;  // channels per lane: 4 or 2
    using Cv = F16<T>;
    const int r = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_wait();
    pdl_trigger();
    if (r == 0 && blockIdx.x == 0 && threadIdx.x == 0 &&
        (a.q_offsets[0] != 0 || a.q_offsets[a.num_reqs] != a.total_q_tokens))
        set_error(a.err, PKV_DEVERR_TOKENS);
    const int qlen = __ldg(a.q_lens + r);
    const int start = __ldg(a.q_offsets + r);
    const int ctx = __ldg(a.context_lens + r);
    const int tok0 = blockIdx.x * kTokPerBlock;
    if (tok0 >= qlen) return;
    if (__ldg(a.q_offsets + r + 1) - start != qlen || ctx < 0 || qlen > a.max_q_len ||
        start < 0 || start + qlen > a.total_q_tokens) {
        if (threadIdx.x == 0) set_error(a.err, PKV_DEVERR_TOKENS);
        return;
    }
    const int ntok = min(kTokPerBlock, qlen - tok0);
    const int32_t* bt = a.block_table + static_cast<int64_t>(r) * a.max_pages;
    auto quant = [](float x, float s) { return int8_code(x, s); };
    for (int w = warp; w < ntok * a.num_kv_heads; w += blockDim.x / 32) {
        const int i = tok0 + w / a.num_kv_heads, h = w % a.num_kv_heads;
        const int t = start + i;
        const int pos = ctx + i;
        const int lp = pos / kPage;
        if (lp >= a.max_pages) {
            if (lane == 0) set_error(a.err, PKV_DEVERR_TABLE_RANGE);
            continue;
        }
        const int page = __ldg(bt + lp);
        if (page < 0 || page >= a.num_pages) {
            if (lane == 0) set_error(a.err, PKV_DEVERR_PAGE_RANGE);
            continue;
        }
        const int slot = pos % kPage;
        if (h == 0 && lane == 0 && a.slot_mapping)
            a.slot_mapping[t] = static_cast<int64_t>(page) * kPage + slot;
        const int64_t src = (static_cast<int64_t>(t) * a.num_kv_heads + h) * D + lane * DPL;
        const int64_t block = (static_cast<int64_t>(page) * a.num_kv_heads + h) * kPage * D;
        const int chan = h * D + lane * DPL;
        uint32_t kq[DPL], vq[DPL];
        {
            const uint16_t* ks = static_cast<const uint16_t*>(a.k_new) + src;
            const uint16_t* vs = static_cast<const uint16_t*>(a.v_new) + src;
            const float* ksc = a.k_scale + chan;
            const float* vsc = a.v_scale + chan;
            if constexpr (DPL == 4) {
                const uint2 kw = __ldg(reinterpret_cast<const uint2*>(ks));
                const uint2 vw = __ldg(reinterpret_cast<const uint2*>(vs));
                const float4 k4 = __ldg(reinterpret_cast<const float4*>(ksc));
                const float4 v4 = __ldg(reinterpret_cast<const float4*>(vsc));
                const float2 k01 = Cv::unpack(kw.x), k23 = Cv::unpack(kw.y);
                const float2 v01 = Cv::unpack(vw.x), v23 = Cv::unpack(vw.y);
                kq[0] = quant(k01.x, k4.x); kq[1] = quant(k01.y, k4.y);
                kq[2] = quant(k23.x, k4.z); kq[DPL - 1] = quant(k23.y, k4.w);
                vq[0] = quant(v01.x, v4.x); vq[1] = quant(v01.y, v4.y);
                vq[2] = quant(v23.x, v4.z); vq[DPL - 1] = quant(v23.y, v4.w);
            } else {
                const float2 k01 = Cv::unpack(__ldg(reinterpret_cast<const uint32_t*>(ks)));
                const float2 v01 = Cv::unpack(__ldg(reinterpret_cast<const uint32_t*>(vs)));
                const float2 k2 = __ldg(reinterpret_cast<const float2*>(ksc));
                const float2 v2 = __ldg(reinterpret_cast<const float2*>(vsc));
                kq[0] = quant(k01.x, k2.x); kq[DPL - 1] = quant(k01.y, k2.y);
                vq[0] = quant(v01.x, v2.x); vq[DPL - 1] = quant(v01.y, v2.y);
            }
        }
        uint8_t* kd = static_cast<uint8_t*>(a.k_cache) + block + slot * D + lane * DPL;
        uint32_t kword = 0;
#pragma unroll
        for (int e = 0; e < DPL; ++e) kword |= kq[e] << (8 * e);
        if constexpr (DPL == 4) *reinterpret_cast<uint32_t*>(kd) = kword;
        else *reinterpret_cast<uint16_t*>(kd) = static_cast<uint16_t>(kword);
        uint8_t* vd = static_cast<uint8_t*>(a.v_cache) + block + slot;
#pragma unroll
        for (int e = 0; e < DPL; ++e) vd[(lane * DPL + e) * kPage] = static_cast<uint8_t>(vq[e]);
    }
}

int launch_kv_append_int8(const AppendArgs& a, cudaStream_t stream) {
    if (a.total_q_tokens == 0 || a.num_reqs == 0) return PKV_OK;
    if (a.num_reqs > 65535) return PKV_ERR_UNSUPPORTED;
    const dim3 grid(cdiv(a.max_q_len, kTokPerBlock), a.num_reqs);
    const bool bf = a.dtype == PKV_BF16, d128 = a.head_dim == 128;
    auto* k = bf ? (d128 ? kv_append_int8_kernel<__nv_bfloat16, 128>
                         : kv_append_int8_kernel<__nv_bfloat16, 64>)
                 : (d128 ? kv_append_int8_kernel<__half, 128> : kv_append_int8_kernel<__half, 64>);
    return launch_pdl(k, grid, dim3(256), 0, stream, a) == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

// context_lens[r] += q_lens[r]: the step's tokens are now cached.  Earlier kernels on the
// stream (the attention step) read the lengths, so the update waits for them.  The next
// step's kernels read the lengths before their own dependency wait, so the update is
// fenced to the device's point of coherence before they may launch.
__global__ void __launch_bounds__(256) advance_context_kernel(const int32_t* q_lens,
                                                              int32_t* context_lens, int n) {
    pdl_wait();
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r < n) context_lens[r] += q_lens[r];
    __threadfence();
    pdl_trigger();
}

int launch_advance_context(const int32_t* q_lens, int32_t* context_lens, int num_reqs,
                           cudaStream_t stream) {
    if (num_reqs == 0) return PKV_OK;
    return launch_pdl(advance_context_kernel, dim3(cdiv(num_reqs, 256)), dim3(256), 0, stream,
                      q_lens, context_lens, num_reqs) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

// Copy-on-write of shared pages: page src[i] -> dst[i], K and V, every KV head, bit for bit
// (a page is one contiguous block of page_bytes in each pool, for 16-bit and INT8 pools
// alike).  grid.x = copy, grid.y = slice of the page; 16 bytes per thread and load.
__global__ void __launch_bounds__(256) copy_pages_kernel(const int32_t* src, const int32_t* dst,
                                                         int n, int64_t page_bytes,
                                                         int num_pages, uint8_t* k_cache,
                                                         uint8_t* v_cache, int32_t* err) {
    // earlier kernels on the stream (the previous step) may still read the destination,
    // a page that was free before this step
    pdl_wait();
    pdl_trigger();
    const int c = blockIdx.x;
    if (c >= n) return;
    const int s = __ldg(src + c), d = __ldg(dst + c);
    if (s < 0 || s >= num_pages || d < 0 || d >= num_pages) {
        if (threadIdx.x == 0 && blockIdx.y == 0) set_error(err, PKV_DEVERR_PAGE_RANGE);
        return;
    }
    if (s == d) return;
    const int64_t words = page_bytes / 16;
    const uint4* ks = reinterpret_cast<const uint4*>(k_cache + s * page_bytes);
    const uint4* vs = reinterpret_cast<const uint4*>(v_cache + s * page_bytes);
    uint4* kd = reinterpret_cast<uint4*>(k_cache + d * page_bytes);
    uint4* vd = reinterpret_cast<uint4*>(v_cache + d * page_bytes);
    for (int64_t w = blockIdx.y * blockDim.x + threadIdx.x; w < words;
         w += static_cast<int64_t>(gridDim.y) * blockDim.x) {
        const uint4 kw = ks[w], vw = vs[w];
        kd[w] = kw;
        vd[w] = vw;
    }
}

int launch_copy_pages(const int32_t* src, const int32_t* dst, int n, int64_t page_bytes,
                      int num_pages, void* k_cache, void* v_cache, int32_t* err,
                      cudaStream_t stream) {
    if (n <= 0) return PKV_OK;
    const int64_t words = page_bytes / 16;
    const int slices = static_cast<int>(std::min<int64_t>(8, (words + 255) / 256));
    const dim3 grid(n, slices);
    return launch_pdl(copy_pages_kernel, grid, dim3(256), 0, stream, src, dst, n, page_bytes,
                      num_pages, static_cast<uint8_t*>(k_cache), static_cast<uint8_t*>(v_cache),
                      err) == cudaSuccess
               ? PKV_OK
               : PKV_ERR_CUDA;
}

int launch_kv_append(const AppendArgs& a, cudaStream_t stream) {
    if (a.total_q_tokens == 0 || a.num_reqs == 0) return PKV_OK;
    if (a.num_reqs > 65535) return PKV_ERR_UNSUPPORTED;
    const dim3 grid(cdiv(a.max_q_len, kTokPerBlock), a.num_reqs);
    const cudaError_t e = a.head_dim == 128
                              ? launch_pdl(kv_append_kernel<128>, grid, dim3(256), 0, stream, a)
                              : launch_pdl(kv_append_kernel<64>, grid, dim3(256), 0, stream, a);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

}  // namespace pkv
