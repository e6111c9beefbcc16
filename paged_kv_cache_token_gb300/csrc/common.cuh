// Shared device helpers for the paged-KV attention library (sm_103a).
// PTX wrappers for mbarriers and bulk async copies, 16-bit float traits, error flags.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

constexpr int kPage = PKV_PAGE_SIZE;  // tokens per page
constexpr uint32_t kFull = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;
// Bounded waits: ~2^24 polls of an mbarrier is far beyond any copy latency; after it the
// kernel records PKV_DEVERR_TIMEOUT and stops instead of spinning forever.
constexpr uint32_t kWaitLimit = 1u << 24;

// ---------------------------------------------------------------- 16-bit float traits
template <typename T> struct F16;
template <> struct F16<__nv_bfloat16> {
    // two packed bf16 -> two floats (exact: bf16 is the top half of an fp32)
    static __device__ __forceinline__ float2 unpack(uint32_t w) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // round to nearest even
        return *reinterpret_cast<uint32_t*>(&h);
    }
    static __device__ __forceinline__ float to_float(uint16_t b) {
        return __uint_as_float(static_cast<uint32_t>(b) << 16);
    }
};
template <> struct F16<__half> {
    static __device__ __forceinline__ float2 unpack(uint32_t w) {
        __half2 h = *reinterpret_cast<__half2*>(&w);
        return __half22float2(h);
    }
    static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t*>(&h);
    }
    static __device__ __forceinline__ float to_float(uint16_t b) {
        return __half2float(__ushort_as_half(b));
    }
};

// ---------------------------------------------------------------- error flag
__device__ __forceinline__ void set_error(int32_t* flag, int32_t bits) {
    if (flag) atomicOr(flag, bits);
}

// ---------------------------------------------------------------- shared-memory addresses
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}
// Make initialised barriers visible to the asynchronous (TMA / tensor-core) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Wait for the phase with the given parity to complete; false after kWaitLimit polls.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < kWaitLimit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}
// Whole-warp wait: lane 0 polls, the other lanes stay parked in the warp barrier instead of
// spinning on the mbarrier; every lane returns lane 0's result, converged.
__device__ __forceinline__ bool mbar_wait_warp(uint64_t* bar, uint32_t parity) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity) ? 1 : 0;
    __syncwarp();
    return __shfl_sync(kFull, ok, 0) != 0;
}

// Generic-proxy shared-memory writes of this thread -> ordered before later async-proxy
// (bulk copy) accesses of the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// One INT8 code of a KV element: the element divided by its channel's fixed scale (IEEE
// division), rounded to the nearest integer (ties to even), clamped to [-127, 127], as the
// code's two's-complement byte.  The quantiser of wmrh.cn/news/64708 §4.3, the same in
// every kernel that writes INT8 pages.
__device__ __forceinline__ uint32_t int8_code(float x, float s) {
    const int c = max(-127, min(127, __float2int_rn(__fdiv_rn(x, s))));
    return static_cast<uint32_t>(c) & 0xFFu;
}

// ---------------------------------------------------------------- bulk async copy (TMA, 1-D)
// Global -> shared copy of `bytes` (multiple of 16, both addresses 16-byte aligned) that
// signals completion on `bar` through the transaction count.
__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                         uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_u32(smem_dst)), "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Same, with an L2 eviction policy (from l2_policy_evict_first and the like) for the source
// lines.
__device__ __forceinline__ void bulk_g2s_hint(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                              uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        ::"r"(smem_u32(smem_dst)), "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}
// L2 policy: lines read through it are the first evicted (a stream read once, so it does not
// push out data that is read again soon).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ---------------------------------------------------------------- programmatic dependent launch
// Kernels of one step are launched so each may start while its predecessor drains.
// pdl_wait: block until every preceding kernel in the stream has completed and its memory
// is visible (a no-op for a launch without the attribute).  pdl_trigger: allow the next
// kernel in the stream to be scheduled.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- misc
__device__ __forceinline__ float fast_exp2(float x) { return exp2f(x); }

__host__ __device__ constexpr int cdiv(int a, int b) { return (a + b - 1) / b; }

}  // namespace pkv
