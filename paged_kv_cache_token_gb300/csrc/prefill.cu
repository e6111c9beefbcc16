// Prefill-chunk path of the paged attention step, host side: the tensor maps the
// tensor-core kernels load with, and the dispatch between them.
//
// Rows of a request that advances by many tokens (a chunked prefill) form a causal block:
// query row i at position ctx + i scores keys 0..ctx+i (hotelren.com/news/6181127 §1.1,
// §2.1: row softmax of the masked score matrix, times V; §2.1 also notes that blocked
// computation avoids materialising the S x S matrix).  A chunk reads the earlier chunks'
// K/V like a decode and writes its own (niuwancheng.cn "11. chunked prefill and unified
// scheduling"), so the keys of every tile come from the pages through the block table.
// Prefill is a dense contraction (wmrh.cn §2.2, hotelren.com §1.2), so QK^T and PV run on
// tcgen05 with fp32 accumulators in tensor memory: prefill_pair.cu over 16-bit pages,
// prefill_q8.cu over INT8 pages, each CTA working on two chains of 128 query rows (two
// query heads of a KV group, or two query tiles of one head; see prefill_tile.cuh).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "launch.h"

namespace pkv {

namespace {
constexpr int kBM = 128;          // query rows per tile (the Q box height)
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

int launch_prefill(const StepArgs& a, cudaStream_t stream, cudaEvent_t e0, cudaEvent_t e1) {
    if (a.kv_int8) return launch_prefill_q8(a, stream, e0, e1);
    return launch_prefill_pair(a, stream, e0, e1);
}

}  // namespace pkv
