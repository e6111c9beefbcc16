// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

namespace pkv {

struct AppendArgs {
    int num_reqs, num_kv_heads, head_dim, num_pages, max_pages, total_q_tokens, max_q_len;
    int dtype;                 // of k_new / v_new
    const float* k_scale;      // [Hkv][D] per-channel INT8 scales (INT8 pools only)
    const float* v_scale;
    const int32_t* q_lens;
    const int32_t* q_offsets;
    const int32_t* context_lens;
    const int32_t* block_table;
    const void* k_new;
    const void* v_new;
    void* k_cache;
    void* v_cache;
    int64_t* slot_mapping;
    int32_t* err;
};

// Workspace layout for one attention step, all offsets 256-byte aligned.
//   ctrl      int32[64]        [0] decode work counter, [1] decode items, [2] decode rows,
//                              [3] pages per split, [9] prefill tiles
//   req_info  int4[num_reqs]   {first decode row, decode rows, q_len, first prefill tile}
//   rows      int4[max_rows]   decode rows {token, slot of the first split, keys, splits}
//   items     2 x int4[max_items]  work queue, largest first: {token, KV head | split << 16,
//                              first page, pages}, {keys, splits, request, slot of split 0}
//   tiles     int4[max_tiles]  prefill tiles {request, q tile, query head (pair), 0}
//   part_ml   float2[max_items * G]      per slot (running max in log2 units, sum)
//   part_o    float[max_items * G * D]   per slot un-normalised outputs
//   (a self-planned step -- self_plan below -- uses req_info for {token, first segment
//   page, keys, pages per head} of every request, ctrl[1] / [2] / [4] for the total pages,
//   the requests and the warps sharing them, and two partial slots per decode warp)
struct WorkspaceLayout {
    size_t ctrl, req_info, rows, items, tiles, part_ml, part_o;
    size_t pair_ctr;  // self-planned steps: an arrival count per (request, KV head)
    size_t total;
    int max_rows, max_items, max_tiles, target_items;
    int self_plan;  // every request advances by <= 1 token, at most kSelfPlanMaxReqs of them
};

// requests a decode CTA plans for itself (one int per request in three shared arrays)
constexpr int kSelfPlanMaxReqs = 256;

struct StepArgs {
    int num_reqs, num_q_heads, num_kv_heads, head_dim, num_pages, max_pages;
    int total_q_tokens, max_q_len, max_context_len, dtype;
    int num_sms;
    const int32_t* q_lens;
    const int32_t* q_offsets;
    const int32_t* context_lens;
    const int32_t* block_table;
    const void* q;
    const void* k_cache;
    const void* v_cache;
    void* out;
    float scale_log2;  // scale * log2(e): scores are kept in base-2 units
    uint8_t* ws;
    WorkspaceLayout lay;
    int prefill_min_q;  // requests with q_len >= this go to the tensor-core prefill path
    int heads_per_tile; // query heads per prefill tile (2 when a KV group has an even size)
    int32_t* err;
    int kv_int8;        // K/V pools hold INT8 codes with per-channel scales
    // the prefill grid runs before the decode grid of this step: the prefill lets the decode
    // launch once its CTAs have all started, and the decode waits for it at its end
    int overlap;
    // the plan waits for the preceding kernel before it reads the lengths: set when the plan
    // is launched on its own (pkv_plan_attention), where that kernel may be the one that
    // wrote them (pkv_advance_context); a full step's plan follows kv_append instead, which
    // waited for that writer before letting the plan start
    int plan_wait_first;
    // the work list in the workspace was planned before this call (pkv_paged_attention_run):
    // the decode kernel may read it (and the block table) before its dependency wait.  The
    // plan kernel of pkv_plan_attention never lets its successor launch before it completes,
    // so the list is complete by the time any later kernel launches.
    int plan_ready;
    // the decode kernel plans the step itself (WorkspaceLayout::self_plan): no plan launch
    int self_plan;
    // this call's tag for the self-planned step's chunk counter: 40 bits, never 0, a new
    // value for every call (a CUDA graph replays the captured values; the combine parks the
    // counter at 0 after every call, so a replayed tag still starts afresh)
    unsigned long long epoch;
    // self-planned steps over 16-bit pools may also append the step's new K/V rows
    // (pkv_append_attention): the warp that reads a (request, KV head)'s last page writes the
    // request's new row into it first
    int fused_append;
    const void* k_new;  // [T][Hkv][D], with fused_append
    const void* v_new;
    int64_t* slot_mapping;  // [T] or null, with fused_append
    const float* k_scale;  // [Hkv][D], INT8 pools only
    const float* v_scale;
};

WorkspaceLayout workspace_layout(int num_reqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int total_q_tokens, int max_q_len, int max_context_len,
                                 int num_sms, int prefill_min_q);
// What the second chain of a prefill CTA is: 2 = the next query head of the KV group (an
// even group), 1 = the next 128-row query tile of the same head (one head per KV head)
inline int prefill_heads_per_tile(int num_q_heads, int num_kv_heads) {
    return ((num_q_heads / num_kv_heads) % 2 == 0) ? 2 : 1;
}

// Launch with the programmatic-stream-serialization attribute (see pdl_wait / pdl_trigger).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

int launch_kv_append(const AppendArgs& a, cudaStream_t stream);
int launch_kv_append_int8(const AppendArgs& a, cudaStream_t stream);
int launch_copy_pages(const int32_t* src, const int32_t* dst, int n, int64_t page_bytes,
                      int num_pages, void* k_cache, void* v_cache, int32_t* err,
                      cudaStream_t stream);
int launch_advance_context(const int32_t* q_lens, int32_t* context_lens, int num_reqs,
                           cudaStream_t stream);
int launch_plan(const StepArgs& a, cudaStream_t stream);
// ev_start / ev_stop (may be null) are recorded around the main kernel only.
int launch_decode(const StepArgs& a, cudaStream_t stream, cudaEvent_t ev_start,
                  cudaEvent_t ev_stop);
int launch_prefill(const StepArgs& a, cudaStream_t stream, cudaEvent_t ev_start,
                   cudaEvent_t ev_stop);
int launch_prefill_pair(const StepArgs& a, cudaStream_t stream, cudaEvent_t ev_start,
                        cudaEvent_t ev_stop);
// INT8 pools
int launch_prefill_q8(const StepArgs& a, cudaStream_t stream, cudaEvent_t ev_start,
                      cudaEvent_t ev_stop);
// Q ([T][Hq][D], 128-row boxes) and K/V pool (16-row page boxes) tensor maps, 128-byte
// swizzle, 64-element-wide boxes.
bool make_prefill_maps(const StepArgs& a, CUtensorMap* mq, CUtensorMap* mk, CUtensorMap* mv);
bool make_q_map(const StepArgs& a, CUtensorMap* mq);

}  // namespace pkv
