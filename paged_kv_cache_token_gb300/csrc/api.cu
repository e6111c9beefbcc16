// C ABI of libpkv.so: argument checks on the host, then kernel launches on the caller's
// stream.  Declarations and the contract of every entry point are in include/pkv.h.
#include <algorithm>
#include <atomic>
#include <climits>
#include <random>
#include <cstdint>

#include "launch.h"
#include "pkv.h"

namespace {

constexpr int kMaxDevices = 64;

int num_sms_current_device() {
    static int cache[kMaxDevices] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return -1;
        cache[dev] = n;
    }
    return cache[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Whether p is device memory (or managed memory, which the device maps as its own).  Pinned
// host memory is mapped into the device's address space too (unified addressing), and the
// kernels' plain loads and stores reach it over the CPU-GPU link -- but the tensor-memory
// accelerator copies of the prefill kernels need device memory.
bool device_memory(const void* p) {
    cudaPointerAttributes at{};
    if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
        cudaGetLastError();  // an unregistered host pointer: clear the sticky-free error
        return false;
    }
    return at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged;
}

// Checks shared by both calls.  Returns PKV_OK or the first problem found.
int check_desc(const pkv_step_desc* d) {
    if (!d) return PKV_ERR_INVALID_ARG;
    if (d->page_size != PKV_PAGE_SIZE) return PKV_ERR_INVALID_ARG;
    if (d->num_reqs < 0 || d->total_q_tokens < 0 || d->max_q_len < 0 ||
        d->max_context_len < 0 || d->num_pages <= 0 || d->max_pages_per_req <= 0)
        return PKV_ERR_INVALID_ARG;
    if (d->num_q_heads <= 0 || d->num_kv_heads <= 0) return PKV_ERR_INVALID_ARG;
    if (d->dtype != PKV_BF16 && d->dtype != PKV_FP16) return PKV_ERR_UNSUPPORTED;
    if (d->head_dim != 64 && d->head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (d->num_q_heads % d->num_kv_heads) return PKV_ERR_UNSUPPORTED;
    const int g = d->num_q_heads / d->num_kv_heads;
    if (g != 1 && g != 2 && g != 4 && g != 8) return PKV_ERR_UNSUPPORTED;
    if (d->num_reqs == 0 && d->total_q_tokens != 0) return PKV_ERR_INVALID_ARG;
    if (d->total_q_tokens > 0 && d->max_q_len == 0) return PKV_ERR_INVALID_ARG;
    if (static_cast<int64_t>(d->max_q_len) > d->total_q_tokens) return PKV_ERR_INVALID_ARG;
    // a request of max_q_len tokens cannot fit a block-table row at all
    if (static_cast<int64_t>(d->max_q_len) > static_cast<int64_t>(d->max_pages_per_req) * 16)
        return PKV_ERR_CAPACITY;
    // positions are int32 on the device
    if (static_cast<int64_t>(d->max_context_len) + d->max_q_len >= INT_MAX / 2)
        return PKV_ERR_CAPACITY;
    if (static_cast<int64_t>(d->num_pages) * d->num_kv_heads * 16 * d->head_dim >
        (int64_t(1) << 40))
        return PKV_ERR_INVALID_ARG;
    // the prefill's tensor maps address pool rows (page x KV head x 16 tokens) with 32-bit
    // coordinates
    if (static_cast<int64_t>(d->num_pages) * d->num_kv_heads * 16 > INT_MAX)
        return PKV_ERR_UNSUPPORTED;
    if (d->num_reqs > 0 &&
        (!d->q_lens || !d->q_offsets || !d->context_lens || !d->block_table))
        return PKV_ERR_INVALID_ARG;
    return PKV_OK;
}

// Requests with at least this many new tokens take the tensor-core prefill path (128-row
// query tiles); shorter multi-token requests run row by row on the streaming path.
int prefill_min_q() { return 16; }

// Tags of attention calls (see StepArgs::epoch): 40-bit values, never 0, from a start chosen
// at random per process so that a workspace's earlier contents are unlikely to hold one.
unsigned long long next_epoch() {
    static std::atomic<unsigned long long> counter{[] {
        std::random_device rd;
        return (static_cast<unsigned long long>(rd()) << 20) ^ rd();
    }()};
    const unsigned long long kMask = (1ull << 40) - 1;
    unsigned long long e;
    do {
        e = counter.fetch_add(1, std::memory_order_relaxed) & kMask;
    } while (e == 0);
    return e;
}

thread_local cudaEvent_t g_events[2][2] = {{nullptr, nullptr}, {nullptr, nullptr}};

// Requests with at least this many new tokens take the tensor-core prefill path (16-bit
// and INT8 pools alike).
int prefill_min_q_for(const pkv_step_desc*, bool) { return prefill_min_q(); }

pkv::WorkspaceLayout layout_for(const pkv_step_desc* d, int num_sms, bool int8 = false) {
    return pkv::workspace_layout(d->num_reqs, d->num_q_heads, d->num_kv_heads, d->head_dim,
                                 d->total_q_tokens, d->max_q_len, d->max_context_len, num_sms,
                                 prefill_min_q_for(d, int8));
}

int kv_append_impl(const pkv_step_desc* desc, const void* k_new, const void* v_new,
                   void* k_cache, void* v_cache, int64_t* slot_mapping_out,
                   int32_t* dev_err_flag, void* stream, const float* k_scale,
                   const float* v_scale) {
    const int rc = check_desc(desc);
    if (rc != PKV_OK) return rc;
    if (desc->total_q_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache))
        return PKV_ERR_INVALID_ARG;
    if (slot_mapping_out && (reinterpret_cast<uintptr_t>(slot_mapping_out) & 7u))
        return PKV_ERR_INVALID_ARG;
    const bool int8 = k_scale != nullptr;
    if (int8 && (!v_scale || !aligned16(k_scale) || !aligned16(v_scale)))
        return PKV_ERR_INVALID_ARG;
    pkv::AppendArgs a{};
    a.num_reqs = desc->num_reqs;
    a.num_kv_heads = desc->num_kv_heads;
    a.head_dim = desc->head_dim;
    a.num_pages = desc->num_pages;
    a.max_pages = desc->max_pages_per_req;
    a.total_q_tokens = desc->total_q_tokens;
    a.max_q_len = desc->max_q_len;
    a.dtype = desc->dtype;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.q_lens = desc->q_lens;
    a.q_offsets = desc->q_offsets;
    a.context_lens = desc->context_lens;
    a.block_table = desc->block_table;
    a.k_new = k_new;
    a.v_new = v_new;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.slot_mapping = slot_mapping_out;
    a.err = dev_err_flag;
    return int8 ? pkv::launch_kv_append_int8(a, static_cast<cudaStream_t>(stream))
                : pkv::launch_kv_append(a, static_cast<cudaStream_t>(stream));
}

}  // namespace

extern "C" {

int pkv_version(void) { return 100; }

const char* pkv_status_string(int status) {
    switch (status) {
        case PKV_OK: return "PKV_OK";
        case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
        case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
        case PKV_ERR_CAPACITY: return "PKV_ERR_CAPACITY";
        case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE";
        case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
        case PKV_ERR_DEVICE: return "PKV_ERR_DEVICE";
        case PKV_ERR_NO_PAGES: return "PKV_ERR_NO_PAGES";
        default: return "PKV_UNKNOWN_STATUS";
    }
}

int pkv_kv_append(const pkv_step_desc* desc, const void* k_new, const void* v_new,
                  void* k_cache, void* v_cache, int64_t* slot_mapping_out,
                  int32_t* dev_err_flag, void* stream) {
    return kv_append_impl(desc, k_new, v_new, k_cache, v_cache, slot_mapping_out, dev_err_flag,
                          stream, nullptr, nullptr);
}

int pkv_kv_append_int8(const pkv_step_desc* desc, const void* k_new, const void* v_new,
                       const float* k_scale, const float* v_scale, int8_t* k_cache,
                       int8_t* v_cache, int64_t* slot_mapping_out, int32_t* dev_err_flag,
                       void* stream) {
    if (!k_scale) return PKV_ERR_INVALID_ARG;
    return kv_append_impl(desc, k_new, v_new, k_cache, v_cache, slot_mapping_out, dev_err_flag,
                          stream, k_scale, v_scale);
}

int pkv_copy_pages(const pkv_step_desc* desc, const int32_t* src_pages,
                   const int32_t* dst_pages, int32_t num_copies, void* k_cache, void* v_cache,
                   int kv_int8, int32_t* dev_err_flag, void* stream) {
    if (!desc || num_copies < 0) return PKV_ERR_INVALID_ARG;
    if (desc->page_size != PKV_PAGE_SIZE || desc->num_pages <= 0 || desc->num_kv_heads <= 0)
        return PKV_ERR_INVALID_ARG;
    if (desc->dtype != PKV_BF16 && desc->dtype != PKV_FP16) return PKV_ERR_UNSUPPORTED;
    if (desc->head_dim != 64 && desc->head_dim != 128) return PKV_ERR_UNSUPPORTED;
    if (kv_int8 != 0 && kv_int8 != 1) return PKV_ERR_INVALID_ARG;
    if (num_copies == 0) return PKV_OK;
    if (!src_pages || !dst_pages || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
    if (!aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(src_pages) & 3u) ||
        (reinterpret_cast<uintptr_t>(dst_pages) & 3u))
        return PKV_ERR_INVALID_ARG;
    const int64_t page_bytes = static_cast<int64_t>(desc->num_kv_heads) * PKV_PAGE_SIZE *
                               desc->head_dim * (kv_int8 ? 1 : 2);
    return pkv::launch_copy_pages(src_pages, dst_pages, num_copies, page_bytes, desc->num_pages,
                                  k_cache, v_cache, dev_err_flag,
                                  static_cast<cudaStream_t>(stream));
}

int pkv_advance_context(const pkv_step_desc* desc, int32_t* context_lens, void* stream) {
    const int rc = check_desc(desc);
    if (rc != PKV_OK) return rc;
    if (desc->num_reqs == 0) return PKV_OK;
    if (!context_lens || (reinterpret_cast<uintptr_t>(context_lens) & 3u))
        return PKV_ERR_INVALID_ARG;
    return pkv::launch_advance_context(desc->q_lens, context_lens, desc->num_reqs,
                                       static_cast<cudaStream_t>(stream));
}

size_t pkv_attention_workspace_bytes(const pkv_step_desc* desc) {
    if (check_desc(desc) != PKV_OK) return 0;
    const int sms = num_sms_current_device();
    if (sms <= 0) return 0;
    return layout_for(desc, sms).total;
}

size_t pkv_attention_workspace_bytes_int8(const pkv_step_desc* desc) {
    if (check_desc(desc) != PKV_OK) return 0;
    const int sms = num_sms_current_device();
    if (sms <= 0) return 0;
    return layout_for(desc, sms, true).total;
}

}  // extern "C"

namespace {

// What one attention call launches: the plan and the attention kernels (a whole step), the
// plan alone, or the attention kernels over a plan already in the workspace.
enum class Phase { kPlanAndRun, kPlanOnly, kRunOnly };

// New K/V rows for an attention call that appends them itself (pkv_append_attention).
struct FusedAppend {
    const void* k_new;
    const void* v_new;
    int64_t* slot_mapping;
};

int attention_impl(const pkv_step_desc* desc, const void* q, const void* k_cache,
                   const void* v_cache, void* out, float scale, void* workspace,
                   size_t workspace_bytes, int32_t* dev_err_flag, void* stream,
                   const float* k_scale, const float* v_scale,
                   Phase phase = Phase::kPlanAndRun, const FusedAppend* fused = nullptr) {
    int rc = check_desc(desc);
    if (rc != PKV_OK) return rc;
    if (desc->total_q_tokens == 0) return PKV_OK;
    const bool int8 = k_scale != nullptr;
    if (phase != Phase::kPlanOnly) {
        if (!q || !k_cache || !v_cache || !out) return PKV_ERR_INVALID_ARG;
        if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
            return PKV_ERR_INVALID_ARG;
        if (int8 && (!v_scale || !aligned16(k_scale) || !aligned16(v_scale)))
            return PKV_ERR_INVALID_ARG;
    }
    const int sms = num_sms_current_device();
    if (sms <= 0) return PKV_ERR_CUDA;
    const pkv::WorkspaceLayout lay = layout_for(desc, sms, int8);
    if (!workspace || workspace_bytes < lay.total) return PKV_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return PKV_ERR_WORKSPACE;
    // steps that can have prefill tiles read q with TMA: it must be device memory
    if (phase != Phase::kPlanOnly && lay.max_tiles > 0 && !device_memory(q))
        return PKV_ERR_INVALID_ARG;

    pkv::StepArgs a{};
    a.num_reqs = desc->num_reqs;
    a.num_q_heads = desc->num_q_heads;
    a.num_kv_heads = desc->num_kv_heads;
    a.head_dim = desc->head_dim;
    a.num_pages = desc->num_pages;
    a.max_pages = desc->max_pages_per_req;
    a.total_q_tokens = desc->total_q_tokens;
    a.max_q_len = desc->max_q_len;
    a.max_context_len = desc->max_context_len;
    a.dtype = desc->dtype;
    a.num_sms = sms;
    a.q_lens = desc->q_lens;
    a.q_offsets = desc->q_offsets;
    a.context_lens = desc->context_lens;
    a.block_table = desc->block_table;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.out = out;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.ws = static_cast<uint8_t*>(workspace);
    a.lay = lay;
    a.prefill_min_q = prefill_min_q_for(desc, int8);
    a.heads_per_tile = pkv::prefill_heads_per_tile(desc->num_q_heads, desc->num_kv_heads);
    a.err = dev_err_flag;
    a.kv_int8 = int8 ? 1 : 0;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // with both paths possible the prefill goes first and the decode fills the SMs its last
    // wave leaves idle
    a.overlap = lay.max_tiles > 0 && lay.max_items > 0 ? 1 : 0;
    a.plan_wait_first = phase == Phase::kPlanOnly ? 1 : 0;
    a.plan_ready = phase == Phase::kRunOnly ? 1 : 0;
    a.self_plan = lay.self_plan;
    a.epoch = a.self_plan ? next_epoch() : 0;
    if (fused) {
        a.fused_append = 1;
        a.k_new = fused->k_new;
        a.v_new = fused->v_new;
        a.slot_mapping = fused->slot_mapping;
    }
    // a self-planned step has nothing to plan ahead: its decode kernel plans for itself
    if (phase != Phase::kRunOnly && !a.self_plan && (rc = pkv::launch_plan(a, s)) != PKV_OK)
        return rc;
    if (phase == Phase::kPlanOnly) return PKV_OK;
    if (a.overlap &&
        (rc = pkv::launch_prefill(a, s, g_events[1][0], g_events[1][1])) != PKV_OK)
        return rc;
    if ((rc = pkv::launch_decode(a, s, g_events[0][0], g_events[0][1])) != PKV_OK) return rc;
    if (!a.overlap && lay.max_tiles > 0 &&
        (rc = pkv::launch_prefill(a, s, g_events[1][0], g_events[1][1])) != PKV_OK)
        return rc;
    return PKV_OK;
}

}  // namespace

extern "C" {

int pkv_paged_attention_step(const pkv_step_desc* desc, const void* q, const void* k_cache,
                             const void* v_cache, void* out, float scale, void* workspace,
                             size_t workspace_bytes, int32_t* dev_err_flag, void* stream) {
    return attention_impl(desc, q, k_cache, v_cache, out, scale, workspace, workspace_bytes,
                          dev_err_flag, stream, nullptr, nullptr);
}

int pkv_paged_attention_step_int8(const pkv_step_desc* desc, const void* q,
                                  const int8_t* k_cache, const int8_t* v_cache,
                                  const float* k_scale, const float* v_scale, void* out,
                                  float scale, void* workspace, size_t workspace_bytes,
                                  int32_t* dev_err_flag, void* stream) {
    if (!k_scale) return PKV_ERR_INVALID_ARG;
    return attention_impl(desc, q, k_cache, v_cache, out, scale, workspace, workspace_bytes,
                          dev_err_flag, stream, k_scale, v_scale);
}

int pkv_append_attention(const pkv_step_desc* desc, const void* k_new, const void* v_new,
                         void* k_cache, void* v_cache, int64_t* slot_mapping_out, const void* q,
                         void* out, float scale, void* workspace, size_t workspace_bytes,
                         int32_t* dev_err_flag, void* stream) {
    int rc = check_desc(desc);
    if (rc != PKV_OK) return rc;
    if (desc->total_q_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return PKV_ERR_INVALID_ARG;
    if (slot_mapping_out && (reinterpret_cast<uintptr_t>(slot_mapping_out) & 7u))
        return PKV_ERR_INVALID_ARG;
    const int sms = num_sms_current_device();
    if (sms <= 0) return PKV_ERR_CUDA;
    if (layout_for(desc, sms).self_plan) {
        // one decode grid appends and attends (after the argument checks of both calls)
        if (!k_cache || !v_cache || !aligned16(k_cache) || !aligned16(v_cache))
            return PKV_ERR_INVALID_ARG;
        const FusedAppend f{k_new, v_new, slot_mapping_out};
        return attention_impl(desc, q, k_cache, v_cache, out, scale, workspace, workspace_bytes,
                              dev_err_flag, stream, nullptr, nullptr, Phase::kPlanAndRun, &f);
    }
    if ((rc = kv_append_impl(desc, k_new, v_new, k_cache, v_cache, slot_mapping_out,
                             dev_err_flag, stream, nullptr, nullptr)) != PKV_OK)
        return rc;
    return attention_impl(desc, q, k_cache, v_cache, out, scale, workspace, workspace_bytes,
                          dev_err_flag, stream, nullptr, nullptr);
}

int pkv_append_attention_int8(const pkv_step_desc* desc, const void* k_new, const void* v_new,
                              const float* k_scale, const float* v_scale, int8_t* k_cache,
                              int8_t* v_cache, int64_t* slot_mapping_out, const void* q,
                              void* out, float scale, void* workspace, size_t workspace_bytes,
                              int32_t* dev_err_flag, void* stream) {
    int rc = check_desc(desc);
    if (rc != PKV_OK) return rc;
    if (desc->total_q_tokens == 0) return PKV_OK;
    if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return PKV_ERR_INVALID_ARG;
    if (!k_scale || !v_scale || !aligned16(k_scale) || !aligned16(v_scale))
        return PKV_ERR_INVALID_ARG;
    if (slot_mapping_out && (reinterpret_cast<uintptr_t>(slot_mapping_out) & 7u))
        return PKV_ERR_INVALID_ARG;
    const int sms = num_sms_current_device();
    if (sms <= 0) return PKV_ERR_CUDA;
    if (layout_for(desc, sms, true).self_plan) {
        // one decode grid quantises, appends and attends
        if (!k_cache || !v_cache || !aligned16(k_cache) || !aligned16(v_cache))
            return PKV_ERR_INVALID_ARG;
        const FusedAppend f{k_new, v_new, slot_mapping_out};
        return attention_impl(desc, q, k_cache, v_cache, out, scale, workspace, workspace_bytes,
                              dev_err_flag, stream, k_scale, v_scale, Phase::kPlanAndRun, &f);
    }
    if ((rc = kv_append_impl(desc, k_new, v_new, k_cache, v_cache, slot_mapping_out,
                             dev_err_flag, stream, k_scale, v_scale)) != PKV_OK)
        return rc;
    return attention_impl(desc, q, k_cache, v_cache, out, scale, workspace, workspace_bytes,
                          dev_err_flag, stream, k_scale, v_scale);
}

int pkv_plan_attention(const pkv_step_desc* desc, void* workspace, size_t workspace_bytes,
                       int32_t* dev_err_flag, void* stream) {
    return attention_impl(desc, nullptr, nullptr, nullptr, nullptr, 1.f, workspace,
                          workspace_bytes, dev_err_flag, stream, nullptr, nullptr,
                          Phase::kPlanOnly);
}

int pkv_paged_attention_run(const pkv_step_desc* desc, const void* q, const void* k_cache,
                            const void* v_cache, void* out, float scale, void* workspace,
                            size_t workspace_bytes, int32_t* dev_err_flag, void* stream) {
    return attention_impl(desc, q, k_cache, v_cache, out, scale, workspace, workspace_bytes,
                          dev_err_flag, stream, nullptr, nullptr, Phase::kRunOnly);
}

int pkv_paged_attention_run_int8(const pkv_step_desc* desc, const void* q,
                                 const int8_t* k_cache, const int8_t* v_cache,
                                 const float* k_scale, const float* v_scale, void* out,
                                 float scale, void* workspace, size_t workspace_bytes,
                                 int32_t* dev_err_flag, void* stream) {
    if (!k_scale) return PKV_ERR_INVALID_ARG;
    return attention_impl(desc, q, k_cache, v_cache, out, scale, workspace, workspace_bytes,
                          dev_err_flag, stream, k_scale, v_scale, Phase::kRunOnly);
}

int pkv_set_kernel_events(int which, void* start, void* stop) {
    if (which != 0 && which != 1) return PKV_ERR_INVALID_ARG;
    g_events[which][0] = static_cast<cudaEvent_t>(start);
    g_events[which][1] = static_cast<cudaEvent_t>(stop);
    return PKV_OK;
}

int pkv_read_device_error(const int32_t* dev_err_flag, int32_t* host_value, void* stream) {
    if (!dev_err_flag || !host_value) return PKV_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(host_value, dev_err_flag, sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
        cudaSuccess)
        return PKV_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return PKV_ERR_CUDA;
    return *host_value == 0 ? PKV_OK : PKV_ERR_DEVICE;
}

}  // extern "C"
