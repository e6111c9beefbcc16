// Attention step whose scratch memory is a fixed array inside the library, for callers
// that cannot allocate device memory at call time (see pkv_paged_attention_step_static_ws
// in pkv.h).  No cudaMalloc, cudaFree or allocating library routine is called here.
#include <cuda_runtime.h>

#include <mutex>

#include "pkv.h"

namespace {

// One copy per device that loads the library; kept until the process exits.
static __device__ __align__(256) unsigned char g_static_ws[PKV_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_static_ws_addr[kMaxDevices] = {nullptr};

// Device address of g_static_ws on the current device.  In host code the symbol name is
// only a host-side handle, so the address is looked up once per device (with that device
// current) and cached.  Returns nullptr when the lookup fails.
void* static_ws_address() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_static_ws_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return nullptr;
        g_static_ws_addr[dev] = p;
    }
    return g_static_ws_addr[dev];
}

}  // namespace

extern "C" int pkv_paged_attention_step_static_ws(const pkv_step_desc* desc, const void* q,
                                                  const void* k_cache, const void* v_cache,
                                                  void* out, float scale,
                                                  int32_t* dev_err_flag, void* stream) {
    if (!desc) return PKV_ERR_INVALID_ARG;
    if (desc->total_q_tokens == 0)  // same early exit as the allocating entry point
        return pkv_paged_attention_step(desc, q, k_cache, v_cache, out, scale, nullptr, 0,
                                        dev_err_flag, stream);
    const size_t need = pkv_attention_workspace_bytes(desc);
    if (need == 0)  // invalid description: let the regular checks name the error
        return pkv_paged_attention_step(desc, q, k_cache, v_cache, out, scale, nullptr, 0,
                                        dev_err_flag, stream);
    if (need > PKV_STATIC_WORKSPACE_BYTES) return PKV_ERR_WORKSPACE;
    void* ws = static_ws_address();
    if (!ws) return PKV_ERR_CUDA;
    return pkv_paged_attention_step(desc, q, k_cache, v_cache, out, scale, ws,
                                    PKV_STATIC_WORKSPACE_BYTES, dev_err_flag, stream);
}
