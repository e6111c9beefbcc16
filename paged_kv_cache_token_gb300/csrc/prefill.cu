// Tensor-core prefill path (q_len > 1 rows): not enabled yet; every row takes the
// streaming path until this kernel lands.
#include "common.cuh"
#include "launch.h"

namespace pkv {

int launch_prefill(const StepArgs& a, cudaStream_t stream, cudaEvent_t e0, cudaEvent_t e1) {
    (void)a;
    (void)stream;
    (void)e0;
    (void)e1;
    return PKV_ERR_UNSUPPORTED;
}

}  // namespace pkv
