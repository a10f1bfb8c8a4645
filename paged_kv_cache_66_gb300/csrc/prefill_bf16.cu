// Paged prefill instantiations for bf16 pools.
#include "prefill_dispatch.cuh"

namespace pa {

cudaError_t launch_prefill_bf16(const PrefillParams& p, const void* k_pool, const void* v_pool, int d, int max_q,
                               cudaStream_t stream) {
    return dispatch_prefill<__nv_bfloat16>(p, k_pool, v_pool, d, max_q, stream);
}

}  // namespace pa
