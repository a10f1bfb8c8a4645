// Paged prefill instantiations for f16 pools.
#include "prefill_dispatch.cuh"

namespace pa {

cudaError_t launch_prefill_f16(const PrefillParams& p, const void* k_pool, const void* v_pool, int d, int max_q,
                               cudaStream_t stream) {
    return dispatch_prefill<__half>(p, k_pool, v_pool, d, max_q, stream);
}

}  // namespace pa
