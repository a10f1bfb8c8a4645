// Instantiations of the paged decode kernel for FP8 (E4M3) pools with f16 or
// bf16 queries (one translation unit so the build compiles it in parallel).
#include "decode_dispatch.cuh"

namespace pa {

cudaError_t launch_decode_fp8_f16(const DecodeParams& p, cudaStream_t stream) {
    return dispatch_decode_fp8<__half>(p, stream);
}

cudaError_t launch_decode_fp8_bf16(const DecodeParams& p, cudaStream_t stream) {
    return dispatch_decode_fp8<__nv_bfloat16>(p, stream);
}

}  // namespace pa
