// Instantiations of the paged decode kernels for __nv_bfloat16 pools (one translation
// unit per dtype so the build compiles them in parallel).
#include "decode_dispatch.cuh"

namespace pa {

cudaError_t launch_decode_bf16(const DecodeParams& p, cudaStream_t stream) { return dispatch_decode<__nv_bfloat16>(p, stream); }

}  // namespace pa
