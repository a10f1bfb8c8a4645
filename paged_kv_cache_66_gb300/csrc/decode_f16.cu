// Instantiations of the paged decode kernels for __half pools (one translation
// unit per dtype so the build compiles them in parallel).
#include "decode_dispatch.cuh"

namespace pa {

cudaError_t launch_decode_f16(const DecodeParams& p, cudaStream_t stream) { return dispatch_decode<__half>(p, stream); }

}  // namespace pa
