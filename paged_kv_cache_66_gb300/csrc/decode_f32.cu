// Instantiations of the paged decode kernels for float pools (one translation
// unit per dtype so the build compiles them in parallel).
#include "decode_dispatch.cuh"

namespace pa {

cudaError_t launch_decode_f32(const DecodeParams& p, cudaStream_t stream) { return dispatch_decode<float>(p, stream); }

}  // namespace pa
