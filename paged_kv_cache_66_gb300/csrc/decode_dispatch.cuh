// Choice between the decode kernels for one pa_decode call.
//
// fp16 / bf16 pools use the tensor-core kernel (decode_mma.cuh) unless the
// caller forced the CUDA-core kernel or the pool has too many rows for a
// 32-bit TMA coordinate; fp32 pools use the CUDA-core kernel
// (decode_simt.cuh).  Both write the same partials and share the merge.
#pragma once

#include <type_traits>

#include "decode_mma.cuh"
#include "decode_simt.cuh"

namespace pa {

template <typename T, int D, int G>
cudaError_t launch_decode_path(const DecodeParams& p, cudaStream_t stream) {
    if constexpr (sizeof(T) == 2) {
        const uint64_t rows = static_cast<uint64_t>(p.num_blocks) * p.hkv * p.block_size;
        if (p.kernel != PA_DECODE_SIMT && rows < (1ull << 31)) {
            CUtensorMap km, vm;
            if (!encode_pool_tmap(&km, p.k_pool, rows, D, 2) || !encode_pool_tmap(&vm, p.v_pool, rows, D, 2))
                return cudaErrorInvalidValue;
            return launch_mma<T, T, D, G>(p, km, vm, stream);
        }
        if (p.kernel == PA_DECODE_MMA) return cudaErrorNotSupported;
    } else {
        if (p.kernel == PA_DECODE_MMA) return cudaErrorNotSupported;
    }
    return launch_simt<T, D, G>(p, stream);
}

template <typename T, int D>
cudaError_t dispatch_group(const DecodeParams& p, cudaStream_t stream) {
    switch (p.hq / p.hkv) {
        case 1: return launch_decode_path<T, D, 1>(p, stream);
        case 2: return launch_decode_path<T, D, 2>(p, stream);
        case 4: return launch_decode_path<T, D, 4>(p, stream);
        case 8: return launch_decode_path<T, D, 8>(p, stream);
        default: return cudaErrorNotSupported;
    }
}

template <typename T>
cudaError_t dispatch_decode(const DecodeParams& p, cudaStream_t stream) {
    switch (p.d) {
        case 64: return dispatch_group<T, 64>(p, stream);
        case 128: return dispatch_group<T, 128>(p, stream);
        case 256: return dispatch_group<T, 256>(p, stream);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace pa

namespace pa {

// FP8 (E4M3) pools: the tensor-core kernel with byte tiles; D = 64 as lines of two 64-byte rows
// (16 tokens = 8 lines of 128 bytes), D = 128, 256 as 128-byte boxes.
template <typename T, int D>
cudaError_t dispatch_fp8_group(const DecodeParams& p, cudaStream_t stream) {
    const uint64_t rows = static_cast<uint64_t>(p.num_blocks) * p.hkv * p.block_size;
    if (rows >= (1ull << 31)) return cudaErrorNotSupported;
    CUtensorMap km, vm;
    const bool ok = D == 64 ? encode_pool_tmap(&km, p.k_pool, rows / 2, 128, 1, 8) &&
                                  encode_pool_tmap(&vm, p.v_pool, rows / 2, 128, 1, 8)
                            : encode_pool_tmap(&km, p.k_pool, rows, D, 1) && encode_pool_tmap(&vm, p.v_pool, rows, D, 1);
    if (!ok) return cudaErrorInvalidValue;
    switch (p.hq / p.hkv) {
        case 1: return launch_mma<T, uint8_t, D, 1>(p, km, vm, stream);
        case 2: return launch_mma<T, uint8_t, D, 2>(p, km, vm, stream);
        case 4: return launch_mma<T, uint8_t, D, 4>(p, km, vm, stream);
        case 8: return launch_mma<T, uint8_t, D, 8>(p, km, vm, stream);
        default: return cudaErrorNotSupported;
    }
}

template <typename T>
cudaError_t dispatch_decode_fp8(const DecodeParams& p, cudaStream_t stream) {
    switch (p.d) {
        case 64: return dispatch_fp8_group<T, 64>(p, stream);
        case 128: return dispatch_fp8_group<T, 128>(p, stream);
        case 256: return dispatch_fp8_group<T, 256>(p, stream);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace pa
