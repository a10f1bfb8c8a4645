// The prefill kernel of one pa_prefill call: one per head dim -- 128-key K/V tiles with two
// query tiles per CTA (prefill_tc05w.cuh) at D in {64, 128}, one query tile with Q in tensor
// memory (prefill_tc05d.cuh) at D = 256.
#pragma once

#include "prefill_tc05d.cuh"
#include "prefill_tc05w.cuh"

namespace pa {

template <typename T, int D, int G>
cudaError_t launch_prefill_path(const PrefillParams& p, const CUtensorMap& km, const CUtensorMap& vm, int max_q,
                                cudaStream_t stream) {
    if constexpr (D <= 128) {
        CUtensorMap qm;
        if (!encode_q_tmap(&qm, p.q, p.total_q, p.hq, D, G)) return cudaErrorInvalidValue;
        return launch_prefill_tc05w<T, D, G>(p, km, vm, qm, max_q, stream);
    } else {
        return launch_prefill_tc05d<T, G>(p, km, vm, max_q, stream);
    }
}

template <typename T, int D>
cudaError_t dispatch_prefill_group(const PrefillParams& p, const CUtensorMap& km, const CUtensorMap& vm, int max_q,
                                   cudaStream_t stream) {
    switch (p.hq / p.hkv) {
        case 1: return launch_prefill_path<T, D, 1>(p, km, vm, max_q, stream);
        case 2: return launch_prefill_path<T, D, 2>(p, km, vm, max_q, stream);
        case 4: return launch_prefill_path<T, D, 4>(p, km, vm, max_q, stream);
        case 8: return launch_prefill_path<T, D, 8>(p, km, vm, max_q, stream);
        default: return cudaErrorNotSupported;
    }
}

template <typename T>
cudaError_t dispatch_prefill(const PrefillParams& p, const void* k_pool, const void* v_pool, int d, int max_q,
                             cudaStream_t stream) {
    const uint64_t rows = static_cast<uint64_t>(p.num_blocks) * p.hkv * p.block_size;
    if (rows >= (1ull << 31)) return cudaErrorNotSupported;
    CUtensorMap km, vm;
    // D = 256: one box spans the row's four 64-dim slices (8 rows of K, 16 of V): 12 copies per
    // 64-key tile instead of 32; D <= 128: boxes of 16 rows x 128 bytes
    const bool ok = d == 256 ? encode_pool_tmap_slices(&km, k_pool, rows, d, 8) &&
                                   encode_pool_tmap_slices(&vm, v_pool, rows, d, 16)
                             : encode_pool_tmap(&km, k_pool, rows, d, 2) && encode_pool_tmap(&vm, v_pool, rows, d, 2);
    if (!ok) return cudaErrorInvalidValue;
    switch (d) {
        case 64: return dispatch_prefill_group<T, 64>(p, km, vm, max_q, stream);
        case 128: return dispatch_prefill_group<T, 128>(p, km, vm, max_q, stream);
        case 256: return dispatch_prefill_group<T, 256>(p, km, vm, max_q, stream);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace pa
