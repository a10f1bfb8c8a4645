// Merge of the split-K partitions of paged decode ("Chapter 7 Paged KV Cache
// and Memory Management", 4.2, "Block Merging Mechanism of Online Softmax"):
// take the largest partition max as the new reference, rescale every
// partition's normaliser and partial output onto it, add, divide.  A partition
// with normaliser 0 (nothing valid) contributes nothing.
//
// One CTA per (query head, sequence), one thread per output dimension.  The
// partition weights exp2(m_p - M) and weighted normalisers are computed once
// into shared memory, then every thread streams its column of partials with
// several independent loads in flight.
#pragma once

#include "pa_common.cuh"
#include "pa_launch.h"

namespace pa {

constexpr int kMergeChunk = 512;  // partitions per shared-memory chunk

template <typename T, int D>
__global__ void __launch_bounds__(D) decode_merge(const DecodeParams p) {
    __shared__ float w[kMergeChunk];
    __shared__ float red[D / 32];
    __shared__ float s_max, s_den;
    const int h = blockIdx.x, s = blockIdx.y, d = threadIdx.x;
    const int cap = p.max_blocks * p.block_size;
    int L = __ldg(p.seq_lens + s);
    L = L < 0 ? 0 : (L > cap ? cap : L);
    const int n_parts = (L + p.partition_tokens - 1) / p.partition_tokens;
    if (n_parts <= 1) return;
    const size_t row0 = (static_cast<size_t>(s) * p.hq + h) * p.max_partitions;
    const float* ml = p.ws_ml + row0 * 2;

    // reference max over the partitions (block reduction)
    float M = -INFINITY;
    for (int i = d; i < n_parts; i += D) M = fmaxf(M, ml[2 * i]);
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if ((d & 31) == 0) red[d >> 5] = M;
    __syncthreads();
    if (d == 0) {
        float m = red[0];
        for (int k = 1; k < D / 32; ++k) m = fmaxf(m, red[k]);
        s_max = m;
        s_den = 0.f;
    }
    __syncthreads();
    M = s_max;
    T* out = static_cast<T*>(p.out) + (static_cast<size_t>(s) * p.hq + h) * D;
    if (M == -INFINITY) {
        out[d] = Elt<T>::from_f32(0.f);
        return;
    }

    const float* acc = p.ws_acc + row0 * D + d;
    float num0 = 0.f, num1 = 0.f, num2 = 0.f, num3 = 0.f;
    float den_part = 0.f;
    for (int c0 = 0; c0 < n_parts; c0 += kMergeChunk) {
        const int nc = min(kMergeChunk, n_parts - c0);
        __syncthreads();  // previous chunk's weights fully used
        for (int i = d; i < nc; i += D) {
            const float f = exp2f(ml[2 * (c0 + i)] - M);
            w[i] = f;
            den_part = fmaf(f, ml[2 * (c0 + i) + 1], den_part);
        }
        __syncthreads();
        const float* a = acc + static_cast<size_t>(c0) * D;
        int i = 0;
        for (; i + 4 <= nc; i += 4) {
            const float x0 = a[static_cast<size_t>(i) * D];
            const float x1 = a[static_cast<size_t>(i + 1) * D];
            const float x2 = a[static_cast<size_t>(i + 2) * D];
            const float x3 = a[static_cast<size_t>(i + 3) * D];
            num0 = fmaf(w[i], x0, num0);
            num1 = fmaf(w[i + 1], x1, num1);
            num2 = fmaf(w[i + 2], x2, num2);
            num3 = fmaf(w[i + 3], x3, num3);
        }
        for (; i < nc; ++i) num0 = fmaf(w[i], a[static_cast<size_t>(i) * D], num0);
    }
    // normaliser: reduce the per-thread partial sums
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) den_part += __shfl_xor_sync(0xffffffffu, den_part, o);
    __syncthreads();
    if ((d & 31) == 0) red[d >> 5] = den_part;
    __syncthreads();
    if (d == 0) {
        float t = 0.f;
        for (int k = 0; k < D / 32; ++k) t += red[k];
        s_den = t;
    }
    __syncthreads();
    const float den = s_den;
    const float num = (num0 + num1) + (num2 + num3);
    out[d] = Elt<T>::from_f32(den > 0.f ? num / den : 0.f);
}

template <typename T, int D>
cudaError_t launch_merge(const DecodeParams& p, cudaStream_t stream) {
    decode_merge<T, D><<<dim3(p.hq, p.batch), D, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace pa
