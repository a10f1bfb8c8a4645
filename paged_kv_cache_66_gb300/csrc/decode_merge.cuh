// Merge of the split-K partitions of paged decode ("Chapter 7 Paged KV Cache
// and Memory Management", 4.2, "Block Merging Mechanism of Online Softmax"):
// take the largest partition max as the new reference, rescale every
// partition's normaliser and partial output onto it, add, divide.  A partition
// with normaliser 0 (nothing valid) contributes nothing.
#pragma once

#include "pa_common.cuh"
#include "pa_launch.h"

namespace pa {

constexpr int kMergeChunk = 256;  // partitions per shared-memory chunk

// Fused merge: every partition CTA of one (sequence, KV head) group bumps a
// counter after publishing its partials; the CTA that arrives last merges the
// group's G heads.  pa_decode zeroes the counters before the partition kernel.
//   nthreads threads (>= 64); `sm` = shared scratch of at least
//   (2 + 2 * kMergeChunk) * G floats.  The reduction order is fixed, so the
//   result does not depend on which CTA merges or on timing.
template <typename T, int D, int G>
__device__ __forceinline__ void merge_if_last(const DecodeParams& p, int s, int kvh, int n_parts, float* sm,
                                              int tid, int nthreads) {
    __shared__ int s_last;
    __threadfence();  // this CTA's partials are visible device-wide before it is counted
    __syncthreads();
    if (tid == 0) {
        const unsigned prev = atomicAdd(p.counters + static_cast<size_t>(s) * p.hq + kvh * G, 1u);
        s_last = prev == static_cast<unsigned>(n_parts - 1);
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();

    const int P = p.max_partitions;
    const size_t row0 = (static_cast<size_t>(s) * p.hq + kvh * G) * P;  // row of (head 0, partition 0)
    const float* ml = p.ws_ml;
    const float* acc = p.ws_acc;
    float* sM = sm;                          // [G] reference max per head
    float* sDen = sm + G;                    // [G] normaliser per head
    float* w = sm + 2 * G;                   // [G][kMergeChunk] partition weights
    float* wl = w + G * kMergeChunk;         // [G][kMergeChunk] weighted normalisers
    const int warp = tid >> 5, lane = tid & 31, nw = nthreads >> 5;

    for (int g = warp; g < G; g += nw) {
        float M = -INFINITY;
        for (int i = lane; i < n_parts; i += 32) M = fmaxf(M, __ldcg(ml + (row0 + g * P + i) * 2));
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        if (lane == 0) {
            sM[g] = M;
            sDen[g] = 0.f;
        }
    }
    constexpr int kMaxOut = (G * D + 63) / 64;  // outputs per thread
    float num[kMaxOut];
#pragma unroll
    for (int k = 0; k < kMaxOut; ++k) num[k] = 0.f;
    for (int c0 = 0; c0 < n_parts; c0 += kMergeChunk) {
        const int nc = min(kMergeChunk, n_parts - c0);
        __syncthreads();  // sM ready; previous chunk consumed
        for (int i = tid; i < G * nc; i += nthreads) {
            const int g = i / nc, j = i - g * nc;
            const size_t r = row0 + g * P + c0 + j;
            const float M = sM[g];
            const float f = (M == -INFINITY) ? 0.f : exp2f(__ldcg(ml + r * 2) - M);
            w[g * kMergeChunk + j] = f;
            wl[g * kMergeChunk + j] = f * __ldcg(ml + r * 2 + 1);
        }
        __syncthreads();
        for (int g = warp; g < G; g += nw) {
            float t = 0.f;
            for (int j = lane; j < nc; j += 32) t += wl[g * kMergeChunk + j];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
            if (lane == 0) sDen[g] += t;
        }
#pragma unroll
        for (int k = 0; k < kMaxOut; ++k) {
            const int idx = tid + k * nthreads;
            if (idx < G * D) {
                const int g = idx / D, d = idx - g * D;
                const float* a = acc + (row0 + g * P + c0) * D + d;
                const float* wg = w + g * kMergeChunk;
                float x0 = 0.f, x1 = 0.f, x2 = 0.f, x3 = 0.f;
                int j = 0;
                for (; j + 4 <= nc; j += 4) {
                    x0 = fmaf(wg[j], __ldcg(a + static_cast<size_t>(j) * D), x0);
                    x1 = fmaf(wg[j + 1], __ldcg(a + static_cast<size_t>(j + 1) * D), x1);
                    x2 = fmaf(wg[j + 2], __ldcg(a + static_cast<size_t>(j + 2) * D), x2);
                    x3 = fmaf(wg[j + 3], __ldcg(a + static_cast<size_t>(j + 3) * D), x3);
                }
                for (; j < nc; ++j) x0 = fmaf(wg[j], __ldcg(a + static_cast<size_t>(j) * D), x0);
                num[k] += (x0 + x1) + (x2 + x3);
            }
        }
    }
    __syncthreads();
    T* out = static_cast<T*>(p.out) + (static_cast<size_t>(s) * p.hq + kvh * G) * D;
#pragma unroll
    for (int k = 0; k < kMaxOut; ++k) {
        const int idx = tid + k * nthreads;
        if (idx < G * D) {
            const float den = sDen[idx / D];
            out[idx] = Elt<T>::from_f32(den > 0.f ? num[k] / den : 0.f);
        }
    }
}

}  // namespace pa
