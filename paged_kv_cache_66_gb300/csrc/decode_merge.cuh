// Merge of the split-K partitions of paged decode ("Chapter 7 Paged KV Cache
// and Memory Management", 4.2, "Block Merging Mechanism of Online Softmax"):
// take the largest partition max as the new reference, rescale every
// partition's normaliser and partial output onto it, add, divide.  A partition
// with normaliser 0 (nothing valid) contributes nothing.
//
// One CTA of 128 threads per (query head, sequence).  The partition weights
// exp2(m_p - M) go to shared memory once; then the CTA's threads form
// 128 / (D/4) "streams" of D/4 lanes, each lane owning 4 output dimensions,
// and stream k walks partitions k, k + streams, ...  When a lane has at most
// 16 partials (up to 64 partitions at D = 128) all of them are requested
// before the reference max is known, so the kernel pays about one memory
// round trip; longer sequences loop with 8 float4 loads in flight per lane.
// Streams are combined in a fixed order, so the result is deterministic.
// (A variant fused into the partition kernel -- the last CTA of a group
// merging -- measured slower: its merge sat on the kernel's tail.)
#pragma once

#include "pa_common.cuh"
#include "pa_launch.h"

namespace pa {

constexpr int kMergeThreads = 128;
constexpr int kMergeChunk = 1024;  // partitions whose weights sit in shared memory at once
constexpr int kPrefetch = 16;      // partials per lane requested up front in the common case

template <typename T, int D>
__global__ void __launch_bounds__(kMergeThreads) decode_merge(const DecodeParams p) {
    constexpr int LPS = D / 4;                       // lanes per stream (4 dims each)
    constexpr int NS = kMergeThreads / LPS;          // streams
    static_assert(NS >= 1 && NS * LPS == kMergeThreads, "stream layout");
    static_assert(kPrefetch * NS <= kMergeThreads, "common case: one (max, normaliser) pair per thread");
    __shared__ float w[kMergeChunk];
    __shared__ float red[kMergeThreads / 32];
    __shared__ float4 part_num[NS > 1 ? NS - 1 : 1][LPS];
    __shared__ float s_max, s_den;

    griddep_wait();
    griddep_launch_dependents();
    const int h = blockIdx.x, s = blockIdx.y, tid = threadIdx.x;
    const int cap = p.max_blocks * p.block_size;
    int L = __ldg(p.seq_lens + s);
    L = L < 0 ? 0 : (L > cap ? cap : L);
    const int n_parts = (L + p.partition_tokens - 1) / p.partition_tokens;
    if (n_parts <= 1) return;  // the partition kernel wrote this row directly
    const size_t row0 = (static_cast<size_t>(s) * p.hq + h) * p.max_partitions;
    const float* ml = p.ws_ml + row0 * 2;
    T* out = static_cast<T*>(p.out) + (static_cast<size_t>(s) * p.hq + h) * D;
    const int stream = tid / LPS, lane4 = tid - stream * LPS;
    const float4* acc = reinterpret_cast<const float4*>(p.ws_acc + row0 * D) + lane4;

    if (n_parts <= kPrefetch * NS) {
        // Common case: every partial of this lane is requested at once, before
        // the reference max is known, together with the (max, normaliser) pairs.
        float4 x[kPrefetch];
#pragma unroll
        for (int u = 0; u < kPrefetch; ++u) {
            const int i = stream + u * NS;
            x[u] = i < n_parts ? __ldcg(acc + static_cast<size_t>(i) * LPS) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float mi = -INFINITY, li = 0.f;
        if (tid < n_parts) {
            mi = __ldcg(ml + 2 * tid);
            li = __ldcg(ml + 2 * tid + 1);
        }
        float M = mi;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        if ((tid & 31) == 0) red[tid >> 5] = M;
        __syncthreads();
        M = red[0];
#pragma unroll
        for (int k = 1; k < kMergeThreads / 32; ++k) M = fmaxf(M, red[k]);
        if (M == -INFINITY) {
            for (int d = tid; d < D; d += kMergeThreads) out[d] = Elt<T>::from_f32(0.f);
            return;
        }
        const float f = tid < n_parts ? exp2f(mi - M) : 0.f;
        if (tid < kMergeChunk) w[tid] = f;
        float dl = f * li;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) dl += __shfl_xor_sync(0xffffffffu, dl, o);
        __syncthreads();  // everyone has read red[] as maxima; w[] written
        if ((tid & 31) == 0) red[tid >> 5] = dl;
        float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < kPrefetch; ++u) {
            const int i = stream + u * NS;
            const float g = i < n_parts ? w[i] : 0.f;
            num.x = fmaf(g, x[u].x, num.x);
            num.y = fmaf(g, x[u].y, num.y);
            num.z = fmaf(g, x[u].z, num.z);
            num.w = fmaf(g, x[u].w, num.w);
        }
        if (stream > 0) part_num[stream - 1][lane4] = num;
        __syncthreads();
        if (stream == 0) {
#pragma unroll
            for (int k = 0; k < NS - 1; ++k) {
                const float4 y = part_num[k][lane4];
                num.x += y.x;
                num.y += y.y;
                num.z += y.z;
                num.w += y.w;
            }
            float den = 0.f;
#pragma unroll
            for (int k = 0; k < kMergeThreads / 32; ++k) den += red[k];
            const float inv = den > 0.f ? 1.f / den : 0.f;
            T* o = out + 4 * lane4;
            o[0] = Elt<T>::from_f32(num.x * inv);
            o[1] = Elt<T>::from_f32(num.y * inv);
            o[2] = Elt<T>::from_f32(num.z * inv);
            o[3] = Elt<T>::from_f32(num.w * inv);
        }
        return;
    }

    // reference max over the partitions
    float M = -INFINITY;
    for (int i = tid; i < n_parts; i += kMergeThreads) M = fmaxf(M, __ldcg(ml + 2 * i));
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    if ((tid & 31) == 0) red[tid >> 5] = M;
    __syncthreads();
    if (tid == 0) {
        float m = red[0];
#pragma unroll
        for (int k = 1; k < kMergeThreads / 32; ++k) m = fmaxf(m, red[k]);
        s_max = m;
    }
    __syncthreads();
    M = s_max;
    if (M == -INFINITY) {
        for (int d = tid; d < D; d += kMergeThreads) out[d] = Elt<T>::from_f32(0.f);
        return;
    }

    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
    float den_part = 0.f;
    for (int c0 = 0; c0 < n_parts; c0 += kMergeChunk) {
        const int nc = min(kMergeChunk, n_parts - c0);
        __syncthreads();  // previous chunk's weights consumed
        for (int i = tid; i < nc; i += kMergeThreads) {
            const float f = exp2f(__ldcg(ml + 2 * (c0 + i)) - M);
            w[i] = f;
            den_part = fmaf(f, __ldcg(ml + 2 * (c0 + i) + 1), den_part);
        }
        __syncthreads();
        int i = stream;
        for (; i + 7 * NS < nc; i += 8 * NS) {
            float4 x[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) x[u] = __ldcg(acc + static_cast<size_t>(c0 + i + u * NS) * LPS);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const float f = w[i + u * NS];
                num.x = fmaf(f, x[u].x, num.x);
                num.y = fmaf(f, x[u].y, num.y);
                num.z = fmaf(f, x[u].z, num.z);
                num.w = fmaf(f, x[u].w, num.w);
            }
        }
        for (; i < nc; i += NS) {
            const float4 x = __ldcg(acc + static_cast<size_t>(c0 + i) * LPS);
            const float f = w[i];
            num.x = fmaf(f, x.x, num.x);
            num.y = fmaf(f, x.y, num.y);
            num.z = fmaf(f, x.z, num.z);
            num.w = fmaf(f, x.w, num.w);
        }
    }
    // normaliser: block sum of the per-thread partial sums
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) den_part += __shfl_xor_sync(0xffffffffu, den_part, o);
    __syncthreads();
    if ((tid & 31) == 0) red[tid >> 5] = den_part;
    if (stream > 0) part_num[stream - 1][lane4] = num;
    __syncthreads();
    if (tid == 0) {
        float t = 0.f;
#pragma unroll
        for (int k = 0; k < kMergeThreads / 32; ++k) t += red[k];
        s_den = t;
    }
    __syncthreads();
    if (stream == 0) {
#pragma unroll
        for (int k = 0; k < NS - 1; ++k) {
            const float4 y = part_num[k][lane4];
            num.x += y.x;
            num.y += y.y;
            num.z += y.z;
            num.w += y.w;
        }
        const float den = s_den;
        const float inv = den > 0.f ? 1.f / den : 0.f;
        T* o = out + 4 * lane4;
        o[0] = Elt<T>::from_f32(num.x * inv);
        o[1] = Elt<T>::from_f32(num.y * inv);
        o[2] = Elt<T>::from_f32(num.z * inv);
        o[3] = Elt<T>::from_f32(num.w * inv);
    }
}

// Batches whose sequences have at most kSmallParts partitions: one CTA of 128
// threads merges 128 / (D/4) query heads of one sequence, each lane holding
// 4 output dimensions and requesting all of its partials at once; the
// (max, normaliser) pairs go through shared memory, so the kernel costs one
// memory round trip and one barrier.  (With one CTA per head, config-5-like
// batches launched 4096 tiny CTAs and the merge took ~12 us.)
constexpr int kSmallParts = 16;

template <typename T, int D>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_small(const DecodeParams p) {
    constexpr int LPS = D / 4;                 // lanes per head
    constexpr int HPC = kMergeThreads / LPS;   // heads per CTA
    __shared__ float sml[HPC][kSmallParts][2];
    griddep_wait();
    griddep_launch_dependents();
    const int s = blockIdx.y, h0 = blockIdx.x * HPC, tid = threadIdx.x;
    const int cap = p.max_blocks * p.block_size;
    int L = __ldg(p.seq_lens + s);
    L = L < 0 ? 0 : (L > cap ? cap : L);
    const int n_parts = (L + p.partition_tokens - 1) / p.partition_tokens;
    if (n_parts <= 1) return;  // the partition kernel wrote these rows directly (uniform per CTA)
    const int hh = tid / LPS, lane4 = tid - hh * LPS, h = h0 + hh;
    const bool active = h < p.hq;
    const int P = p.max_partitions;
    float4 x[kSmallParts];
    if (active) {
        const float4* acc =
            reinterpret_cast<const float4*>(p.ws_acc + (static_cast<size_t>(s) * p.hq + h) * P * D) + lane4;
#pragma unroll
        for (int u = 0; u < kSmallParts; ++u)
            x[u] = u < n_parts ? __ldcg(acc + static_cast<size_t>(u) * LPS) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int i = tid; i < HPC * n_parts; i += kMergeThreads) {
        const int k = i / n_parts, u = i - k * n_parts;
        if (h0 + k < p.hq) {
            const float* ml = p.ws_ml + ((static_cast<size_t>(s) * p.hq + h0 + k) * P + u) * 2;
            sml[k][u][0] = __ldcg(ml);
            sml[k][u][1] = __ldcg(ml + 1);
        }
    }
    __syncthreads();
    if (!active) return;
    float M = -INFINITY;
    for (int u = 0; u < n_parts; ++u) M = fmaxf(M, sml[hh][u][0]);
    T* o = static_cast<T*>(p.out) + (static_cast<size_t>(s) * p.hq + h) * D + 4 * lane4;
    float4 num = make_float4(0.f, 0.f, 0.f, 0.f);
    float den = 0.f;
    if (M != -INFINITY) {
#pragma unroll
        for (int u = 0; u < kSmallParts; ++u) {
            if (u < n_parts) {
                const float f = exp2f(sml[hh][u][0] - M);
                den = fmaf(f, sml[hh][u][1], den);
                num.x = fmaf(f, x[u].x, num.x);
                num.y = fmaf(f, x[u].y, num.y);
                num.z = fmaf(f, x[u].z, num.z);
                num.w = fmaf(f, x[u].w, num.w);
            }
        }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    o[0] = Elt<T>::from_f32(num.x * inv);
    o[1] = Elt<T>::from_f32(num.y * inv);
    o[2] = Elt<T>::from_f32(num.z * inv);
    o[3] = Elt<T>::from_f32(num.w * inv);
}

template <typename T, int D>
cudaError_t launch_merge(const DecodeParams& p, cudaStream_t stream) {
    if (p.max_partitions <= kSmallParts) {
        constexpr int HPC = kMergeThreads / (D / 4);
        return launch_pdl(decode_merge_small<T, D>, dim3((p.hq + HPC - 1) / HPC, p.batch), dim3(kMergeThreads), 0,
                          stream, p);
    }
    return launch_pdl(decode_merge<T, D>, dim3(p.hq, p.batch), dim3(kMergeThreads), 0, stream, p);
}

}  // namespace pa
