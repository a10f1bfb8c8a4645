// Paged decode attention on the CUDA cores (fp32 math), one CTA per
// (partition, kv head, sequence).
//
// What it computes: "25. Paged attention and prefix caching", section
// "Attention that reads through the table" (walk the block table, online
// softmax one block at a time, tail mask from the length, query head h reads
// KV head h // group), with the two production additions that page lists:
// all query heads of one KV group are processed together so each K/V tile is
// read once, and long sequences are split into partitions whose partial
// (max, normaliser, output) are merged afterwards ("Chapter 7 Paged KV Cache
// and Memory Management", 4.2, "Block Merging Mechanism of Online Softmax").
//
// GB300 structure:
//  * each warp owns its own slice of the partition (16-token tiles w, w+NW,
//    ...) and its own STAGES-deep ring of shared-memory buffers;
//  * lane 0 of the warp resolves the physical block of a tile from the block
//    table (staged in shared memory at CTA start, so no dependent global load
//    sits in the loop) and fetches the tile's K and V rows -- each one
//    contiguous 16*D*sizeof(T) chunk of the [N, Hkv, b, D] pool -- with 1-D
//    bulk copies (TMA engine) that complete on an mbarrier, STAGES tiles ahead;
//  * all 32 lanes compute: a token group of TG lanes reads one K row with
//    16-byte shared loads (conflict-free), reduces the G dot products with
//    xor shuffles, then accumulates p * V into per-lane fp32 accumulators;
//  * online softmax in base 2 (q pre-scaled by scale * log2 e) with a lazy
//    rescale: the reference max moves only when a tile's max exceeds it by
//    more than 2^8, which keeps every exponent <= 256 and skips almost all
//    accumulator rescales (exact: the reference cancels in O / l);
//  * warps merge their states through shared memory at the end.
#pragma once

#include "decode_merge.cuh"
#include "pa_common.cuh"
#include "pa_launch.h"

namespace pa {

template <typename T, int D, int G>
struct SimtCfg {
    static constexpr int VEC = 16 / static_cast<int>(sizeof(T));
    static constexpr int TG_RAW = G * D / 64;
    static constexpr int TG_HI = (D / VEC < 32) ? D / VEC : 32;
    static constexpr int TG = TG_RAW < 8 ? 8 : (TG_RAW > TG_HI ? TG_HI : TG_RAW);  // lanes per token
    static constexpr int DPL = D / TG;                                               // dims per lane
    static constexpr int NV = DPL / VEC;                                             // 16-B vectors per lane per row
    static constexpr int TPP = 32 / TG;                                              // tokens per pass
    static constexpr int TILE = 16;                                                  // tokens per pipeline tile
    static constexpr int NPASS = TILE / TPP;
    static constexpr int TILE_BYTES = TILE * D * static_cast<int>(sizeof(T));
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;                               // K tile + V tile
    static constexpr int NW = (4 * 2 * STAGE_BYTES > 200 * 1024) ? 2 : 4;            // warps per CTA
    static constexpr int ST_RAW = (96 * 1024) / (NW * STAGE_BYTES);
    static constexpr int STAGES = ST_RAW < 2 ? 2 : (ST_RAW > 4 ? 4 : ST_RAW);
    static constexpr int RING_BYTES = NW * STAGES * STAGE_BYTES;
    static constexpr int BAR_OFF = RING_BYTES;
    static constexpr int TBL_OFF = BAR_OFF + NW * STAGES * 8;
    static constexpr int RED_BYTES = NW * G * (D + 2) * 4;
    static_assert(NV >= 1 && DPL % VEC == 0, "lane layout");
    static_assert(RED_BYTES <= RING_BYTES, "merge scratch aliases the ring");
    static constexpr size_t smem_bytes(int table_entries) {
        return static_cast<size_t>(TBL_OFF) + static_cast<size_t>(table_entries) * 4;
    }
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(SimtCfg<T, D, G>::NW * 32)
    decode_partition_simt(const DecodeParams p) {
    using C = SimtCfg<T, D, G>;
    constexpr int TG = C::TG, NV = C::NV, VEC = C::VEC, TPP = C::TPP, NPASS = C::NPASS;
    constexpr int NW = C::NW, STAGES = C::STAGES;
    extern __shared__ __align__(128) unsigned char smem[];

    griddep_wait();
    const int part = blockIdx.x, kvh = blockIdx.y, s = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bs = p.block_size, P = p.partition_tokens;
    const int cap = p.max_blocks * bs;
    int L = __ldg(p.seq_lens + s);
    if (L < 0 || L > cap) {
        if (part == 0 && kvh == 0 && tid == 0) flag_error(p.err, PA_DEVERR_SEQLEN);
        L = L < 0 ? 0 : cap;
    }
    const int n_parts = (L + P - 1) / P;
    T* out_rows = static_cast<T*>(p.out) + (static_cast<size_t>(s) * p.hq + kvh * G) * D;
    if (L == 0) {
        if (part == 0)
            for (int i = tid; i < G * D; i += blockDim.x) out_rows[i] = Elt<T>::from_f32(0.f);
        return;
    }
    const int tok0 = part * P;
    if (tok0 >= L) return;
    const int tok1 = min(L, tok0 + P);
    const int n_tiles = (tok1 - tok0 + C::TILE - 1) / C::TILE;

    // ---- stage this partition's block-table entries (validated) in shared memory
    int* tbl = reinterpret_cast<int*>(smem + C::TBL_OFF);
    const int nblk = (tok1 - tok0 + bs - 1) / bs;
    const int32_t* trow = p.block_tables + static_cast<size_t>(s) * p.max_blocks + tok0 / bs;
    for (int i = tid; i < nblk; i += blockDim.x) {
        int e = __ldg(trow + i);
        if (e < 0 || e >= p.num_blocks) {
            flag_error(p.err, PA_DEVERR_TABLE);
            e = -1;
        }
        tbl[i] = e;
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF) + warp * STAGES;
    if (lane == 0) {
#pragma unroll
        for (int st = 0; st < STAGES; ++st) mbar_init(&bars[st], 1);
        fence_mbar_init();
    }
    __syncthreads();

    unsigned char* ring = smem + warp * STAGES * C::STAGE_BYTES;
    const size_t head_stride = static_cast<size_t>(bs) * D;  // elements per (block, head) tile of the pool
    const T* kp = static_cast<const T*>(p.k_pool);
    const T* vp = static_cast<const T*>(p.v_pool);
    const int my_n = warp < n_tiles ? (n_tiles - warp + NW - 1) / NW : 0;

    // producer (lane 0): fetch my j-th tile into stage j % STAGES
    auto issue = [&](int j) {
        const int i = warp + j * NW;
        const int st = j % STAGES;
        const int blk = tbl[(i * C::TILE) / bs];
        if (blk < 0) {
            mbar_arrive_expect_tx(&bars[st], 0);
            return;
        }
        const size_t off = (static_cast<size_t>(blk) * p.hkv + kvh) * head_stride +
                           static_cast<size_t>((i * C::TILE) % bs) * D;
        unsigned char* dst = ring + st * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&bars[st], 2 * C::TILE_BYTES);
        bulk_g2s(dst, kp + off, C::TILE_BYTES, &bars[st]);
        bulk_g2s(dst + C::TILE_BYTES, vp + off, C::TILE_BYTES, &bars[st]);
    };
    if (lane == 0)
        for (int j = 0; j < STAGES && j < my_n; ++j) issue(j);

    // ---- per-lane state
    const int tp = lane / TG, lig = lane % TG;
    float qf[G][NV][VEC];
    const T* qrow = static_cast<const T*>(p.q) + (static_cast<size_t>(s) * p.hq + kvh * G) * D;
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const uint4 u = __ldg(reinterpret_cast<const uint4*>(qrow + g * D + (v * TG + lig) * VEC));
            unpack16<T>(u, qf[g][v]);
#pragma unroll
            for (int e = 0; e < VEC; ++e) qf[g][v][e] *= p.scale_log2;
        }
    float acc[G][NV][VEC];
    float m[G], lsum[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        lsum[g] = 0.f;
#pragma unroll
        for (int v = 0; v < NV; ++v)
#pragma unroll
            for (int e = 0; e < VEC; ++e) acc[g][v][e] = 0.f;
    }

    bool timed_out = false;
    for (int j = 0; j < my_n; ++j) {
        const int st = j % STAGES;
        // one decision for the whole warp: the shuffle reductions below need every lane
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&bars[st], (j / STAGES) & 1))) {
            timed_out = true;
            if (lane == 0) flag_error(p.err, PA_DEVERR_TIMEOUT);
            // let the copies already issued land before the CTA may exit
            for (int r = j; r < my_n && r < j + STAGES; ++r) mbar_wait_bounded(&bars[r % STAGES], (r / STAGES) & 1);
            break;
        }
        const int i = warp + j * NW;
        const int nv = min(C::TILE, tok1 - (tok0 + i * C::TILE));
        const bool present = tbl[(i * C::TILE) / bs] >= 0;
        if (present) {
            const T* Ks = reinterpret_cast<const T*>(ring + st * C::STAGE_BYTES);
            const T* Vs = reinterpret_cast<const T*>(ring + st * C::STAGE_BYTES + C::TILE_BYTES);
            float sc[NPASS][G];
#pragma unroll
            for (int ps = 0; ps < NPASS; ++ps) {
                const int tok = ps * TPP + tp;
                float dot[G];
#pragma unroll
                for (int g = 0; g < G; ++g) dot[g] = 0.f;
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    const uint4 u = *reinterpret_cast<const uint4*>(Ks + tok * D + (v * TG + lig) * VEC);
                    float kf[VEC];
                    unpack16<T>(u, kf);
#pragma unroll
                    for (int g = 0; g < G; ++g)
#pragma unroll
                        for (int e = 0; e < VEC; ++e) dot[g] = fmaf(qf[g][v][e], kf[e], dot[g]);
                }
#pragma unroll
                for (int o = TG / 2; o >= 1; o >>= 1)
#pragma unroll
                    for (int g = 0; g < G; ++g) dot[g] += __shfl_xor_sync(0xffffffffu, dot[g], o);
#pragma unroll
                for (int g = 0; g < G; ++g) sc[ps][g] = (tok < nv) ? dot[g] : -INFINITY;
            }
            // tile max per head over the warp's 16 tokens
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float mx = sc[0][g];
#pragma unroll
                for (int ps = 1; ps < NPASS; ++ps) mx = fmaxf(mx, sc[ps][g]);
#pragma unroll
                for (int o = TG; o < 32; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                if (mx > m[g] + kLazyRescale) {  // warp-uniform
                    const float alpha = exp2f(m[g] - mx);
                    lsum[g] *= alpha;
#pragma unroll
                    for (int v = 0; v < NV; ++v)
#pragma unroll
                        for (int e = 0; e < VEC; ++e) acc[g][v][e] *= alpha;
                    m[g] = mx;
                }
            }
            const bool tail = nv < C::TILE;
#pragma unroll
            for (int ps = 0; ps < NPASS; ++ps) {
                const int tok = ps * TPP + tp;
                float pr[G];
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    pr[g] = exp2f(sc[ps][g] - m[g]);
                    lsum[g] += pr[g];
                }
#pragma unroll
                for (int v = 0; v < NV; ++v) {
                    const uint4 u = *reinterpret_cast<const uint4*>(Vs + tok * D + (v * TG + lig) * VEC);
                    float vf[VEC];
                    unpack16<T>(u, vf);
                    if (tail && tok >= nv) {
#pragma unroll
                        for (int e = 0; e < VEC; ++e) vf[e] = 0.f;  // unwritten slots may hold anything
                    }
#pragma unroll
                    for (int g = 0; g < G; ++g)
#pragma unroll
                        for (int e = 0; e < VEC; ++e) acc[g][v][e] = fmaf(pr[g], vf[e], acc[g][v][e]);
                }
            }
        }
        __syncwarp();
        if (lane == 0 && j + STAGES < my_n) issue(j + STAGES);
    }
    (void)timed_out;

    griddep_launch_dependents();

    // ---- reduce over the token groups of the warp
#pragma unroll
    for (int o = TG; o < 32; o <<= 1) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            lsum[g] += __shfl_xor_sync(0xffffffffu, lsum[g], o);
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int e = 0; e < VEC; ++e) acc[g][v][e] += __shfl_xor_sync(0xffffffffu, acc[g][v][e], o);
        }
    }

    // ---- merge the warps (scratch aliases the ring: wait until every warp is done)
    __syncthreads();
    float* red_m = reinterpret_cast<float*>(smem);
    float* red_l = red_m + NW * G;
    float* red_acc = red_l + NW * G;
    if (lane == 0)
#pragma unroll
        for (int g = 0; g < G; ++g) {
            red_m[warp * G + g] = m[g];
            red_l[warp * G + g] = lsum[g];
        }
    if (tp == 0)
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int v = 0; v < NV; ++v)
#pragma unroll
                for (int e = 0; e < VEC; ++e) red_acc[(warp * G + g) * D + (v * TG + lig) * VEC + e] = acc[g][v][e];
    __syncthreads();

    const bool direct = n_parts == 1;
    for (int idx = tid; idx < G * D; idx += blockDim.x) {
        const int g = idx / D, d = idx - g * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, red_m[w * G + g]);
        float num = 0.f, den = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float f = exp2f(red_m[w * G + g] - M);
                num = fmaf(f, red_acc[(w * G + g) * D + d], num);
                den = fmaf(f, red_l[w * G + g], den);
            }
        }
        if (direct) {
            out_rows[idx] = Elt<T>::from_f32(den > 0.f ? num / den : 0.f);
        } else {
            const size_t row = (static_cast<size_t>(s) * p.hq + kvh * G + g) * p.max_partitions + part;
            p.ws_acc[row * D + d] = num;
            if (d == 0) {
                p.ws_ml[row * 2] = M;
                p.ws_ml[row * 2 + 1] = den;
            }
        }
    }

}

template <typename T, int D, int G>
cudaError_t launch_simt(const DecodeParams& p, cudaStream_t stream) {
    using C = SimtCfg<T, D, G>;
    const int entries = p.partition_tokens / p.block_size;
    const size_t smem = C::smem_bytes(entries);
    static int configured_for = -1;  // device on which the attribute was last set
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_for != dev) {
        cudaError_t e = cudaFuncSetAttribute(decode_partition_simt<T, D, G>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(C::smem_bytes(8192 / 16)));
        if (e != cudaSuccess) return e;
        configured_for = dev;
    }
    dim3 grid(p.max_partitions, p.hkv, p.batch);
    cudaError_t e = launch_pdl(decode_partition_simt<T, D, G>, grid, dim3(C::NW * 32), smem, stream, p);
    if (e != cudaSuccess || p.max_partitions <= 1) return e;
    return launch_merge<T, D>(p, stream);
}

}  // namespace pa
