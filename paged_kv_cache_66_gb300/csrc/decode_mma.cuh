// Paged decode attention with the GQA q-group x 16-token tile on the tensor
// cores (mma.sync m16n8k16, fp32 accumulate), for fp16 and bf16 pools.
//
// Computes the same partition (max, normaliser, output) as the CUDA-core
// kernel -- online softmax over the blocks of one partition for all G query
// heads of one KV head ("25. Paged attention and prefix caching", "Attention
// that reads through the table"; "Chapter 7 Paged KV Cache and Memory
// Management", 4.2) -- and hands it to the same merge.
//
// Why the tensor cores: the CUDA-core kernel needs ~79 instructions per
// (token, KV head) and is issue-bound well below the HBM roofline.  Here one
// 16-token tile costs D/16 MMAs for the scores and D/16 for the output:
//   S^T[16 tok x 8 heads] = K_tile[16 x D] . Q^T[D x 8]      (A = K from smem, B = Q in registers)
//   O^T[D x 8 heads]     += V_tile^T[D x 16] . P^T[16 x 8]    (A = V^T from smem, B = P^T)
// The query group (G <= 8) sits on the N = 8 side; unused columns are zero.
// The score fragment becomes the P^T operand with one movmatrix transpose per
// 8 tokens, so P never touches shared memory.
//
// Data movement: each 16-token K (and V) tile of one (block, KV head) is
// fetched by TMA as D/64 boxes of 16 rows x 128 bytes with the 128-byte
// swizzle, so the ldmatrix reads of the fragments are bank-conflict free.
// Each warp owns every NW-th tile of the partition and a STAGES-deep ring,
// lane 0 issuing the tensor copies STAGES tiles ahead on per-stage mbarriers.
//
// FP8 (E4M3) pools, with one fp32 scale per KV head for K and for V, run the
// same kernel with P = uint8_t: a 128-byte TMA box holds 128 dims, ldmatrix
// moves byte pairs, and cvt.e4m3x2 turns them into f16 operands (exact).  For
// the scores, one ldmatrix of 8 tokens x 16 bytes gives lane (g, t) dims
// 4t..4t+3 of token g; these serve as k = {2t, 2t+1} and {2t+8, 2t+9} of the
// MMA, and q's fragment is loaded with the same permutation (a dot product is
// indifferent to the order of its terms).  For the output, the transposed
// load gives lane (g, t) dims {2g, 2g+1} of tokens {2t, 2t+1}; after a byte
// select, MMA row g stands for dim 2g and row g+8 for dim 2g+1, which the
// write-out undoes.  q is used in f16 (exact for bf16 inputs in f16's normal
// range), the K scale folds into the score scale, the V scale into the
// partial outputs.
#pragma once

#include <cuda.h>
#include <cuda_fp8.h>

#include <type_traits>

#include "decode_merge.cuh"
#include "pa_common.cuh"
#include "pa_launch.h"

namespace pa {

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ void tma_load_2d(void* smem_dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(smem_u32(smem_dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

// 2^x on the MUFU unit (relative error ~2^-22; -inf -> +0)
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t* r) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t* r) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

template <typename T>
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1);
template <>
__device__ __forceinline__ void mma16816<__half>(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
template <>
__device__ __forceinline__ void mma16816<__nv_bfloat16>(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <typename T>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<__half>(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<__nv_bfloat16>(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}

// four E4M3 codes -> two f16x2 (exact): bytes 0, 1 -> lo (byte 0 in the low half), bytes 2, 3 -> hi
__device__ __forceinline__ void e4m3x4_to_h2x2(uint32_t four, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 l16, h16;\n\tmov.b32 {l16, h16}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l16;\n\tcvt.rn.f16x2.e4m3x2 %1, h16;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(four));
}

template <typename T>
__device__ __forceinline__ uint32_t to_h2(T a, T b) {
    return pack2<__half>(Elt<T>::to_f32(a), Elt<T>::to_f32(b));
}

// ------------------------------------------------------------------ configuration
// P = pool element: the 16-bit type of q, or uint8_t (E4M3) with a 16-bit q.
template <typename P, int D, int G>
struct MmaCfg {
    static constexpr int EB = static_cast<int>(sizeof(P));
    static_assert(EB == 2 || EB == 1, "16-bit or FP8 pools");
    static constexpr bool F8 = EB == 1;
    static constexpr int TILE = 16;                    // tokens per tile (M of the score MMA)
    static constexpr int ROW_BYTES = D * EB;
    // 64-byte rows (E4M3 at D = 64): two tokens share one 128-byte swizzled line
    static constexpr bool PAIR = ROW_BYTES == 64;
    static_assert(PAIR || ROW_BYTES % 128 == 0, "rows of whole 128-byte boxes, or token pairs");
    static constexpr int NBOX = PAIR ? 1 : ROW_BYTES / 128;  // 128-byte boxes per 16-token row block
    static constexpr int BOX_ELEMS = 128 / EB;
    static constexpr int CHUNKS = ROW_BYTES / 16;      // 16-byte chunks per row
    static constexpr int BOX_BYTES = TILE * 128 / (PAIR ? 2 : 1);  // 1024-byte aligned in smem
    static constexpr int TILE_BYTES = NBOX * BOX_BYTES;
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES; // K tile + V tile
    // 2 stages x 4 warps (2 warps when a stage is >= 16 KiB; 3 stages for the
    // 4 KiB stages of FP8 at D = 128): 32-64 KiB per CTA, so 3+ CTAs share an
    // SM; deeper rings measured slower on the long-context workload (fewer
    // resident CTAs to cover each CTA's start and end, and to hide the
    // latency of each warp's chain of dependent MMAs).
#ifdef PA_MMA_WARPS
    static constexpr int NW = PA_MMA_WARPS;  // build-time override (tuning sweeps)
#else
    static constexpr int NW = STAGE_BYTES >= 16384 ? 2 : 4;
#endif
#ifdef PA_MMA_STAGES
    static constexpr int STAGES = PA_MMA_STAGES;
#else
    static constexpr int STAGES = (F8 && STAGE_BYTES <= 4096) ? 3 : 2;
#endif
    static constexpr int RING_BYTES = NW * STAGES * STAGE_BYTES;
    static constexpr int BAR_OFF = RING_BYTES;
    static constexpr int BAR_END = BAR_OFF + NW * STAGES * 8;
    static constexpr int KSTEPS = D / 16;
    static constexpr int RED_BYTES = NW * G * (D + 2) * 4;
    static_assert(RED_BYTES <= RING_BYTES, "merge scratch may alias the ring");
    static_assert(G >= 1 && G <= 8, "query group on the N = 8 side");
    static_assert(!F8 || KSTEPS % 2 == 0, "FP8 fragments come in pairs of k-steps");
    // With one KV head per CTA the warps' merge scratch aliases the ring; with two, the ring is
    // still streaming the second head while the first is merged, so the scratch has its own
    // region ahead of the table.
    static constexpr int red_off(int heads_per_cta) { return heads_per_cta > 1 ? BAR_END : 0; }
    static constexpr int tbl_off(int heads_per_cta) { return BAR_END + (heads_per_cta > 1 ? RED_BYTES : 0); }
    // + 1 KiB so the ring can be aligned to 1024 bytes for the 128-byte swizzle
    static constexpr size_t smem_bytes(int table_entries, int heads_per_cta) {
        return 1024 + static_cast<size_t>(tbl_off(heads_per_cta)) + static_cast<size_t>(table_entries) * 4;
    }
};

// Byte offset of (token row r, 16-byte chunk c) of a tile stored as NBOX boxes
// of 16 rows x 128 bytes with the 128-byte swizzle (chunk index XOR row % 8);
// with PAIR (64-byte rows) as 8 lines of two tokens, token r at line r / 2,
// chunks 4 (r % 2) + c, the line index doing the swizzle.
template <bool PAIR = false>
__device__ __forceinline__ uint32_t swz(int r, int c) {
    if constexpr (PAIR) {
        const int line = r >> 1;
        return static_cast<uint32_t>(line * 128 + ((((r & 1) * 4 + c) ^ (line & 7)) << 4));
    } else {
        return static_cast<uint32_t>((c >> 3) * 2048 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
    }
}

template <typename T, typename PE, int D, int G>
__global__ void __launch_bounds__(MmaCfg<PE, D, G>::NW * 32)
    decode_partition_mma(const DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                         const __grid_constant__ CUtensorMap vmap) {
    using C = MmaCfg<PE, D, G>;
    constexpr int NW = C::NW, STAGES = C::STAGES, KSTEPS = C::KSTEPS;
    constexpr bool F8 = C::F8;
    using TM = std::conditional_t<F8, __half, T>;  // MMA operand type
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem =
        smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);  // 1024-byte aligned ring

    griddep_wait();
    const int part = blockIdx.x, s = blockIdx.z;
    const int hpc = p.heads_per_cta;
    const int kvh0 = blockIdx.y * hpc;
    const int nh = min(hpc, p.hkv - kvh0);  // KV heads of this CTA, streamed back to back
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int bs = p.block_size, P = p.partition_tokens;
    const int cap = p.max_blocks * bs;
    const int tok0 = part * P;
    const int32_t* trow = p.block_tables + static_cast<size_t>(s) * p.max_blocks + tok0 / bs;
    // The partition's table entries are requested together with the length (neither depends on
    // the other), so the prologue costs one round trip before the first copy instead of two.
    // Entries past the sequence's end are loaded (they lie inside the table row) but not used.
    constexpr int PRE = (kMaxPartitionTokens / 16 + NW * 32 - 1) / (NW * 32);
    const int ent_cap = min(P / bs, p.max_blocks - tok0 / bs);
    int pre[PRE];
#pragma unroll
    for (int k = 0; k < PRE; ++k) {
        const int i = tid + k * NW * 32;
        pre[k] = i < ent_cap ? __ldg(trow + i) : -1;
    }
    int L = __ldg(p.seq_lens + s);
    if (L < 0 || L > cap) {
        if (part == 0 && kvh0 == 0 && tid == 0) flag_error(p.err, PA_DEVERR_SEQLEN);
        L = L < 0 ? 0 : cap;
    }
    const int n_parts = (L + P - 1) / P;
    if (L == 0) {
        if (part == 0) {
            T* out0 = static_cast<T*>(p.out) + (static_cast<size_t>(s) * p.hq + kvh0 * G) * D;
            for (int i = tid; i < nh * G * D; i += blockDim.x) out0[i] = Elt<T>::from_f32(0.f);
        }
        return;
    }
    if (tok0 >= L) return;
    const int tok1 = min(L, tok0 + P);
    const int n_tiles = (tok1 - tok0 + C::TILE - 1) / C::TILE;

    int* tbl = reinterpret_cast<int*>(smem + C::tbl_off(hpc));
    const int nblk = (tok1 - tok0 + bs - 1) / bs;  // <= ent_cap
    // fused append: the partition holding position L - 1 writes that position's K/V rows of its
    // heads before any of its copies is issued.  Its loads (slot, table entry, the new rows) are
    // issued here, beside the table staging, so that they cost one round trip
    constexpr int VPR = D * static_cast<int>(sizeof(T)) / 16;                  // 16-byte vectors per row
    constexpr int APP_PER = (2 * 2 * VPR + C::NW * 32 - 1) / (C::NW * 32);  // vectors per thread (<= 2 heads)
    bool app = false;
    int64_t app_slot = -1;
    int app_e = -1;
    uint4 app_v[APP_PER];
    if constexpr (!F8) {
        app = p.new_slots != nullptr && tok1 == L;
        if (app) {
            app_slot = __ldg(p.new_slots + s);
            app_e = __ldg(trow + (L - 1) / bs - tok0 / bs);
#pragma unroll
            for (int k = 0; k < APP_PER; ++k) {
                const int x = tid + k * C::NW * 32;
                if (x < nh * 2 * VPR) {
                    const int u = x / (2 * VPR), kind = (x / VPR) & 1, v = x % VPR;
                    app_v[k] = __ldg(static_cast<const uint4*>(kind ? p.v_new : p.k_new) +
                                     (static_cast<size_t>(s) * p.hkv + kvh0 + u) * VPR + v);
                }
            }
        }
    }
#pragma unroll
    for (int k = 0; k < PRE; ++k) {
        const int i = tid + k * NW * 32;
        if (i < nblk) {
            int e = pre[k];
            if (e < 0 || e >= p.num_blocks) {
                flag_error(p.err, PA_DEVERR_TABLE);
                e = -1;
            }
            tbl[i] = e;
        }
    }
    if constexpr (!F8) {
        // the pool stores are fenced against the async proxy, and the barrier below orders them
        // before the TMA loads; no other CTA reads position L - 1 of these heads
        if (app && app_slot >= 0) {
            const int e = app_e;
            if (e < 0 || e >= p.num_blocks || app_slot != static_cast<int64_t>(e) * bs + (L - 1) % bs) {
                if (tid == 0) flag_error(p.err, PA_DEVERR_SLOT);
            } else {
#pragma unroll
                for (int k = 0; k < APP_PER; ++k) {
                    const int x = tid + k * C::NW * 32;
                    if (x < nh * 2 * VPR) {
                        const int u = x / (2 * VPR), kind = (x / VPR) & 1, v = x % VPR;
                        uint4* dst = static_cast<uint4*>(const_cast<void*>(kind ? p.v_pool : p.k_pool)) +
                                     ((static_cast<size_t>(e) * p.hkv + kvh0 + u) * bs + (L - 1) % bs) * VPR + v;
                        *dst = app_v[k];
                    }
                }
                fence_proxy_async_global();
            }
        }
    }
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF) + warp * STAGES;
    if (lane == 0) {
#pragma unroll
        for (int st = 0; st < STAGES; ++st) mbar_init(&bars[st], 1);
        fence_mbar_init();
    }
    __syncthreads();

    unsigned char* ring = smem + warp * STAGES * C::STAGE_BYTES;
    const int my_n = warp < n_tiles ? (n_tiles - warp + NW - 1) / NW : 0;
    const int my_total = nh * my_n;  // this warp's tiles over all heads: one stream through its ring
    // tile i of the partition lies in table entry i / tpb (the partition starts on a block
    // boundary); i < 512 and tpb <= 16, where (i * inv_tpb) >> 16 is that quotient exactly
    const int tpb = bs / C::TILE;
    const uint32_t inv_tpb = (65536u + tpb - 1) / tpb;

    // tile jj of the stream: head jj / my_n, the warp's (jj % my_n)-th tile of the partition.
    // Copies go out in stream order, so lane 0 steps (iss_u, iss_j) instead of dividing.
    int iss_u = 0, iss_j = 0;
    auto issue = [&](int jj) {
        const int u = iss_u, i = warp + iss_j * NW;
        if (++iss_j == my_n) {
            iss_j = 0;
            ++iss_u;
        }
        const int st = jj % STAGES;
        const int bi = static_cast<int>((static_cast<uint32_t>(i) * inv_tpb) >> 16);
        const int blk = tbl[bi];
        if (blk < 0) {
            mbar_arrive_expect_tx(&bars[st], 0);
            return;
        }
        const int row = (blk * p.hkv + kvh0 + u) * bs + (i - bi * tpb) * C::TILE;
        unsigned char* dst = ring + st * C::STAGE_BYTES;
        mbar_arrive_expect_tx(&bars[st], 2 * C::TILE_BYTES);
#pragma unroll
        for (int bx = 0; bx < C::NBOX; ++bx) {
            // token pairs: the maps view the pool as lines of two rows (row is even: b % 16 == 0)
            const int y = C::PAIR ? row >> 1 : row;
            tma_load_2d(dst + bx * C::BOX_BYTES, &kmap, bx * C::BOX_ELEMS, y, &bars[st]);
            tma_load_2d(dst + C::TILE_BYTES + bx * C::BOX_BYTES, &vmap, bx * C::BOX_ELEMS, y, &bars[st]);
        }
    };
    if (lane == 0)
        for (int jj = 0; jj < STAGES && jj < my_total; ++jj) issue(jj);

    const int g = lane >> 2, t = lane & 3;
    // ldmatrix addressing: lane provides row (lane & 7) of matrix (lane >> 3)
    const int lm = lane >> 3, lr = lane & 7;
    float* red_m = reinterpret_cast<float*>(smem + C::red_off(hpc));
    float* red_l = red_m + NW * G;
    float* red_acc = red_l + NW * G;
    const int h0 = 2 * t, h1 = 2 * t + 1;
    bool aborted = false;

    for (int u = 0; u < nh; ++u) {
        const int kvh = kvh0 + u;
        T* out_rows = static_cast<T*>(p.out) + (static_cast<size_t>(s) * p.hq + kvh * G) * D;
        // ---- query fragments (B operand of the score MMA): lane (g, t) holds
        // Q[head g][k0 + 2t, +1] and Q[head g][k0 + 8 + 2t, +1]; heads >= G are zero.
        uint32_t qb[KSTEPS][2];
        {
            const T* qrow = static_cast<const T*>(p.q) + (static_cast<size_t>(s) * p.hq + kvh * G + g) * D;
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
                if (g < G) {
                    if constexpr (F8) {
                        // dims 4t..4t+3 of this 16-dim step, matching the K fragment below
                        const T* q4 = qrow + ks * 16 + 4 * t;
                        qb[ks][0] = to_h2<T>(q4[0], q4[1]);
                        qb[ks][1] = to_h2<T>(q4[2], q4[3]);
                    } else {
                        qb[ks][0] = __ldg(reinterpret_cast<const unsigned int*>(qrow + ks * 16 + 2 * t));
                        qb[ks][1] = __ldg(reinterpret_cast<const unsigned int*>(qrow + ks * 16 + 8 + 2 * t));
                    }
                } else {
                    qb[ks][0] = 0u;
                    qb[ks][1] = 0u;
                }
            }
        }
        // ---- output accumulators O^T: acc[mt] = {O[h0][dim mt*16+g], O[h1][..], O[h0][dim mt*16+g+8], O[h1][..]}
        // with h0 = 2t, h1 = 2t + 1
        float acc[KSTEPS][4];
#pragma unroll
        for (int mt = 0; mt < KSTEPS; ++mt) acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
        const float sl2 = F8 ? p.scale_log2 * __ldg(p.k_scale + kvh) : p.scale_log2;

        for (int j = 0; j < my_n && !aborted; ++j) {
            const int jj = u * my_n + j;
            const int st = jj % STAGES;
            // the warp decides together: ldmatrix / mma / shuffles below are full-warp collectives,
            // so a lane whose own wait ran out must not leave the others behind
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&bars[st], (jj / STAGES) & 1))) {
                if (lane == 0) flag_error(p.err, PA_DEVERR_TIMEOUT);
                // let every copy this warp issued land before the CTA may exit (bounded again)
                for (int r = jj; r < my_total && r < jj + STAGES; ++r)
                    mbar_wait_bounded(&bars[r % STAGES], (r / STAGES) & 1);
                aborted = true;
                break;
            }
            const int i = warp + j * NW;
            const int nv = min(C::TILE, tok1 - (tok0 + i * C::TILE));
            const bool present = tbl[(static_cast<uint32_t>(i) * inv_tpb) >> 16] >= 0;
            unsigned char* kt = ring + st * C::STAGE_BYTES;
            unsigned char* vt = kt + C::TILE_BYTES;
            if (present) {
                // ---- scores S^T = K Q^T (16 tokens x 8 heads)
                // two accumulators (even / odd k-steps) halve the chain of dependent MMAs
                float sc[4] = {0.f, 0.f, 0.f, 0.f}, sc2[4] = {0.f, 0.f, 0.f, 0.f};
                const uint32_t kbase = smem_u32(kt);
                const int krow = lr + (lm & 1) * 8;
                if constexpr (F8) {
#pragma unroll
                    for (int ks = 0; ks < KSTEPS; ks += 2) {
                        uint32_t r[4], a0[4], a1[4];
                        ldsm_x4(kbase + swz<C::PAIR>(lr + (lm & 1) * 8, ks + (lm >> 1)), r);
                        // lane holds dims 4t..4t+3 of rows g and g+8: {r0 lo, r1 lo, r0 hi, r1 hi} per k-step
                        e4m3x4_to_h2x2(r[0], a0[0], a0[2]);
                        e4m3x4_to_h2x2(r[1], a0[1], a0[3]);
                        e4m3x4_to_h2x2(r[2], a1[0], a1[2]);
                        e4m3x4_to_h2x2(r[3], a1[1], a1[3]);
                        mma16816<TM>(sc, a0, qb[ks][0], qb[ks][1]);
                        mma16816<TM>(sc2, a1, qb[ks + 1][0], qb[ks + 1][1]);
                    }
                } else {
#pragma unroll
                    for (int ks = 0; ks < KSTEPS; ++ks) {
                        uint32_t a[4];
                        ldsm_x4(kbase + swz(krow, ks * 2 + (lm >> 1)), a);
                        mma16816<TM>((ks & 1) ? sc2 : sc, a, qb[ks][0], qb[ks][1]);
                    }
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[e] += sc2[e];
                // sc = {S[tok g][h0], S[tok g][h1], S[tok g+8][h0], S[tok g+8][h1]}
#pragma unroll
                for (int e = 0; e < 4; ++e) sc[e] *= sl2;
                if (nv < C::TILE) {  // the partition's last tile only
                    if (g >= nv) sc[0] = sc[1] = -INFINITY;
                    if (g + 8 >= nv) sc[2] = sc[3] = -INFINITY;
                }
                float mx0 = fmaxf(sc[0], sc[2]), mx1 = fmaxf(sc[1], sc[3]);
                // A head's max moves only when one of its 8 token lanes passes the lazy threshold;
                // one vote finds the (rare) tiles where some head's does, and only those reduce.
                if (__any_sync(0xffffffffu, mx0 > m0 + kLazyRescale || mx1 > m1 + kLazyRescale)) {
#pragma unroll
                    for (int o = 4; o < 32; o <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
                    }
                }
                if (mx0 > m0 + kLazyRescale) {
                    const float a0 = ex2_approx(m0 - mx0);
                    l0 *= a0;
#pragma unroll
                    for (int mt = 0; mt < KSTEPS; ++mt) {
                        acc[mt][0] *= a0;
                        acc[mt][2] *= a0;
                    }
                    m0 = mx0;
                }
                if (mx1 > m1 + kLazyRescale) {
                    const float a1 = ex2_approx(m1 - mx1);
                    l1 *= a1;
#pragma unroll
                    for (int mt = 0; mt < KSTEPS; ++mt) {
                        acc[mt][1] *= a1;
                        acc[mt][3] *= a1;
                    }
                    m1 = mx1;
                }
                const float p0 = ex2_approx(sc[0] - m0), p1 = ex2_approx(sc[1] - m1);
                const float p2 = ex2_approx(sc[2] - m0), p3 = ex2_approx(sc[3] - m1);
                l0 += p0 + p2;
                l1 += p1 + p3;
                // P^T operand: transpose the 8x8 (token x head) halves
                const uint32_t pb0 = movmatrix_t(pack2<TM>(p0, p1));
                const uint32_t pb1 = movmatrix_t(pack2<TM>(p2, p3));
                if (nv < C::TILE) {
                    // unwritten slots of the tail may hold anything (NaN * 0 = NaN): zero those V rows
                    for (int e = lane; e < (C::TILE - nv) * C::CHUNKS; e += 32) {
                        const int r = nv + e / C::CHUNKS, c = e % C::CHUNKS;
                        *reinterpret_cast<uint4*>(vt + swz<C::PAIR>(r, c)) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    __syncwarp();
                }
                // ---- O^T += V^T P^T
                const uint32_t vbase = smem_u32(vt);
                const int vrow = lr + (lm >> 1) * 8;
                if constexpr (F8) {
#pragma unroll
                    for (int mt = 0; mt < KSTEPS; mt += 2) {
                        uint32_t r[4], a0[4], a1[4];
                        ldsm_x4_t(vbase + swz<C::PAIR>(lr + (lm & 1) * 8, mt + (lm >> 1)), r);
                        // r[i] bytes: (tok 2t, dim 2g), (tok 2t, dim 2g+1), (tok 2t+1, dim 2g), (tok 2t+1, dim 2g+1);
                        // one byte permute groups each dim's two tokens: [b0 b2 | b1 b3]
                        e4m3x4_to_h2x2(__byte_perm(r[0], 0u, 0x3120u), a0[0], a0[1]);
                        e4m3x4_to_h2x2(__byte_perm(r[1], 0u, 0x3120u), a0[2], a0[3]);
                        e4m3x4_to_h2x2(__byte_perm(r[2], 0u, 0x3120u), a1[0], a1[1]);
                        e4m3x4_to_h2x2(__byte_perm(r[3], 0u, 0x3120u), a1[2], a1[3]);
                        mma16816<TM>(acc[mt], a0, pb0, pb1);
                        mma16816<TM>(acc[mt + 1], a1, pb0, pb1);
                    }
                } else {
#pragma unroll
                    for (int mt = 0; mt < KSTEPS; ++mt) {
                        uint32_t a[4];
                        ldsm_x4_t(vbase + swz(vrow, mt * 2 + (lm & 1)), a);
                        mma16816<TM>(acc[mt], a, pb0, pb1);
                    }
                }
            }
            __syncwarp();
            if (lane == 0 && jj + STAGES < my_total) {
                fence_proxy_async_smem();  // order this warp's shared accesses before the next async copy
                issue(jj + STAGES);
            }
        }
        if (u + 1 == nh) griddep_launch_dependents();

        // ---- normalisers: sum over the 8 token rows held by lanes with the same t
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, o);
            l1 += __shfl_xor_sync(0xffffffffu, l1, o);
        }

        // ---- merge the warps through shared memory (aliasing the ring when one head per CTA)
        __syncthreads();
        if (g == 0) {
            if (h0 < G) {
                red_m[warp * G + h0] = m0;
                red_l[warp * G + h0] = l0;
            }
            if (h1 < G) {
                red_m[warp * G + h1] = m1;
                red_l[warp * G + h1] = l1;
            }
        }
        // MMA rows g and g+8 are dims g and g+8 of the 16-dim tile (FP8: dims 2g, 2g+1)
        const int dA = F8 ? 2 * g : g, dB = F8 ? 2 * g + 1 : g + 8;
        const float vs = F8 ? __ldg(p.v_scale + kvh) : 1.f;
#pragma unroll
        for (int mt = 0; mt < KSTEPS; ++mt) {
            if (h0 < G) {
                red_acc[(warp * G + h0) * D + mt * 16 + dA] = acc[mt][0] * vs;
                red_acc[(warp * G + h0) * D + mt * 16 + dB] = acc[mt][2] * vs;
            }
            if (h1 < G) {
                red_acc[(warp * G + h1) * D + mt * 16 + dA] = acc[mt][1] * vs;
                red_acc[(warp * G + h1) * D + mt * 16 + dB] = acc[mt][3] * vs;
            }
        }
        __syncthreads();

        const bool direct = n_parts == 1;
        for (int idx = tid; idx < G * D; idx += blockDim.x) {
            const int hh = idx / D, d = idx - hh * D;
            float M = -INFINITY;
#pragma unroll
            for (int w = 0; w < NW; ++w) M = fmaxf(M, red_m[w * G + hh]);
            float num = 0.f, den = 0.f;
            if (M != -INFINITY) {
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    const float f = exp2f(red_m[w * G + hh] - M);
                    num = fmaf(f, red_acc[(w * G + hh) * D + d], num);
                    den = fmaf(f, red_l[w * G + hh], den);
                }
            }
            if (direct) {
                out_rows[idx] = Elt<T>::from_f32(den > 0.f ? num / den : 0.f);
            } else {
                const size_t row = (static_cast<size_t>(s) * p.hq + kvh * G + hh) * p.max_partitions + part;
                p.ws_acc[row * D + d] = num;
                if (d == 0) {
                    p.ws_ml[row * 2] = M;
                    p.ws_ml[row * 2 + 1] = den;
                }
            }
        }
        // every thread leaves the merge before the next head's warps write the scratch, and a
        // timeout anywhere ends the CTA after this head (uniform: read after the barrier)
        if (u + 1 < nh) {
            __shared__ int s_abort;
            if (tid == 0) s_abort = 0;
            __syncthreads();
            if (aborted) s_abort = 1;
            __syncthreads();
            if (s_abort) break;
        }
    }
}

template <typename T, typename PE, int D, int G>
cudaError_t launch_mma(const DecodeParams& p_in, const CUtensorMap& kmap, const CUtensorMap& vmap,
                       cudaStream_t stream) {
    using C = MmaCfg<PE, D, G>;
    DecodeParams p = p_in;
    const int entries = p.partition_tokens / p.block_size;
    static int configured_for = -1;  // device on which the attribute was last set
    static int cached_entries = -1, cached_hpc = 1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_for != dev) {
        cudaError_t e = cudaFuncSetAttribute(decode_partition_mma<T, PE, D, G>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(C::smem_bytes(kMaxPartitionTokens / 16, 2)));
        if (e != cudaSuccess) return e;
        configured_for = dev;
        cached_entries = -1;
    }
    if (cached_entries != entries) {
        // two KV heads per CTA (table staged once, the ring streaming on into the second head)
        // when the merge scratch it needs of its own costs no resident CTA
        int occ1 = 0, occ2 = 0;
        cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ1, decode_partition_mma<T, PE, D, G>,
                                                                      C::NW * 32, C::smem_bytes(entries, 1));
        if (e == cudaSuccess)
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ2, decode_partition_mma<T, PE, D, G>, C::NW * 32,
                                                              C::smem_bytes(entries, 2));
        if (e != cudaSuccess) return e;
        if (e != cudaSuccess) return e;
        cached_hpc = occ2 >= occ1 ? 2 : 1;
        cached_entries = entries;
    }
#ifdef PA_MMA_HEADS
    p.heads_per_cta = PA_MMA_HEADS;  // build-time override (tuning sweeps)
#else
    // two heads per CTA when it costs no resident CTA per SM, unless the caller forced 1 or 2
    if (p.heads_per_cta != 1 && p.heads_per_cta != 2) p.heads_per_cta = cached_hpc;
    if (p.hkv < 2) p.heads_per_cta = 1;
#endif
    const size_t smem = C::smem_bytes(entries, p.heads_per_cta);
    dim3 grid(p.max_partitions, (p.hkv + p.heads_per_cta - 1) / p.heads_per_cta, p.batch);
    cudaError_t e =
        launch_pdl(decode_partition_mma<T, PE, D, G>, grid, dim3(C::NW * 32), smem, stream, p, kmap, vmap);
    if (e != cudaSuccess || p.max_partitions <= 1) return e;
    return launch_merge<T, D>(p, stream);
}

}  // namespace pa
