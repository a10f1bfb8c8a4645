// Paged prefill on the fifth-generation tensor cores: tcgen05.mma with the
// accumulators in tensor memory (TMEM), operands staged in shared memory by
// TMA, for fp16 / bf16 pools with D in {64, 128}.
//
// Same operation as prefill_mma.cuh (causal attention of each sequence's
// chunk over its paged history plus the chunk, "25. Paged attention and
// prefix caching", stretch exercise 4; "Chapter 7 Paged KV Cache and Memory
// Management", 4.1 step 3), same packing of rows: one CTA owns 128 query rows
// -- (chunk token, query head of the group) pairs -- of one KV head.
//
// One CTA owns 256 query rows of one KV head as two 128-row tiles X = A, B that
// share every K/V tile staged in shared memory (twice the FLOPs per copied byte
// of a single tile).  Per 64-key tile j of the history (a TMA ring of K/V
// stages, each 16-key sub-tile fetched through the block table), for each X:
//   S_Xj = Q_X . K_j^T   tcgen05.mma M=128 N=64, A = Q_X (smem, K-major), B = K_j (smem,
//                        K-major), into one of two TMEM S buffers of tile X;
//   softmax              one thread per row (group X = warps 4X .. 4X+3): tcgen05.ld of its
//                        64 scores, causal mask, running max (base 2, lazy rescale of O_X
//                        only when the max grows by more than 2^8), P_Xj = exp2(s - m)
//                        rounded to the dtype and stored over the first half of S_Xj;
//   O_X += P_Xj . V_j    tcgen05.mma M=128 N=D, A = P_Xj (tensor memory), B = V_j (smem,
//                        MN-major: keys are the K dimension).
// Warps: 0-7 softmax (warp w: tile w / 4, rows 32 (w % 4) .. +31 = its TMEM lanes),
// 8 producer (TMA, four lanes issuing), 9 MMA issuer (one lane, fixed order one
// K/V tile ahead: S_A(j+1) and S_B(j+1), then P_A(j) . V_j and P_B(j) . V_j; a
// K/V stage is released once both tiles' P . V on it have completed).  The
// 128-key kernel (prefill_tc05w.cuh) is the default at D = 128; this one serves
// D = 64 and D = 128 when forced.
// Hand-offs are mbarriers: TMA bytes (kv_full), MMA completion through
// tcgen05.commit (s_full, o_ready per tile, o_final, kv_empty), softmax arrivals
// (p_full).  Every wait is bounded (1 s of %globaltimer, PA_DEVERR_TIMEOUT), and no
// barrier phase can run two ahead of a waiter's parity.
//
// Shared-memory operands use the 128-byte swizzle (the TMA layout): rows of
// 128 bytes, 8-row atoms of 1024 bytes.  Descriptor: start >> 4, leading
// byte offset >> 4 at bit 16, stride byte offset (8-row atom step) >> 4 at
// bit 32, version 1 at bit 46, layout 2 (128B swizzle) at bit 61; K-steps of
// 16 elements advance the start address by 32 bytes inside the atom.
#pragma once

#include "prefill_mma.cuh"

namespace pa {
namespace tc05 {

__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

template <typename T>
struct Fmt;
template <>
struct Fmt<__half> {
    static constexpr uint32_t v = 0;
};
template <>
struct Fmt<__nv_bfloat16> {
    static constexpr uint32_t v = 1;
};

// instruction descriptor of kind::f16: fp32 accumulate, A K-major, M = 128
template <typename T>
constexpr uint32_t idesc(int n, bool b_mn_major) {
    return (1u << 4) | (Fmt<T>::v << 7) | (Fmt<T>::v << 10) | ((b_mn_major ? 1u : 0u) << 16) |
           (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(128 >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t id, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(id), "r"(accumulate)
        : "memory");
}

// A operand in tensor memory: row m at lane m, two 16-bit values per column (low half = even k)
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t id,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b), "r"(id), "r"(accumulate)
        : "memory");
}

// arrives on `bar` once every tcgen05 operation this thread issued before has completed
__device__ __forceinline__ void commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void ld32(uint32_t addr, uint32_t* r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(addr));
}

__device__ __forceinline__ void st32(uint32_t addr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(addr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void st16(uint32_t addr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16};" ::"r"(addr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// non-blocking test of a phase (try_wait may suspend the thread for a while when the phase is
// not complete, which a loop polling two barriers cannot afford)
__device__ __forceinline__ bool test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// 2^x by the MUFU approximation (relative error ~2^-22; 2^-inf = 0)
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// barrier `id` over `count` threads that also ANDs `pred` over them
__device__ __forceinline__ bool bar_and(int id, int count, bool pred) {
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.and.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(out)
        : "r"(static_cast<uint32_t>(pred)), "r"(id), "r"(count)
        : "memory");
    return out != 0;
}

__device__ __forceinline__ void named_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace tc05

template <int D>
struct Tc05Cfg {
    static constexpr int BM = 256, BN = 64;  // two 128-row query tiles; 64 keys per K/V tile
    static constexpr int NSB = 2;            // S buffers per query tile (P_j overwrites the first half of S_j)
#ifdef PA_TC05_STAGES
    static constexpr int STAGES = PA_TC05_STAGES;  // build-time override (tuning sweeps)
#else
    static constexpr int STAGES = D == 64 ? 8 : 4;
#endif
    static constexpr int NBOX = D / 64;
    static constexpr int QBOX = 128 * 128;           // 128 rows x 128 B
    static constexpr int Q_BYTES = 2 * NBOX * QBOX;  // both tiles
    static constexpr int KV_BOX = BN * 128;          // 64 keys x 128 B
    static constexpr int K_BYTES = NBOX * KV_BOX;
    static constexpr int STAGE_BYTES = 2 * K_BYTES;  // K then V
    static constexpr int KV_OFF = Q_BYTES;
    static constexpr int BAR_OFF = KV_OFF + STAGES * STAGE_BYTES;
    // kv_full, kv_empty [STAGES]; s_full, p_full [2 tiles x NSB]; o_ready [2]; o_final; q_full
    static constexpr int NBARS = 2 * STAGES + 4 * NSB + 2 + 2;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr size_t smem_bytes = 1024 + MISC_OFF + 16 + 4 * STAGES;
    // tensor memory columns: O_A [0, D), O_B [D, 2D), S buffers of tile X at 2D + (X NSB + b) 64
    static constexpr int O_COL = 0, S_COL = 2 * D;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int NSW = 8;  // softmax warps: two groups of four, one thread per row
    static constexpr int PRODUCER = NSW, ISSUER = NSW + 1;
    static constexpr int THREADS = (NSW + 2) * 32;
    static_assert(D == 64 || D == 128, "D in {64, 128}");
    static_assert(S_COL + 2 * NSB * BN <= 512, "tensor memory columns");
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(Tc05Cfg<D>::THREADS, 1)
    prefill_tc05(const PrefillParams p, const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap vmap) {
    using C = Tc05Cfg<D>;
    constexpr int STAGES = C::STAGES, NBOX = C::NBOX, BN = C::BN, NSB = C::NSB;
    constexpr int QT = C::BM / G;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint64_t* kv_full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* kv_empty = kv_full + STAGES;
    uint64_t* s_full = kv_empty + STAGES;  // [X * NSB + b]
    uint64_t* p_full = s_full + 2 * NSB;
    uint64_t* o_ready = p_full + 2 * NSB;  // [X]
    uint64_t* o_final = o_ready + 2;
    uint64_t* q_full = o_final + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
    int* stage_ok = reinterpret_cast<int*>(smem + C::MISC_OFF + 16);  // loaded 16-key sub-tiles (bit mask)

    griddep_wait();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = blockIdx.z, kvh = blockIdx.y;
    const int tile = gridDim.x - 1 - blockIdx.x;  // the tiles with the most keys start first
    const int q0 = __ldg(p.qstart + s), q1 = __ldg(p.qstart + s + 1);
    const int L = __ldg(p.seq_lens + s);
    const int Cq = q1 - q0;
    if (L < 0 || L > p.max_blocks * p.block_size || Cq < 0 || Cq > L || q0 < 0 || q1 > p.total_q) {
        if (tid == 0 && blockIdx.x == 0 && kvh == 0) flag_error(p.err, PA_DEVERR_SEQLEN);
        return;  // uniform over the CTA
    }
    const int tok0 = tile * QT;
    if (tok0 >= Cq) return;  // uniform
    const int base = L - Cq;  // position of chunk token 0
    const int kv_end = base + min(Cq, tok0 + QT);
    const int n_kv = (kv_end + BN - 1) / BN;

    if (tid == 0) {
#pragma unroll
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&kv_full[i], 1);
            mbar_init(&kv_empty[i], 1);
        }
#pragma unroll
        for (int i = 0; i < 2 * NSB; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 128);
        }
        mbar_init(&o_ready[0], 1);
        mbar_init(&o_ready[1], 1);
        mbar_init(o_final, 1);
        mbar_init(q_full, C::NSW * 32);
        fence_mbar_init();
    }
    if (warp == C::ISSUER) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                     "r"(C::TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc05::fence_before();
    __syncthreads();
    tc05::fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sbase = smem_u32(smem);

    if (warp == C::PRODUCER) {
        // ------------------------------------------------------------ producer
        const int32_t* trow = p.block_tables + static_cast<size_t>(s) * p.max_blocks;
        const int n_sub = n_kv * 4;
        bool ok = true;
        for (int u0 = 0; u0 < n_sub && ok; u0 += 32) {
            // lane i resolves 16-key sub-tile u0 + i (-1: beyond the sequence or a bad entry)
            int row = -1;
            const int u = u0 + lane;
            if (u < n_sub && u * 16 < L) {
                const int e = __ldg(trow + (u * 16) / p.block_size);
                if (e >= 0 && e < p.num_blocks) {
                    row = (e * p.hkv + kvh) * p.block_size + (u * 16) % p.block_size;
                } else {
                    flag_error(p.err, PA_DEVERR_TABLE);
                }
            }
            for (int t0 = 0; t0 < 32 && u0 + t0 < n_sub; t0 += 4) {  // one 64-key tile per 4 lanes
                const int j = (u0 + t0) / 4;
                const int st = j % STAGES;
                const int my_row = __shfl_sync(0xffffffffu, row, t0 + (lane & 3));
                const unsigned mask = __ballot_sync(0xffffffffu, my_row >= 0) & 0xFu;
                if (lane == 0 && ok) {
                    if (!mbar_wait_bounded(&kv_empty[st], ((j / STAGES) & 1) ^ 1)) {
                        flag_error(p.err, PA_DEVERR_TIMEOUT);
                        ok = false;
                    } else {
                        stage_ok[st] = static_cast<int>(mask);
                        // the stage's byte count is posted before any of its copies is issued
                        mbar_arrive_expect_tx(&kv_full[st], static_cast<uint32_t>(__popc(mask) * 2 * NBOX * 2048));
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                // lanes 0-3 issue the copies of sub-tiles 0-3 side by side
                if (ok && lane < 4 && my_row >= 0) {
                    unsigned char* kd = smem + C::KV_OFF + st * C::STAGE_BYTES + lane * 2048;
#pragma unroll
                    for (int bx = 0; bx < NBOX; ++bx) {
                        tma_load_2d(kd + bx * C::KV_BOX, &kmap, bx * 64, my_row, &kv_full[st]);
                        tma_load_2d(kd + C::K_BYTES + bx * C::KV_BOX, &vmap, bx * 64, my_row, &kv_full[st]);
                    }
                }
                __syncwarp();
            }
        }
        return;  // every copy issued is waited for by the MMA warp before the kernel ends
    }

    if (warp == C::ISSUER) {
        // ------------------------------------------------------------ MMA issuer (one lane)
        // Fixed order, one K/V tile ahead: S_A(j+1) and S_B(j+1) back to back as soon as K_(j+1)
        // has landed, then O_A += P_Aj V_j and O_B += P_Bj V_j as each softmax group delivers.
        // The softmax of tile j then overlaps P.V of tile j-1 and the scores of tile j+1 on the
        // tensor pipe.  S buffer (j+1) % NSB held P_(j-1), whose P.V was issued before (the
        // pipe executes one thread's MMAs in order).
        if (lane == 0) {
            constexpr uint32_t ID_S = tc05::idesc<T>(BN, false);
            constexpr uint32_t ID_PV = tc05::idesc<T>(D, true);
            bool ok = mbar_wait_bounded(q_full, 0);
            tc05::fence_after();
            // Descriptors are formed once; an operand at byte offset o from a base has the base's
            // descriptor plus o / 16 (shared addresses stay below 2^18, so the 14-bit start field
            // never carries).  This keeps the issuing thread's instructions per MMA few: it shares
            // its scheduler with two softmax warps.
            const uint64_t q_desc = tc05::sdesc(sbase, 16, 1024);
            const uint64_t k_desc = tc05::sdesc(sbase + C::KV_OFF, 16, 1024);
            const uint64_t v_desc = tc05::sdesc(sbase + C::KV_OFF + C::K_BYTES, C::KV_BOX, 1024);
            auto issue_s = [&](int j) {
                const uint64_t kst = k_desc + static_cast<uint64_t>((j % STAGES) * (C::STAGE_BYTES >> 4));
#pragma unroll
                for (int X = 0; X < 2; ++X) {
                    const uint32_t sd = tmem + C::S_COL + (X * NSB + j % NSB) * BN;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint64_t a = q_desc + static_cast<uint64_t>((X * NBOX * C::QBOX + (ks >> 2) * C::QBOX + (ks & 3) * 32) >> 4);
                        const uint64_t b = kst + static_cast<uint64_t>(((ks >> 2) * C::KV_BOX + (ks & 3) * 32) >> 4);
                        tc05::mma(sd, a, b, ID_S, ks > 0);
                    }
                    tc05::commit(&s_full[X * NSB + j % NSB]);
                }
            };
            // kv_full of tile j cannot complete another phase before kv_empty of tile j is
            // committed (below, after both P.V of tile j), so each wait's parity is unambiguous
            if (ok && n_kv > 0) {
                ok = mbar_wait_bounded(&kv_full[0], 0);
                if (ok) {
                    tc05::fence_after();
                    issue_s(0);
                }
            }
            for (int j = 0; ok && j < n_kv; ++j) {
                if (j + 1 < n_kv) {
                    ok = mbar_wait_bounded(&kv_full[(j + 1) % STAGES], ((j + 1) / STAGES) & 1);
                    if (!ok) break;
                    tc05::fence_after();
                    issue_s(j + 1);
                }
                const int st = j % STAGES;
                const uint64_t vst = v_desc + static_cast<uint64_t>(st * (C::STAGE_BYTES >> 4));
#pragma unroll
                for (int X = 0; X < 2; ++X) {
                    // P_X(j + NSB) needs S_X(j + NSB), issued after this P.V: at most one phase ahead
                    ok = mbar_wait_bounded(&p_full[X * NSB + j % NSB], (j / NSB) & 1);
                    if (!ok) break;
                    tc05::fence_after();
                    const uint32_t pa = tmem + C::S_COL + (X * NSB + j % NSB) * BN;  // key k at column k / 2
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk) {
                        // N = D in one MMA: the 64-dim boxes of V are KV_BOX apart (leading byte offset)
                        const uint64_t b = vst + static_cast<uint64_t>((kk * 2048) >> 4);
                        tc05::mma_ts(tmem + C::O_COL + X * D, pa + kk * 8, b, ID_PV, (j > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc05::commit(&o_ready[X]);
                }
                if (!ok) break;
                tc05::commit(&kv_empty[st]);  // the stage is free once both tiles' P.V on it complete
            }
            if (ok) tc05::commit(o_final);
            else flag_error(p.err, PA_DEVERR_TIMEOUT);
        }
        __syncwarp();
        tc05::named_sync(1, (C::NSW + 1) * 32);
        tc05::fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS)
                     : "memory");
        return;
    }

    // ------------------------------------------------------------ softmax warps (thread = row)
    const int X = warp >> 2, r = tid & 127;  // query tile, row within it
    const int wq = warp & 3;
    const int prow_id = X * 128 + r;  // packed row of the CTA
    const int tok = tok0 + prow_id / G;
    const bool valid = tok < Cq;
    const int pos = valid ? base + tok : -1;
    const int head = kvh * G + prow_id % G;
    // position of the first row of this warp's 32 (every valid row of the warp is at or after it)
    const int warp_tok = tok0 + (X * 128 + wq * 32) / G;
    const int warp_pos_min = warp_tok < Cq ? base + warp_tok : -1;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t o_addr = lane_addr + C::O_COL + X * D;
    {
        // Q row into tile X's K-major swizzled operand (zeros past the chunk)
        const uint4* qrow =
            reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) + (static_cast<size_t>(q0 + (valid ? tok : 0)) * p.hq + head) * D);
        unsigned char* qx = smem + X * NBOX * C::QBOX;
#pragma unroll
        for (int cc = 0; cc < D / 8; ++cc) {
            const int bx = cc >> 3, c = cc & 7;
            const uint4 v = valid ? __ldg(qrow + cc) : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(qx + bx * C::QBOX + r * 128 + ((c ^ (r & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
        mbar_arrive(q_full);
    }
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
        const int st = j % STAGES, sb = X * NSB + j % NSB;
        // decisions that guard a tcgen05.ld / st are warp-uniform (those are .sync.aligned)
        // neither can run two phases ahead: tile j + STAGES is loaded, and S_X(j + NSB) issued,
        // only after this thread's P_Xj has been consumed
        const bool got = mbar_wait_bounded(&kv_full[st], (j / STAGES) & 1) && mbar_wait_bounded(&s_full[sb], (j / NSB) & 1);
        if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
        }
        tc05::fence_after();
        const int key0 = j * BN;
        const int okmask = stage_ok[st];
        const uint32_t sa = lane_addr + C::S_COL + sb * BN;
        uint32_t sr[64];
        tc05::ld32(sa, sr);
        tc05::ld32(sa + 32, sr + 32);
        tc05::wait_ld();
        // interior tile: every valid row of the warp sees all 64 keys and the scale is positive,
        // so the row max is the raw max times the scale; masked tiles keep their scores
        // pre-scaled (masked: -inf) in sr
        const bool interior = okmask == 0xF && key0 + BN - 1 <= warp_pos_min && sl2 > 0.f;
        float mx;
        {
            float t[8];
            if (interior) {
#pragma unroll
                for (int i = 0; i < 8; ++i) t[i] = __uint_as_float(sr[i]);
#pragma unroll
                for (int c = 8; c < 64; ++c) t[c & 7] = fmaxf(t[c & 7], __uint_as_float(sr[c]));
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) t[i] = -INFINITY;
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    const bool vis = key0 + c <= pos && ((okmask >> (c >> 4)) & 1);
                    const float x = vis ? __uint_as_float(sr[c]) * sl2 : -INFINITY;
                    sr[c] = __float_as_uint(x);
                    t[c & 7] = fmaxf(t[c & 7], x);
                }
            }
            mx = fmaxf(fmaxf(fmaxf(t[0], t[1]), fmaxf(t[2], t[3])), fmaxf(fmaxf(t[4], t[5]), fmaxf(t[6], t[7])));
            if (interior) mx *= sl2;
        }
        // lazy rescale per row; O_X (in TMEM) is rescaled for the whole warp when any row needs
        // it, once P_X(j-1) . V_(j-1) has landed, each lane by its own factor
        const bool grow = mx > m + kLazyRescale;
        const bool scale_o = grow && m != -INFINITY;
        const float a = scale_o ? tc05::fast_exp2(m - mx) : 1.f;
        if (j > 0 && __any_sync(0xffffffffu, scale_o)) {
            // o_ready[X] counts tile X's P . V in order: the one of tile j needs this thread's P_Xj,
            // and the one of tile j - 2 completed before S_Xj (issued after it)
            if (!__all_sync(0xffffffffu, mbar_wait_bounded(&o_ready[X], (j - 1) & 1))) {
                ok = false;
                break;
            }
            tc05::fence_after();
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tc05::ld32(o_addr + c0, o);
                tc05::wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * a);
                tc05::st32(o_addr + c0, o);
            }
        }
        if (grow) {
            l *= a;
            m = mx;
        }
        const float ms = m == -INFINITY ? 0.f : m;
        // P = 2^(v * mul - m) in one FFMA and one ex2 (interior: v raw, mul = scale; masked: v
        // pre-scaled, mul = 1); key c at column c / 2 of S buffer sb, over this lane's own scores
        const float mul = interior ? sl2 : 1.f;
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int hq = 0; hq < 2; ++hq) {
            uint32_t pw[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int c = hq * 32 + 2 * i;
                const float e0 = tc05::fast_exp2(fmaf(__uint_as_float(sr[c]), mul, -ms));
                const float e1 = tc05::fast_exp2(fmaf(__uint_as_float(sr[c + 1]), mul, -ms));
                ls[i & 3] += e0 + e1;
                pw[i] = pack2<T>(e0, e1);
            }
            tc05::st16(sa + hq * 16, pw);
        }
        l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        // V rows of keys past the sequence or of sub-tiles not loaded may hold anything: zero
        // them (both groups write the same zeros; each P . V waits only for its own group's)
        if (key0 + BN > L || okmask != 0xF) {
            unsigned char* vt = smem + C::KV_OFF + st * C::STAGE_BYTES + C::K_BYTES;
            for (int e = r; e < BN * NBOX * 8; e += 128) {
                const int key = e / (NBOX * 8), rest = e % (NBOX * 8);
                if (key0 + key >= L || !((okmask >> (key >> 4)) & 1))
                    *reinterpret_cast<uint4*>(vt + (rest >> 3) * C::KV_BOX + key * 128 + (rest & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
        }
        tc05::wait_st();
        tc05::fence_before();
        mbar_arrive(&p_full[sb]);
    }
    griddep_launch_dependents();
    const bool all_ok = tc05::bar_and(2, C::NSW * 32, ok);
    const bool done = all_ok && mbar_wait_bounded(o_final, 0);
    if (__all_sync(0xffffffffu, done)) {
        tc05::fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        T* orow = static_cast<T*>(p.out) + (static_cast<size_t>(q0 + (valid ? tok : 0)) * p.hq + head) * D;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tc05::ld32(o_addr + c0, o);
            tc05::wait_ld();
            if (valid) {
#pragma unroll
                for (int i = 0; i < 32; i += 8) {
                    uint4 u;
                    u.x = pack2<T>(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv);
                    u.y = pack2<T>(__uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv);
                    u.z = pack2<T>(__uint_as_float(o[i + 4]) * inv, __uint_as_float(o[i + 5]) * inv);
                    u.w = pack2<T>(__uint_as_float(o[i + 6]) * inv, __uint_as_float(o[i + 7]) * inv);
                    *reinterpret_cast<uint4*>(orow + c0 + i) = u;
                }
            }
        }
    } else if (lane == 0) {
        flag_error(p.err, PA_DEVERR_TIMEOUT);
    }
    tc05::fence_before();
    tc05::named_sync(1, (C::NSW + 1) * 32);
}

template <typename T, int D, int G>
cudaError_t launch_prefill_tc05(const PrefillParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                int max_query_len, cudaStream_t stream) {
    using C = Tc05Cfg<D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc05<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(C::smem_bytes));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int64_t rows = static_cast<int64_t>(max_query_len) * G;
    const unsigned tiles = static_cast<unsigned>((rows + C::BM - 1) / C::BM);
    return launch_pdl(prefill_tc05<T, D, G>, dim3(tiles, p.hkv, p.batch), dim3(C::THREADS), C::smem_bytes, stream,
                      p, kmap, vmap);
}

}  // namespace pa
