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
// Per 64-key tile j of the history (a 3-stage TMA ring, each 16-key sub-tile
// fetched through the block table):
//   S_j = Q . K_j^T     tcgen05.mma M=128 N=64, A = Q (smem, K-major), B = K_j (smem, K-major)
//                       into one of two TMEM S buffers, so the tensor core
//                       computes S_{j+1} while the softmax threads read S_j;
//   softmax             one thread per row: tcgen05.ld of its 64 scores,
//                       causal mask, running max (base 2, lazy rescale of O
//                       in TMEM only when the max grows by more than 2^8),
//                       P_j = exp2(s - m) rounded to the dtype into shared
//                       memory as a K-major operand;
//   O += P_j . V_j      tcgen05.mma M=128 N=64 per 64 dims, A = P_j (smem),
//                       B = V_j (smem, MN-major: keys are the K dimension).
// Warps: 0-3 softmax (thread = row = TMEM lane), 4 producer (TMA), 5 MMA
// issuer (one lane).  Hand-offs are mbarriers: TMA bytes (kv_full), MMA
// completion through tcgen05.commit (s_full, o_ready, kv_empty), softmax
// arrivals (p_full).  Barriers whose phases a waiter may skip come in pairs
// by tile parity, so a parity wait never meets a barrier two phases ahead.
// Every wait is bounded (1 s of %globaltimer, PA_DEVERR_TIMEOUT).
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

__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void named_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

}  // namespace tc05

template <int D>
struct Tc05Cfg {
    static constexpr int BM = 128, BN = 64, STAGES = 3;
    static constexpr int NBOX = D / 64;
    static constexpr int Q_BYTES = NBOX * BM * 128;  // boxes of 128 rows x 128 B
    static constexpr int KV_BOX = BN * 128;          // 64 keys x 128 B
    static constexpr int K_BYTES = NBOX * KV_BOX;
    static constexpr int STAGE_BYTES = 2 * K_BYTES;  // K then V
    static constexpr int P_BYTES = BM * BN * 2;      // 128 rows x 64 keys x 16 bit
    static constexpr int KV_OFF = Q_BYTES;
    static constexpr int P_OFF = KV_OFF + STAGES * STAGE_BYTES;
    static constexpr int BAR_OFF = P_OFF + 2 * P_BYTES;
    static constexpr int NBARS = 2 * STAGES + 2 + 2 + 2 + 1;  // kv_full, kv_empty, s_full, p_full, o_ready, q_full
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr size_t smem_bytes = 1024 + MISC_OFF + 16 + STAGES * 4;
    static constexpr int O_COL = 2 * BN;
    static constexpr uint32_t TMEM_COLS = 2 * BN + D <= 256 ? 256u : 512u;
    static constexpr int THREADS = 192;
    static_assert(D == 64 || D == 128, "D in {64, 128}");
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(Tc05Cfg<D>::THREADS, 1)
    prefill_tc05(const PrefillParams p, const __grid_constant__ CUtensorMap kmap,
                 const __grid_constant__ CUtensorMap vmap) {
    using C = Tc05Cfg<D>;
    constexpr int STAGES = C::STAGES, NBOX = C::NBOX, BN = C::BN;
    constexpr int QT = C::BM / G;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint64_t* kv_full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* kv_empty = kv_full + STAGES;
    uint64_t* s_full = kv_empty + STAGES;
    uint64_t* p_full = s_full + 2;
    uint64_t* o_ready = p_full + 2;
    uint64_t* q_full = o_ready + 2;
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
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&p_full[i], 128);
            mbar_init(&o_ready[i], 1);
        }
        mbar_init(q_full, 128);
        fence_mbar_init();
    }
    if (warp == 5) {
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

    if (warp == 4) {
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
                int r4[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) r4[i] = __shfl_sync(0xffffffffu, row, t0 + i);
                if (lane == 0 && ok) {
                    const int st = j % STAGES;
                    if (!mbar_wait_bounded(&kv_empty[st], ((j / STAGES) & 1) ^ 1)) {
                        flag_error(p.err, PA_DEVERR_TIMEOUT);
                        ok = false;
                    } else {
                        int mask = 0, n = 0;
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (r4[i] >= 0) {
                                mask |= 1 << i;
                                ++n;
                            }
                        stage_ok[st] = mask;
                        mbar_arrive_expect_tx(&kv_full[st], static_cast<uint32_t>(n * 2 * NBOX * 2048));
                        unsigned char* kd = smem + C::KV_OFF + st * C::STAGE_BYTES;
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            if (r4[i] < 0) continue;
#pragma unroll
                            for (int bx = 0; bx < NBOX; ++bx) {
                                tma_load_2d(kd + bx * C::KV_BOX + i * 2048, &kmap, bx * 64, r4[i], &kv_full[st]);
                                tma_load_2d(kd + C::K_BYTES + bx * C::KV_BOX + i * 2048, &vmap, bx * 64, r4[i],
                                            &kv_full[st]);
                            }
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
            }
        }
        return;  // every copy issued is waited for by the MMA warp before the kernel ends
    }

    if (warp == 5) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t ID_S = tc05::idesc<T>(BN, false);
            constexpr uint32_t ID_PV = tc05::idesc<T>(64, true);
            bool ok = mbar_wait_bounded(q_full, 0);
            tc05::fence_after();
            for (int j = 0; j <= n_kv && ok; ++j) {
                if (j < n_kv) {
                    const int st = j % STAGES;
                    if (!mbar_wait_bounded(&kv_full[st], (j / STAGES) & 1)) {
                        ok = false;
                        break;
                    }
                    tc05::fence_after();
                    const uint32_t kb = sbase + C::KV_OFF + st * C::STAGE_BYTES;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        const uint64_t a = tc05::sdesc(sbase + (ks >> 2) * (C::BM * 128) + (ks & 3) * 32, 16, 1024);
                        const uint64_t b = tc05::sdesc(kb + (ks >> 2) * C::KV_BOX + (ks & 3) * 32, 16, 1024);
                        tc05::mma(tmem + (j & 1) * BN, a, b, ID_S, ks > 0);
                    }
                    tc05::commit(&s_full[j & 1]);
                }
                if (j >= 1) {
                    const int jj = j - 1;
                    if (!mbar_wait_bounded(&p_full[jj & 1], (jj >> 1) & 1)) {
                        ok = false;
                        break;
                    }
                    tc05::fence_after();
                    const int st = jj % STAGES;
                    const uint32_t vb = sbase + C::KV_OFF + st * C::STAGE_BYTES + C::K_BYTES;
                    const uint32_t pb = sbase + C::P_OFF + (jj & 1) * C::P_BYTES;
#pragma unroll
                    for (int kk = 0; kk < BN / 16; ++kk) {
                        const uint64_t a = tc05::sdesc(pb + kk * 32, 16, 1024);
#pragma unroll
                        for (int bx = 0; bx < NBOX; ++bx) {
                            const uint64_t b = tc05::sdesc(vb + bx * C::KV_BOX + kk * 2048, C::KV_BOX, 1024);
                            tc05::mma(tmem + C::O_COL + bx * 64, a, b, ID_PV, (jj > 0 || kk > 0) ? 1u : 0u);
                        }
                    }
                    tc05::commit(&o_ready[jj & 1]);
                    tc05::commit(&kv_empty[st]);
                }
            }
            if (!ok) flag_error(p.err, PA_DEVERR_TIMEOUT);
        }
        __syncwarp();
        tc05::named_sync(1, 160);
        tc05::fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(C::TMEM_COLS)
                     : "memory");
        return;
    }

    // ------------------------------------------------------------ softmax warps (thread = row)
    const int r = tid;
    const int tok = tok0 + r / G;
    const bool valid = tok < Cq;
    const int pos = valid ? base + tok : -1;
    const int head = kvh * G + r % G;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    {
        // this row of Q into the K-major swizzled operand (zeros for rows past the chunk)
        const uint4* qrow =
            reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) + (static_cast<size_t>(q0 + (valid ? tok : 0)) * p.hq + head) * D);
#pragma unroll
        for (int bx = 0; bx < NBOX; ++bx)
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 v = valid ? __ldg(qrow + bx * 8 + c) : make_uint4(0u, 0u, 0u, 0u);
                *reinterpret_cast<uint4*>(smem + bx * (C::BM * 128) + r * 128 + ((c ^ (r & 7)) << 4)) = v;
            }
        fence_proxy_async_smem();
        mbar_arrive(q_full);
    }
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
        const int st = j % STAGES;
        // every decision that guards a tcgen05.ld / st is warp-uniform (those are .sync.aligned)
        bool got = mbar_wait_bounded(&kv_full[st], (j / STAGES) & 1) && mbar_wait_bounded(&s_full[j & 1], (j >> 1) & 1);
        if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
        }
        tc05::fence_after();
        const int key0 = j * BN;
        const int okmask = stage_ok[st];
        uint32_t sr[64];
        tc05::ld32(lane_addr + (j & 1) * BN, sr);
        tc05::ld32(lane_addr + (j & 1) * BN + 32, sr + 32);
        tc05::wait_ld();
        float sv[64];
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
            const bool vis = key0 + c <= pos && ((okmask >> (c >> 4)) & 1);
            sv[c] = vis ? __uint_as_float(sr[c]) * sl2 : -INFINITY;
            mx = fmaxf(mx, sv[c]);
        }
        // lazy rescale per row; O (in TMEM) is rescaled for the whole warp when any row needs it,
        // once P_{j-1} . V_{j-1} has landed, each lane by its own factor (1 when it keeps its max)
        const bool grow = mx > m + kLazyRescale;
        const bool scale_o = grow && m != -INFINITY;
        const float a = scale_o ? exp2f(m - mx) : 1.f;
        if (j > 0 && __any_sync(0xffffffffu, scale_o)) {
            got = mbar_wait_bounded(&o_ready[(j - 1) & 1], ((j - 1) >> 1) & 1);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc05::fence_after();
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                uint32_t o[32];
                tc05::ld32(lane_addr + C::O_COL + c0, o);
                tc05::wait_ld();
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * a);
                tc05::st32(lane_addr + C::O_COL + c0, o);
            }
            tc05::wait_st();
        }
        if (grow) {
            l *= a;
            m = mx;
        }
        const float ms = m == -INFINITY ? 0.f : m;
        unsigned char* prow = smem + C::P_OFF + (j & 1) * C::P_BYTES + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float e0 = exp2f(sv[c * 8 + 2 * i] - ms), e1 = exp2f(sv[c * 8 + 2 * i + 1] - ms);
                l += e0 + e1;
                w[i] = pack2<T>(e0, e1);
            }
            *reinterpret_cast<uint4*>(prow + ((c ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        // V rows of keys past the sequence or of sub-tiles not loaded may hold anything: zero them
        if (key0 + BN > L || okmask != 0xF) {
            unsigned char* vt = smem + C::KV_OFF + st * C::STAGE_BYTES + C::K_BYTES;
            for (int e = r; e < BN * NBOX * 8; e += 128) {
                const int key = e / (NBOX * 8), rest = e % (NBOX * 8);
                if (key0 + key >= L || !((okmask >> (key >> 4)) & 1))
                    *reinterpret_cast<uint4*>(vt + (rest >> 3) * C::KV_BOX + key * 128 + (rest & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
            }
        }
        fence_proxy_async_smem();
        tc05::fence_before();
        mbar_arrive(&p_full[j & 1]);
    }
    griddep_launch_dependents();
    if (ok) ok = mbar_wait_bounded(&o_ready[(n_kv - 1) & 1], ((n_kv - 1) >> 1) & 1);
    if (__all_sync(0xffffffffu, ok)) {
        tc05::fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        T* orow = static_cast<T*>(p.out) + (static_cast<size_t>(q0 + (valid ? tok : 0)) * p.hq + head) * D;
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tc05::ld32(lane_addr + C::O_COL + c0, o);
            tc05::wait_ld();
            if (valid) {
#pragma unroll
                for (int i = 0; i < 32; i += 8) {
                    uint4 v;
                    v.x = pack2<T>(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv);
                    v.y = pack2<T>(__uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv);
                    v.z = pack2<T>(__uint_as_float(o[i + 4]) * inv, __uint_as_float(o[i + 5]) * inv);
                    v.w = pack2<T>(__uint_as_float(o[i + 6]) * inv, __uint_as_float(o[i + 7]) * inv);
                    *reinterpret_cast<uint4*>(orow + c0 + i) = v;
                }
            }
        }
    } else {
        if (threadIdx.x % 32 == 0) flag_error(p.err, PA_DEVERR_TIMEOUT);
    }
    tc05::fence_before();
    tc05::named_sync(1, 160);
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
