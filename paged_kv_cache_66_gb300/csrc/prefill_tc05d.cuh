// Paged prefill on tcgen05 for D = 256: the operation, row packing, masking and
// base-2 lazy-rescale softmax of prefill_tc05w.cuh ("25. Paged attention and
// prefix caching", stretch exercise 4; "Chapter 7 Paged KV Cache and Memory
// Management", 4.1 step 3), laid out for the wide head.
//
// One CTA owns 128 query rows of one KV head.  Tensor memory holds O (256
// columns, fp32), the query tile Q as the A operand of the score MMAs (128
// columns, two 16-bit values per column, written once by the softmax threads)
// and two 64-column S buffers; shared memory then holds only the K/V ring, three
// stages of 64 keys (64 KiB each).  A K/V copy takes every 64-dim slice of its
// rows at once (a 3-D box: 8 rows of K, 16 of V), so the 64-key tile is 12 TMA
// copies: K as eight 8-key groups of [slice][8 rows][128 B] (4 KiB apart, the
// score MMA's 8-row step), V as four 16-key sub-tiles of [slice][16 rows][128 B]
// (8 KiB apart, one P . V K-step each; slices 2 KiB apart).  Per 64-key tile j:
//   S_j = Q . K_j^T   tcgen05.mma M=128 N=64, A = Q (tensor memory), B = K_j (smem, K-major)
//   softmax           one thread per row: tcgen05.ld of its 64 scores, causal mask, running
//                     max, P_j = 2^(s - m) rounded to the dtype over the first half of S_j
//   O += P_j . V_j    tcgen05.mma M=128 N=256, A = P_j (tensor memory), B = V_j (smem, MN-major)
// The MMA issuer polls both inputs and issues whichever is ready: S(j+1) as soon
// as K_(j+1) has landed (its S buffer held P(j-1), whose P . V was issued before;
// one thread's MMAs run in issue order), P(j) . V_j once the softmax has written
// P(j), so a P . V never waits behind a later tile's copy.
// kmap / vmap are the pools' 3-D maps (element, row, 64-dim slice) with boxes of
// 8 (K) and 16 (V) rows by every slice.
// Warps: 0-3 softmax (thread = row = TMEM lane), 4 producer (TMA, four lanes
// issuing), 5 MMA issuer (the whole warp walks the issue loop, one elected lane
// issues the MMAs).  Every wait is bounded (1 s); no barrier can run two
// phases ahead of a waiter (comments at each wait); every warp-collective
// tcgen05 load / store sits behind warp-uniform decisions.
#pragma once

#include "prefill_tc05_common.cuh"

namespace pa {

struct Tc05dCfg {
    static constexpr int D = 256, BM = 128, BN = 64, NSB = 2, STAGES = 3;
    static constexpr int NBOX = D / 64;              // 64-dim (128-byte) boxes per row
    static constexpr int KV_BOX = BN * 128;          // 64 keys x 128 B
    static constexpr int K_BYTES = NBOX * KV_BOX;    // 32 KiB
    static constexpr int KG_BYTES = 8 * NBOX * 128;  // one 8-key group of K, all slices (4 KiB)
    static constexpr int VS_BYTES = 16 * NBOX * 128; // one 16-key sub-tile of V, all slices (8 KiB)
    static constexpr int STAGE_BYTES = 2 * K_BYTES;  // K then V
    static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
    // kv_full, kv_empty [STAGES]; s_full, p_full [NSB]; o_ready; o_final; q_full
    static constexpr int NBARS = 2 * STAGES + 2 * NSB + 3;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr size_t smem_bytes = 1024 + MISC_OFF + 16 + 4 * STAGES;
    // tensor memory: O [0, 256), Q [256, 384), S buffers [384 + 64 b, +64)
    static constexpr int O_COL = 0, Q_COL = D, S_COL = D + D / 2;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int NSW = 4;
    static constexpr int PRODUCER = NSW, ISSUER = NSW + 1;
    static constexpr int THREADS = (NSW + 2) * 32;
    static_assert(S_COL + NSB * BN <= 512, "tensor memory columns");
};

template <typename T, int G>
__global__ void __launch_bounds__(Tc05dCfg::THREADS, 1)
    prefill_tc05d(const PrefillParams p, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap) {
    using C = Tc05dCfg;
    constexpr int D = C::D, NBOX = C::NBOX, BN = C::BN, NSB = C::NSB, STAGES = C::STAGES;
    constexpr int QT = C::BM / G;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint64_t* kv_full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* kv_empty = kv_full + STAGES;
    uint64_t* s_full = kv_empty + STAGES;  // [b]
    uint64_t* p_full = s_full + NSB;       // [b]
    uint64_t* o_ready = p_full + NSB;
    uint64_t* o_final = o_ready + 1;
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
        for (int b = 0; b < NSB; ++b) {
            mbar_init(&s_full[b], 1);
            mbar_init(&p_full[b], 128);
        }
        mbar_init(o_ready, 1);
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
                    // the stage's previous tile is released after both its MMAs consumed it, which
                    // needs this tile's predecessors' copies: at most one phase ahead
                    if (!tc05::wait_bounded(&kv_empty[st], ((j / STAGES) & 1) ^ 1)) {
                        flag_error(p.err, PA_DEVERR_TIMEOUT);
                        ok = false;
                    } else {
                        stage_ok[st] = static_cast<int>(mask);
                        // the stage's byte count is posted before any of its copies is issued
                        mbar_arrive_expect_tx(&kv_full[st], static_cast<uint32_t>(__popc(mask) * 2 * NBOX * 2048));
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                // lanes 0-3 issue the copies of sub-tiles 0-3 side by side: K as its two 8-key
                // groups, V whole
                if (ok && lane < 4 && my_row >= 0) {
                    unsigned char* kd = smem + st * C::STAGE_BYTES + lane * 2 * C::KG_BYTES;
                    tma_load_3d(kd, &kmap, 0, my_row, 0, &kv_full[st]);
                    tma_load_3d(kd + C::KG_BYTES, &kmap, 0, my_row + 8, 0, &kv_full[st]);
                    tma_load_3d(smem + st * C::STAGE_BYTES + C::K_BYTES + lane * C::VS_BYTES, &vmap, 0, my_row, 0,
                                &kv_full[st]);
                }
                __syncwarp();
            }
        }
        return;  // every copy issued is waited for by the MMA warp before the kernel ends
    }

    if (warp == C::ISSUER) {
        // ------------------------------------------------------------ MMA issuer (one elected lane)
        // The whole warp walks the issue loop, so operands are formed in warp-uniform code and only
        // the MMAs and commits sit behind the elected lane: issued from a lane-0 branch instead, an
        // N = 64 score MMA measured ~45 cycles against 32 (every decision below is warp-uniform)
        const bool leader = tc05::elect_one();
        constexpr uint32_t ID_S = tc05::idesc<T>(BN, false);
        constexpr uint32_t ID_PV = tc05::idesc<T>(D, true);
        // Q in tensor memory: written by the softmax threads (tcgen05.st) before q_full
        bool ok = __all_sync(0xffffffffu, tc05::wait_bounded(q_full, 0));
        tc05::fence_after();
        // descriptors formed once; an operand at byte offset o from a base has the base's
        // descriptor plus o / 16 (shared addresses stay below 2^18: no carry out of the field).
        // K: 8-key groups KG_BYTES apart; V: 8-key groups 1 KiB apart, 64-dim slices 2 KiB apart
        const uint64_t k_desc = tc05::sdesc(sbase, 16, C::KG_BYTES);
        const uint64_t v_desc = tc05::sdesc(sbase + C::K_BYTES, 2048, 1024);
        auto issue_s = [&](int j) {
            const uint64_t kst = k_desc + static_cast<uint64_t>((j % STAGES) * (C::STAGE_BYTES >> 4));
            const uint32_t sd = tmem + C::S_COL + (j % NSB) * BN;
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
                const uint64_t b = kst + static_cast<uint64_t>(((ks >> 2) * 1024 + (ks & 3) * 32) >> 4);
                if (leader) tc05::mma_ts(sd, tmem + C::Q_COL + ks * 8, b, ID_S, ks > 0);
            }
            if (leader) tc05::commit(&s_full[j % NSB]);
        };
        auto issue_pv = [&](int j) {
            const int st = j % STAGES;
            const uint64_t vst = v_desc + static_cast<uint64_t>(st * (C::STAGE_BYTES >> 4));
            const uint32_t pt = tmem + C::S_COL + (j % NSB) * BN;  // key k at column k / 2
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {
                // N = D in one MMA (the four 64-dim slices 2 KiB apart: leading byte offset);
                // K-step kk is V sub-tile kk
                const uint64_t b = vst + static_cast<uint64_t>((kk * C::VS_BYTES) >> 4);
                if (leader) tc05::mma_ts(tmem + C::O_COL, pt + kk * 8, b, ID_PV, (j > 0 || kk > 0) ? 1u : 0u);
            }
            if (leader) {
                tc05::commit(o_ready);
                tc05::commit(&kv_empty[st]);  // the stage is free once this P . V completes
            }
        };
        // S(ns) and P(np) . V go out as their inputs arrive, whichever is first, so that a P . V
        // never waits behind a later tile's copy: S(ns) once K(ns) has landed and the P . V of
        // the tile whose P its S buffer holds (ns - NSB) is issued; P(np) . V once the softmax
        // has published P(np).  Parities: kv_full of tile j completes no other phase before
        // kv_empty of tile j is committed (after its P . V), nor p_full of tile j before S(j + NSB)
        // is issued (after P(j) . V).  A phase counts as seen once every lane has seen it.  No
        // progress for 1 s ends the walk
        int ns = 0, np = 0;
        uint32_t idle = 0;
        uint64_t t0 = 0;
        while (ok && np < n_kv) {
            bool moved = false;
            if (ns < n_kv && ns < np + NSB &&
                __all_sync(0xffffffffu, tc05::test_wait(&kv_full[ns % STAGES], (ns / STAGES) & 1))) {
                tc05::fence_after();
                issue_s(ns++);
                moved = true;
            }
            if (np < ns && __all_sync(0xffffffffu, tc05::test_wait(&p_full[np % NSB], (np / NSB) & 1))) {
                tc05::fence_after();
                issue_pv(np++);
                moved = true;
            }
            if (moved) {
                idle = 0;
            } else if ((++idle & 255u) == 0) {
                const uint64_t t = __shfl_sync(0xffffffffu, global_timer_ns(), 0);
                if (idle == 256u) t0 = t;
                else if (t - t0 > 1000000000ull) ok = false;
            }
        }
        if (leader) {
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
    const int r = tid;  // row of the query tile = TMEM lane
    const int tok = tok0 + r / G;
    const bool valid = tok < Cq;
    const int pos = valid ? base + tok : -1;
    const int head = kvh * G + r % G;
    // position of the first row of this warp's 32 (every valid row of the warp is at or after it)
    const int warp_tok = tok0 + (warp * 32) / G;
    const int warp_pos_min = warp_tok < Cq ? base + warp_tok : -1;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const uint32_t o_addr = lane_addr + C::O_COL;
    {
        // the Q row into tensor memory, the A operand of the score MMAs: column c holds dims 2c and
        // 2c + 1 (low half even), which is the row's own memory order (zeros past the chunk)
        const uint4* qrow = reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) +
                                                           (static_cast<size_t>(q0 + (valid ? tok : 0)) * p.hq + head) * D);
#pragma unroll
        for (int c0 = 0; c0 < D / 2; c0 += 32) {
            uint32_t w[32];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint4 v = valid ? __ldg(qrow + c0 / 4 + i) : make_uint4(0u, 0u, 0u, 0u);
                w[4 * i] = v.x;
                w[4 * i + 1] = v.y;
                w[4 * i + 2] = v.z;
                w[4 * i + 3] = v.w;
            }
            tc05::st32(lane_addr + C::Q_COL + c0, w);
        }
        tc05::wait_st();
        tc05::fence_before();
        mbar_arrive(q_full);
    }
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
        const int st = j % STAGES, sb = j % NSB;
        // decisions that guard a tcgen05.ld / st are warp-uniform (those are .sync.aligned).
        // Neither barrier can run two phases ahead: tile j + STAGES is loaded, and S(j + NSB)
        // issued, only after this thread's P_j has been consumed
        const bool got = tc05::wait_bounded(&kv_full[st], (j / STAGES) & 1) && tc05::wait_bounded(&s_full[sb], (j / NSB) & 1);
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
        // so the row max is the raw max times the scale; masked tiles keep their scores pre-scaled
        // (masked: -inf) in sr
        const bool interior = okmask == 0xF && key0 + BN - 1 <= warp_pos_min && sl2 > 0.f;
        float mx;
        {
            float t[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) t[i] = -INFINITY;
            if (interior) {
#pragma unroll
                for (int c = 0; c < 64; ++c) t[c & 7] = fmaxf(t[c & 7], __uint_as_float(sr[c]));
            } else {
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
        // lazy rescale per row; O (in TMEM) is rescaled for the whole warp when any row needs it,
        // once P(j-1) . V_(j-1) has landed, each lane by its own factor
        const bool grow = mx > m + kLazyRescale;
        const bool scale_o = grow && m != -INFINITY;
        const float a = scale_o ? tc05::fast_exp2(m - mx) : 1.f;
        if (j > 0 && __any_sync(0xffffffffu, scale_o)) {
            // o_ready counts the P . V launches in order: the one of tile j needs this thread's P_j,
            // and the one of tile j - 2 completed before S(j) (issued after it)
            if (!__all_sync(0xffffffffu, tc05::wait_bounded(o_ready, (j - 1) & 1))) {
                ok = false;
                break;
            }
            tc05::fence_after();
#pragma unroll 1
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
        // P = 2^(v * mul - m), pairs of keys in one packed FMA and add (interior: v raw, mul =
        // scale; masked: v pre-scaled, mul = 1); key c at column c / 2 of S buffer sb, over this
        // lane's own scores, in 8-word stores (each issued before the next words' exponentials)
        const float mul = interior ? sl2 : 1.f;
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int hq = 0; hq < 4; ++hq) {
            uint32_t pw[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int c = hq * 16 + 2 * i;
                float x0, x1;
                tc05::fma2(x0, x1, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]), mul, -ms);
                const float e0 = tc05::fast_exp2(x0);
                const float e1 = tc05::fast_exp2(x1);
                tc05::add2(ls[(i & 1) * 2], ls[(i & 1) * 2 + 1], e0, e1);
                pw[i] = pack2<T>(e0, e1);
            }
            tc05::st8(sa + hq * 8, pw);
        }
        l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        // V rows of keys past the sequence or of sub-tiles not loaded may hold anything: zero them
        if (key0 + BN > L || okmask != 0xF) {
            unsigned char* vt = smem + st * C::STAGE_BYTES + C::K_BYTES;
            for (int e = r; e < BN * NBOX * 8; e += 128) {
                const int key = e / (NBOX * 8), rest = e % (NBOX * 8);
                if (key0 + key >= L || !((okmask >> (key >> 4)) & 1))
                    *reinterpret_cast<uint4*>(vt + (key >> 4) * C::VS_BYTES + (rest >> 3) * 2048 + (key & 15) * 128 +
                                              (rest & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
        }
        tc05::wait_st();
        tc05::fence_before();
        mbar_arrive(&p_full[sb]);
    }
    griddep_launch_dependents();
    const bool all_ok = tc05::bar_and(2, C::NSW * 32, ok);
    const bool done = all_ok && tc05::wait_bounded(o_final, 0);
    if (__all_sync(0xffffffffu, done)) {
        tc05::fence_after();
        const float inv = l > 0.f ? 1.f / l : 0.f;
        const bool out32 = (reinterpret_cast<uintptr_t>(p.out) & 31) == 0;  // rows are 2 D bytes apart
        T* orow = static_cast<T*>(p.out) + (static_cast<size_t>(q0 + (valid ? tok : 0)) * p.hq + head) * D;
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            tc05::ld32(o_addr + c0, o);
            tc05::wait_ld();
            if (valid) {
#pragma unroll
                for (int i = 0; i < 32; i += 16) {
                    uint32_t pw[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        pw[k] = pack2<T>(__uint_as_float(o[i + 2 * k]) * inv, __uint_as_float(o[i + 2 * k + 1]) * inv);
                    // lanes hold different rows: 32 bytes per lane write whole sectors
                    if (out32) {
                        st_global_v8(orow + c0 + i, pw);
                    } else {
                        *reinterpret_cast<uint4*>(orow + c0 + i) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
                        *reinterpret_cast<uint4*>(orow + c0 + i + 8) = make_uint4(pw[4], pw[5], pw[6], pw[7]);
                    }
                }
            }
        }
    } else if (lane == 0) {
        flag_error(p.err, PA_DEVERR_TIMEOUT);
    }
    tc05::fence_before();
    tc05::named_sync(1, (C::NSW + 1) * 32);
}

template <typename T, int G>
cudaError_t launch_prefill_tc05d(const PrefillParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                 int max_query_len, cudaStream_t stream) {
    using C = Tc05dCfg;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc05d<T, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(C::smem_bytes));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int64_t rows = static_cast<int64_t>(max_query_len) * G;
    const unsigned tiles = static_cast<unsigned>((rows + C::BM - 1) / C::BM);
    return launch_pdl(prefill_tc05d<T, G>, dim3(tiles, p.hkv, p.batch), dim3(C::THREADS), C::smem_bytes, stream, p,
                      kmap, vmap);
}

}  // namespace pa
