// Paged prefill on the fifth-generation tensor cores (tcgen05.mma, accumulators in tensor
// memory, operands staged in shared memory by TMA) for fp16 / bf16 pools with D in {64, 128}.
//
// A chunk of C new query tokens of one sequence -- its last C positions, whose K/V rows were
// appended before the call -- attends causally to the sequence's paged history plus the chunk
// ("25. Paged attention and prefix caching", stretch exercise 4; "Chapter 7 Paged KV Cache and
// Memory Management", 4.1 step 3: the key at position p is visible to the query at position i
// iff p <= i).  A row is a (chunk token, query head of the group) pair, the G heads of a token
// side by side, so every K/V tile staged in shared memory serves all G heads of its KV head.
// The softmax runs in base 2 with the scale folded in, and rescales O only when a row's max
// grows by more than 2^8 (the reference cancels exactly in O / l).  Keys at or past a row's
// position are masked; V rows past the sequence length (unwritten slots may hold anything) are
// zeroed before they are used.  The score MMAs run at N = 128 keys.
//
// One CTA owns 256 query rows of one KV head as two 128-row tiles X = A, B that
// share every 128-key K/V tile j.  Tensor memory holds O_A, O_B and one S buffer
// per tile (2 D + 2 x 128 columns); P_Xj (two 16-bit values per column) overwrites
// the first 64 columns of S_X.  P_Xj is published in two halves (keys 0-31 and 64-95,
// then 32-63 and 96-127: each softmax thread's first and second 32 keys), and the
// P . V k-steps of the first half start while the second is computed.  The MMA
// issuer keeps one fixed order:
//   O_A += P_Aj V_j (two halves),  S_A(j+1) = Q_A K_(j+1)^T,  O_B += P_Bj V_j,  S_B(j+1) = Q_B K_(j+1)^T
// so the softmax of one tile overlaps the other tile's MMAs.  S_X(j+1) follows
// P_Xj . V_j on the tensor pipe, which performs one thread's MMAs in issue order;
// and the commit that reports S_X(j+1) done reports every earlier MMA of the
// thread done, so the softmax may rescale O_X (no P . V of tile X in flight) as
// soon as it sees S_X(j+1).
//
// K and V slots (two of each at D = 128, three at D = 64; 128 keys x D per tile) are released separately:
// K_j once both S_j have completed, V_j once both P . V_j have, each refilled by
// its own producer warp; every slot then has about two iterations to land.
// Warps: 0-15 softmax (group X = warp / 8; two threads per row, one per 64-key
// half, meeting once per tile to combine the row max), 16 K producer, 17 MMA
// issuer, 18 V producer.  Every wait is bounded (1 s), each barrier a waiter may
// skip phases of is at most one phase ahead of it (comments at each wait), and
// every warp-collective tcgen05 load / store sits behind warp-uniform decisions.
#pragma once

#include "prefill_tc05_common.cuh"

namespace pa {

template <int D_>
struct Tc05wCfg {
    static constexpr int D = D_, BM = 256, BN = 128;
    static_assert(D == 64 || D == 128, "D in {64, 128}");
    static constexpr int NBOX = D / 64;              // 64-dim (128-byte) boxes per row
    static constexpr int QBOX = 128 * 128;           // 128 rows x 128 B
    static constexpr int Q_BYTES = 2 * NBOX * QBOX;  // both tiles
    static constexpr int KV_BOX = BN * 128;          // 128 keys x 128 B
    static constexpr int SLOT_BYTES = NBOX * KV_BOX; // one K or V tile
#ifdef PA_TC05W_SLOTS64
    static constexpr int SLOTS = D == 64 ? PA_TC05W_SLOTS64 : 2;  // build-time override (tuning sweeps)
#else
    static constexpr int SLOTS = D == 64 ? 3 : 2;  // per operand (as many as shared memory holds at D = 128)
#endif
    static constexpr int K_OFF = Q_BYTES;
    static constexpr int V_OFF = K_OFF + SLOTS * SLOT_BYTES;
    static constexpr int BAR_OFF = V_OFF + SLOTS * SLOT_BYTES;
    // k_full, k_empty, v_full, v_empty [SLOTS]; s_full [2]; p_full [2][2] (tile, half); o_final; q_full
    static constexpr int NBARS = 4 * SLOTS + 6 + 2;
    static constexpr int MISC_OFF = BAR_OFF + NBARS * 8;
    static constexpr int RED_OFF = MISC_OFF + 64;  // row max exchange [2][2][2][128], row sums [2][2][128]
    static constexpr size_t smem_bytes = 1024 + RED_OFF + (8 + 4) * 128 * 4;
    // tensor memory: O_A [0, D), O_B [D, 2D), S_A [2D, 2D + 128), S_B [2D + 128, 2D + 256)
    static constexpr int O_COL = 0, S_COL = 2 * D;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr int NSW = 16;  // two groups of eight: two threads (key halves) per row
    static constexpr int PRODUCER_K = NSW, ISSUER = NSW + 1, PRODUCER_V = NSW + 2;
    static constexpr int THREADS = (NSW + 3) * 32;
    static constexpr int SUB = BN / 16;  // 16-key sub-tiles (one block row each) per tile
};

template <typename T, int D_, int G>
__global__ void __launch_bounds__(Tc05wCfg<D_>::THREADS, 1)
    prefill_tc05w(const PrefillParams p, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap) {
    using C = Tc05wCfg<D_>;
    constexpr int D = C::D, NBOX = C::NBOX, BN = C::BN, SLOTS = C::SLOTS, SUB = C::SUB;
    constexpr int DH = D / 2;  // O columns (dims) per thread of a row
    constexpr int QT = C::BM / G;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint64_t* k_full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* k_empty = k_full + SLOTS;
    uint64_t* v_full = k_empty + SLOTS;
    uint64_t* v_empty = v_full + SLOTS;
    uint64_t* s_full = v_empty + SLOTS;  // [X]
    uint64_t* p_full = s_full + 2;       // [X][half]: keys 32 q .. of each 64-key half, q = half
    uint64_t* o_final = p_full + 4;
    uint64_t* q_full = o_final + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
    int* slot_ok = reinterpret_cast<int*>(smem + C::MISC_OFF + 16);  // loaded sub-tiles of each V slot (bit mask)

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
        for (int i = 0; i < SLOTS; ++i) {
            mbar_init(&k_full[i], 1);
            mbar_init(&k_empty[i], 1);
            mbar_init(&v_full[i], 1);
            mbar_init(&v_empty[i], 1);
        }
#pragma unroll
        for (int X = 0; X < 2; ++X) {
            mbar_init(&s_full[X], 1);
            mbar_init(&p_full[X * 2], 256);
            mbar_init(&p_full[X * 2 + 1], 256);
        }
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

    if (warp == C::PRODUCER_K || warp == C::PRODUCER_V) {
        // ------------------------------------------------------------ producers (K: warp 8, V: warp 10)
        const bool is_v = warp == C::PRODUCER_V;
        uint64_t* full = is_v ? v_full : k_full;
        uint64_t* empty = is_v ? v_empty : k_empty;
        const CUtensorMap* map = is_v ? &vmap : &kmap;
        const int32_t* trow = p.block_tables + static_cast<size_t>(s) * p.max_blocks;
        const int n_sub = n_kv * SUB;
        bool ok = true;
        for (int u0 = 0; u0 < n_sub && ok; u0 += 32) {
            // lane i resolves 16-key sub-tile u0 + i (-1: beyond the sequence or a bad entry)
            int row = -1;
            const int u = u0 + lane;
            if (u < n_sub && u * 16 < L) {
                const int e = __ldg(trow + (u * 16) / p.block_size);
                if (e >= 0 && e < p.num_blocks) {
                    row = (e * p.hkv + kvh) * p.block_size + (u * 16) % p.block_size;
                } else if (!is_v) {
                    flag_error(p.err, PA_DEVERR_TABLE);
                }
            }
            for (int t0 = 0; t0 < 32 && u0 + t0 < n_sub; t0 += SUB) {  // one 128-key tile per 8 lanes
                const int j = (u0 + t0) / SUB;
                const int sl = j % SLOTS;
                const int my_row = __shfl_sync(0xffffffffu, row, t0 + (lane & (SUB - 1)));
                const unsigned mask = __ballot_sync(0xffffffffu, my_row >= 0) & ((1u << SUB) - 1u);
                if (lane == 0 && ok) {
                    // the slot's previous tile (j - SLOTS) is released after its MMAs have consumed it,
                    // which needs this tile's predecessor copies: at most one phase ahead
                    if (!tc05::wait_bounded(&empty[sl], ((j / SLOTS) & 1) ^ 1)) {
                        flag_error(p.err, PA_DEVERR_TIMEOUT);
                        ok = false;
                    } else {
                        // the softmax reads the mask of tile j after v_full; the V slot is refilled only
                        // after both groups have delivered P of tile j
                        if (is_v) slot_ok[sl] = static_cast<int>(mask);
                        // the slot's byte count is posted before any of its copies is issued
                        mbar_arrive_expect_tx(&full[sl], static_cast<uint32_t>(__popc(mask) * NBOX * 2048));
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                // lanes 0-7 issue the copies of sub-tiles 0-7 side by side
                if (ok && lane < SUB && my_row >= 0) {
                    unsigned char* d = smem + (is_v ? C::V_OFF : C::K_OFF) + sl * C::SLOT_BYTES + lane * 2048;
#pragma unroll
                    for (int bx = 0; bx < NBOX; ++bx) tma_load_2d(d + bx * C::KV_BOX, map, bx * 64, my_row, &full[sl]);
                }
                __syncwarp();
            }
        }
        return;  // every copy issued is waited for by the MMA warp before the kernel ends
    }

    if (warp == C::ISSUER) {
        // ------------------------------------------------------------ MMA issuer (one lane)
        if (lane == 0) {
            constexpr uint32_t ID_S = tc05::idesc<T>(BN, false);
            constexpr uint32_t ID_PV = tc05::idesc<T>(D, true);
            bool ok = tc05::wait_bounded(q_full, 0);
            tc05::fence_after();
            // descriptors formed once; an operand at byte offset o from a base has the base's
            // descriptor plus o / 16 (shared addresses stay below 2^18: no carry out of the field)
            const uint64_t q_desc = tc05::sdesc(sbase, 16, 1024);
            const uint64_t k_desc = tc05::sdesc(sbase + C::K_OFF, 16, 1024);
            const uint64_t v_desc = tc05::sdesc(sbase + C::V_OFF, C::KV_BOX, 1024);
            auto issue_s = [&](int X, int j) {
                const uint64_t kst = k_desc + static_cast<uint64_t>((j % SLOTS) * (C::SLOT_BYTES >> 4));
                const uint32_t sd = tmem + C::S_COL + X * BN;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint64_t a = q_desc + static_cast<uint64_t>((X * NBOX * C::QBOX + (ks >> 2) * C::QBOX + (ks & 3) * 32) >> 4);
                    const uint64_t b = kst + static_cast<uint64_t>(((ks >> 2) * C::KV_BOX + (ks & 3) * 32) >> 4);
                    tc05::mma(sd, a, b, ID_S, ks > 0);
                }
                // reports S_X(j) and every earlier MMA of this thread (P_X(j-1) . V_(j-1) included) done
                tc05::commit(&s_full[X]);
            };
            // the k-steps of half q of P_Xj: keys 32 q .. 32 q + 31 and 64 + 32 q .. (k-steps 2q, 2q+1, 4+2q, 5+2q)
            auto issue_pv = [&](int X, int j, int q) {
                const uint64_t vst = v_desc + static_cast<uint64_t>((j % SLOTS) * (C::SLOT_BYTES >> 4));
                const uint32_t pa = tmem + C::S_COL + X * BN;  // key k at column k / 2
#pragma unroll
                for (int i = 0; i < BN / 32; ++i) {
                    const int kk = (i >> 1) * 4 + 2 * q + (i & 1);
                    const uint64_t b = vst + static_cast<uint64_t>((kk * 2048) >> 4);
                    tc05::mma_ts(tmem + C::O_COL + X * D, pa + kk * 8, b, ID_PV, (j > 0 || q > 0 || i > 0) ? 1u : 0u);
                }
            };
            // k_full / v_full of tile j cannot complete the next phase of their slot before k_empty /
            // v_empty of tile j is committed (below), so each wait's parity is unambiguous
            if (ok && n_kv > 0) {
                ok = tc05::wait_bounded(&k_full[0], 0);
                if (ok) {
                    tc05::fence_after();
                    issue_s(0, 0);
                    issue_s(1, 0);
                    tc05::commit(&k_empty[0]);  // K_0 is free once both S_0 complete
                }
            }
            for (int j = 0; ok && j < n_kv; ++j) {
                const int sl = j % SLOTS;
                const bool more = j + 1 < n_kv;
                ok = tc05::wait_bounded(&v_full[sl], (j / SLOTS) & 1);
                // P_X(j+1) needs S_X(j+1), issued below after both waits of P_Xj: each half's
                // p_full is at most one phase ahead
                ok = ok && tc05::wait_bounded(&p_full[0], j & 1);
                if (!ok) break;
                tc05::fence_after();
                issue_pv(0, j, 0);
                ok = tc05::wait_bounded(&p_full[1], j & 1);
                if (!ok) break;
                tc05::fence_after();
                issue_pv(0, j, 1);
                if (more) {
                    ok = tc05::wait_bounded(&k_full[(j + 1) % SLOTS], ((j + 1) / SLOTS) & 1);
                    if (!ok) break;
                    tc05::fence_after();
                    issue_s(0, j + 1);  // after P_A(j) . V_j on the pipe: overwrites P_A(j) in S_A
                }
                ok = tc05::wait_bounded(&p_full[2], j & 1);
                if (!ok) break;
                tc05::fence_after();
                issue_pv(1, j, 0);
                ok = tc05::wait_bounded(&p_full[3], j & 1);
                if (!ok) break;
                tc05::fence_after();
                issue_pv(1, j, 1);
                tc05::commit(&v_empty[sl]);  // V_j is free once both P . V_j complete
                if (more) {
                    issue_s(1, j + 1);
                    tc05::commit(&k_empty[(j + 1) % SLOTS]);
                }
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

    // ------------------------------------------------------------ softmax warps (two threads per row)
    // warp w: tile X = w / 8, key half hh = (w / 4) % 2 (columns 64 hh .. 64 hh + 63 of S, 32 hh ..
    // of P, dims 64 hh .. of O), rows 32 (w % 4) .. +31 = its TMEM lanes; warps w and w + 4 share
    // their rows and meet once per tile to combine the row max
    const int X = warp >> 3, hh = (warp >> 2) & 1, wq = warp & 3;
    const int r = wq * 32 + lane;     // row within tile X
    const int prow_id = X * 128 + r;  // packed row of the CTA
    const int tok = tok0 + prow_id / G;
    const bool valid = tok < Cq;
    const int pos = valid ? base + tok : -1;
    const int head = kvh * G + prow_id % G;
    // position of the first row of this warp's 32 (every valid row of the warp is at or after it)
    const int warp_tok = tok0 + (X * 128 + wq * 32) / G;
    const int warp_pos_min = warp_tok < Cq ? base + warp_tok : -1;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t o_addr = lane_addr + C::O_COL + X * D + hh * DH;
    const uint32_t sa = lane_addr + C::S_COL + X * BN;
    float* xmax = reinterpret_cast<float*>(smem + C::RED_OFF);  // [tile parity][X][half][row]
    float* xl = xmax + 2 * 2 * 2 * 128;                          // [X][half][row]
    const int gbar = 3 + X;                                      // the group's named barrier (256 threads)
    {
        // this half of the Q row into tile X's K-major swizzled operand (zeros past the chunk)
        const uint4* qrow = reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) +
                                                           (static_cast<size_t>(q0 + (valid ? tok : 0)) * p.hq + head) * D);
        unsigned char* qx = smem + X * NBOX * C::QBOX;
#pragma unroll
        for (int i = 0; i < D / 16; ++i) {
            const int cc = hh * (D / 16) + i, bx = cc >> 3, c = cc & 7;  // 16-byte chunk of the row
            const uint4 v = valid ? __ldg(qrow + cc) : make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(qx + bx * C::QBOX + r * 128 + ((c ^ (r & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
        mbar_arrive(q_full);
    }
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.f;  // l: this half's share of the row sum
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
        const int sl = j % SLOTS;
        // decisions that guard a tcgen05.ld / st are warp-uniform (those are .sync.aligned).
        // Neither barrier can run two phases ahead: V of tile j + SLOTS is loaded, and S_X(j + 1)
        // issued, only after this thread's P_Xj has been consumed
        const bool got = __all_sync(0xffffffffu, tc05::wait_bounded(&v_full[sl], (j / SLOTS) & 1) &&
                                                     tc05::wait_bounded(&s_full[X], j & 1));
        const int key0 = j * BN;
        int okmask = 0;
        bool interior = false;
        uint32_t sr[64];
        float pmx = -INFINITY;
        if (got) {
            tc05::fence_after();
            okmask = slot_ok[sl];
            // interior tile: every valid row of the warp sees all 128 keys and the scale is positive
            interior = okmask == (1 << SUB) - 1 && key0 + BN - 1 <= warp_pos_min && sl2 > 0.f;
            // this half's 64 scores in registers; masked tiles are scaled and masked in place
            // (invisible keys: -inf), so the exponentials below are branch-free
            tc05::ld32(sa + hh * 64, sr);
            tc05::ld32(sa + hh * 64 + 32, sr + 32);
            tc05::wait_ld();
            float t[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) t[i] = -INFINITY;
            if (interior) {
#pragma unroll
                for (int c = 0; c < 64; c += 2)
                    t[(c >> 1) & 7] = tc05::max3(t[(c >> 1) & 7], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
            } else {
#pragma unroll
                for (int c = 0; c < 64; ++c) {
                    const int key = hh * 64 + c;
                    const bool vis = key0 + key <= pos && ((okmask >> (key >> 4)) & 1);
                    const float x = vis ? __uint_as_float(sr[c]) * sl2 : -INFINITY;
                    sr[c] = __float_as_uint(x);
                    t[c & 7] = fmaxf(t[c & 7], x);
                }
            }
            pmx = fmaxf(fmaxf(fmaxf(t[0], t[1]), fmaxf(t[2], t[3])), fmaxf(fmaxf(t[4], t[5]), fmaxf(t[6], t[7])));
            if (interior) pmx *= sl2;
            xmax[(((j & 1) * 2 + X) * 2 + hh) * 128 + r] = pmx;
        }
        // every thread of the group arrives here once per tile, so a timeout ends the loop for the
        // whole group at the same tile; the partner's max of tile j sits in the parity-j buffer,
        // which is written again (tile j + 2) only after both have passed tile j + 1's barrier
        if (!tc05::bar_and(gbar, 256, got)) {
            ok = false;
            break;
        }
        const float mx = fmaxf(pmx, xmax[(((j & 1) * 2 + X) * 2 + (hh ^ 1)) * 128 + r]);
        // lazy rescale per row (both threads of a row decide alike); O_X is rescaled for the whole
        // warp when any row needs it.  No P . V of tile X is in flight: S_X(j) was issued after
        // P_X(j-1) . V_(j-1), and its completion, seen above, reports that one's too
        const bool grow = mx > m + kLazyRescale;
        const bool scale_o = grow && m != -INFINITY;
        const float a = scale_o ? tc05::fast_exp2(m - mx) : 1.f;
        if (j > 0 && __any_sync(0xffffffffu, scale_o)) {
#pragma unroll
            for (int c0 = 0; c0 < DH; c0 += 32) {
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
        const float mul = interior ? sl2 : 1.f;
        // V rows of keys past the sequence or of sub-tiles not loaded may hold anything: zero them
        // before the first half of P is published (both groups write the same zeros; each
        // P . V waits only for its own group's)
        if (key0 + BN > L || okmask != (1 << SUB) - 1) {
            unsigned char* vt = smem + C::V_OFF + sl * C::SLOT_BYTES;
            for (int e = hh * 128 + r; e < BN * NBOX * 8; e += 256) {
                const int key = e / (NBOX * 8), rest = e % (NBOX * 8);
                if (key0 + key >= L || !((okmask >> (key >> 4)) & 1))
                    *reinterpret_cast<uint4*>(vt + (rest >> 3) * C::KV_BOX + key * 128 + (rest & 7) * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
        }
        // ---- P = 2^(v * mul - m): keys 64 hh + 32 q .. +31 go to columns 32 hh + 16 q .. +15
        // (two 16-bit values per column), over scores already in registers
        // (pairs of keys in packed fp32 FMAs and adds: the softmax is issue-bound here)
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int qq = 0; qq < 2; ++qq) {
            // the half's 16 words leave in two 8-word stores, the first issued before the second's
            // exponentials (measured faster than one 16-word store, and than four 4-word ones)
#pragma unroll
            for (int hv = 0; hv < 2; ++hv) {
                uint32_t pw[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int c = qq * 32 + hv * 16 + 2 * i;
                    float x0, x1;
                    tc05::fma2(x0, x1, __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]), mul, -ms);
                    // fp32 exponentials (with the 8-word stores, the f16x2 form -- one MUFU op per
                    // pair, three conversions more -- measured slower at every share of the pairs)
                    const float e0 = tc05::fast_exp2(x0), e1 = tc05::fast_exp2(x1);
                    pw[i] = pack2<T>(e0, e1);
                    tc05::add2(ls[(i & 1) * 2], ls[(i & 1) * 2 + 1], e0, e1);
                }
                tc05::st8(sa + hh * 32 + qq * 16 + hv * 8, pw);
            }
            tc05::wait_st();
            tc05::fence_before();
            mbar_arrive(&p_full[X * 2 + qq]);
        }
        l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
    }
    griddep_launch_dependents();
    const bool all_ok = tc05::bar_and(2, C::NSW * 32, ok);
    const bool done = all_ok && tc05::wait_bounded(o_final, 0);
    // the row sum: this half's share plus the partner's (every softmax thread passed the barrier
    // above, so the exchange below is reached by the whole group)
    xl[(X * 2 + hh) * 128 + r] = l;
    tc05::named_sync(gbar, 256);
    const float lt = l + xl[(X * 2 + (hh ^ 1)) * 128 + r];
    if (__all_sync(0xffffffffu, done)) {
        tc05::fence_after();
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        T* orow = static_cast<T*>(p.out) + (static_cast<size_t>(q0 + (valid ? tok : 0)) * p.hq + head) * D + hh * DH;
#pragma unroll
        for (int c0 = 0; c0 < DH; c0 += 32) {
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
cudaError_t launch_prefill_tc05w(const PrefillParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                 int max_query_len, cudaStream_t stream) {
    using C = Tc05wCfg<D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc05w<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(C::smem_bytes));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int64_t rows = static_cast<int64_t>(max_query_len) * G;
    const unsigned tiles = static_cast<unsigned>((rows + C::BM - 1) / C::BM);
    return launch_pdl(prefill_tc05w<T, D, G>, dim3(tiles, p.hkv, p.batch), dim3(C::THREADS), C::smem_bytes, stream, p,
                      kmap, vmap);
}

}  // namespace pa
