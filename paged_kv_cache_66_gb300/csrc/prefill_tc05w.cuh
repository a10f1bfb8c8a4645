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
// A unit of work is 256 query rows of one KV head, two 128-row tiles X = A, B that
// share every 128-key K/V tile j.  The kernel is persistent: one CTA per SM walks
// its units back to back (dealt round by round in a snake over the CTAs), its producers running
// on into the next unit's K/V tiles, the next unit's Q tiles loaded by TMA as soon as
// the unit before has no score MMA left, and tensor memory allocated once.  Each
// unit ends with its O read, normalised and stored by the softmax warps before they
// publish any P of the next unit (whose first P . V overwrites O).  Tensor memory holds O_A, O_B and one S buffer
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
// half, meeting once per tile to combine the row max), 16 K and Q producer, 17 MMA
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
    // k_full, k_empty, v_full, v_empty [SLOTS]; s_full [2]; p_full [2][2] (tile, half); o_final; q_full; q_empty
    static constexpr int NBARS = 4 * SLOTS + 6 + 3;
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
    prefill_tc05w(const PrefillParams p, const int q_tiles, const __grid_constant__ CUtensorMap kmap,
                  const __grid_constant__ CUtensorMap vmap, const __grid_constant__ CUtensorMap qmap) {
    using C = Tc05wCfg<D_>;
    constexpr int D = C::D, NBOX = C::NBOX, BN = C::BN, SLOTS = C::SLOTS, SUB = C::SUB;
    constexpr int DH = D / 2;  // O columns (dims) per thread of a row
    constexpr int QT = C::BM / G;   // chunk tokens of one unit
    constexpr int QTX = QT / 2;     // chunk tokens of one query tile
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint64_t* k_full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* k_empty = k_full + SLOTS;
    uint64_t* v_full = k_empty + SLOTS;
    uint64_t* v_empty = v_full + SLOTS;
    uint64_t* s_full = v_empty + SLOTS;  // [X]
    uint64_t* p_full = s_full + 2;       // [X][half]: keys 32 q .. of each 64-key half, q = half
    uint64_t* o_final = p_full + 4;      // one phase per unit: its last P . V done
    uint64_t* q_full = o_final + 1;      // one phase per unit: its Q tiles landed
    uint64_t* q_empty = q_full + 1;      // one phase per unit: its last score MMA done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::MISC_OFF);
    int* slot_ok = reinterpret_cast<int*>(smem + C::MISC_OFF + 16);  // loaded sub-tiles of each V slot (bit mask)

    griddep_wait();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // Work units: (query tile pair, KV head, sequence) with the tile pair fastest, the pairs with the
    // most keys first; in round r CTA c takes unit r * grid + c (r even) or r * grid + grid - 1 - c
    // (r odd).  The CTAs at work at any time hold all tile pairs of a few (sequence, KV head)s, which
    // read the same K/V blocks (one DRAM read, the rest from L2).  Every role walks the same units and
    // skips the same ones, so the barrier phases below count the same K/V tiles and units everywhere.
    const int n_units = q_tiles * p.hkv * p.batch;  // < 2^31 (the launcher checks)
    struct Unit {
        int s, kvh, q0, Cq, L, base, tok0, n_kv;
    };
    // the unit of this CTA's round r: rounds alternate direction over the CTAs (a snake), which
    // evens out the per-CTA work when the tile pairs' key counts grow with their index
    auto unit_of = [&](int rnd) -> int {
        return rnd * static_cast<int>(gridDim.x) +
               ((rnd & 1) ? static_cast<int>(gridDim.x) - 1 - static_cast<int>(blockIdx.x) : static_cast<int>(blockIdx.x));
    };
    // n_kv = 0: a unit with no rows (past its sequence's chunk, or an inconsistent sequence)
    auto unit_at = [&](int u) -> Unit {
        Unit w{};
        const int pair = u / q_tiles;
        const int t = q_tiles - 1 - (u - pair * q_tiles);
        w.s = pair / p.hkv;
        w.kvh = pair - w.s * p.hkv;
        w.q0 = __ldg(p.qstart + w.s);
        const int q1 = __ldg(p.qstart + w.s + 1);
        w.L = __ldg(p.seq_lens + w.s);
        w.Cq = q1 - w.q0;
        if (w.L < 0 || w.L > p.max_blocks * p.block_size || w.Cq < 0 || w.Cq > w.L || w.q0 < 0 || q1 > p.total_q) {
            if (tid == 0 && t == q_tiles - 1 && w.kvh == 0) flag_error(p.err, PA_DEVERR_SEQLEN);
            return w;
        }
        w.tok0 = t * QT;
        if (w.tok0 >= w.Cq) return w;
        w.base = w.L - w.Cq;  // position of chunk token 0
        const int kv_end = w.base + min(w.Cq, w.tok0 + QT);
        w.n_kv = (kv_end + BN - 1) / BN;
        return w;
    };

    // the next unit with rows at or after round `rnd` (rnd is advanced past it; n_kv = 0: none)
    auto next_unit = [&](int& rnd) -> Unit {
        for (int u = unit_of(rnd); u < n_units; u = unit_of(rnd)) {
            ++rnd;
            const Unit w = unit_at(u);
            if (w.n_kv > 0) return w;
        }
        return Unit{};
    };

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
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
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
        // ------------------------------------------------------------ producers (K and Q: warp 16, V: warp 18)
        // Each runs on into the next unit's tiles as its slots free up; the K producer also loads
        // each unit's two Q tiles once every score MMA of the unit before has completed.
        const bool is_v = warp == C::PRODUCER_V;
        uint64_t* full = is_v ? v_full : k_full;
        uint64_t* empty = is_v ? v_empty : k_empty;
        const CUtensorMap* map = is_v ? &vmap : &kmap;
        bool ok = true;
        int jg = 0, nu = 0;  // K/V tiles and units of this CTA so far
        for (int rnd = 0, u = unit_of(0); u < n_units && ok; u = unit_of(++rnd)) {
            const Unit w = unit_at(u);
            if (w.n_kv == 0) continue;
            if (!is_v) {
                if (lane == 0) {
                    // q_empty of the previous unit: its phase completes only after this unit's
                    // predecessor Q landed and was consumed, so it is at most one phase ahead
                    if (nu > 0 && !tc05::wait_bounded(q_empty, (nu - 1) & 1)) {
                        flag_error(p.err, PA_DEVERR_TIMEOUT);
                        ok = false;
                    } else {
                        // rows = (token, head of the group), the G heads of a token side by side: the
                        // box's own order; rows past the chunk load other rows (or zeros past total_q),
                        // which only rows that are never stored see
                        mbar_arrive_expect_tx(q_full, static_cast<uint32_t>(2 * NBOX * C::QBOX));
#pragma unroll
                        for (int X = 0; X < 2; ++X)
#pragma unroll
                            for (int bx = 0; bx < NBOX; ++bx)
                                tma_load_3d(smem + (X * NBOX + bx) * C::QBOX, &qmap, bx * 64, w.kvh * G,
                                            w.q0 + w.tok0 + X * QTX, q_full);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (lane == 0) {
                    // the next unit's Q tiles into L2 now, so that its TMA load, issued only once this
                    // unit's score MMAs are done, finds them there
                    int r2 = rnd + 1;
                    const Unit w2 = next_unit(r2);
                    if (w2.n_kv > 0) {
#pragma unroll
                        for (int X = 0; X < 2; ++X)
#pragma unroll
                            for (int bx = 0; bx < NBOX; ++bx)
                                tma_prefetch_3d(&qmap, bx * 64, w2.kvh * G, w2.q0 + w2.tok0 + X * QTX);
                    }
                }
            }
            const int32_t* trow = p.block_tables + static_cast<size_t>(w.s) * p.max_blocks;
            const int n_sub = w.n_kv * SUB;
            for (int u0 = 0; u0 < n_sub && ok; u0 += 32) {
                // lane i resolves 16-key sub-tile u0 + i (-1: beyond the sequence or a bad entry)
                int row = -1;
                const int su = u0 + lane;
                if (su < n_sub && su * 16 < w.L) {
                    const int e = __ldg(trow + (su * 16) / p.block_size);
                    if (e >= 0 && e < p.num_blocks) {
                        row = (e * p.hkv + w.kvh) * p.block_size + (su * 16) % p.block_size;
                    } else if (!is_v) {
                        flag_error(p.err, PA_DEVERR_TABLE);
                    }
                }
                for (int t0 = 0; t0 < 32 && u0 + t0 < n_sub; t0 += SUB) {  // one 128-key tile per 8 lanes
                    const int j = jg + (u0 + t0) / SUB;  // tile of this CTA's stream
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
                            // the softmax reads the mask of tile j after v_full; the V slot is refilled
                            // only after both groups have delivered P of tile j
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
                        for (int bx = 0; bx < NBOX; ++bx)
                            tma_load_2d(d + bx * C::KV_BOX, map, bx * 64, my_row, &full[sl]);
                    }
                    __syncwarp();
                }
            }
            jg += w.n_kv;
            ++nu;
        }
        return;  // every copy issued is waited for by the MMA warp before the kernel ends
    }

    if (warp == C::ISSUER) {
        // ------------------------------------------------------------ MMA issuer (one lane)
        if (lane == 0) {
            constexpr uint32_t ID_S = tc05::idesc<T>(BN, false);
            constexpr uint32_t ID_PV = tc05::idesc<T>(D, true);
            // descriptors formed once; an operand at byte offset o from a base has the base's
            // descriptor plus o / 16 (shared addresses stay below 2^18: no carry out of the field)
            const uint64_t q_desc = tc05::sdesc(sbase, 16, 1024);
            const uint64_t k_desc = tc05::sdesc(sbase + C::K_OFF, 16, 1024);
            const uint64_t v_desc = tc05::sdesc(sbase + C::V_OFF, C::KV_BOX, 1024);
            auto issue_s = [&](int X, int g) {
                const uint64_t kst = k_desc + static_cast<uint64_t>((g % SLOTS) * (C::SLOT_BYTES >> 4));
                const uint32_t sd = tmem + C::S_COL + X * BN;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint64_t a = q_desc + static_cast<uint64_t>((X * NBOX * C::QBOX + (ks >> 2) * C::QBOX + (ks & 3) * 32) >> 4);
                    const uint64_t b = kst + static_cast<uint64_t>(((ks >> 2) * C::KV_BOX + (ks & 3) * 32) >> 4);
                    tc05::mma(sd, a, b, ID_S, ks > 0);
                }
                // reports S_X(g) and every earlier MMA of this thread (P_X(g-1) . V_(g-1) included) done
                tc05::commit(&s_full[X]);
            };
            // the k-steps of half q of P_Xg: keys 32 q .. 32 q + 31 and 64 + 32 q .. (k-steps 2q, 2q+1, 4+2q, 5+2q);
            // `first`: the unit's first tile, whose first k-step overwrites O_X
            auto issue_pv = [&](int X, int g, int q, bool first) {
                const uint64_t vst = v_desc + static_cast<uint64_t>((g % SLOTS) * (C::SLOT_BYTES >> 4));
                const uint32_t pa = tmem + C::S_COL + X * BN;  // key k at column k / 2
#pragma unroll
                for (int i = 0; i < BN / 32; ++i) {
                    const int kk = (i >> 1) * 4 + 2 * q + (i & 1);
                    const uint64_t b = vst + static_cast<uint64_t>((kk * 2048) >> 4);
                    tc05::mma_ts(tmem + C::O_COL + X * D, pa + kk * 8, b, ID_PV, (!first || q > 0 || i > 0) ? 1u : 0u);
                }
            };
            // Per unit: S_A(0), S_B(0), then for each tile j: P_A(j) . V_j, S_A(j+1), P_B(j) . V_j,
            // S_B(j+1).  A unit's first P . V (which overwrites O_X) waits for P_X of its first tile,
            // which each softmax thread publishes only after it has read O_X of the unit before.
            // k_full / v_full of tile g cannot complete the next phase of their slot before k_empty /
            // v_empty of tile g is committed (below), so each wait's parity is unambiguous.
            bool ok = true;
            int jg = 0, nu = 0;
            // the next unit is found while the current one runs (its loads off the unit boundary)
            int rnd_is = 0;
            Unit w_is = next_unit(rnd_is);
            while (w_is.n_kv > 0 && ok) {
                const Unit w_after = next_unit(rnd_is);
                const int n_kv = w_is.n_kv;
                ok = tc05::wait_bounded(q_full, nu & 1) && tc05::wait_bounded(&k_full[jg % SLOTS], (jg / SLOTS) & 1);
                if (!ok) break;
                tc05::fence_after();
                issue_s(0, jg);
                issue_s(1, jg);
                tc05::commit(&k_empty[jg % SLOTS]);  // K of the unit's first tile is free once both S complete
                if (n_kv == 1) tc05::commit(q_empty);  // the unit's last score MMA is issued
                for (int j = 0; ok && j < n_kv; ++j) {
                    const int g = jg + j, sl = g % SLOTS;
                    const bool more = j + 1 < n_kv;
                    ok = tc05::wait_bounded(&v_full[sl], (g / SLOTS) & 1);
                    // P_X(g+1) needs S_X(g+1), issued below after both waits of P_Xg: each half's
                    // p_full is at most one phase ahead
                    ok = ok && tc05::wait_bounded(&p_full[0], g & 1);
                    if (!ok) break;
                    tc05::fence_after();
                    issue_pv(0, g, 0, j == 0);
                    ok = tc05::wait_bounded(&p_full[1], g & 1);
                    if (!ok) break;
                    tc05::fence_after();
                    issue_pv(0, g, 1, j == 0);
                    if (more) {
                        ok = tc05::wait_bounded(&k_full[(g + 1) % SLOTS], ((g + 1) / SLOTS) & 1);
                        if (!ok) break;
                        tc05::fence_after();
                        issue_s(0, g + 1);  // after P_A(g) . V_g on the pipe: overwrites P_A(g) in S_A
                    }
                    ok = tc05::wait_bounded(&p_full[2], g & 1);
                    if (!ok) break;
                    tc05::fence_after();
                    issue_pv(1, g, 0, j == 0);
                    ok = tc05::wait_bounded(&p_full[3], g & 1);
                    if (!ok) break;
                    tc05::fence_after();
                    issue_pv(1, g, 1, j == 0);
                    tc05::commit(&v_empty[sl]);  // V_g is free once both P . V_g complete
                    if (more) {
                        issue_s(1, g + 1);
                        tc05::commit(&k_empty[(g + 1) % SLOTS]);
                        if (j + 2 == n_kv) tc05::commit(q_empty);  // the unit's last score MMA is issued
                    }
                }
                if (!ok) break;
                tc05::commit(o_final);
                jg += n_kv;
                ++nu;
                w_is = w_after;
            }
            if (!ok) flag_error(p.err, PA_DEVERR_TIMEOUT);
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
    const int prow_id = X * 128 + r;  // packed row of the unit
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t o_addr = lane_addr + C::O_COL + X * D + hh * DH;
    const uint32_t sa = lane_addr + C::S_COL + X * BN;
    float* xmax = reinterpret_cast<float*>(smem + C::RED_OFF);  // [tile parity][X][half][row]
    float* xl = xmax + 2 * 2 * 2 * 128;                          // [X][half][row]
    const int gbar = 3 + X;                                      // the group's named barrier (256 threads)
    const float sl2 = p.scale_log2;
    const bool out32 = (reinterpret_cast<uintptr_t>(p.out) & 31) == 0;  // rows are 2 D bytes apart
    bool ok = true;
    int jg = 0, nu = 0;
    for (int rnd = 0, u = unit_of(0); u < n_units && ok; u = unit_of(++rnd)) {
        const Unit w = unit_at(u);
        if (w.n_kv == 0) continue;
        const int n_kv = w.n_kv, L = w.L;
        const int tok = w.tok0 + prow_id / G;
        const bool valid = tok < w.Cq;
        const int pos = valid ? w.base + tok : -1;
        // this thread's output row (-1: a row past the chunk, never stored)
        const int64_t orow_off =
            valid ? (static_cast<int64_t>(w.q0 + tok) * p.hq + w.kvh * G + prow_id % G) * D + hh * DH : -1;
        // position of the first row of this warp's 32 (every valid row of the warp is at or after it)
        const int warp_tok = w.tok0 + (X * 128 + wq * 32) / G;
        const int warp_pos_min = warp_tok < w.Cq ? w.base + warp_tok : -1;
        float m = -INFINITY, l = 0.f;  // l: this half's share of the row sum
        for (int j = 0; j < n_kv; ++j) {
            const int g = jg + j, sl = g % SLOTS;
            // decisions that guard a tcgen05.ld / st are warp-uniform (those are .sync.aligned).
            // Neither barrier can run two phases ahead: V of tile g + SLOTS is loaded, and S_X(g + 1)
            // issued, only after this thread's P_Xg has been consumed
            const bool got = __all_sync(0xffffffffu, tc05::wait_bounded(&v_full[sl], (g / SLOTS) & 1) &&
                                                         tc05::wait_bounded(&s_full[X], g & 1));
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
                float t[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) t[i] = -INFINITY;
                if (interior) {
#pragma unroll
                    for (int c = 0; c < 64; c += 2)
                        t[(c >> 1) & 3] = tc05::max3(t[(c >> 1) & 3], __uint_as_float(sr[c]), __uint_as_float(sr[c + 1]));
                } else {
#pragma unroll
                    for (int c = 0; c < 64; ++c) {
                        const int key = hh * 64 + c;
                        const bool vis = key0 + key <= pos && ((okmask >> (key >> 4)) & 1);
                        const float x = vis ? __uint_as_float(sr[c]) * sl2 : -INFINITY;
                        sr[c] = __float_as_uint(x);
                        t[c & 3] = fmaxf(t[c & 3], x);
                    }
                }
                pmx = fmaxf(fmaxf(t[0], t[1]), fmaxf(t[2], t[3]));
                if (interior) pmx *= sl2;
                xmax[(((g & 1) * 2 + X) * 2 + hh) * 128 + r] = pmx;
            }
            // every thread of the group arrives here once per tile, so a timeout ends the loop for the
            // whole group at the same tile; the partner's max of tile g sits in the parity-g buffer,
            // which is written again (tile g + 2) only after both have passed tile g + 1's barrier
            if (!tc05::bar_and(gbar, 256, got)) {
                ok = false;
                break;
            }
            const float mx = fmaxf(pmx, xmax[(((g & 1) * 2 + X) * 2 + (hh ^ 1)) * 128 + r]);
            // lazy rescale per row (both threads of a row decide alike); O_X is rescaled for the whole
            // warp when any row needs it.  No P . V of tile X is in flight: S_X(g) was issued after
            // P_X(g-1) . V_(g-1), and its completion, seen above, reports that one's too
            const bool grow = mx > m + kLazyRescale;
            const bool scale_o = grow && m != -INFINITY;
            const float a = scale_o ? tc05::fast_exp2(m - mx) : 1.f;
            if (j > 0 && __any_sync(0xffffffffu, scale_o)) tc05::scale_tmem_cols<DH>(o_addr, a);
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
            float ls[2] = {0.f, 0.f};
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
                        tc05::add2(ls[0], ls[1], e0, e1);
                    }
                    tc05::st8(sa + hh * 32 + qq * 16 + hv * 8, pw);
                }
                tc05::wait_st();
                tc05::fence_before();
                mbar_arrive(&p_full[X * 2 + qq]);
            }
            l += ls[0] + ls[1];
        }
        // ---- the unit's end: both groups meet (a timeout anywhere ends every softmax warp's walk here)
        if (!tc05::bar_and(2, C::NSW * 32, ok)) {
            ok = false;
            break;
        }
        const bool done = tc05::bar_and(2, C::NSW * 32, tc05::wait_bounded(o_final, nu & 1));
        if (!done) {
            ok = false;
            break;
        }

        // the row sum: this half's share plus the partner's; xl is written again only after every
        // softmax thread has passed the next unit's first barrier above
        xl[(X * 2 + hh) * 128 + r] = l;
        tc05::named_sync(gbar, 256);
        const float lt = l + xl[(X * 2 + (hh ^ 1)) * 128 + r];
        tc05::fence_after();
        const float inv = lt > 0.f ? 1.f / lt : 0.f;
        T* orow = static_cast<T*>(p.out) + (orow_off < 0 ? 0 : orow_off);
        // O_X is read here before this thread publishes any P of the next unit, whose first P . V
        // overwrites it
#pragma unroll
        for (int c0 = 0; c0 < DH; c0 += 16) {
            uint32_t o[16];
            tc05::ld16(o_addr + c0, o);
            tc05::wait_ld();
            if (orow_off >= 0) {
                uint32_t pw[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    pw[i] = pack2<T>(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
                // lanes hold different rows: a 32-byte store per lane writes whole sectors, half as
                // many L2 transactions as 16-byte ones (the epilogue's stores were its whole cost)
                if (out32) {
                    st_global_v8(orow + c0, pw);
                } else {
                    *reinterpret_cast<uint4*>(orow + c0) = make_uint4(pw[0], pw[1], pw[2], pw[3]);
                    *reinterpret_cast<uint4*>(orow + c0 + 8) = make_uint4(pw[4], pw[5], pw[6], pw[7]);
                }
            }
        }
        jg += n_kv;
        ++nu;
    }
    if (!ok && lane == 0) flag_error(p.err, PA_DEVERR_TIMEOUT);
    griddep_launch_dependents();
    tc05::fence_before();
    tc05::named_sync(1, (C::NSW + 1) * 32);
}

template <typename T, int D, int G>
cudaError_t launch_prefill_tc05w(const PrefillParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                 const CUtensorMap& qmap, int max_query_len, cudaStream_t stream) {
    using C = Tc05wCfg<D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc05w<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(C::smem_bytes));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int64_t rows = static_cast<int64_t>(max_query_len) * G;
    const int q_tiles = static_cast<int>((rows + C::BM - 1) / C::BM);
    const int64_t units = static_cast<int64_t>(q_tiles) * p.hkv * p.batch;
    if (units >= (1LL << 31)) return cudaErrorNotSupported;
    const int ctas = static_cast<int>(units < sm_count() ? units : sm_count());  // one CTA per SM, persistent
    if (ctas <= 0) return cudaSuccess;
    return launch_pdl(prefill_tc05w<T, D, G>, dim3(ctas), dim3(C::THREADS), C::smem_bytes, stream, p, q_tiles, kmap,
                      vmap, qmap);
}

}  // namespace pa
