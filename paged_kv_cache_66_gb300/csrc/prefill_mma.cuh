// Paged prefill attention on the tensor cores (mma.sync m16n8k16, fp32
// accumulate) for fp16 / bf16 pools.
//
// A chunk of C new query tokens of one sequence attends causally to the
// sequence's paged history plus the chunk itself ("25. Paged attention and
// prefix caching", stretch exercise 4; "Chapter 7 Paged KV Cache and Memory
// Management", 4.1 step 3: the key at position p is visible to the query at
// position i iff p <= i).  The chunk is the last C positions of the
// sequence; its K/V rows are appended to the pool before the call.
//
// One CTA: one KV head of one sequence and BM = 64 query rows, a row being a
// (chunk token, query head of the group) pair with the G heads of a token
// side by side, so every K/V tile staged in shared memory serves all G heads.
// Four consumer warps own 16 rows each:
//   S[16 rows x 16 keys] = Q[16 x D] . K_tile^T     (A = Q in registers, B = K by ldmatrix)
//   O[16 rows x D]      += P[16 x 16 keys] . V_tile  (A = P from the S fragments, B = V by ldmatrix.trans)
// with the online softmax per row (base 2, lazy rescale).  A fifth warp
// produces: its lanes read 32 block-table entries at a time, and lane 0
// issues the TMA copies of each 16-key K and V tile -- the decode kernel's
// tile format, D/64 boxes of 16 rows x 128 bytes with the 128-byte swizzle --
// into a ring shared by the consumers (full barriers count the transaction
// bytes, empty barriers one arrival per consumer warp).  Every wait is
// bounded (1 s of %globaltimer) and reports PA_DEVERR_TIMEOUT.
//
// Keys at or past the sequence length are masked by position; their V rows
// (unwritten slots may hold anything) are zeroed in the B fragments, so a
// NaN there cannot reach the output.
#pragma once

#include "decode_mma.cuh"

namespace pa {

template <int D>
struct PrefillCfg {
    static constexpr int NWC = 4;                   // consumer warps
    static constexpr int THREADS = (NWC + 1) * 32;  // + one producer warp
    static constexpr int BM = NWC * 16;             // query rows per CTA
    static constexpr int ROW_BYTES = D * 2;
    static constexpr int NBOX = ROW_BYTES / 128;
    static constexpr int BOX_ELEMS = 64;
    static constexpr int TILE_BYTES = NBOX * 2048;  // 16 keys
    static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
    static constexpr int STAGES = D == 256 ? 4 : 8;
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int FULL_OFF = RING_BYTES;
    static constexpr int EMPTY_OFF = FULL_OFF + STAGES * 8;
    static constexpr int OK_OFF = EMPTY_OFF + STAGES * 8;
    static constexpr int KSTEPS = D / 16;
    static constexpr int DN = D / 8;  // n8 blocks of the output
    static constexpr size_t smem_bytes = 1024 + OK_OFF + STAGES * 4;
};

// keeps the 16-bit halves of x (keys k and k + 1) whose key is below nv
__device__ __forceinline__ uint32_t keep_keys(uint32_t x, int k, int nv) {
    return k + 1 < nv ? x : (k < nv ? (x & 0xFFFFu) : 0u);
}

template <typename T, int D, int G>
__global__ void __launch_bounds__(PrefillCfg<D>::THREADS)
    prefill_mma(const PrefillParams p, const __grid_constant__ CUtensorMap kmap,
                const __grid_constant__ CUtensorMap vmap) {
    using C = PrefillCfg<D>;
    constexpr int STAGES = C::STAGES, KSTEPS = C::KSTEPS, DN = C::DN;
    constexpr int QT = C::BM / G;  // chunk tokens per CTA
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::FULL_OFF);
    uint64_t* empty = reinterpret_cast<uint64_t*>(smem + C::EMPTY_OFF);
    int* stage_ok = reinterpret_cast<int*>(smem + C::OK_OFF);

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
    const int n_sub = (kv_end + 15) / 16;

    if (tid == 0) {
#pragma unroll
        for (int st = 0; st < STAGES; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], C::NWC);
        }
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == C::NWC) {
        // ------------------------------------------------------------ producer
        const int32_t* trow = p.block_tables + static_cast<size_t>(s) * p.max_blocks;
        int issued = 0;
        bool ok = true;
        for (int j0 = 0; j0 < n_sub && ok; j0 += 32) {
            int row = -1;
            const int j = j0 + lane;
            if (j < n_sub) {
                const int e = __ldg(trow + (j * 16) / p.block_size);
                if (e >= 0 && e < p.num_blocks) {
                    row = (e * p.hkv + kvh) * p.block_size + (j * 16) % p.block_size;
                } else {
                    flag_error(p.err, PA_DEVERR_TABLE);
                }
            }
            const int cnt = min(32, n_sub - j0);
            for (int i = 0; i < cnt; ++i) {
                const int r = __shfl_sync(0xffffffffu, row, i);
                if (lane == 0 && ok) {
                    const int st = issued % STAGES;
                    if (!mbar_wait_bounded(&empty[st], ((issued / STAGES) & 1) ^ 1)) {
                        flag_error(p.err, PA_DEVERR_TIMEOUT);
                        ok = false;
                    } else {
                        stage_ok[st] = r >= 0;
                        if (r < 0) {
                            mbar_arrive_expect_tx(&full[st], 0);
                        } else {
                            unsigned char* dst = smem + st * C::STAGE_BYTES;
                            mbar_arrive_expect_tx(&full[st], C::STAGE_BYTES);
#pragma unroll
                            for (int bx = 0; bx < C::NBOX; ++bx) {
                                tma_load_2d(dst + bx * 2048, &kmap, bx * C::BOX_ELEMS, r, &full[st]);
                                tma_load_2d(dst + C::TILE_BYTES + bx * 2048, &vmap, bx * C::BOX_ELEMS, r, &full[st]);
                            }
                        }
                        ++issued;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
            }
        }
        // the last STAGES copies land before this warp leaves (they normally have: the
        // consumers waited for them)
        if (lane == 0) {
            for (int k = max(0, issued - STAGES); k < issued; ++k)
                mbar_wait_bounded(&full[k % STAGES], (k / STAGES) & 1);
        }
        return;
    }

    // -------------------------------------------------------------- consumers
    const int g = lane >> 2, t = lane & 3;
    const int lm = lane >> 3, lr = lane & 7;
    const int rA = warp * 16 + g, rB = rA + 8;  // this lane's two rows of the CTA
    const int tokA = tok0 + rA / G, tokB = tok0 + rB / G;
    const bool validA = tokA < Cq, validB = tokB < Cq;
    const int posA = validA ? base + tokA : -1;
    const int posB = validB ? base + tokB : -1;
    const int headA = kvh * G + rA % G, headB = kvh * G + rB % G;
    const int warp_last = min(Cq - 1, tok0 + (warp * 16 + 15) / G);
    const int warp_pos = tok0 + (warp * 16) / G < Cq ? base + warp_last : -1;  // largest visible key

    // Q fragments (A operand): rows rA / rB, k = dims
    uint32_t qa[KSTEPS][4];
    {
        const T* qA = static_cast<const T*>(p.q) + (static_cast<size_t>(q0 + (validA ? tokA : 0)) * p.hq + headA) * D;
        const T* qB = static_cast<const T*>(p.q) + (static_cast<size_t>(q0 + (validB ? tokB : 0)) * p.hq + headB) * D;
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks) {
            const int d0 = ks * 16 + 2 * t;
            qa[ks][0] = validA ? __ldg(reinterpret_cast<const unsigned int*>(qA + d0)) : 0u;
            qa[ks][1] = validB ? __ldg(reinterpret_cast<const unsigned int*>(qB + d0)) : 0u;
            qa[ks][2] = validA ? __ldg(reinterpret_cast<const unsigned int*>(qA + d0 + 8)) : 0u;
            qa[ks][3] = validB ? __ldg(reinterpret_cast<const unsigned int*>(qB + d0 + 8)) : 0u;
        }
    }
    float o[DN][4];
#pragma unroll
    for (int nd = 0; nd < DN; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
    float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
    const float sl2 = p.scale_log2;

    for (int j = 0; j < n_sub; ++j) {
        const int st = j % STAGES;
        // one decision for the whole warp: ldmatrix, mma and the shuffles below are collectives
        if (!__all_sync(0xffffffffu, mbar_wait_bounded(&full[st], (j / STAGES) & 1))) {
            if (lane == 0) flag_error(p.err, PA_DEVERR_TIMEOUT);
            break;
        }
        const int key0 = j * 16;
        if (key0 <= warp_pos && stage_ok[st]) {
            const uint32_t kb = smem_u32(smem + st * C::STAGE_BYTES);
            const uint32_t vb = kb + C::TILE_BYTES;
            // ---- S = Q K^T: sc[nb] covers keys nb*8 .. nb*8+7; two accumulator sets per n-block
            float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            float sd[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int ks = 0; ks < KSTEPS; ++ks) {
                uint32_t r[4];
                ldsm_x4(kb + swz(lr + (lm >> 1) * 8, ks * 2 + (lm & 1)), r);
                mma16816<T>((ks & 1) ? sd[0] : sc[0], qa[ks], r[0], r[1]);
                mma16816<T>((ks & 1) ? sd[1] : sc[1], qa[ks], r[2], r[3]);
            }
            // sc[nb] = {S[rA][k], S[rA][k+1], S[rB][k], S[rB][k+1]} with k = nb*8 + 2t
#pragma unroll
            for (int nb = 0; nb < 2; ++nb) {
                const int k = key0 + nb * 8 + 2 * t;
                sc[nb][0] = k <= posA ? (sc[nb][0] + sd[nb][0]) * sl2 : -INFINITY;
                sc[nb][1] = k + 1 <= posA ? (sc[nb][1] + sd[nb][1]) * sl2 : -INFINITY;
                sc[nb][2] = k <= posB ? (sc[nb][2] + sd[nb][2]) * sl2 : -INFINITY;
                sc[nb][3] = k + 1 <= posB ? (sc[nb][3] + sd[nb][3]) * sl2 : -INFINITY;
            }
            float mxA = fmaxf(fmaxf(sc[0][0], sc[0][1]), fmaxf(sc[1][0], sc[1][1]));
            float mxB = fmaxf(fmaxf(sc[0][2], sc[0][3]), fmaxf(sc[1][2], sc[1][3]));
            mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 1));
            mxA = fmaxf(mxA, __shfl_xor_sync(0xffffffffu, mxA, 2));
            mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 1));
            mxB = fmaxf(mxB, __shfl_xor_sync(0xffffffffu, mxB, 2));
            if (mxA > mA + kLazyRescale) {
                const float a = exp2f(mA - mxA);
                lA *= a;
#pragma unroll
                for (int nd = 0; nd < DN; ++nd) {
                    o[nd][0] *= a;
                    o[nd][1] *= a;
                }
                mA = mxA;
            }
            if (mxB > mB + kLazyRescale) {
                const float a = exp2f(mB - mxB);
                lB *= a;
#pragma unroll
                for (int nd = 0; nd < DN; ++nd) {
                    o[nd][2] *= a;
                    o[nd][3] *= a;
                }
                mB = mxB;
            }
            // a row with no visible key yet keeps m = -inf: use 0 so exp2(-inf - 0) = 0
            const float mAs = mA == -INFINITY ? 0.f : mA, mBs = mB == -INFINITY ? 0.f : mB;
            float pr[2][4];
#pragma unroll
            for (int nb = 0; nb < 2; ++nb) {
                pr[nb][0] = exp2f(sc[nb][0] - mAs);
                pr[nb][1] = exp2f(sc[nb][1] - mAs);
                pr[nb][2] = exp2f(sc[nb][2] - mBs);
                pr[nb][3] = exp2f(sc[nb][3] - mBs);
                lA += pr[nb][0] + pr[nb][1];
                lB += pr[nb][2] + pr[nb][3];
            }
            // P as the A operand over the 16 keys
            const uint32_t pa[4] = {pack2<T>(pr[0][0], pr[0][1]), pack2<T>(pr[0][2], pr[0][3]),
                                    pack2<T>(pr[1][0], pr[1][1]), pack2<T>(pr[1][2], pr[1][3])};
            // ---- O += P V; V fragments b0 = keys 2t, 2t+1 and b1 = keys 8+2t, 9+2t of dim nd*8 + g
            const int nv = L - key0;  // keys of this tile inside the sequence (>= 16 except at the end)
#pragma unroll
            for (int nd = 0; nd < DN; nd += 2) {
                uint32_t r[4];
                ldsm_x4_t(vb + swz(lr + (lm & 1) * 8, nd + (lm >> 1)), r);
                if (nv < 16) {
                    r[0] = keep_keys(r[0], 2 * t, nv);
                    r[1] = keep_keys(r[1], 8 + 2 * t, nv);
                    r[2] = keep_keys(r[2], 2 * t, nv);
                    r[3] = keep_keys(r[3], 8 + 2 * t, nv);
                }
                mma16816<T>(o[nd], pa, r[0], r[1]);
                mma16816<T>(o[nd + 1], pa, r[2], r[3]);
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
    griddep_launch_dependents();

    // ---- normalise and write: o[nd] = {O[rA][c], O[rA][c+1], O[rB][c], O[rB][c+1]}, c = nd*8 + 2t
    lA += __shfl_xor_sync(0xffffffffu, lA, 1);
    lA += __shfl_xor_sync(0xffffffffu, lA, 2);
    lB += __shfl_xor_sync(0xffffffffu, lB, 1);
    lB += __shfl_xor_sync(0xffffffffu, lB, 2);
    const float iA = lA > 0.f ? 1.f / lA : 0.f, iB = lB > 0.f ? 1.f / lB : 0.f;
    T* out = static_cast<T*>(p.out);
    if (validA) {
        T* oA = out + (static_cast<size_t>(q0 + tokA) * p.hq + headA) * D;
#pragma unroll
        for (int nd = 0; nd < DN; ++nd)
            *reinterpret_cast<uint32_t*>(oA + nd * 8 + 2 * t) = pack2<T>(o[nd][0] * iA, o[nd][1] * iA);
    }
    if (validB) {
        T* oB = out + (static_cast<size_t>(q0 + tokB) * p.hq + headB) * D;
#pragma unroll
        for (int nd = 0; nd < DN; ++nd)
            *reinterpret_cast<uint32_t*>(oB + nd * 8 + 2 * t) = pack2<T>(o[nd][2] * iB, o[nd][3] * iB);
    }
}

template <typename T, int D, int G>
cudaError_t launch_prefill(const PrefillParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           int max_query_len, cudaStream_t stream) {
    using C = PrefillCfg<D>;
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(prefill_mma<T, D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(C::smem_bytes));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    const int64_t rows = static_cast<int64_t>(max_query_len) * G;
    const unsigned tiles = static_cast<unsigned>((rows + C::BM - 1) / C::BM);
    return launch_pdl(prefill_mma<T, D, G>, dim3(tiles, p.hkv, p.batch), dim3(C::THREADS), C::smem_bytes, stream, p,
                      kmap, vmap);
}

}  // namespace pa
