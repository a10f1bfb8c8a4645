// KV append ("reshape_and_cache") and block copy-on-write kernels.
//
// "25. Paged attention and prefix caching", section "The paged cache":
// update scatters each new key/value row to (table[p // b], :, p % b) of the
// [num_blocks, kv_heads, b, head_dim] pool; reserve copies a shared block into
// a fresh one in every layer's K and V pool before it is written.
//
// Both are pure byte movement.  They move 16-byte vectors: consecutive threads
// touch consecutive vectors of one row (append) or one block (copy), so every
// warp access is a fully used, coalesced span, with several independent loads
// in flight per thread before the stores.
#include <cuda_fp8.h>

#include "pa_common.cuh"
#include "pa_launch.h"

namespace pa {

// A CTA of 256 threads moves 256 / vpr (token, head) rows per iteration, one
// 16-byte vector of K and one of V per thread per row (vpr = vectors per
// row); each thread keeps two rows -- four 16-byte loads -- in flight.  Index
// arithmetic is 32-bit (the host splits calls so that T * Hkv < 2^31).
__global__ void __launch_bounds__(256) kv_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                                        uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                                                        const int64_t* __restrict__ slots, int rows,
                                                        int64_t num_slots, int hkv, int vpr, int block_size,
                                                        int* err) {
    griddep_wait();
    griddep_launch_dependents();
    const int rpi = blockDim.x / vpr;  // rows per CTA iteration
    const int lr = threadIdx.x / vpr, c = threadIdx.x - lr * vpr;
    if (lr >= rpi) return;
    const bool narrow = num_slots < (1LL << 31);
    const int step = gridDim.x * rpi;
    auto place = [&](int r, size_t& dst) -> bool {
        const int t = r / hkv, h = r - t * hkv;
        const int64_t slot = __ldg(slots + t);
        if (slot < 0) return false;  // padding row
        if (slot >= num_slots) {
            if (c == 0 && h == 0) flag_error(err, PA_DEVERR_SLOT);
            return false;
        }
        int64_t blk, off;
        if (narrow) {
            const int s32 = static_cast<int>(slot);
            blk = s32 / block_size;
            off = s32 - static_cast<int>(blk) * block_size;
        } else {
            blk = slot / block_size;
            off = slot - blk * block_size;
        }
        dst = ((static_cast<size_t>(blk) * hkv + h) * block_size + off) * vpr + c;
        return true;
    };
    int r = blockIdx.x * rpi + lr;
    for (; r + step < rows; r += 2 * step) {
        // the rows' data is requested together with their slots (the rows lie inside k and v
        // whatever the slots say); only the stores wait for the slots
        const size_t s0 = static_cast<size_t>(r) * vpr + c, s1 = static_cast<size_t>(r + step) * vpr + c;
        const uint4 k0 = __ldg(k + s0), v0 = __ldg(v + s0);
        const uint4 k1 = __ldg(k + s1), v1 = __ldg(v + s1);
        size_t d0 = 0, d1 = 0;
        const bool ok0 = place(r, d0), ok1 = place(r + step, d1);
        if (ok0) {
            k_pool[d0] = k0;
            v_pool[d0] = v0;
        }
        if (ok1) {
            k_pool[d1] = k1;
            v_pool[d1] = v1;
        }
    }
    if (r < rows) {
        size_t d0 = 0;
        if (place(r, d0)) {
            const size_t s0 = static_cast<size_t>(r) * vpr + c;
            k_pool[d0] = __ldg(k + s0);
            v_pool[d0] = __ldg(v + s0);
        }
    }
}

// One CTA per (pair, layer, K|V) and 32 KiB of the block: every thread loads
// 8 vectors (strided by the CTA width) before storing them.
__global__ void __launch_bounds__(256) copy_blocks_kernel(PoolPtrs pools, int num_layers,
                                                          const int64_t* __restrict__ pairs, int64_t num_blocks,
                                                          int64_t vec_per_block, int* err) {
    griddep_wait();
    griddep_launch_dependents();
    // grid.y = (layer, kind) x pair with the pair fastest: CTAs resident together copy within few
    // pools, so they touch few pages (the copy runs at ~0.5 of the HBM rate when its concurrent
    // CTAs spread over 64 pools of 128 MB, at ~0.93 within a few)
    const int64_t y = blockIdx.y;
    const int64_t np = gridDim.y / (2 * num_layers);
    const int lk = static_cast<int>(y / np);
    const int64_t pair = y - static_cast<int64_t>(lk) * np;
    const int layer = lk >> 1;
    const int kind = lk & 1;
    const int64_t src = __ldg(pairs + 2 * pair);
    const int64_t dst = __ldg(pairs + 2 * pair + 1);
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
        if (blockIdx.x == 0 && threadIdx.x == 0 && layer == 0 && kind == 0) flag_error(err, PA_DEVERR_PAIR);
        return;
    }
    uint4* base = reinterpret_cast<uint4*>(kind == 0 ? pools.k[layer] : pools.v[layer]);
    const uint4* s = base + src * vec_per_block;
    uint4* d = base + dst * vec_per_block;
    constexpr int U = 8;
    const int64_t i0 = static_cast<int64_t>(blockIdx.x) * (U * 256) + threadIdx.x;
    uint4 x[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (i0 + u * 256 < vec_per_block) x[u] = s[i0 + u * 256];
#pragma unroll
    for (int u = 0; u < U; ++u)
        if (i0 + u * 256 < vec_per_block) d[i0 + u * 256] = x[u];
}

// FP8 append: the same scatter, quantising on the way.  Each thread turns 16
// input elements of one (token, head) row of K or V into 16 E4M3 bytes:
// code = e4m3(x / scale[h]) with an IEEE fp32 division, rounding to nearest
// even and saturating to +-448 (cvt.rn.satfinite), then one 16-byte store.
template <typename Tin>
__global__ void __launch_bounds__(256) kv_append_fp8_kernel(const Tin* __restrict__ k, const Tin* __restrict__ v,
                                                            uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                                                            const float* __restrict__ k_scale,
                                                            const float* __restrict__ v_scale,
                                                            const int64_t* __restrict__ slots, int rows,
                                                            int64_t num_slots, int hkv, int vpr, int block_size,
                                                            int* err) {
    griddep_wait();
    griddep_launch_dependents();
    const int total = rows * 2 * vpr;  // (row, K|V, 16-byte output chunk)
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const int c = i % vpr;
        const int rk = i / vpr;
        const int kind = rk & 1, r = rk >> 1;
        const int t = r / hkv, h = r - t * hkv;
        // the row's 16 inputs and its scale are requested together with the slot (they lie inside
        // k / v and the scale array whatever the slot says); only the store waits for the slot
        const Tin* src = (kind == 0 ? k : v) + (static_cast<size_t>(r) * vpr + c) * 16;
        float x[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) x[j] = Elt<Tin>::to_f32(src[j]);
        const float sc = __ldg((kind == 0 ? k_scale : v_scale) + h);
        const int64_t slot = __ldg(slots + t);
        if (slot < 0) continue;
        if (slot >= num_slots) {
            if (c == 0 && kind == 0 && h == 0) flag_error(err, PA_DEVERR_SLOT);
            continue;
        }
        const int64_t blk = slot / block_size, off = slot - blk * block_size;
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const float a = x[4 * j] / sc, b = x[4 * j + 1] / sc;
            const float cc = x[4 * j + 2] / sc, d = x[4 * j + 3] / sc;
            const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
            const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(cc, d), __NV_SATFINITE, __NV_E4M3);
            w[j] = (lo & 0xFFFFu) | (hi << 16);
        }
        const size_t dst = ((static_cast<size_t>(blk) * hkv + h) * block_size + off) * vpr + c;
        (kind == 0 ? k_pool : v_pool)[dst] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

cudaError_t launch_kv_append_fp8(const void* k, const void* v, pa_dtype in_dtype, void* k_pool, void* v_pool,
                                 const float* k_scale, const float* v_scale, const int64_t* slots,
                                 int64_t num_tokens, int64_t num_blocks, int hkv, int d, int block_size, int* err,
                                 cudaStream_t stream) {
    const int vpr = d / 16;  // 16-byte output chunks per row
    const int64_t chunk = ((1LL << 29) / (hkv * 2LL * vpr)) > 0 ? ((1LL << 29) / (hkv * 2LL * vpr)) : 1;
    const int es = in_dtype == PA_F32 ? 4 : 2;
    for (int64_t t0 = 0; t0 < num_tokens; t0 += chunk) {
        const int64_t nt = (num_tokens - t0 < chunk) ? (num_tokens - t0) : chunk;
        const int rows = static_cast<int>(nt * hkv);
        int64_t blocks = (static_cast<int64_t>(rows) * 2 * vpr + 255) / 256;
        if (blocks > 152LL * 12) blocks = 152LL * 12;
        if (blocks < 1) blocks = 1;
        const size_t off = static_cast<size_t>(t0) * hkv * d * es;
        const char* kb = static_cast<const char*>(k) + off;
        const char* vb = static_cast<const char*>(v) + off;
        cudaError_t e;
        const int64_t ns = num_blocks * block_size;
        uint4* kp = static_cast<uint4*>(k_pool);
        uint4* vp = static_cast<uint4*>(v_pool);
        dim3 grid(static_cast<unsigned>(blocks)), block(256);
        if (in_dtype == PA_F16)
            e = launch_pdl(kv_append_fp8_kernel<__half>, grid, block, 0, stream, reinterpret_cast<const __half*>(kb),
                           reinterpret_cast<const __half*>(vb), kp, vp, k_scale, v_scale, slots + t0, rows, ns, hkv,
                           vpr, block_size, err);
        else if (in_dtype == PA_BF16)
            e = launch_pdl(kv_append_fp8_kernel<__nv_bfloat16>, grid, block, 0, stream,
                           reinterpret_cast<const __nv_bfloat16*>(kb), reinterpret_cast<const __nv_bfloat16*>(vb), kp,
                           vp, k_scale, v_scale, slots + t0, rows, ns, hkv, vpr, block_size, err);
        else
            e = launch_pdl(kv_append_fp8_kernel<float>, grid, block, 0, stream, reinterpret_cast<const float*>(kb),
                           reinterpret_cast<const float*>(vb), kp, vp, k_scale, v_scale, slots + t0, rows, ns, hkv,
                           vpr, block_size, err);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Failure-path check of the bounded waits, in the shape the decode and
// prefill kernels use them: each lane of one warp waits, for at most
// `limit_ns`, on one of two mbarriers -- odd lanes on one whose phase 0 is
// completed here, even lanes on one that nothing completes -- so the lanes'
// own results differ.  The warp then decides together (__all_sync) and runs a
// full-mask shuffle reduction, as the kernels do after their waits.  Lane 0
// records PA_DEVERR_TIMEOUT only if the vote failed and the reduction saw all
// 32 lanes with the expected split (16 waits met, 16 given up); nothing hangs
// and nothing faults.
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns, int* err) {
    __shared__ uint64_t bar[2];
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (threadIdx.x == 0) mbar_arrive(&bar[1]);  // completes phase 0 of bar[1]; bar[0] stays open
    __syncwarp();
    const bool mine = mbar_wait_bounded(&bar[lane & 1], 0, limit_ns);
    const bool all_ok = __all_sync(0xffffffffu, mine);
    int met = mine ? 1 : 0, present = 1;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        met += __shfl_xor_sync(0xffffffffu, met, o);
        present += __shfl_xor_sync(0xffffffffu, present, o);
    }
    if (lane == 0 && !all_ok && met == 16 && present == 32) flag_error(err, PA_DEVERR_TIMEOUT);
}

cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, int* err, cudaStream_t stream) {
    wait_timeout_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns, err);
    return cudaGetLastError();
}

cudaError_t launch_kv_append(const void* k, const void* v, void* k_pool, void* v_pool, const int64_t* slots,
                             int64_t num_tokens, int64_t num_blocks, int hkv, int row_bytes, int block_size,
                             int* err, cudaStream_t stream) {
    const int vpr = row_bytes / 16;
    if (vpr > 256) return cudaErrorNotSupported;
    const int rpi = 256 / vpr;
    // chunks of tokens keep T * Hkv (the row index) below 2^31
    const int64_t chunk = ((1LL << 30) / hkv) > 0 ? ((1LL << 30) / hkv) : 1;
    for (int64_t t0 = 0; t0 < num_tokens; t0 += chunk) {
        const int64_t nt = (num_tokens - t0 < chunk) ? (num_tokens - t0) : chunk;
        const int rows = static_cast<int>(nt * hkv);
        int64_t blocks = (rows + 2LL * rpi - 1) / (2LL * rpi);
        const int64_t cap = 152LL * 12;
        if (blocks > cap) blocks = cap;
        if (blocks < 1) blocks = 1;
        const size_t off = static_cast<size_t>(t0) * hkv * vpr;
        cudaError_t e = launch_pdl(kv_append_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream,
                                   static_cast<const uint4*>(k) + off, static_cast<const uint4*>(v) + off,
                                   static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), slots + t0, rows,
                                   num_blocks * block_size, hkv, vpr, block_size, err);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_copy_blocks(const PoolPtrs& pools, int num_layers, const int64_t* pairs, int64_t num_pairs,
                               int64_t num_blocks, size_t block_bytes, int* err, cudaStream_t stream) {
    const int64_t vec = static_cast<int64_t>(block_bytes / 16);
    const int64_t gx = (vec + 8 * 256 - 1) / (8 * 256);
    // grid.y is limited to 65535: split the pairs into chunks
    const int64_t per_pair = 2LL * num_layers;
    const int64_t max_pairs = 65535 / per_pair;
    for (int64_t p0 = 0; p0 < num_pairs; p0 += max_pairs) {
        const int64_t np = (num_pairs - p0 < max_pairs) ? (num_pairs - p0) : max_pairs;
        dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(np * per_pair));
        cudaError_t e = launch_pdl(copy_blocks_kernel, grid, dim3(256), 0, stream, pools, num_layers,
                                   pairs + 2 * p0, num_blocks, vec, err);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace pa
