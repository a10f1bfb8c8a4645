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
        size_t d0 = 0, d1 = 0;
        const bool ok0 = place(r, d0), ok1 = place(r + step, d1);
        const size_t s0 = static_cast<size_t>(r) * vpr + c, s1 = static_cast<size_t>(r + step) * vpr + c;
        uint4 k0, v0, k1, v1;
        if (ok0) {
            k0 = __ldg(k + s0);
            v0 = __ldg(v + s0);
        }
        if (ok1) {
            k1 = __ldg(k + s1);
            v1 = __ldg(v + s1);
        }
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
    const int64_t y = blockIdx.y;
    const int64_t pair = y / (2 * num_layers);
    const int rem = static_cast<int>(y - pair * 2 * num_layers);
    const int layer = rem >> 1;
    const int kind = rem & 1;
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

// Failure-path check of the bounded waits: one warp initialises an mbarrier
// that nothing will ever complete and waits on it with the same helper the
// decode kernels use, for at most `limit_ns`.  The wait gives up, the kernel
// records PA_DEVERR_TIMEOUT and returns; nothing hangs and nothing faults.
__global__ void wait_timeout_selftest_kernel(uint64_t limit_ns, int* err) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncwarp();
    if (!mbar_wait_bounded(&bar, 0, limit_ns) && threadIdx.x == 0) flag_error(err, PA_DEVERR_TIMEOUT);
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
