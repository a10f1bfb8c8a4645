// KV append ("reshape_and_cache") and block copy-on-write kernels.
//
// "25. Paged attention and prefix caching", section "The paged cache":
// update scatters each new key/value row to (table[p // b], :, p % b) of the
// [num_blocks, kv_heads, b, head_dim] pool; reserve copies a shared block into
// a fresh one in every layer's K and V pool before it is written.
//
// Both are pure byte movement.  They move 16-byte vectors: consecutive threads
// touch consecutive vectors of one row (append) or one block (copy), so every
// warp access is a fully used, coalesced 512-byte span.
#include "pa_common.cuh"
#include "pa_launch.h"

namespace pa {

// One thread per 16-byte vector of a (token, head, {K,V}) row.
// rows are enumerated as (t * Hkv + h) * 2 + kind; vpr = vectors per row.
__global__ void __launch_bounds__(256) kv_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                                        uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                                                        const int64_t* __restrict__ slots, int64_t num_tokens,
                                                        int64_t num_slots, int hkv, int vpr, int block_size,
                                                        int* err) {
    griddep_wait();
    griddep_launch_dependents();
    const int64_t total = num_tokens * hkv * 2 * vpr;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t row = i / vpr;
        const int c = static_cast<int>(i - row * vpr);
        const int kind = static_cast<int>(row & 1);
        const int64_t th = row >> 1;  // t * hkv + h
        const int64_t t = th / hkv;
        const int h = static_cast<int>(th - t * hkv);
        const int64_t slot = __ldg(slots + t);
        if (slot < 0) continue;  // padding row
        if (slot >= num_slots) {
            if (c == 0 && kind == 0 && h == 0) flag_error(err, PA_DEVERR_SLOT);
            continue;
        }
        const int64_t blk = slot / block_size;
        const int64_t off = slot - blk * block_size;
        const int64_t dst = ((blk * hkv + h) * block_size + off) * vpr + c;
        const int64_t src = th * vpr + c;
        if (kind == 0)
            k_pool[dst] = __ldg(k + src);
        else
            v_pool[dst] = __ldg(v + src);
    }
}

// grid.y = pair * (2 * layers) + layer * 2 + kind; grid.x strides over the
// block's 16-byte vectors with 4 independent vectors in flight per thread.
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
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    for (; i + 3 * stride < vec_per_block; i += 4 * stride) {
        uint4 a0 = s[i], a1 = s[i + stride], a2 = s[i + 2 * stride], a3 = s[i + 3 * stride];
        d[i] = a0;
        d[i + stride] = a1;
        d[i + 2 * stride] = a2;
        d[i + 3 * stride] = a3;
    }
    for (; i < vec_per_block; i += stride) d[i] = s[i];
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
    const int64_t total = num_tokens * hkv * 2 * vpr;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = 152LL * 16;
    if (blocks > cap) blocks = cap;
    return launch_pdl(kv_append_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, stream,
                      static_cast<const uint4*>(k), static_cast<const uint4*>(v), static_cast<uint4*>(k_pool),
                      static_cast<uint4*>(v_pool), slots, num_tokens, num_blocks * block_size, hkv, vpr,
                      block_size, err);
}

cudaError_t launch_copy_blocks(const PoolPtrs& pools, int num_layers, const int64_t* pairs, int64_t num_pairs,
                               int64_t num_blocks, size_t block_bytes, int* err, cudaStream_t stream) {
    const int64_t vec = static_cast<int64_t>(block_bytes / 16);
    const int threads = 256;
    int64_t gx = (vec + threads * 4 - 1) / (threads * 4);
    if (gx < 1) gx = 1;
    if (gx > 64) gx = 64;
    // grid.y is limited to 65535: split the pairs into chunks
    const int64_t per_pair = 2LL * num_layers;
    const int64_t max_pairs = 65535 / per_pair;
    for (int64_t p0 = 0; p0 < num_pairs; p0 += max_pairs) {
        const int64_t np = (num_pairs - p0 < max_pairs) ? (num_pairs - p0) : max_pairs;
        dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(np * per_pair));
        cudaError_t e = launch_pdl(copy_blocks_kernel, grid, dim3(threads), 0, stream, pools, num_layers,
                                   pairs + 2 * p0, num_blocks, vec, err);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace pa
