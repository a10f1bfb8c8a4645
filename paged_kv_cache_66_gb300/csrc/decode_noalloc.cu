// pa_decode_noalloc: paged decode whose split-K scratch lives in a fixed
// device array inside this library, for callers that cannot allocate device
// memory themselves.
//
// Who needs it: code that runs where a device allocation is not an option at
// the moment it wants to decode -- a host application that hands this
// library only its own tensors and owns every other byte of device memory
// through its own allocator, a real-time loop that forbids allocation after
// start-up, or a plugin/ABI consumer with no allocator handle at all.  Such a
// caller still passes q, the pools, the tables and the output; only the
// scratch of the partition merge comes from here.
//
// The array below is reserved on a GPU when the module holding it is loaded
// there -- under CUDA's default lazy loading, by the first call's address
// lookup on that device -- and stays reserved until the process exits.
#include <cstdint>
#include <mutex>

#include "../../include/pagedkv.h"
#include "pa_launch.h"

namespace {

static __device__ __align__(256) unsigned char g_decode_scratch[PA_DECODE_NOALLOC_MAX_BYTES];

constexpr int kMaxDev = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDev] = {};

// Device address of g_decode_scratch on the current device.  The name of a
// __device__ array in host code is only a host-side shadow, never a device
// address, so it is looked up once per device with that device current.
pa_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return PA_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(void* out, const void* q, const void* k_pool, const void* v_pool,
                                       int64_t num_blocks, const int32_t* block_tables, int max_blocks,
                                       const int32_t* seq_lens, int batch, int num_q_heads, int num_kv_heads,
                                       int head_dim, int block_size, float scale, int partition_tokens,
                                       pa_dtype dtype, void* stream) {
    const size_t need =
        pa_decode_workspace_size(batch, num_q_heads, head_dim, max_blocks, block_size, partition_tokens);
    if (need > static_cast<size_t>(PA_DECODE_NOALLOC_MAX_BYTES)) return PA_ERR_INVALID;
    void* scratch = nullptr;
    if (need > 0) {
        pa_status st = scratch_address(&scratch);
        if (st != PA_OK) return st;
    }
    // The partition kernel writes every scratch entry the merge kernel reads in
    // the same call, so nothing has to be cleared between calls.
    return pa_decode(out, q, k_pool, v_pool, num_blocks, block_tables, max_blocks, seq_lens, batch, num_q_heads,
                     num_kv_heads, head_dim, block_size, scale, partition_tokens, scratch,
                     static_cast<size_t>(PA_DECODE_NOALLOC_MAX_BYTES), dtype, stream);
}
