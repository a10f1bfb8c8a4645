// C ABI of the paged KV-cache device library: argument validation, the
// device error word, and dispatch to the kernels.  See include/pagedkv.h for
// the contract of every entry point.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include <cudaTypedefs.h>

#include "pa_common.cuh"
#include "pa_launch.h"

namespace {

__device__ int g_pa_error_word;

constexpr int kMaxDevices = 64;
constexpr int kDefaultPartition = 512;
// E4M3 pools: a token carries half the bytes, and the byte-tile kernel measured fastest at 2048-token
// partitions on the long-context workload (512: 0.83, 1024: 0.84, 2048: 0.87, 4096: 0.84 of the
// HBM peak), with the unit threshold halved so that 2048 holds there
constexpr int kDefaultPartitionE4M3 = 2048;
constexpr int kMaxPartition = pa::kMaxPartitionTokens;
constexpr int kMinAutoPartition = 128;
// partition_tokens = 0: 512 tokens, halved (down to 128) while the launch would have fewer than
// this many (sequence, KV head, partition) units -- about four per SM of a GB300 (152 SMs).
// Short histories then still fill the GPU, and each CTA's serial chain of tiles is shorter.
constexpr int64_t kAutoMinUnits = 4 * 152;

std::mutex g_mu;
int* g_err_ptr[kMaxDevices] = {};

// Device address of the error word on the current device (looked up once).
int* error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_pa_error_word) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<int*>(p);
    }
    return g_err_ptr[dev];
}

std::atomic<int> g_decode_kernel{PA_DECODE_AUTO};
std::atomic<int> g_decode_heads{0};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

inline bool al(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

inline int elt_size(pa_dtype t) {
    switch (t) {
        case PA_F32: return 4;
        case PA_F16: return 2;
        case PA_BF16: return 2;
        default: return 0;
    }
}

inline pa_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return PA_OK;
    if (e == cudaErrorNotSupported) return PA_ERR_UNSUPPORTED;
    return PA_ERR_CUDA;
}

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Decode scratch: [(max, normaliser) B*Hq*P*2 f32 | partials B*Hq*P*D f32],
// the second region 256-byte aligned.
struct WsLayout {
    int partitions;
    size_t acc_off;
    size_t total;
};

// The automatic partition size.  It depends only on arguments that pa_decode_workspace_size
// also receives, so the two always agree.  The number of KV heads is not among them: the unit
// count takes hq / 8 (the fewest KV heads a supported group allows) as a lower estimate.
// With `e4m3` the result is never smaller than the 16-bit one (it starts higher and stops at a
// lower unit count), so a workspace sized by pa_decode_workspace_size(..., 0) always suffices.
int auto_partition(int batch, int hq, int max_blocks, int b, bool e4m3 = false) {
    int part = e4m3 ? kDefaultPartitionE4M3 : kDefaultPartition;
    const int64_t min_units = e4m3 ? kAutoMinUnits / 2 : kAutoMinUnits;
    if (b > 0 && part % b != 0) part = b * (part / b > 0 ? part / b : 1);
    const int64_t ctx = static_cast<int64_t>(max_blocks) * b;
    const int64_t rows = static_cast<int64_t>(batch) * ((hq + 7) / 8);
    while (part / 2 >= kMinAutoPartition && (part / 2) % b == 0 && (part / 2) % 16 == 0 &&
           rows * ((ctx + part - 1) / part) < min_units)
        part /= 2;
    return part;
}

WsLayout ws_layout(int batch, int hq, int d, int max_blocks, int b, int part) {
    WsLayout w{};
    w.partitions = static_cast<int>(ceil_div(static_cast<int64_t>(max_blocks) * b, part));
    if (w.partitions <= 1) return w;
    const size_t rows = static_cast<size_t>(batch) * hq * w.partitions;
    w.acc_off = align256(rows * 2 * sizeof(float));
    w.total = w.acc_off + rows * static_cast<size_t>(d) * sizeof(float);
    return w;
}

}  // namespace

namespace pa {

static PFN_cuTensorMapEncodeTiled_v12000 encoder() {
    std::call_once(g_encode_once, [] {
        void* fn = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    });
    return g_encode;
}

bool encode_pool_tmap(CUtensorMap* map, const void* pool, uint64_t rows, int d, int elt_bytes, int box_rows) {
    auto enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(d) * elt_bytes};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / elt_bytes), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, elt_bytes == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, const_cast<void*>(pool), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_pool_tmap_slices(CUtensorMap* map, const void* pool, uint64_t rows, int d, int box_rows) {
    auto enc = encoder();
    if (!enc || d % 64 != 0 || d / 64 > 256 || box_rows <= 0 || box_rows > 256) return false;
    // dims (element in the slice, row, slice): the row's stride is the whole row, the slice's 128 B,
    // so one box lands as [slice][box_rows rows][128 B], each slice its own run of 128-byte rows
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(d / 64)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, 128};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), static_cast<cuuint32_t>(d / 64)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(pool), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_q_tmap(CUtensorMap* map, const void* q, int total_q, int hq, int d, int g) {
    auto enc = encoder();
    if (!enc || g <= 0 || 128 % g != 0 || d % 64 != 0) return false;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(hq),
                                static_cast<cuuint64_t>(total_q)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(hq) * d * 2};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(g), static_cast<cuuint32_t>(128 / g)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<void*>(q), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (dev >= 0 && dev < 64) {
        const int c = cache[dev].load(std::memory_order_relaxed);
        if (c > 0) return c;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace pa

extern "C" {

pa_status pa_set_decode_kernel(pa_decode_kernel kernel) {
    if (kernel != PA_DECODE_AUTO && kernel != PA_DECODE_SIMT && kernel != PA_DECODE_MMA) return PA_ERR_INVALID;
    g_decode_kernel.store(kernel);
    return PA_OK;
}

pa_status pa_set_decode_heads_per_cta(int heads) {
    if (heads < 0 || heads > 2) return PA_ERR_INVALID;
    g_decode_heads.store(heads);
    return PA_OK;
}


pa_status pa_kv_append(const void* k, const void* v, void* k_pool, void* v_pool, const int64_t* slot_mapping,
                       int64_t num_tokens, int64_t num_blocks, int num_kv_heads, int head_dim, int block_size,
                       pa_dtype dtype, void* stream) {
    const int es = elt_size(dtype);
    if (es == 0 || num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0)
        return PA_ERR_INVALID;
    if (!k_pool || !v_pool || !al(k_pool, 16) || !al(v_pool, 16)) return PA_ERR_INVALID;
    if ((static_cast<int64_t>(head_dim) * es) % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !slot_mapping || !al(k, 16) || !al(v, 16) || !al(slot_mapping, 8)) return PA_ERR_INVALID;
    int* err = error_word();
    if (!err) return PA_ERR_CUDA;
    return from_cuda(pa::launch_kv_append(k, v, k_pool, v_pool, slot_mapping, num_tokens, num_blocks, num_kv_heads,
                                          head_dim * es, block_size, err, static_cast<cudaStream_t>(stream)));
}

pa_status pa_copy_blocks(void* const* k_pools, void* const* v_pools, int num_layers, const int64_t* pairs,
                         int64_t num_pairs, int64_t num_blocks, size_t block_bytes, void* stream) {
    if (!k_pools || !v_pools || num_layers <= 0 || num_pairs < 0 || num_blocks <= 0 || block_bytes == 0 ||
        block_bytes % 16 != 0)
        return PA_ERR_INVALID;
    for (int l = 0; l < num_layers; ++l)
        if (!k_pools[l] || !v_pools[l] || !al(k_pools[l], 16) || !al(v_pools[l], 16)) return PA_ERR_INVALID;
    if (num_pairs == 0) return PA_OK;
    if (!pairs || !al(pairs, 8)) return PA_ERR_INVALID;
    int* err = error_word();
    if (!err) return PA_ERR_CUDA;
    for (int l0 = 0; l0 < num_layers; l0 += pa::kMaxLayersPerLaunch) {
        const int nl = (num_layers - l0 < pa::kMaxLayersPerLaunch) ? num_layers - l0 : pa::kMaxLayersPerLaunch;
        pa::PoolPtrs pp{};
        for (int l = 0; l < nl; ++l) {
            pp.k[l] = k_pools[l0 + l];
            pp.v[l] = v_pools[l0 + l];
        }
        pa_status st = from_cuda(pa::launch_copy_blocks(pp, nl, pairs, num_pairs, num_blocks, block_bytes, err,
                                                        static_cast<cudaStream_t>(stream)));
        if (st != PA_OK) return st;
    }
    return PA_OK;
}

size_t pa_decode_workspace_size(int batch, int num_q_heads, int head_dim, int max_blocks, int block_size,
                                int partition_tokens) {
    if (batch <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_blocks <= 0 || block_size <= 0) return 0;
    const int part =
        partition_tokens == 0 ? auto_partition(batch, num_q_heads, max_blocks, block_size) : partition_tokens;
    if (part <= 0) return 0;
    return ws_layout(batch, num_q_heads, head_dim, max_blocks, block_size, part).total;
}

namespace {

// pa_decode with, optionally, the fused append of each sequence's newest row (k_new, v_new,
// new_slots non-null: tensor-core kernel only, the caller has checked that it applies)
pa_status decode_impl(void* out, const void* q, const void* k_pool, const void* v_pool, int64_t num_blocks,
                      const int32_t* block_tables, int max_blocks, const int32_t* seq_lens, int batch, int num_q_heads,
                      int num_kv_heads, int head_dim, int block_size, float scale, int partition_tokens,
                      void* workspace, size_t workspace_bytes, pa_dtype dtype, void* stream, const void* k_new,
                      const void* v_new, const int64_t* new_slots) {
    const int es = elt_size(dtype);
    if (es == 0 || batch < 0 || batch > 65535 || num_q_heads <= 0 || num_kv_heads <= 0 || num_kv_heads > 65535 ||
        head_dim <= 0 || block_size <= 0 || max_blocks <= 0 || num_blocks <= 0 || !std::isfinite(scale))
        return PA_ERR_INVALID;
    if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID;
    const int group = num_q_heads / num_kv_heads;
    if (group != 1 && group != 2 && group != 4 && group != 8) return PA_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return PA_ERR_UNSUPPORTED;
    if (block_size % 16 != 0 || block_size > 256) return PA_ERR_UNSUPPORTED;
    const int part =
        partition_tokens == 0 ? auto_partition(batch, num_q_heads, max_blocks, block_size) : partition_tokens;
    if (part <= 0 || part > kMaxPartition || part % 16 != 0 || part % block_size != 0) return PA_ERR_INVALID;
    if (static_cast<int64_t>(max_blocks) * block_size > (1LL << 30)) return PA_ERR_INVALID;
    if (batch == 0) return PA_OK;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !seq_lens) return PA_ERR_INVALID;
    if (!al(out, 16) || !al(q, 16) || !al(k_pool, 16) || !al(v_pool, 16) || !al(block_tables, 4) ||
        !al(seq_lens, 4))
        return PA_ERR_INVALID;
    const WsLayout ws = ws_layout(batch, num_q_heads, head_dim, max_blocks, block_size, part);
    if (ws.partitions > 1 && (!workspace || !al(workspace, 16) || workspace_bytes < ws.total))
        return PA_ERR_INVALID;
    int* err = error_word();
    if (!err) return PA_ERR_CUDA;

    pa::DecodeParams p{};
    p.out = out;
    p.q = q;
    p.k_pool = k_pool;
    p.v_pool = v_pool;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    char* wsb = static_cast<char*>(workspace);
    p.ws_ml = ws.partitions > 1 ? reinterpret_cast<float*>(wsb) : nullptr;
    p.ws_acc = ws.partitions > 1 ? reinterpret_cast<float*>(wsb + ws.acc_off) : nullptr;
    p.err = err;
    p.num_blocks = num_blocks;
    p.max_blocks = max_blocks;
    p.batch = batch;
    p.hq = num_q_heads;
    p.hkv = num_kv_heads;
    p.d = head_dim;
    p.block_size = block_size;
    p.partition_tokens = part;
    p.max_partitions = ws.partitions < 1 ? 1 : ws.partitions;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.k_new = k_new;
    p.v_new = v_new;
    p.new_slots = new_slots;
    p.kernel = g_decode_kernel.load();
    p.heads_per_cta = g_decode_heads.load();  // 0: the launcher chooses
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    switch (dtype) {
        case PA_F32: return from_cuda(pa::launch_decode_f32(p, st));
        case PA_F16: return from_cuda(pa::launch_decode_f16(p, st));
        case PA_BF16: return from_cuda(pa::launch_decode_bf16(p, st));
        default: return PA_ERR_INVALID;
    }
}

}  // namespace

pa_status pa_decode(void* out, const void* q, const void* k_pool, const void* v_pool, int64_t num_blocks,
                    const int32_t* block_tables, int max_blocks, const int32_t* seq_lens, int batch, int num_q_heads,
                    int num_kv_heads, int head_dim, int block_size, float scale, int partition_tokens,
                    void* workspace, size_t workspace_bytes, pa_dtype dtype, void* stream) {
    return decode_impl(out, q, k_pool, v_pool, num_blocks, block_tables, max_blocks, seq_lens, batch, num_q_heads,
                       num_kv_heads, head_dim, block_size, scale, partition_tokens, workspace, workspace_bytes, dtype,
                       stream, nullptr, nullptr, nullptr);
}

pa_status pa_decode_append(void* out, const void* q, const void* k_new, const void* v_new,
                           const int64_t* slot_mapping, void* k_pool, void* v_pool, int64_t num_blocks,
                           const int32_t* block_tables, int max_blocks, const int32_t* seq_lens, int batch,
                           int num_q_heads, int num_kv_heads, int head_dim, int block_size, float scale,
                           int partition_tokens, void* workspace, size_t workspace_bytes, pa_dtype dtype,
                           void* stream) {
    if (batch > 0 && (!k_new || !v_new || !slot_mapping || !al(k_new, 16) || !al(v_new, 16) || !al(slot_mapping, 8)))
        return PA_ERR_INVALID;
    const bool fuse = (dtype == PA_F16 || dtype == PA_BF16) && g_decode_kernel.load() != PA_DECODE_SIMT &&
                      num_blocks > 0 && num_kv_heads > 0 && block_size > 0 &&
                      static_cast<uint64_t>(num_blocks) * num_kv_heads * block_size < (1ull << 31);
    if (!fuse) {
        // the CUDA-core kernel writes nothing itself: the append kernel, then the decode
        if (batch > 0) {
            const pa_status st = pa_kv_append(k_new, v_new, k_pool, v_pool, slot_mapping, batch, num_blocks,
                                              num_kv_heads, head_dim, block_size, dtype, stream);
            if (st != PA_OK) return st;
        }
        return pa_decode(out, q, k_pool, v_pool, num_blocks, block_tables, max_blocks, seq_lens, batch, num_q_heads,
                         num_kv_heads, head_dim, block_size, scale, partition_tokens, workspace, workspace_bytes,
                         dtype, stream);
    }
    return decode_impl(out, q, k_pool, v_pool, num_blocks, block_tables, max_blocks, seq_lens, batch, num_q_heads,
                       num_kv_heads, head_dim, block_size, scale, partition_tokens, workspace, workspace_bytes, dtype,
                       stream, k_new, v_new, slot_mapping);
}

pa_status pa_kv_append_fp8(const void* k, const void* v, pa_dtype in_dtype, void* k_pool, void* v_pool,
                           const float* k_scale, const float* v_scale, const int64_t* slot_mapping,
                           int64_t num_tokens, int64_t num_blocks, int num_kv_heads, int head_dim, int block_size,
                           void* stream) {
    if (elt_size(in_dtype) == 0 || num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        block_size <= 0)
        return PA_ERR_INVALID;
    if (!k_pool || !v_pool || !al(k_pool, 16) || !al(v_pool, 16)) return PA_ERR_INVALID;
    if (head_dim % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !k_scale || !v_scale || !slot_mapping || !al(k, 16) || !al(v, 16) || !al(slot_mapping, 8) ||
        !al(k_scale, 4) || !al(v_scale, 4))
        return PA_ERR_INVALID;
    int* err = error_word();
    if (!err) return PA_ERR_CUDA;
    return from_cuda(pa::launch_kv_append_fp8(k, v, in_dtype, k_pool, v_pool, k_scale, v_scale, slot_mapping,
                                              num_tokens, num_blocks, num_kv_heads, head_dim, block_size, err,
                                              static_cast<cudaStream_t>(stream)));
}

pa_status pa_decode_fp8(void* out, const void* q, pa_dtype q_dtype, const void* k_pool, const void* v_pool,
                        const float* k_scale, const float* v_scale, int64_t num_blocks, const int32_t* block_tables,
                        int max_blocks, const int32_t* seq_lens, int batch, int num_q_heads, int num_kv_heads,
                        int head_dim, int block_size, float scale, int partition_tokens, void* workspace,
                        size_t workspace_bytes, void* stream) {
    if ((q_dtype != PA_F16 && q_dtype != PA_BF16) || batch < 0 || batch > 65535 || num_q_heads <= 0 ||
        num_kv_heads <= 0 || num_kv_heads > 65535 || head_dim <= 0 || block_size <= 0 || max_blocks <= 0 ||
        num_blocks <= 0 || !std::isfinite(scale))
        return PA_ERR_INVALID;
    if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID;
    const int group = num_q_heads / num_kv_heads;
    if (group != 1 && group != 2 && group != 4 && group != 8) return PA_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return PA_ERR_UNSUPPORTED;
    if (block_size % 16 != 0 || block_size > 256) return PA_ERR_UNSUPPORTED;
    if (static_cast<uint64_t>(num_blocks) * num_kv_heads * block_size >= (1ull << 31)) return PA_ERR_UNSUPPORTED;
    const int part =
        partition_tokens == 0 ? auto_partition(batch, num_q_heads, max_blocks, block_size, true) : partition_tokens;
    if (part <= 0 || part > kMaxPartition || part % 16 != 0 || part % block_size != 0) return PA_ERR_INVALID;
    if (static_cast<int64_t>(max_blocks) * block_size > (1LL << 30)) return PA_ERR_INVALID;
    if (batch == 0) return PA_OK;
    if (!out || !q || !k_pool || !v_pool || !k_scale || !v_scale || !block_tables || !seq_lens) return PA_ERR_INVALID;
    if (!al(out, 16) || !al(q, 16) || !al(k_pool, 16) || !al(v_pool, 16) || !al(block_tables, 4) ||
        !al(seq_lens, 4) || !al(k_scale, 4) || !al(v_scale, 4))
        return PA_ERR_INVALID;
    const WsLayout ws = ws_layout(batch, num_q_heads, head_dim, max_blocks, block_size, part);
    if (ws.partitions > 1 && (!workspace || !al(workspace, 16) || workspace_bytes < ws.total))
        return PA_ERR_INVALID;
    int* err = error_word();
    if (!err) return PA_ERR_CUDA;
    pa::DecodeParams p{};
    p.out = out;
    p.q = q;
    p.k_pool = k_pool;
    p.v_pool = v_pool;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    char* wsb = static_cast<char*>(workspace);
    p.ws_ml = ws.partitions > 1 ? reinterpret_cast<float*>(wsb) : nullptr;
    p.ws_acc = ws.partitions > 1 ? reinterpret_cast<float*>(wsb + ws.acc_off) : nullptr;
    p.err = err;
    p.num_blocks = num_blocks;
    p.max_blocks = max_blocks;
    p.batch = batch;
    p.hq = num_q_heads;
    p.hkv = num_kv_heads;
    p.d = head_dim;
    p.block_size = block_size;
    p.partition_tokens = part;
    p.max_partitions = ws.partitions < 1 ? 1 : ws.partitions;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.kernel = PA_DECODE_MMA;
    p.heads_per_cta = g_decode_heads.load();  // 0: the launcher chooses
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return from_cuda(q_dtype == PA_F16 ? pa::launch_decode_fp8_f16(p, st) : pa::launch_decode_fp8_bf16(p, st));
}

pa_status pa_prefill(void* out, const void* q, const void* k_pool, const void* v_pool, int64_t num_blocks,
                     const int32_t* block_tables, int max_blocks, const int32_t* seq_lens, const int32_t* qstart,
                     int batch, int total_q, int max_query_len, int num_q_heads, int num_kv_heads, int head_dim,
                     int block_size, float scale, pa_dtype dtype, void* stream) {
    if (elt_size(dtype) == 0 || batch < 0 || batch > 65535 || total_q < 0 || max_query_len < 0 ||
        num_q_heads <= 0 || num_kv_heads <= 0 || num_kv_heads > 65535 || head_dim <= 0 || block_size <= 0 ||
        max_blocks <= 0 || num_blocks <= 0 || !std::isfinite(scale))
        return PA_ERR_INVALID;
    if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID;
    if (dtype == PA_F32) return PA_ERR_UNSUPPORTED;
    const int group = num_q_heads / num_kv_heads;
    if (group != 1 && group != 2 && group != 4 && group != 8) return PA_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return PA_ERR_UNSUPPORTED;
    if (block_size % 16 != 0 || block_size > 256) return PA_ERR_UNSUPPORTED;
    if (static_cast<uint64_t>(num_blocks) * num_kv_heads * block_size >= (1ull << 31)) return PA_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(max_blocks) * block_size > (1LL << 30)) return PA_ERR_INVALID;
    if (static_cast<int64_t>(total_q) * num_q_heads * head_dim >= (1LL << 40)) return PA_ERR_INVALID;
    if (batch == 0 || total_q == 0 || max_query_len == 0) return PA_OK;
    if (!out || !q || !k_pool || !v_pool || !block_tables || !seq_lens || !qstart) return PA_ERR_INVALID;
    if (!al(out, 16) || !al(q, 16) || !al(k_pool, 16) || !al(v_pool, 16) || !al(block_tables, 4) ||
        !al(seq_lens, 4) || !al(qstart, 4))
        return PA_ERR_INVALID;
    int* err = error_word();
    if (!err) return PA_ERR_CUDA;
    pa::PrefillParams p{};
    p.out = out;
    p.q = q;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.qstart = qstart;
    p.err = err;
    p.num_blocks = num_blocks;
    p.max_blocks = max_blocks;
    p.batch = batch;
    p.total_q = total_q;
    p.hq = num_q_heads;
    p.hkv = num_kv_heads;
    p.block_size = block_size;
    p.scale_log2 = scale * 1.4426950408889634f;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    return from_cuda(dtype == PA_F16 ? pa::launch_prefill_f16(p, k_pool, v_pool, head_dim, max_query_len, st)
                                     : pa::launch_prefill_bf16(p, k_pool, v_pool, head_dim, max_query_len, st));
}

pa_status pa_selftest_wait_timeout(int limit_us, void* stream) {
    if (limit_us <= 0 || limit_us > 100000) return PA_ERR_INVALID;
    int* err = error_word();
    if (!err) return PA_ERR_CUDA;
    return from_cuda(pa::launch_wait_timeout_selftest(static_cast<uint64_t>(limit_us) * 1000ull, err,
                                                      static_cast<cudaStream_t>(stream)));
}

pa_status pa_get_device_error(int* code, void* stream) {
    if (!code) return PA_ERR_INVALID;
    *code = 0;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return PA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_pa_error_word, sizeof(int)) != cudaSuccess) return PA_ERR_CUDA;
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_pa_error_word, &zero, sizeof(int)) != cudaSuccess) return PA_ERR_CUDA;
    *code = v;
    if (v & ~PA_DEVERR_TIMEOUT) return PA_ERR_DEVICE_CHECK;
    if (v & PA_DEVERR_TIMEOUT) return PA_ERR_TIMEOUT;
    return PA_OK;
}

const char* pa_status_string(pa_status s) {
    switch (s) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID: return "PA_ERR_INVALID";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        case PA_ERR_DEVICE_CHECK: return "PA_ERR_DEVICE_CHECK";
        case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT";
        case PA_ERR_POOL_EXHAUSTED: return "PA_ERR_POOL_EXHAUSTED";
        case PA_ERR_OVER_RELEASE: return "PA_ERR_OVER_RELEASE";
        case PA_ERR_EXISTS: return "PA_ERR_EXISTS";
        case PA_ERR_NOT_FOUND: return "PA_ERR_NOT_FOUND";
        default: return "PA_ERR_UNKNOWN";
    }
}

}  // extern "C"
