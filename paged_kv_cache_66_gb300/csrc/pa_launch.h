// Internal launcher interface between the C ABI (pa_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "../../include/pagedkv.h"

namespace pa {

constexpr int kMaxLayersPerLaunch = 64;
constexpr int kMaxPartitionTokens = 8192;  // largest decode partition (a multiple of 16 and of b)

struct PoolPtrs {
    void* k[kMaxLayersPerLaunch];
    void* v[kMaxLayersPerLaunch];
};

// Everything one pa_decode call needs on the device.
struct DecodeParams {
    void* out;                  // [B, Hq, D] dtype
    const void* q;              // [B, Hq, D] dtype
    const void* k_pool;         // [N, Hkv, b, D] dtype
    const void* v_pool;
    const int32_t* block_tables;  // [B, max_blocks]
    const int32_t* seq_lens;      // [B]
    float* ws_ml;               // [B, Hq, P, 2] running max (log2 units) and normaliser
    float* ws_acc;              // [B, Hq, P, D] unnormalised partial outputs
    int* err;
    int64_t num_blocks;
    int max_blocks;
    int batch;
    int hq, hkv, d, block_size;
    int partition_tokens;
    int max_partitions;         // P = ceil(max_blocks * b / partition_tokens)
    float scale_log2;           // scale * log2(e)
    int kernel;                 // pa_decode_kernel choice (PA_DECODE_AUTO / _SIMT / _MMA)
    const float* k_scale;       // FP8 pools: [Hkv] scale of K codes (else null)
    const float* v_scale;       // FP8 pools: [Hkv] scale of V codes (else null)
    int heads_per_cta;          // tensor-core kernel: KV heads one CTA streams back to back (1 or 2;
                                // 0 on entry: the launcher chooses)
    // fused append (16-bit pools, tensor-core kernel): the row of position seq_lens[s] - 1 of
    // every sequence, written by the CTA that streams it (null: plain decode)
    const void* k_new;          // [B, Hkv, D] dtype
    const void* v_new;
    const int64_t* new_slots;   // [B] slot of position seq_lens[s] - 1 (negative: nothing to write)
};

// Everything one pa_prefill call needs on the device.
struct PrefillParams {
    void* out;                    // [total_q, Hq, D] dtype
    const void* q;                // [total_q, Hq, D] dtype
    const int32_t* block_tables;  // [B, max_blocks]
    const int32_t* seq_lens;      // [B] total length (history + chunk)
    const int32_t* qstart;        // [B + 1] first query row of each sequence
    int* err;
    int64_t num_blocks;
    int max_blocks;
    int batch;
    int total_q;
    int hq, hkv, block_size;
    float scale_log2;             // scale * log2(e)
};

// Launch `kernel` on `stream` allowing programmatic dependent launch (the
// kernel itself waits for its predecessor with griddepcontrol.wait).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// 2-D TMA descriptor of a pool viewed as [rows, D] elements of `elt_bytes`
// (2, or 1 for FP8), boxes of 16 rows x 128 bytes with the 128-byte swizzle.
// 2-D map over a pool viewed as `rows` rows of `d` elements: boxes of 128 bytes x box_rows rows,
// 128-byte swizzle
bool encode_pool_tmap(CUtensorMap* map, const void* pool, uint64_t rows, int d, int elt_bytes, int box_rows = 16);
// 3-D map over a 16-bit pool viewed as `rows` rows of `d` elements, in which one box is box_rows
// rows of every 64-element (128-byte) slice of the row: it lands as d / 64 runs of box_rows
// 128-byte rows, one run per slice, with the 128-byte swizzle.  d a multiple of 64.
bool encode_pool_tmap_slices(CUtensorMap* map, const void* pool, uint64_t rows, int d, int box_rows);
// Tensor map over a packed 16-bit query tensor [total_q, hq, d] whose box is one 128-row query tile
// of the prefill kernels: 64 dims x g heads x 128 / g tokens (rows token-major, the g heads of a token
// side by side), 128-byte swizzle, zeros past total_q.  q 16-byte aligned.
bool encode_q_tmap(CUtensorMap* map, const void* q, int total_q, int hq, int d, int g);
// Streaming multiprocessors of the current device (cached per device).
int sm_count();

cudaError_t launch_kv_append(const void* k, const void* v, void* k_pool, void* v_pool, const int64_t* slots,
                             int64_t num_tokens, int64_t num_blocks, int hkv, int row_bytes, int block_size,
                             int* err, cudaStream_t stream);

cudaError_t launch_wait_timeout_selftest(uint64_t limit_ns, int* err, cudaStream_t stream);

cudaError_t launch_copy_blocks(const PoolPtrs& pools, int num_layers, const int64_t* pairs, int64_t num_pairs,
                               int64_t num_blocks, size_t block_bytes, int* err, cudaStream_t stream);

// Returns cudaErrorNotSupported when (dtype, D, G) has no compiled kernel.
cudaError_t launch_decode_f32(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_decode_f16(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_decode_bf16(const DecodeParams& p, cudaStream_t stream);
// FP8 (E4M3) pools; q / out in f16 or bf16.
cudaError_t launch_decode_fp8_f16(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_decode_fp8_bf16(const DecodeParams& p, cudaStream_t stream);

// Paged prefill (fp16 / bf16 pools, D in {64, 128, 256}, G in {1, 2, 4, 8}).
cudaError_t launch_prefill_f16(const PrefillParams& p, const void* k_pool, const void* v_pool, int d, int max_q,
                               cudaStream_t stream);
cudaError_t launch_prefill_bf16(const PrefillParams& p, const void* k_pool, const void* v_pool, int d, int max_q,
                                cudaStream_t stream);
cudaError_t launch_kv_append_fp8(const void* k, const void* v, pa_dtype in_dtype, void* k_pool, void* v_pool,
                                 const float* k_scale, const float* v_scale, const int64_t* slots,
                                 int64_t num_tokens, int64_t num_blocks, int hkv, int d, int block_size, int* err,
                                 cudaStream_t stream);

}  // namespace pa
