/*
 * pagedkv.h -- C ABI of the paged KV-cache device library (libpagedkv.so).
 *
 * The KV cache of every sequence lives in fixed-size blocks of b tokens taken
 * from one pool per layer, laid out [num_blocks, kv_heads, b, head_dim]
 * ("25. Paged attention and prefix caching", section "Paging").  A
 * per-sequence block table maps logical block j (tokens [j*b, (j+1)*b)) to a
 * physical block of the pool.  Three device operations act on the pools:
 *
 *   pa_kv_append    write each step's new K/V rows into their slots
 *                   (same page, section "The paged cache": update's scatter)
 *   pa_copy_blocks  copy-on-write duplication of shared blocks in every layer
 *                   (same page, "The paged cache": reserve; "Sharing blocks")
 *   pa_decode       one query per sequence attends over its paged history
 *                   (same page, "Attention that reads through the table";
 *                   "Chapter 7 Paged KV Cache and Memory Management", 4.1-4.2,
 *                   for the blockwise online softmax and the split merge)
 *
 * Conventions shared by every call:
 *   - All tensors are dense, row-major, owned by the caller and resident on
 *     the current CUDA device unless stated otherwise.  The library allocates
 *     no memory, keeps no state except one device error word, and never
 *     synchronises the stream (pa_get_device_error excepted).
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).
 *   - Arguments are validated on the host before any launch: null pointers,
 *     non-positive sizes, pointers not 16-byte aligned, and inconsistent
 *     shapes return PA_ERR_INVALID; shapes that are valid but not compiled
 *     (head_dim, block size, dtype or query group) return PA_ERR_UNSUPPORTED.
 *     Nothing is launched in either case.  A failed launch returns PA_ERR_CUDA.
 *   - Data-dependent errors (a block-table entry or slot outside the pool, a
 *     sequence length above the table's capacity, a copy pair outside the
 *     pool) are caught on the device: the offending access is skipped and a
 *     bit is OR-ed into the device error word, which pa_get_device_error reads.
 *     No kernel traps or reads out of bounds on bad data.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
    PA_OK = 0,
    PA_ERR_INVALID = 1,        /* bad argument; nothing launched                   */
    PA_ERR_UNSUPPORTED = 2,    /* valid shape that is not compiled; nothing launched */
    PA_ERR_CUDA = 3,           /* a CUDA runtime call or kernel launch failed       */
    PA_ERR_DEVICE_CHECK = 4,   /* a device-side check flagged bad data              */
    PA_ERR_TIMEOUT = 5,        /* a bounded device wait gave up                     */
    PA_ERR_POOL_EXHAUSTED = 6, /* host block manager: no free block (MemoryError)   */
    PA_ERR_OVER_RELEASE = 7,   /* host block manager: refcount already 0            */
    PA_ERR_EXISTS = 8,         /* host block manager: sequence id already exists    */
    PA_ERR_NOT_FOUND = 9       /* host block manager: unknown sequence id           */
} pa_status;

typedef enum pa_dtype {
    PA_F32 = 0,
    PA_F16 = 1,
    PA_BF16 = 2
} pa_dtype;

/* Bits of the device error word (see pa_get_device_error). */
#define PA_DEVERR_SLOT 1         /* pa_kv_append: slot >= num_blocks * b;
                                    pa_decode_append: slot not position L - 1's */
#define PA_DEVERR_TABLE 2        /* pa_decode: table entry outside [0, num_blocks) */
#define PA_DEVERR_SEQLEN 4       /* pa_decode: seq_len < 0 or > max_blocks * b  */
#define PA_DEVERR_PAIR 8         /* pa_copy_blocks: src or dst outside the pool */
#define PA_DEVERR_TIMEOUT 16     /* a bounded mbarrier wait gave up            */

/*
 * pa_kv_append -- "reshape_and_cache": scatter new K/V rows into the pools.
 *
 *   k, v          [T, Hkv, D] in `dtype`; row t holds token t's key/value.
 *   k_pool,v_pool [num_blocks, Hkv, b, D] in `dtype`.
 *   slot_mapping  [T] int64 on the device; slot = physical_block * b + offset,
 *                 i.e. logical position p of a sequence maps to
 *                 table[p / b] * b + p % b.  A negative slot skips the row
 *                 (padding).  Slots of one call must be distinct (otherwise
 *                 which row lands is unspecified).
 *   Effect: k_pool[slot / b, h, slot % b, :] = k[t, h, :] (same for v), bit
 *   exact.  A slot >= num_blocks * b is skipped and flags PA_DEVERR_SLOT.
 *   Supported: any D with D * sizeof(dtype) a multiple of 16, any b >= 1,
 *   any dtype.  T may be 0 (no launch).
 */
pa_status pa_kv_append(const void* k, const void* v, void* k_pool, void* v_pool,
                       const int64_t* slot_mapping, int64_t num_tokens, int64_t num_blocks,
                       int num_kv_heads, int head_dim, int block_size, pa_dtype dtype,
                       void* stream);

/*
 * pa_copy_blocks -- copy-on-write: for every pair (src, dst) and every layer,
 * K_pool[layer][dst] = K_pool[layer][src] and V_pool[layer][dst] = V_pool[layer][src].
 *
 *   k_pools, v_pools  HOST arrays of `num_layers` device pointers, one pool per layer.
 *   pairs             DEVICE int64 [num_pairs, 2] of (src, dst) physical blocks.
 *                     Destinations must be distinct and disjoint from sources.
 *   block_bytes       Hkv * b * D * sizeof(dtype): the bytes of one block of one
 *                     pool; a multiple of 16.
 *   A pair outside [0, num_blocks) is skipped and flags PA_DEVERR_PAIR.
 *   num_pairs may be 0 (no launch).
 */
pa_status pa_copy_blocks(void* const* k_pools, void* const* v_pools, int num_layers,
                         const int64_t* pairs, int64_t num_pairs, int64_t num_blocks,
                         size_t block_bytes, void* stream);

/*
 * pa_decode_workspace_size -- bytes of fp32 scratch pa_decode needs for a
 * batch of B sequences with Hq query heads whose block tables have
 * `max_blocks` columns: per (sequence, query head, partition) one running
 * max, one normaliser and D partial output values.  Returns 0 when every
 * sequence fits one partition (max_blocks * b <= partition tokens).
 * partition_tokens = 0 selects the automatic size, the same one pa_decode
 * then uses (see pa_decode).  The contents need no initialisation.
 */
size_t pa_decode_workspace_size(int batch, int num_q_heads, int head_dim, int max_blocks,
                                int block_size, int partition_tokens);

/*
 * pa_decode -- paged decode attention, one query token per sequence.
 *
 *   out           [B, Hq, D] in `dtype` (written).
 *   q             [B, Hq, D] in `dtype`.
 *   k_pool,v_pool [num_blocks, Hkv, b, D] in `dtype`.
 *   block_tables  [B, max_blocks] int32; row s lists the physical blocks of
 *                 sequence s in logical order; entries past ceil(L_s / b) are
 *                 never used (the whole row must be readable: a partition's
 *                 entries may be loaded before L_s is known; pad with anything).
 *   seq_lens      [B] int32; L_s >= 1 tokens of history (the token appended
 *                 this step included).  L_s = 0 writes a zero row.
 *   scale         multiplies q . k (the pages use 1 / sqrt(D)).
 *   Query head h reads KV head h / (Hq / Hkv) (contiguous GQA groups).
 *   Computes out[s, h] = sum_t softmax_t(scale * q[s,h] . K[t]) V[t] over
 *   t < L_s with fp32 accumulation, rounded once to `dtype`.
 *   Sequences longer than `partition_tokens` (a multiple of 16 and of b) are
 *   split into partitions whose (max, normaliser, partial output) go to
 *   `workspace` and are merged by a second kernel.  partition_tokens = 0
 *   picks the size: 512 tokens (rounded down to a multiple of b), halved down
 *   to 128 while B * ceil(Hq / 8) * ceil(max_blocks * b / size) stays below
 *   608 (about four units per SM), so that short histories still spread over
 *   the GPU.  It depends only on B, Hq, max_blocks and b, as the workspace
 *   size does.
 *   workspace     device scratch of at least pa_decode_workspace_size(...)
 *                 bytes, 16-byte aligned; may be NULL when that size is 0.
 *   Supported: D in {64, 128, 256}; Hq / Hkv in {1, 2, 4, 8}; b a multiple of
 *   16 up to 256; any dtype.
 */
pa_status pa_decode(void* out, const void* q, const void* k_pool, const void* v_pool,
                    int64_t num_blocks, const int32_t* block_tables, int max_blocks,
                    const int32_t* seq_lens, int batch, int num_q_heads, int num_kv_heads,
                    int head_dim, int block_size, float scale, int partition_tokens,
                    void* workspace, size_t workspace_bytes, pa_dtype dtype, void* stream);

/*
 * pa_decode_append -- pa_kv_append of each sequence's newest row followed by
 * pa_decode, for the decode step where every sequence appends exactly one
 * token ("25. Paged attention and prefix caching", "The paged cache": update
 * writes the step's K/V, then attention reads the history including it).
 *   k_new, v_new   [batch, Hkv, D] `dtype`, device: the rows of position
 *                  seq_lens[s] - 1 (the newest) of sequence s.
 *   slot_mapping   int64 [batch], device: the slot of that position, i.e.
 *                  table[s][(L-1) / b] * b + (L-1) % b; negative: no row
 *                  (give a negative slot for a sequence with L_s = 0).
 *   Other arguments and the workspace as for pa_decode.
 * The pools end bit for bit as after pa_kv_append, and the outputs equal
 * pa_decode's.  fp16 / bf16 pools with the tensor-core kernel do both in one
 * launch: the CTA whose partition holds position L - 1 writes the rows of its
 * KV heads before it streams that position.  A slot that is not the table's
 * slot of position L - 1 is skipped and flags PA_DEVERR_SLOT (its row is then
 * not written).  fp32 pools, the CUDA-core kernel forced by
 * pa_set_decode_kernel, or pools of 2^31 rows or more run pa_kv_append and
 * then pa_decode (the slot is then not checked against the table).
 */
pa_status pa_decode_append(void* out, const void* q, const void* k_new, const void* v_new,
                           const int64_t* slot_mapping, void* k_pool, void* v_pool, int64_t num_blocks,
                           const int32_t* block_tables, int max_blocks, const int32_t* seq_lens, int batch,
                           int num_q_heads, int num_kv_heads, int head_dim, int block_size, float scale,
                           int partition_tokens, void* workspace, size_t workspace_bytes, pa_dtype dtype,
                           void* stream);

/*
 * pa_decode_noalloc -- pa_decode for callers that cannot allocate device
 * memory: the same arguments minus the workspace, which comes instead from a
 * fixed array of PA_DECODE_NOALLOC_MAX_BYTES inside this library.  The pages
 * have no counterpart; it exists because some callers (an application that
 * owns all device memory through its own allocator, a loop that must not
 * allocate after start-up, an ABI consumer without an allocator) cannot
 * provide scratch.
 *   - Returns PA_ERR_INVALID, launching nothing, when the call needs more
 *     scratch than the array holds (pa_decode_workspace_size(...) >
 *     PA_DECODE_NOALLOC_MAX_BYTES); use pa_decode with caller scratch then.
 *   - Allocates nothing (no cudaMalloc / cudaFree, no allocating library call).
 *   - The first call on a device, with that device current, looks up the
 *     array's device address (cudaGetSymbolAddress) and caches it; make that
 *     first call before any stream capture.
 *   - Under CUDA's default lazy module loading, that first lookup is also
 *     what loads the array onto the device: the driver reserves its
 *     PA_DECODE_NOALLOC_MAX_BYTES then (with CUDA_MODULE_LOADING=EAGER, when
 *     the context is created).  So make the first call on each device before
 *     the application hands all device memory to its own allocator; a first
 *     call that finds no room returns PA_ERR_CUDA.  Later calls take no
 *     device memory at all.
 *   - Every call on a device shares the one array and leaves its contents
 *     behind.  Calls whose kernels overlap on the GPU (different streams
 *     without ordering between them) race on it and give wrong results;
 *     serialise them.  No clearing is needed between ordered calls.
 *   - Once loaded, the array stays reserved on that GPU until the process
 *     exits.
 */
#define PA_DECODE_NOALLOC_MAX_BYTES (16u << 20)
pa_status pa_decode_noalloc(void* out, const void* q, const void* k_pool, const void* v_pool,
                            int64_t num_blocks, const int32_t* block_tables, int max_blocks,
                            const int32_t* seq_lens, int batch, int num_q_heads,
                            int num_kv_heads, int head_dim, int block_size, float scale,
                            int partition_tokens, pa_dtype dtype, void* stream);

/*
 * FP8 (E4M3) KV cache -- the pools hold one byte per element, halving the
 * bytes every decode reads ("25. Paged attention and prefix caching",
 * "Attention that reads through the table": FP8 KV caches; "Модуль 09",
 * "6. Квантование KV-кэша по блокам": E4M3 halves KV memory, the scale kept
 * per head).  Layout of the pools as above, [num_blocks, Hkv, b, D] bytes;
 * k_scale, v_scale are DEVICE fp32 arrays [Hkv] (one scale per KV head of
 * the layer).  A stored code c of head h stands for e4m3(c) * scale[h].
 *
 * pa_kv_append_fp8 -- like pa_kv_append, quantising on the way: rows k, v
 *   [T, Hkv, D] in `in_dtype` (f32, f16 or bf16) are stored as
 *   e4m3(x / scale[h]), the quotient an IEEE fp32 division, rounded to the
 *   nearest code (ties to even) and saturated to +-448.  D a multiple of 16.
 *
 * pa_decode_fp8 -- like pa_decode over FP8 pools: q and out [B, Hq, D] in
 *   `q_dtype` (f16 or bf16); the attention is taken over the dequantised
 *   history, with q used in f16 (exact for bf16 values in f16's normal range)
 *   and fp32 accumulation.  Tensor-core kernel only: D in {64, 128, 256}, Hq/Hkv in
 *   {1, 2, 4, 8}, b a multiple of 16, num_blocks * Hkv * b < 2^31 (else
 *   PA_ERR_UNSUPPORTED).  Workspace as for pa_decode.  partition_tokens = 0
 *   takes the automatic size for E4M3 pools: 2048 tokens (a token carries
 *   half the bytes), halved down to 128 while the launch would have fewer
 *   than ~2 units per SM; it is never smaller than pa_decode's automatic
 *   size, so pa_decode_workspace_size(..., 0) bytes always suffice.
 */
pa_status pa_kv_append_fp8(const void* k, const void* v, pa_dtype in_dtype, void* k_pool, void* v_pool,
                           const float* k_scale, const float* v_scale, const int64_t* slot_mapping,
                           int64_t num_tokens, int64_t num_blocks, int num_kv_heads, int head_dim,
                           int block_size, void* stream);

pa_status pa_decode_fp8(void* out, const void* q, pa_dtype q_dtype, const void* k_pool, const void* v_pool,
                        const float* k_scale, const float* v_scale, int64_t num_blocks,
                        const int32_t* block_tables, int max_blocks, const int32_t* seq_lens, int batch,
                        int num_q_heads, int num_kv_heads, int head_dim, int block_size, float scale,
                        int partition_tokens, void* workspace, size_t workspace_bytes, void* stream);

/*
 * pa_prefill -- paged prefill (chunked prefill) attention.  A chunk of new
 * query tokens of each sequence attends causally to that sequence's paged
 * history plus the chunk itself ("25. Paged attention and prefix caching",
 * stretch exercise 4; "Chapter 7 Paged KV Cache and Memory Management", 4.1
 * step 3: the key at position p is visible to the query at position i iff
 * p <= i, the score scaled, masked keys weighted 0).
 *
 *   q, out        [total_q, Hq, D] `dtype` (f16 or bf16), device.  The rows of
 *                 sequence s are qstart[s] .. qstart[s+1]-1 (its chunk, in
 *                 position order).
 *   qstart        int32 [batch + 1], device: cumulative query rows
 *                 (qstart[0] = 0, qstart[batch] = total_q).
 *   seq_lens      int32 [batch], device: each sequence's TOTAL length, the
 *                 chunk included.  The chunk is the last C = qstart[s+1] -
 *                 qstart[s] positions: chunk row r sits at position
 *                 seq_lens[s] - C + r and sees positions 0 .. seq_lens[s] - C + r.
 *                 The chunk's K/V rows must already be in the pools
 *                 (pa_kv_append).
 *   k_pool, v_pool, block_tables, max_blocks, num_blocks, block_size: as for
 *                 pa_decode.
 *   max_query_len the largest C of the batch: it sizes the work, units of
 *                 256 (D <= 128) or 128 (D = 256) query rows of one KV head
 *                 (a row = a chunk token x a query head of the group); a
 *                 smaller value leaves the rows past it unwritten.  At
 *                 D <= 128 one persistent CTA per SM walks the units.
 *   scale         multiplies q . k (typically 1/sqrt(D)).
 *
 * Output rows are rounded once from fp32 to `dtype`.  Tensor-core kernel
 * only: D in {64, 128, 256}, Hq/Hkv in {1, 2, 4, 8}, b a multiple of 16 up to
 * 256, num_blocks * Hkv * b < 2^31; other shapes, and f32, give
 * PA_ERR_UNSUPPORTED.  No workspace.  On the device, a sequence whose
 * length, chunk or qstart entries are inconsistent (C < 0, C > length,
 * length above the table's capacity, rows outside [0, total_q]) is skipped
 * and flagged PA_DEVERR_SEQLEN; a table entry outside the pool is skipped
 * and flagged PA_DEVERR_TABLE.
 */
pa_status pa_prefill(void* out, const void* q, const void* k_pool, const void* v_pool, int64_t num_blocks,
                     const int32_t* block_tables, int max_blocks, const int32_t* seq_lens, const int32_t* qstart,
                     int batch, int total_q, int max_query_len, int num_q_heads, int num_kv_heads, int head_dim,
                     int block_size, float scale, pa_dtype dtype, void* stream);

/*
 * pa_set_decode_kernel -- process-wide choice of the pa_decode partition
 * kernel (both compute the same result within the attention tolerance):
 *   PA_DECODE_AUTO  (default) tensor cores for fp16/bf16 pools, CUDA cores for fp32;
 *   PA_DECODE_SIMT  CUDA cores (fp32 FMAs) for every dtype;
 *   PA_DECODE_MMA   tensor cores (mma m16n8k16, fp32 accumulate, TMA-fed) --
 *                   pa_decode then returns PA_ERR_UNSUPPORTED for fp32 pools
 *                   or pools of 2^31 rows (num_blocks * Hkv * b) or more.
 * Returns PA_ERR_INVALID for any other value.
 */
typedef enum pa_decode_kernel {
    PA_DECODE_AUTO = 0,
    PA_DECODE_SIMT = 1,
    PA_DECODE_MMA = 2
} pa_decode_kernel;

pa_status pa_set_decode_kernel(pa_decode_kernel kernel);

/*
 * pa_set_decode_heads_per_cta -- process-wide choice of how many KV heads one
 * CTA of the tensor-core decode kernel streams back to back (its block-table
 * slice staged once): 0 (default) takes two when that costs no resident CTA
 * per SM (by the occupancy calculator), else one; 1 or 2 force it.  Results
 * are identical either way.
 * Returns PA_ERR_INVALID for any other value.
 */
pa_status pa_set_decode_heads_per_cta(int heads);


/*
 * pa_selftest_wait_timeout -- exercise the failure path of the bounded
 * device waits: launch one warp whose odd lanes wait on an mbarrier that is
 * completed and whose even lanes wait on one that nothing completes, giving
 * up after `limit_us` microseconds (1..100000).  As in the decode and prefill
 * kernels, the warp then takes one decision for all lanes (a vote over the
 * lanes' own results) before a full-warp shuffle.  Afterwards
 * pa_get_device_error reports PA_DEVERR_TIMEOUT (status PA_ERR_TIMEOUT) --
 * set only when the vote failed and the shuffle saw every lane -- and the
 * context stays usable.  The kernels use the same wait with a 1-second limit.
 */
pa_status pa_selftest_wait_timeout(int limit_us, void* stream);

/*
 * pa_get_device_error -- synchronise `stream`, then read and clear the device
 * error word of the current device.  *code receives the OR of PA_DEVERR_* bits
 * raised since the last call (0 when none).  Returns PA_ERR_DEVICE_CHECK when
 * a data bit is set, PA_ERR_TIMEOUT when only the timeout bit is set, PA_OK
 * otherwise.
 */
pa_status pa_get_device_error(int* code, void* stream);

/* pa_status_string -- static, human-readable name of a status. */
const char* pa_status_string(pa_status status);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
