/*
 * pagedkv_host.h -- C ABI of the host-side block manager (in libpagedkv.so).
 *
 * Host bookkeeping that builds the integer arrays the device calls take
 * (block tables, sequence lengths, slot mappings, copy-on-write pairs).  It
 * touches no GPU memory and launches nothing.  Semantics follow
 * "25. Paged attention and prefix caching", sections "The allocator",
 * "The paged cache", "Sharing blocks: forks and copy-on-write" and
 * "Prefix caching", with these readings:
 *   - the free list is first-in first-out: allocation takes the head, a block
 *     whose refcount drops to 0 goes to the tail; the initial order is the
 *     caller's permutation (or 0..N-1);
 *   - releasing a block whose refcount is already 0 fails with
 *     PA_ERR_OVER_RELEASE and changes nothing;
 *   - pa_host_reserve is all-or-nothing: if the pool lacks the blocks it needs
 *     it returns PA_ERR_POOL_EXHAUSTED before changing any state;
 *   - blocks are not zeroed when allocated.
 *
 * A handle is not thread-safe; use one per thread or lock around it.
 * Sequence ids are arbitrary int64 values chosen by the caller.
 * Every output array is caller-owned host memory.
 */
#ifndef PAGEDKV_HOST_H
#define PAGEDKV_HOST_H

#include <stdint.h>

#include "pagedkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_host pa_host;

/* New manager over `num_blocks` blocks of `block_size` tokens.  `initial_order`
 * (may be NULL) is a permutation of 0..num_blocks-1 giving the initial free
 * list.  Returns NULL on bad arguments (non-permutation, sizes <= 0). */
pa_host* pa_host_create(int64_t num_blocks, int block_size, const int32_t* initial_order);
void pa_host_destroy(pa_host* h);

/* New empty sequence; PA_ERR_EXISTS if the id is taken. */
pa_status pa_host_seq_create(pa_host* h, int64_t seq);

/* Make blocks exist for positions [len, len + new_tokens) of `seq`.  Any
 * table entry in that range whose block is shared (refcount > 1) is replaced
 * by a fresh block; each such copy is reported as a (src, dst) pair in
 * pairs_out[2*i], pairs_out[2*i+1] (capacity `pairs_cap` pairs; at most
 * ceil(new_tokens / b) + 1 pairs occur).  The length is not changed. */
pa_status pa_host_reserve(pa_host* h, int64_t seq, int64_t new_tokens, int64_t* pairs_out,
                          int64_t pairs_cap, int64_t* num_pairs);

/* slots_out[i] = table[p / b] * b + p % b for p = start + i, i < n.  Every
 * position must have a block (PA_ERR_INVALID otherwise). */
pa_status pa_host_slots(pa_host* h, int64_t seq, int64_t start, int64_t n, int64_t* slots_out);

/* Commit n written tokens: len += n (blocks must already exist). */
pa_status pa_host_advance(pa_host* h, int64_t seq, int64_t n);

/* `child` starts as an alias of `parent`: same table, same length, every
 * block's refcount + 1. */
pa_status pa_host_fork(pa_host* h, int64_t parent, int64_t child);

/* Release every block of `seq` and forget it. */
pa_status pa_host_free(pa_host* h, int64_t seq);

/* Roll back to `length` tokens, releasing blocks past ceil(length / b). */
pa_status pa_host_truncate(pa_host* h, int64_t seq, int64_t length);

pa_status pa_host_length(const pa_host* h, int64_t seq, int64_t* length);

/* Copy the block table of `seq` into out (capacity cap); *n = its length. */
pa_status pa_host_table(const pa_host* h, int64_t seq, int32_t* out, int64_t cap, int64_t* n);

int64_t pa_host_num_free(const pa_host* h);
int64_t pa_host_num_blocks(const pa_host* h);
/* Refcount of a block, or -1 when out of range. */
int32_t pa_host_refcount(const pa_host* h, int64_t block);

/* Rows of the batch's block tables, padded with 0, into tables_out
 * [B, stride] (stride >= the longest table) and lengths into lens_out [B];
 * *width = the longest table. */
pa_status pa_host_batch(const pa_host* h, const int64_t* seqs, int64_t batch, int32_t* tables_out,
                        int64_t stride, int32_t* lens_out, int64_t* width);

/* One decode step for a batch, in batch order: reserve one position per
 * sequence (collecting copy-on-write pairs), slot of position len, len += 1,
 * then the padded tables and new lengths as in pa_host_batch.  On
 * PA_ERR_POOL_EXHAUSTED no length has been advanced; reservations made for
 * earlier sequences stay (reserving again is a no-op). */
pa_status pa_host_decode_step(pa_host* h, const int64_t* seqs, int64_t batch,
                              int64_t* slots_out, int64_t* pairs_out, int64_t pairs_cap,
                              int64_t* num_pairs, int32_t* tables_out, int64_t stride,
                              int32_t* lens_out, int64_t* width);

/* Prefix table ("Prefix caching"): keys are whole token prefixes ending at a
 * block boundary; the table holds its own reference on each cached block.
 * attach: create `seq` with the longest cached prefix of `prompt`, always
 * leaving at least one prompt token to prefill; *reused = tokens reused.
 * remember: publish the full blocks of `seq` (tokens = its token ids).
 * evict: drop least-recently-used entries held by nobody else until
 * `blocks_wanted` blocks are free (or none is left to drop). */
pa_status pa_host_prefix_attach(pa_host* h, int64_t seq, const int64_t* prompt, int64_t n,
                                int64_t* reused);
pa_status pa_host_prefix_remember(pa_host* h, int64_t seq, const int64_t* tokens, int64_t n);
pa_status pa_host_prefix_evict(pa_host* h, int64_t blocks_wanted);
int64_t pa_host_prefix_entries(const pa_host* h);

/* Hash-chain prefix table ("Prefix caching": production engines hash the
 * chain of block contents instead of keeping token tuples, and the key also
 * covers whatever changes the activations: model revision, adapter,
 * multimodal inputs).  Readings, since the pages fix no hash or layout:
 *   root  = SHA-256("pagedkv.prefix.v1" || u64le(salt_len) || salt)
 *   key_i = SHA-256(key_{i-1} || u32le(block_size) || i64le(token) for the
 *           block_size tokens of full block i),  key_{-1} = root
 * (SHA-256 of FIPS PUB 180-4).  `salt` is caller-owned bytes that identify
 * everything besides the tokens that a block's K/V depend on; the same salt
 * must be given to attach and remember.  attach / remember / evict follow the
 * rules of the tuple-keyed table above; this table has its own entries and
 * its own least-recently-used order, and the two tables never see each
 * other's entries.  NULL handles or negative sizes give PA_ERR_INVALID. */

/* Keys of the n / block_size full blocks of `tokens`: 32 bytes each, written
 * to keys_out (caller-owned, (n / block_size) * 32 bytes). */
pa_status pa_prefix_chain_keys(const int64_t* tokens, int64_t n, int block_size, const void* salt, int64_t salt_len,
                               uint8_t* keys_out);
pa_status pa_host_hprefix_attach(pa_host* h, int64_t seq, const int64_t* prompt, int64_t n, const void* salt,
                                 int64_t salt_len, int64_t* reused);
/* PA_ERR_INVALID when `seq` holds fewer than n / block_size blocks. */
pa_status pa_host_hprefix_remember(pa_host* h, int64_t seq, const int64_t* tokens, int64_t n, const void* salt,
                                   int64_t salt_len);
pa_status pa_host_hprefix_evict(pa_host* h, int64_t blocks_wanted);
int64_t pa_host_hprefix_entries(const pa_host* h);
/* Cached block ids, least recently used first; writes at most `capacity`
 * and returns the number of entries (-1 on invalid arguments). */
int64_t pa_host_hprefix_blocks(const pa_host* h, int32_t* blocks_out, int64_t capacity);

/* Block prefix tree: the radix-tree form of the prefix table ("Prefix caching",
 * closing paragraph: a radix tree over all cached prefixes; "Модуль 09",
 * RadixAttention: the shared prefixes of all past requests form a tree kept
 * by least-recently-used eviction).  One node per cached full block, reached
 * from its parent by an edge labelled with the block's token ids.
 * attach / remember follow the rules of the tuple-keyed table above (with no
 * eviction the two make the same decisions): attach walks the prompt's full
 * blocks from the root, leaving at least one token to prefill, shares each
 * matched block and marks the matched nodes most recently used in walk
 * order; remember descends through cached blocks (recency unchanged) and
 * hangs the sequence's remaining full blocks below them, taking the tree's
 * own reference.  evict drops only leaves -- nodes no cached block extends --
 * least recently used first and only while the tree alone holds the block,
 * until `blocks_wanted` blocks are free; a parent whose last child went
 * becomes a leaf in turn.  The tree is independent of the other two tables.
 * NULL handles or negative sizes give PA_ERR_INVALID; remember gives
 * PA_ERR_INVALID when `seq` holds fewer than n / block_size blocks. */
pa_status pa_host_tprefix_attach(pa_host* h, int64_t seq, const int64_t* prompt, int64_t n, int64_t* reused);
pa_status pa_host_tprefix_remember(pa_host* h, int64_t seq, const int64_t* tokens, int64_t n);
pa_status pa_host_tprefix_evict(pa_host* h, int64_t blocks_wanted);
/* Number of cached nodes (-1 for a NULL handle). */
int64_t pa_host_tprefix_nodes(const pa_host* h);
/* Cached block ids in ascending order; writes at most `capacity` and returns
 * the number of cached blocks (-1 on invalid arguments). */
int64_t pa_host_tprefix_blocks(const pa_host* h, int32_t* blocks_out, int64_t capacity);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_HOST_H */
