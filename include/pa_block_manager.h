/*
 * pa_block_manager.h -- host-side allocator of the paged KV pool, with prefix caching.
 *
 * It produces what the attention path consumes: per-sequence block tables, the slot mapping of
 * each step's new tokens, and copy-on-write block copies (run on the device by pa_copy_blocks).
 *   - "Local_LLM_03_vLLM_Architecture", paged-KV slide: the cache is a pool of fixed-size blocks
 *     reached through a per-sequence block table; prefix-caching slide: each block's token
 *     content is hashed, and requests whose first N tokens agree share those N / block_size
 *     physical blocks instead of recomputing their K/V.
 *   - "Scaling inference with vLLM": requests that start the same way (one system prompt)
 *     physically share those pages; memory and compute are paid once.
 *   - "vLLM: LLM Inference That Doesn't Waste Your GPU", "PagedAttention: virtual memory for KV":
 *     blocks make eviction cheap and prefixes shareable without copies; "Prefix caching": the
 *     sharing can leak across requests, hence the per-request cache salt below.
 *
 * Model (this library's reading; the pages fix no details):
 *   - A block is FULL when it holds block_size tokens.  Only full blocks enter the prefix cache.
 *     A full block's key is a 128-bit chained hash of (key of the previous block of the same
 *     sequence, the sequence's cache salt, the block's tokens), so two blocks match only when the
 *     whole prefix up to them matches; a match also compares the block's own tokens exactly.
 *   - Every physical block has a reference count (sequences using it).  A block whose count
 *     drops to 0 returns to the free list, unless it is cached: then it stays findable in the
 *     prefix cache and becomes EVICTABLE (least recently released first).  Allocation takes free
 *     blocks first, then evicts.
 *   - Adding a prompt reuses the longest run of cached leading full blocks, but never the block
 *     holding the prompt's last token (that token is always computed, to produce logits);
 *     num_cached_tokens reports how many leading tokens need no K/V computation.
 *   - Appending into a partial last block that another sequence also uses copies it first
 *     (copy-on-write): the caller must copy K/V of block src into block dst (pa_copy_blocks)
 *     before the step's reshape_and_cache.  A partial last block that is cached but used only by
 *     this sequence (after a truncation) leaves the cache and is written in place.
 *   - Every call either succeeds completely or changes nothing.
 *
 * Not thread-safe: one manager is driven by one scheduler thread (use one manager per pool).
 * Sequence ids are caller-chosen int64 values.  All pointers here are HOST pointers.
 */
#ifndef PA_BLOCK_MANAGER_H_
#define PA_BLOCK_MANAGER_H_

#include <stdint.h>

#include "pa.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_block_manager pa_block_manager;

/* A manager of physical blocks 0 .. num_blocks-1 of block_size tokens.  prefix_caching = 0
 * turns sharing off (every block private, nothing cached).  Returns NULL for bad sizes
 * (num_blocks < 1, block_size < 1) or when out of host memory. */
pa_block_manager* pa_bm_create(int32_t num_blocks, int32_t block_size, int32_t prefix_caching);
void pa_bm_destroy(pa_block_manager* bm);

/* Register sequence seq_id with its n prompt tokens (n >= 1).  cache_salt separates requests
 * that must not share blocks (different tenants): blocks match only under the same salt.
 * *num_cached_tokens (may be NULL) receives the count of leading tokens whose K/V already sit
 * in reused blocks (a multiple of block_size, < n).  Errors: PA_ERR_INVALID_ARG (unknown
 * arguments, seq_id already present), PA_ERR_NO_BLOCKS (pool exhausted; nothing changed). */
int pa_bm_add_sequence(pa_block_manager* bm, int64_t seq_id, const int32_t* tokens, int32_t n,
                       int64_t cache_salt, int32_t* num_cached_tokens);

/* Append n >= 1 tokens to seq_id (a decode step: n = 1; accepted speculative tokens: n > 1).
 * Copy-on-write pairs go to copies[2*i] (src) and copies[2*i + 1] (dst), i < *num_copies; at
 * most one pair per call, so copies needs room for 2 entries (may be NULL when the caller knows
 * no sharing happens: a needed copy then fails with PA_ERR_INVALID_ARG and nothing changes). */
int pa_bm_append(pa_block_manager* bm, int64_t seq_id, const int32_t* tokens, int32_t n,
                 int32_t* copies, int32_t* num_copies);

/* Shorten seq_id to new_len tokens (1 <= new_len <= length): rejected speculative tokens.
 * Blocks past the new end are released. */
int pa_bm_truncate(pa_block_manager* bm, int64_t seq_id, int32_t new_len);

/* child becomes a copy of parent that shares all of parent's blocks (parallel sampling). */
int pa_bm_fork(pa_block_manager* bm, int64_t parent, int64_t child);

/* Release seq_id and all its block references. */
int pa_bm_free(pa_block_manager* bm, int64_t seq_id);

/* Counts: free blocks (not cached, unused), evictable blocks (cached, unused), cached blocks
 * (in the prefix cache, used or not), live sequences.  Any pointer may be NULL. */
int pa_bm_stats(const pa_block_manager* bm, int32_t* free_blocks, int32_t* evictable_blocks,
                int32_t* cached_blocks, int32_t* num_seqs);

/* Length (tokens) of seq_id and its block table: block_table[i], i < ceil(len / block_size),
 * written to out (room for max_blocks entries).  *num_blocks may be NULL. */
int pa_bm_sequence(const pa_block_manager* bm, int64_t seq_id, int32_t* length, int32_t* out,
                   int32_t max_blocks, int32_t* num_blocks);

/* The batch descriptor of one step over n sequences, the last query_lens[i] tokens of sequence
 * seq_ids[i] being that step's new tokens (0 <= query_lens[i] <= length):
 *   block_tables     int32 [n, max_blocks], entries past a sequence's blocks set to pad_block,
 *   seq_lens         int32 [n],
 *   query_start_loc  int32 [n + 1] (prefix sums of query_lens),
 *   slot_mapping     int64 [sum query_lens]: block * block_size + offset of each new token.
 * PA_ERR_INVALID_ARG when a sequence is unknown, a query length is out of range or a table
 * does not fit max_blocks. */
int pa_bm_step_descriptor(const pa_block_manager* bm, const int64_t* seq_ids,
                          const int32_t* query_lens, int32_t n, int32_t max_blocks,
                          int32_t pad_block, int32_t* block_tables, int32_t* seq_lens,
                          int32_t* query_start_loc, int64_t* slot_mapping);

/* pa_step_slot_mapping -- the same descriptor arithmetic for a scheduler that keeps its own
 * block tables (no manager): from host arrays of n sequences (seq_lens[i] keys after the step,
 * the last query_lens[i] of them new; block_tables int32 rows of max_blocks entries, bt_stride
 * apart) it writes
 *   query_start_loc  int32 [n + 1] (prefix sums of query_lens),
 *   slot_mapping     int64 [sum query_lens]: block_tables[i][p / block_size] * block_size +
 *                    p % block_size for p = seq_lens[i] - query_lens[i] .. seq_lens[i] - 1
 *                    ("Local_LLM_03_vLLM_Architecture", paged-KV slide: logical position p of a
 *                    sequence lives at offset p % block_size of its (p / block_size)-th block).
 * Block ids are copied, not checked (the device checks them against the pool).
 * PA_ERR_INVALID_ARG (nothing written) when a query length is outside 0 .. seq_len, a sequence
 * with new tokens needs more than max_blocks blocks, or slot_capacity is below the row count. */
int pa_step_slot_mapping(int32_t n, const int32_t* seq_lens, const int32_t* query_lens,
                         const int32_t* block_tables, int64_t bt_stride, int32_t max_blocks,
                         int32_t block_size, int32_t* query_start_loc, int64_t* slot_mapping,
                         int64_t slot_capacity);

#ifdef __cplusplus
}
#endif

#endif /* PA_BLOCK_MANAGER_H_ */
