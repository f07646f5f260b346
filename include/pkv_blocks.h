/*
 * pkv_blocks.h -- host-side KV block manager of libpkv.so (C ABI).
 *
 * The paged KV cache is a pool of num_blocks physical blocks of block_size
 * token slots.  Each sequence owns a block table: logical block i of the
 * sequence lives in physical block table[i], so token position p sits in
 * slot table[p / block_size] * block_size + p % block_size.  Blocks are
 * taken from the pool only when a sequence crosses a block boundary.
 * ("How to design an LLM serving system (a vLLM deep dive)", "PagedAttention
 * (vLLM KV manager)" and "Latency and scaling knobs"; nanoserve, "Prefix
 * caching" and the block_manager.py row of its file table.)
 *
 * Prefix caching: every full block is content-addressed by a chained hash of
 * its parent block's hash and its own token ids.  A new sequence whose prompt
 * starts with the same full blocks shares those physical blocks (reference
 * counts) instead of recomputing them.  Blocks whose count drops to zero go
 * back to the free queue in release order but keep their content and hash,
 * so a later prompt can still hit them; allocation takes the least recently
 * released block and forgets its hash (eviction).  A hash hit is confirmed by
 * comparing the block's token ids, so two different prefixes never share a
 * block even if their hashes collide.
 *
 * The manager is plain host memory and host code: it never touches the GPU.
 * Its outputs (slot mapping, block tables, lengths) are the inputs of
 * pkv_append and pkv_attention.  A manager is not thread-safe: one thread (or
 * one lock) per manager.
 *
 * Errors: PKV_ERR_INVALID_ARGUMENT for unknown or duplicate sequence ids and
 * bad sizes; PKV_ERR_OUT_OF_BLOCKS when the pool cannot hold the request, in
 * which case nothing is changed.  pkv_last_error() gives the detail.
 */
#ifndef PKV_BLOCKS_H
#define PKV_BLOCKS_H

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_block_manager pkv_block_manager; /* opaque */

typedef struct {
  int32_t num_blocks;      /* pool size */
  int32_t free_blocks;     /* reference count 0 (including cached ones) */
  int32_t cached_blocks;   /* full blocks whose hash is registered (in use or free) */
  int32_t num_sequences;   /* live sequences */
  int64_t prefix_hit_blocks; /* blocks shared through the prefix cache so far */
  int64_t evictions;       /* cached free blocks reallocated so far */
} pkv_bm_stats_t;

/* Creates a manager for a pool of num_blocks blocks of block_size slots.
 * num_blocks * block_size must fit in int32 (slot numbers are int32). */
PKV_API pkv_status pkv_bm_create(int32_t num_blocks, int32_t block_size, pkv_block_manager** out);

/* Frees the manager (NULL is ignored). */
PKV_API void pkv_bm_destroy(pkv_block_manager* bm);

/*
 * Registers sequence seq_id with its prompt (n token ids, not yet in the
 * cache) and matches its longest cached prefix of full blocks.  Matched
 * blocks are shared; *cached_tokens (a multiple of block_size, at most
 * n - 1 so that the last prompt token is always computed) tells the caller
 * how many prompt tokens are already in the cache: the sequence's length
 * starts there and the remaining prompt tokens are appended with
 * pkv_bm_append.  The prompt is kept to hash the blocks it fills later.
 */
PKV_API pkv_status pkv_bm_add_sequence(pkv_block_manager* bm, int64_t seq_id, const int32_t* prompt, int32_t n,
                                       int32_t* cached_tokens);

/*
 * Appends n tokens (their ids) to sequence seq_id, taking new blocks when a
 * block boundary is crossed, and writes each token's cache slot into
 * slots[n].  Blocks that become full are registered in the prefix cache.
 * All or nothing: PKV_ERR_OUT_OF_BLOCKS leaves everything unchanged.
 */
PKV_API pkv_status pkv_bm_append(pkv_block_manager* bm, int64_t seq_id, const int32_t* tokens, int32_t n,
                                 int32_t* slots);

/* Releases a sequence: its blocks' counts drop; blocks reaching zero return
 * to the free queue (cached ones keep their content for later hits). */
PKV_API pkv_status pkv_bm_free_sequence(pkv_block_manager* bm, int64_t seq_id);

/* Copies a sequence's block table (at most capacity entries) and reports its
 * block and token counts. */
PKV_API pkv_status pkv_bm_block_table(const pkv_block_manager* bm, int64_t seq_id, int32_t* table, int32_t capacity,
                                      int32_t* n_blocks, int32_t* n_tokens);

/*
 * One engine step for B sequences: appends n_new[b] tokens to sequence
 * seq_ids[b] (token ids packed in order in tokens[sum n_new]) and writes the
 * inputs of pkv_append / pkv_attention for the packed batch:
 *   cu_seqlens_q [B+1]                prefix sums of n_new
 *   seq_lens     [B]                  each sequence's length after the append
 *   block_tables [B, max_blocks]      row-major, padded with -1
 *   slot_mapping [sum n_new]          the new tokens' slots, packed
 * All or nothing: the blocks the whole step needs are checked first.
 * Sequence ids must be distinct within a step.
 */
PKV_API pkv_status pkv_bm_build_step(pkv_block_manager* bm, const int64_t* seq_ids, const int32_t* n_new,
                                     const int32_t* tokens, int32_t B, int32_t max_blocks, int32_t* cu_seqlens_q,
                                     int32_t* seq_lens, int32_t* block_tables, int32_t* slot_mapping);

/* Counters of the pool. */
PKV_API pkv_status pkv_bm_stats(const pkv_block_manager* bm, pkv_bm_stats_t* out);

#ifdef __cplusplus
}
#endif

#endif /* PKV_BLOCKS_H */
