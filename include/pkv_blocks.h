/*
 * pkv_blocks.h — host-side KV block manager: the step before paged attention.
 *
 * The engine keeps the KV cache in fixed-size blocks handed out by a block
 * manager ("How lunaryes/nano-vllm works", Components: KV Block Manager;
 * Connections: the scheduler asks the KV block manager for cached blocks),
 * with prefix caching (nano-vllm-sansho README, "Key Features") and a block
 * size set by the deployment (nano-vllm-rs README, "Notes":
 * NANO_VLLM_KVCACHE_BLOCK_SIZE). This manager produces exactly what the
 * kernels of pkv.h consume: each sequence's block-table row and the cache slot
 * of every token to store (slot = block * block_size + position % block_size).
 *
 * Policy (the pages give no more detail; these are the plainest readings):
 *  - Blocks are reference counted. A block with no reference is on a free
 *    list, oldest freed first.
 *  - A full block (block_size tokens) is identified by a chained hash: the
 *    64-bit FNV-1a hash of the previous full block's hash and its own token
 *    ids. A new prompt's leading full blocks that are found by hash, with the
 *    same stored token ids and the same previous-block hash, are shared with
 *    their current holders (or taken back from the free list) instead of being
 *    allocated: their K/V are already in the cache, and their tokens get no
 *    slot. At least one prompt token is always left to compute.
 *  - A freed full block stays findable until it is handed out again for other
 *    tokens.
 *  - A block becomes findable as soon as it is full: when a prompt is added
 *    (the caller stores its tokens in the same step, before attention) or when
 *    an appended token fills it.
 * Identical prompts thus share physical blocks; the kernels never write a
 * shared block, because only tokens past a sequence's cached prefix get slots.
 *
 * Ownership and threading: the manager owns its host memory; it touches no
 * device memory. Calls on one manager must not run concurrently.
 * Errors: PKV_ERR_INVALID_ARG for bad arguments (unknown or duplicate
 * sequence id, positions outside a sequence, a row too short),
 * PKV_ERR_OUT_OF_BLOCKS when the free list cannot cover a request; a failed
 * call changes nothing.
 */
#ifndef PKV_BLOCKS_H
#define PKV_BLOCKS_H

#include <stdint.h>

#include "pkv.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pkv_block_manager pkv_block_manager;

/* A manager of num_blocks blocks of block_size token slots, all free.
 * NULL for non-positive sizes, for num_blocks * block_size above INT32_MAX
 * (slots are int32) or when host memory runs out. */
pkv_block_manager *pkv_bm_create(int32_t num_blocks, int32_t block_size);

/* Frees the manager (NULL is allowed). */
void pkv_bm_destroy(pkv_block_manager *bm);

/* Blocks with no reference (including freed blocks still findable by hash). */
int32_t pkv_bm_num_free_blocks(const pkv_block_manager *bm);

/* References to block b (-1 if b is outside the pool). */
int32_t pkv_bm_ref_count(const pkv_block_manager *bm, int32_t b);

/* Admit sequence seq_id with its num_tokens (>= 1) prompt token ids.
 * *num_cached_tokens receives how many leading tokens are already in the
 * cache (a multiple of block_size, below num_tokens); the caller stores and
 * computes positions num_cached_tokens .. num_tokens - 1. */
pkv_status pkv_bm_add_sequence(pkv_block_manager *bm, int64_t seq_id, const int32_t *token_ids,
                               int32_t num_tokens, int32_t *num_cached_tokens);

/* Append one token (a decode step) to seq_id; a new block is taken when the
 * sequence's last block is full. The new token is at position num_tokens - 1. */
pkv_status pkv_bm_append_token(pkv_block_manager *bm, int64_t seq_id, int32_t token_id);

/* Release seq_id: each of its blocks loses one reference; blocks left with
 * none go to the back of the free list. */
pkv_status pkv_bm_free_sequence(pkv_block_manager *bm, int64_t seq_id);

/* Number of tokens of seq_id in *num_tokens. */
pkv_status pkv_bm_num_tokens(const pkv_block_manager *bm, int64_t seq_id, int32_t *num_tokens);

/* Block-table row of seq_id: its block ids in order, then -1 up to max_blocks.
 * *num_blocks receives the sequence's block count; PKV_ERR_INVALID_ARG (row
 * untouched) if max_blocks is smaller. */
pkv_status pkv_bm_block_table(const pkv_block_manager *bm, int64_t seq_id, int32_t *row,
                              int32_t max_blocks, int32_t *num_blocks);

/* Cache slots of positions first .. first + count - 1 of seq_id (all inside
 * the sequence), for pkv_kv_store's slot_mapping. */
pkv_status pkv_bm_slots(const pkv_block_manager *bm, int64_t seq_id, int32_t first,
                        int32_t count, int32_t *slots);

#ifdef __cplusplus
}
#endif

#endif /* PKV_BLOCKS_H */
