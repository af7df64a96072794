/*
 * wf_blocks.h -- host-side block manager for the paged KV cache of libwf.
 *
 * The bookkeeping that produces what the attention calls consume: which block of
 * the pool holds which positions of which sequence (the block tables), the slot
 * of every new token (slot_mapping for wf_reshape_and_cache), and the
 * copy-on-write block pairs for wf_copy_blocks when sequences share a prefix.
 *
 * Sources (page title, section):
 *   ember, "The core idea, in one picture": a sequence's positions live in the
 *     blocks its block table lists, position p in block table[p / P] at p % P.
 *   weft, "Cache layouts": blocks are handed out to requests from a shared pool.
 *   tiny-vllm-py, "Mental Model" and "Prefix Sharing": a request grows block by
 *     block; requests with a common prefix share its blocks, and a shared block
 *     that is only partly filled is copied before a request appends to it.
 *
 * Conventions
 *   - Host memory only: every pointer here is a host pointer.  No CUDA call is
 *     made; the caller uploads the tables and slots it needs.
 *   - One manager is not safe for concurrent use from several threads.
 *   - A sequence is named by any int64 id; it exists from its first append (or
 *     fork) until it is freed.
 *   - Blocks are reference counted: a block returns to the free list when the
 *     last sequence holding it is freed.  Free blocks are handed out last-freed
 *     first.
 *   - A call that fails changes nothing.
 */
#ifndef WF_BLOCKS_H
#define WF_BLOCKS_H

#include <stdint.h>

#include "wf.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct wf_block_manager wf_block_manager;

/*
 * A manager of num_blocks blocks of block_size tokens (1 .. 1024).  The free list
 * starts as the ids 0 .. N-1 in ascending order (shuffle_seed == 0) or shuffled by
 * a splitmix64 stream seeded with shuffle_seed.  *out receives the handle.
 * WF_ERR_INVALID_ARG on bad sizes or a null out.
 */
wf_status wf_bm_create(int32_t num_blocks, int32_t block_size, uint64_t shuffle_seed, wf_block_manager** out);

/* Releases the manager (NULL is a no-op). */
void wf_bm_destroy(wf_block_manager* bm);

/* Free blocks; -1 for a null manager. */
int32_t wf_bm_num_free(const wf_block_manager* bm);

/* Tokens sequence seq holds; -1 if it does not exist. */
int64_t wf_bm_seq_len(const wf_block_manager* bm, int64_t seq);

/* Reference count of block `block` (0 = free); -1 if out of range. */
int32_t wf_bm_ref_count(const wf_block_manager* bm, int32_t block);

/*
 * Appends n >= 0 tokens to sequence seq (created if new) and writes the slot of
 * each, slot = block * block_size + offset, into slots[0 .. n).  Blocks are taken
 * from the free list as the sequence crosses block boundaries.  If the sequence's
 * last block is partly filled and shared with another sequence, it is first
 * copied on write: a fresh block replaces it in this sequence's table, and
 * (src, dst) is written to cow_pair[0..1] with *n_cow = 1 (else *n_cow = 0); the
 * caller copies the block (wf_copy_blocks) before scattering the new tokens.
 * WF_ERR_NO_BLOCKS if the free list is too short; WF_ERR_INVALID_ARG on null
 * pointers (slots may be NULL when n == 0) or n < 0.
 */
wf_status wf_bm_append(wf_block_manager* bm, int64_t seq, int32_t n, int64_t* slots, int32_t* cow_pair,
                       int32_t* n_cow);

/*
 * Sequence child (which must not exist) starts as a copy of parent's table and
 * length, sharing every block (prefix sharing).  WF_ERR_INVALID_ARG if parent does
 * not exist or child does.
 */
wf_status wf_bm_fork(wf_block_manager* bm, int64_t parent, int64_t child);

/* Drops sequence seq; its blocks' reference counts go down.  WF_ERR_INVALID_ARG if
 * it does not exist. */
wf_status wf_bm_free(wf_block_manager* bm, int64_t seq);

/*
 * The batch arrays of sequences seqs[0 .. B): block_tables [B, M] row-major (row b
 * lists seqs[b]'s blocks, then pad_block up to M) and seq_lens [B].
 * WF_ERR_INVALID_ARG if a sequence does not exist or holds more than M blocks.
 */
wf_status wf_bm_tables(const wf_block_manager* bm, const int64_t* seqs, int32_t B, int32_t M, int32_t pad_block,
                       int32_t* block_tables, int32_t* seq_lens);

#ifdef __cplusplus
}
#endif

#endif /* WF_BLOCKS_H */
