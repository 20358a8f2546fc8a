/*
 * pkv_blocks.h -- C ABI of the host-side KV block manager in libpkv.
 *
 * This is the bookkeeping that produces the block tables the GPU path consumes.
 * What it implements, and where the pages state it:
 *  - "vLLM's PagedAttention" teardown (arcyou-site), section "PagedAttention: the KV
 *    cache is paged, like virtual memory":
 *    - one fixed pool of 16-token blocks;
 *    - allocate_slots hands out ceil(new tokens / 16) blocks, or nothing at all (None,
 *      here -1) if the pool is short;
 *    - the hash of a request's block i depends on blocks 0..i, so two requests
 *      with equal hashes at block i have equal prefixes up to there;
 *    - a hit hands out the cached physical block again and counts one more user;
 *    - at zero users a block is free again, but freed blocks that still carry a
 *      hash are handed out only after blocks that never did, oldest first;
 *  - same page, section "What happens when the blocks run out": a freed request's
 *    blocks are queued last block first, so its first blocks are the last reused;
 *  - "The 1960s Operating System Trick ..." page, Technical Details: samples of one
 *    prompt use the same blocks, and the one block about to change is copied first.
 *
 * All calls are host-only and not thread-safe (one manager per scheduler thread).
 * Requests are named by caller-chosen int64 ids.  Functions returning int return
 * a negative value on error: -1 = pool too small (nothing changed), -2 = unknown or
 * already-existing request, -3 = bad argument.
 */
#ifndef PKV_BLOCKS_H_
#define PKV_BLOCKS_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PKV_BM_API __attribute__((visibility("default")))
#else
#define PKV_BM_API
#endif

typedef struct pkv_block_manager pkv_block_manager;

/* A pool of num_blocks 16-token blocks, all free.  enable_prefix_cache != 0 turns on
 * hashing of full blocks and reuse of cached prefixes.  NULL on bad arguments. */
PKV_BM_API pkv_block_manager* pkv_bm_create(int64_t num_blocks, int32_t enable_prefix_cache);
PKV_BM_API void pkv_bm_destroy(pkv_block_manager* bm);

/* Blocks with reference count zero (including cached-but-free ones). */
PKV_BM_API int64_t pkv_bm_num_free(const pkv_block_manager* bm);

/* Starts request `req` and looks up the longest cached prefix of its prompt tokens
 * (full blocks only, hashes chained from the first block, token ids compared on a hit).
 * Each hit block is referenced by the request.  Returns the number of hit blocks
 * (computed tokens = 16 x that), -2 if the request exists. */
PKV_BM_API int32_t pkv_bm_get_computed_blocks(pkv_block_manager* bm, int64_t req, const int32_t* tokens,
                                              int64_t num_tokens);

/* Grows request `req` so that its blocks hold `total_tokens` tokens: takes
 * ceil(total_tokens / 16) - (blocks held) blocks from the head of the free queue
 * (evicting the cached hash of any cached-but-free block it takes).  Returns the
 * number of blocks added (0 if none were needed), -1 if the pool cannot cover them
 * (then nothing is taken), -2 if the request does not exist. */
PKV_BM_API int32_t pkv_bm_allocate_slots(pkv_block_manager* bm, int64_t req, int64_t total_tokens);

/* Registers the hashes of the request's blocks that `tokens` (the request's first
 * num_tokens token ids) fills completely and that are not registered yet.  A hash
 * that already names another block leaves this block uncached.  Returns the number
 * of blocks newly cached, or a negative error. */
PKV_BM_API int32_t pkv_bm_cache_full_blocks(pkv_block_manager* bm, int64_t req, const int32_t* tokens,
                                            int64_t num_tokens);

/* Copies the request's block table (physical block ids in logical order) into out
 * (capacity max_out).  Returns the number of blocks, or a negative error. */
PKV_BM_API int32_t pkv_bm_block_table(const pkv_block_manager* bm, int64_t req, int32_t* out, int32_t max_out);

/* Ends request `req`: every block loses one reference, and blocks reaching zero join
 * the tail of the free queue, the request's last block first.  Returns 0 or -2. */
PKV_BM_API int32_t pkv_bm_free(pkv_block_manager* bm, int64_t req);

/* Starts request `child` sharing every block of `parent` (one more reference each),
 * with the same token count and hash chain -- a parallel sample.  Returns 0 or -2. */
PKV_BM_API int32_t pkv_bm_fork(pkv_block_manager* bm, int64_t parent, int64_t child);

/* Copy-on-write before writing into logical block `logical_block` of `req`: if that
 * block is shared (reference count > 1), a free block replaces it in the request's
 * table, *src / *dst receive the old and new physical ids (for pkv_copy_blocks), and
 * 1 is returned; 0 if the block is already exclusive; -1 if no block is free. */
PKV_BM_API int32_t pkv_bm_cow(pkv_block_manager* bm, int64_t req, int32_t logical_block, int32_t* src,
                              int32_t* dst);

/* Usage of the live requests: blocks referenced (each distinct block once), and the
 * slots they leave unused beyond each request's token count (the only waste of
 * paging is each request's last partial block). */
PKV_BM_API int32_t pkv_bm_usage(const pkv_block_manager* bm, int64_t* blocks_in_use, int64_t* tokens_held,
                                int64_t* unused_slots);

/* Shared-prefix groups of a batch, for paged_attention_cascade: requests reqs[0..n) (the batch
 * order) whose block tables start with the same physical block form a group, and the group's prefix
 * is the longest run of leading blocks that all its members share (at most max_prefix_blocks).
 * Groups of a single request, or whose members share no block, are left out.  Writes group g's
 * prefix block ids to prefix_tables[g * max_prefix_blocks ...], its length in blocks to
 * prefix_num_blocks[g], and its members' batch indices to member_seqs[member_start[g] ..
 * member_start[g + 1]) (member_start holds max_groups + 1 entries, member_seqs n).  The kernel
 * admits only decodes whose context goes past the prefix; the rest of a group is attended the
 * ordinary way.  Returns the number of groups (at most max_groups; further groups are dropped),
 * -2 if a request is unknown, -3 on bad arguments. */
PKV_BM_API int32_t pkv_bm_prefix_groups(const pkv_block_manager* bm, const int64_t* reqs, int32_t n,
                                        int32_t max_prefix_blocks, int32_t max_groups, int32_t* prefix_tables,
                                        int32_t* prefix_num_blocks, int32_t* member_start, int32_t* member_seqs);

/* The chained hash of one full block: 64-bit hash of (parent_hash, 16 token ids,
 * extra_key).  Exposed for tests.  The first block of a request chains from 0. */
PKV_BM_API uint64_t pkv_bm_block_hash(uint64_t parent_hash, const int32_t* tokens16, uint64_t extra_key);

#ifdef __cplusplus
}
#endif

#endif /* PKV_BLOCKS_H_ */
