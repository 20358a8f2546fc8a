/*
 * pkv.h -- C ABI of libpkv: the PagedAttention hot path on one GB300 (sm_103a).
 *
 * The KV cache of every request lives in fixed 16-token physical blocks reached
 * through a per-request block table; requests that share a prefix point at the
 * same physical blocks ("vLLM's PagedAttention" teardown, section "PagedAttention:
 * the KV cache is paged, like virtual memory").  One batch mixes chunked prefills
 * and decodes freely (same page, section "Continuous batching").  This library
 * implements the data-parallel steps of that path as CUDA kernels:
 *
 *   pkv_slot_mapping  logical position -> physical slot through the block table
 *   pkv_write         scatter new tokens' K/V rows into their slots
 *   pkv_copy_blocks   copy-on-write block copy ("The 1960s Operating System
 *                     Trick ..." page, Technical Details: Copy-on-Write)
 *   paged_attention   attention for one continuously-batched step: split-KV GQA
 *                     decode with online softmax and a cross-split merge, plus
 *                     causal chunked prefill, gathering K/V through block tables
 *   paged_attention_cascade  the same, reading each shared prompt prefix once
 *   paged_attention_step     slot mapping + K/V scatter + attention in one call
 *   paged_attention_step_cow the same, after the step's copy-on-write block copies
 *
 * Conventions for every call
 *  - Pointers named as device pointers must point to device memory of the current
 *    CUDA device; `stream` is a cudaStream_t (NULL = legacy default stream).  All
 *    compute calls are asynchronous on `stream`.
 *  - Ownership: the caller owns every buffer it passes.  The library owns only a
 *    per-device workspace for split-KV partials and a per-device error word; both
 *    are created on first use and released by pkv_shutdown().
 *  - Errors: an argument error found on the host returns a non-zero pkv_status
 *    and launches nothing.  Data errors found on the device (a block id outside
 *    [0, num_blocks), a slot past the pool, seq_len < q_len, more blocks than a
 *    table row holds) never trap: they set bits in the device error word, the
 *    affected outputs are zeroed or skipped, and pkv_get_last_error() reports them.
 *  - No call allocates device memory except paged_attention(), which grows the
 *    workspace when a larger batch needs it (never during stream capture).
 *
 * Cache layout (a reading where the pages are silent): k_cache and v_cache are
 * each [num_blocks][num_kv_heads][16][head_dim], row-major, so that one
 * (block, kv head) is a contiguous 16 x head_dim tile.
 * Supported element types: fp32 with head_dim 64 or 128; bf16 with head_dim 128.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1, /* null pointer, bad size, inconsistent shape */
  PKV_ERR_UNSUPPORTED = 2, /* dtype / head_dim / group size not built */
  PKV_ERR_INDEX = 3,       /* device saw a bad block id, slot or length */
  PKV_ERR_CUDA = 4,        /* a CUDA runtime call failed */
  PKV_ERR_NO_MEMORY = 5,   /* workspace could not be grown */
  PKV_ERR_TIMEOUT = 6      /* a kernel gave up a bounded wait (internal error) */
} pkv_status;

typedef enum { PKV_F32 = 0, PKV_BF16 = 1 } pkv_dtype;

#define PKV_BLOCK_SIZE 16

/* Shape of the paged KV pool (host struct). */
typedef struct {
  int64_t num_blocks;   /* physical blocks in the pool */
  int32_t block_size;   /* tokens per block; must be 16 */
  int32_t num_kv_heads; /* KV heads */
  int32_t head_dim;     /* elements per head row */
  int32_t dtype;        /* pkv_dtype of the cache, q, k, v and out */
} pkv_cache_desc;

/*
 * Slot mapping ("vLLM's PagedAttention" teardown, section "PagedAttention": the
 * block table maps logical token positions to physical block ids).
 * For request i with q_i = query_start_loc[i+1] - query_start_loc[i] new tokens
 * and context length seq_lens[i] (which counts those new tokens), new token j sits
 * at position p = seq_lens[i] - q_i + j and gets
 *     slot_mapping[query_start_loc[i] + j] = block_tables[i][p / 16] * 16 + p % 16.
 * block_tables    device int32 [num_seqs][max_blocks_per_seq], row-major
 * seq_lens        device int32 [num_seqs]
 * query_start_loc device int32 [num_seqs + 1], non-decreasing, [0] == 0,
 *                 [num_seqs] == num_tokens
 * slot_mapping    device int64 [num_tokens], written
 * Device errors: p / 16 >= max_blocks_per_seq or a negative block id give slot -1
 * and PKV_ERR_INDEX in the error word.
 */
PKV_API int pkv_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                     const int32_t* query_start_loc, int32_t num_seqs, int64_t num_tokens,
                     int64_t* slot_mapping, void* stream);

/*
 * KV-slot scatter (same section: new tokens go to the slots their block table
 * names).  For each token t with slot_mapping[t] >= 0 and each kv head h:
 *     k_cache[slot / 16][h][slot % 16][:] = k[t][h][:]   (and v into v_cache)
 * Bit-exact copy.  A negative slot skips the token (padding).
 * k, v            device [num_tokens][num_kv_heads][head_dim], cache dtype, contiguous
 * slot_mapping    device int64 [num_tokens]
 * k_cache,v_cache device pool, layout above
 * Duplicate non-negative slots are a caller error (the surviving row is unspecified).
 * Device errors: slot >= num_blocks * 16 is skipped and flagged PKV_ERR_INDEX.
 */
PKV_API int pkv_write(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens, void* k_cache,
              void* v_cache, const pkv_cache_desc* cache, void* stream);

/*
 * Copy-on-write block copy ("The 1960s Operating System Trick ..." page, Technical
 * Details: samples share blocks until they diverge; only the blocks that change are
 * duplicated).  For i in [0, n): k_cache[dst[i]] = k_cache[src[i]] and the same for
 * v_cache, all heads and all 16 slots, bit-exact.
 * src, dst        device int32 [n]
 * Caller contract: dst entries are distinct and none appears in src, so the pairs
 * are independent and may run in any order.
 * Device errors: an id outside [0, num_blocks) skips the pair and flags PKV_ERR_INDEX.
 */
PKV_API int pkv_copy_blocks(const int32_t* src, const int32_t* dst, int64_t n, void* k_cache, void* v_cache,
                    const pkv_cache_desc* cache, void* stream);

/*
 * Attention for one continuously-batched step ("vLLM's PagedAttention" teardown,
 * sections "PagedAttention" and "Continuous batching": the kernel is handed a
 * per-request block table and gathers K/V from wherever the blocks live; one pass
 * mixes chunked prefills and decodes).
 * For request i (q_i query tokens, context seq_lens[i] including them), query token
 * j at position p = seq_lens[i] - q_i + j and query head h (kv head g = h / G,
 * G = num_q_heads / num_kv_heads):
 *     out[t][h][:] = sum_{u<=p} softmax_u(scale * q[t][h] . K_u) V_u
 * with K_u, V_u = cache[block_tables[i][u / 16]][g][u % 16][:].  Causal masking is
 * bottom-right aligned inside a chunk; a decode token (q_i == 1) sees all seq_lens[i]
 * keys.  Accumulation is fp32; out has the dtype of q.
 * q               device [num_tokens][num_q_heads][head_dim]
 * block_tables    device int32 [num_seqs][max_blocks_per_seq]
 * seq_lens        device int32 [num_seqs]
 * query_start_loc device int32 [num_seqs + 1]
 * max_query_len, max_seq_len  host upper bounds over the batch, used only to plan
 *                 the launch; results never depend on them beyond being bounds
 * out             device [num_tokens][num_q_heads][head_dim], written
 * Device errors: a bad block id, seq_len < q_len or ceil(seq_len/16) >
 * max_blocks_per_seq flags PKV_ERR_INDEX and zeroes the affected output rows.
 */
PKV_API int paged_attention(const void* q, const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                    const int32_t* query_start_loc, int32_t num_seqs, int32_t num_q_heads, int64_t num_tokens,
                    int32_t max_query_len, int32_t max_seq_len, float scale, void* out, void* stream);

/*
 * Shared-prefix groups for paged_attention_cascade (host struct of device arrays).
 * Requests that share a prompt prefix point at the same physical blocks ("vLLM's
 * PagedAttention" teardown, section "PagedAttention": a new request whose prefix
 * hashes match reuses the cached blocks), so those blocks need to be read only once
 * per step for all of them.  Group g is a prefix of prefix_num_blocks[g] full blocks
 * (P_g = 16 x that many tokens) whose physical ids are row g of prefix_block_tables;
 * its members are the request indices member_seqs[member_start[g] ..
 * member_start[g + 1]).
 *   prefix_block_tables  device int32 [num_groups][max_prefix_blocks]
 *   prefix_num_blocks    device int32 [num_groups], each in [1, max_prefix_blocks]
 *   member_start         device int32 [num_groups + 1], 0 = first <= ... <= last = num_members
 *   member_seqs          device int32 [num_members]
 */
typedef struct {
  const int32_t* prefix_block_tables;
  int32_t max_prefix_blocks;
  const int32_t* prefix_num_blocks;
  const int32_t* member_start;
  const int32_t* member_seqs;
  int32_t num_groups;
  int32_t num_members;
} pkv_prefix_groups;

/*
 * paged_attention_cascade -- paged_attention() with shared-prefix groups as a hint.
 * The output is paged_attention()'s (up to fp32 rounding order): the groups only
 * change how the work is done.  A member whose request is a decode (one query
 * token), whose context goes past the prefix (seq_len > P_g), which is listed once
 * in all groups, and whose block table starts with the group's prefix blocks has
 * its first P_g keys attended together with the other members of its group: one
 * tensor-core pass per (group, kv head) reads the prefix once and leaves a partial
 * softmax state per member, which the split merge folds with the member's own keys
 * (log-sum-exp merge, prefix first).  Any other listed request -- a prefill chunk,
 * a shorter context, a duplicate, a table that does not match, a malformed group --
 * is attended the ordinary way.  No counterpart on the pages beyond the sharing
 * itself; this is the cascade reading of it.
 * groups: NULL or num_groups == 0 or num_members == 0 = paged_attention().  The fp32
 * path ignores the groups.  Host errors as paged_attention(), plus PKV_ERR_INVALID_ARG
 * for negative counts, null group arrays or max_prefix_blocks < 1.
 */
PKV_API int paged_attention_cascade(const void* q, const void* k_cache, const void* v_cache,
                                    const pkv_cache_desc* cache, const int32_t* block_tables,
                                    int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                    const int32_t* query_start_loc, int32_t num_seqs, int32_t num_q_heads,
                                    int64_t num_tokens, int32_t max_query_len, int32_t max_seq_len, float scale,
                                    const pkv_prefix_groups* groups, void* out, void* stream);

/*
 * paged_attention_step -- the new tokens' slot mapping and K/V scatter, then
 * attention, in one call: pkv_slot_mapping + pkv_write + paged_attention_cascade
 * with the same results, bit for bit ("vLLM's PagedAttention" teardown, section
 * "Continuous batching": every step appends each running request's new tokens to
 * its blocks and attends over them).  On the bf16 path the mapping and the scatter
 * run in extra CTAs of the planning launch, so the step has two launches fewer and
 * no slot array round trip; the kernel boundary orders the writes before every
 * attention read.  On an fp32 cache with max_query_len == 1 (every request brings
 * one token) the attention launch itself stores each token's rows before it reads
 * them, one launch in all; a request with more query tokens than that bound is then
 * flagged (PKV_ERR_INDEX), its rows zeroed and its tokens not written.
 * Copy-on-write copies (pkv_copy_blocks) go before this call.
 * k_new, v_new    device [num_tokens][num_kv_heads][head_dim], cache dtype, required
 * k_cache, v_cache  written at the new tokens' slots, then read
 * groups          NULL for none (see paged_attention_cascade)
 * slot_mapping    optional device int64 [num_tokens]: receives the slots (NULL: not stored)
 * Everything else and the errors: as paged_attention() and pkv_write().
 */
PKV_API int paged_attention_step(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                                 const pkv_cache_desc* cache, const int32_t* block_tables,
                                 int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                 const int32_t* query_start_loc, int32_t num_seqs, int32_t num_q_heads,
                                 int64_t num_tokens, int32_t max_query_len, int32_t max_seq_len, float scale,
                                 const pkv_prefix_groups* groups, int64_t* slot_mapping, void* out, void* stream);

/*
 * paged_attention_step_cow -- pkv_copy_blocks(cow_src, cow_dst, num_cow) followed by
 * paged_attention_step, in one call, with the same results bit for bit.  The copies
 * are the copy-on-write of the "vLLM's PagedAttention" teardown, section
 * "PagedAttention": a request about to write into a block another request still
 * shares gets a fresh copy first.  Taking them in the same call lets the step plan
 * its work while the copies run, instead of after them; only the new tokens' writes,
 * which may land in a copied block, wait for the copies.
 * cow_src, cow_dst  device int32 [num_cow] block ids (as pkv_copy_blocks)
 * num_cow          0: no copies (exactly paged_attention_step)
 * Everything else and the errors: as paged_attention_step() and pkv_copy_blocks().
 */
PKV_API int paged_attention_step_cow(const void* q, const void* k_new, const void* v_new, void* k_cache,
                                     void* v_cache, const pkv_cache_desc* cache, const int32_t* block_tables,
                                     int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                     const int32_t* query_start_loc, int32_t num_seqs, int32_t num_q_heads,
                                     int64_t num_tokens, int32_t max_query_len, int32_t max_seq_len, float scale,
                                     const pkv_prefix_groups* groups, const int32_t* cow_src,
                                     const int32_t* cow_dst, int64_t num_cow, int64_t* slot_mapping, void* out,
                                     void* stream);

/*
 * paged_attention_noalloc -- paged_attention() for callers that cannot let a library
 * allocate device memory.  The pages have no counterpart for this call; it exists
 * for deployment.  paged_attention() grows a workspace with cudaMalloc when a batch
 * needs more split-KV scratch; a caller whose allocator must account for every byte
 * of device memory, or a service that reserves its memory at start-up and forbids
 * allocation afterwards, cannot accept that.  This call computes the same result
 * with its scratch in a fixed 16 MiB static device array that the library holds on
 * every GPU that loads it, until the process exits.
 *  - Same arguments and results as paged_attention(), bf16 with head_dim 128 only.
 *  - error_bits: optional device uint32 the kernels OR their data-error bits into
 *    (the bits of pkv_peek_error_bits); NULL discards them.  The caller clears it.
 *  - A batch whose scratch need exceeds the array returns PKV_ERR_NO_MEMORY and
 *    launches nothing.  The need is about num_seqs * num_kv_heads *
 *    ceil(max_seq_len / 1024) * GP * 520 bytes plus a few arrays per request, GP
 *    being the query-head group size rounded up to 4, 8 or 16.  A batch that
 *    paged_attention() refuses as unsupported (2^31 or more split items) returns
 *    PKV_ERR_UNSUPPORTED here too.
 *  - The first call on a device looks up the array's device address (with that
 *    device current); make it before any stream capture.
 *  - All calls share the array and the library re-zeroes what each call needs, but
 *    calls whose kernels overlap on the GPU race on it: serialise them.
 *  - Calls no cudaMalloc, cudaFree or other allocating routine.
 */
PKV_API int paged_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                    const pkv_cache_desc* cache, const int32_t* block_tables,
                                    int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                    const int32_t* query_start_loc, int32_t num_seqs, int32_t num_q_heads,
                                    int64_t num_tokens, int32_t max_query_len, int32_t max_seq_len, float scale,
                                    void* out, uint32_t* error_bits, void* stream);

/* Synchronises `stream`, returns the device error word of the current device as a
 * pkv_status (PKV_OK, PKV_ERR_INDEX or PKV_ERR_TIMEOUT) and clears it. */
PKV_API int pkv_get_last_error(void* stream);

/* Raw device error bits of the current device (bit 0 bad block id, bit 1 bad slot,
 * bit 2 bad length, bit 3 wait timeout); synchronises `stream`; does not clear. */
PKV_API int pkv_peek_error_bits(void* stream, uint32_t* bits);

/* Human-readable name of a pkv_status value (static string). */
PKV_API const char* pkv_status_string(int status);

/* Number of persistent CTAs the attention kernels launch on the current device
 * (a multiple of the SM count); split boundaries depend only on it and the lengths. */
PKV_API int pkv_num_workers(int32_t* workers);

/* Releases the library-owned workspace and error word on every device used. */
PKV_API void pkv_shutdown(void);

/*
 * Launch tracing.  While enabled, every kernel the library launches is bracketed
 * by CUDA events on its stream.  pkv_trace_read() synchronises the device and
 * returns, per kernel kind, the launch count and the summed device time in ms,
 * then resets the counters.  Kinds: 0 slot mapping, 1 write, 2 copy, 3 plan,
 * 4 decode, 5 prefill, 6 generic attention, 7 split merge, 8 shared-prefix (cascade)
 * pass.  Arrays hold PKV_TRACE_KINDS entries.
 */
#define PKV_TRACE_KINDS 9
PKV_API int pkv_trace_enable(int on);
PKV_API int pkv_trace_read(int64_t* launches, double* total_ms);
PKV_API const char* pkv_trace_kind_name(int kind);

/*
 * Diagnostics for the tensor-core operand layouts (no counterpart in the pages).
 * pkv_umma_selftest copies two operand images (a_img, b_img: device bytes, already
 * in shared-memory order) into shared memory, runs k_steps tcgen05 bf16 MMAs with
 * an fp32 accumulator in TMEM, and writes D ([M][N] fp32 row-major) to d_out.
 * params (host int32[29]): M, N, a_mn_major, b_mn_major, a_layout, a_lbo, a_sbo,
 * b_layout, b_lbo, b_sbo, a_bytes, b_bytes, k_steps, a_off[8], b_off[8] -- layouts
 * use the descriptor codes (0 none, 2 128B, 4 64B, 6 32B), offsets are bytes.
 * a_layout = -1 reads A from TMEM instead (M must be 128, A K-major): a_img is then
 * [128 rows][a_bytes / 512] 32-bit columns, two bf16 each, stored to the rows' lanes
 * after the N accumulator columns, and a_off[k] is k step k's first column (a multiple
 * of 8) within them.
 * pkv_tma_selftest loads rows [row0, row0+16) of a bf16 [rows][128] matrix with two
 * 16 x 64 boxes in the 128-byte swizzle and copies the 4 KiB of shared memory they
 * land in to dump.
 */
PKV_API int pkv_umma_selftest(const int32_t* params, const void* a_img, const void* b_img, float* d_out, void* stream);
PKV_API int pkv_tma_selftest(const void* src, int64_t rows, int32_t row0, void* dump, void* stream);
/*
 * pkv_wait_selftest launches one CTA that waits on an mbarrier nothing arrives on.
 * The bounded wait every kernel of the library uses gives up after its limit (1 s),
 * the CTA sets the timeout bit of the device error word and exits: the next
 * pkv_get_last_error() returns PKV_ERR_TIMEOUT, and the context stays usable.
 */
PKV_API int pkv_wait_selftest(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
