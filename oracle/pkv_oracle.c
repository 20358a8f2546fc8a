/*
 * pkv_oracle.c -- plain, slow, fp64 CPU oracle for the PagedAttention hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the tests, the package's smoke check and the timed CPU
 * baseline of the benchmark load it.  It shares no code, header, table or
 * constant with the CUDA path.
 *
 * What it follows (page titles and sections):
 *  - "vLLM's PagedAttention ... teardown" (arcyou-site), section "PagedAttention:
 *    the KV cache is paged, like virtual memory": KV memory is cut into 16-token
 *    blocks; each request holds a block table that maps logical token positions
 *    to physical block ids; the attention step gathers K/V from wherever those
 *    blocks are.  Shared prefixes point at the same physical blocks.
 *  - same page, section "Continuous batching": one forward pass mixes prompts
 *    (chunked prefill) and generations (decode) freely.
 *  - "The 1960s Operating System Trick ..." (aitrending), "Technical Details":
 *    logical blocks map to scattered physical pages; copy-on-write duplicates only
 *    the blocks that change.
 *  - "Introduction" (kenhuang), "PagedAttention (intuition)": the logical context
 *    is contiguous, the physical pages need not be.
 *
 * Because paging only moves bytes, the attention result is, by definition, ordinary
 * attention over each request's logical context.  So the oracle is that definition
 * written out: gather each key/value through the block table, compute
 * softmax(scale * q.k) with a plain two-pass softmax in fp64, and sum the values.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - cache layout [num_blocks][num_kv_heads][16][head_dim] for K and for V;
 *  - seq_lens[i] counts the whole context including this step's query tokens;
 *  - query token j of a request with q_i query tokens sits at position
 *    seq_len - q_i + j and sees keys 0..that position (bottom-right causal);
 *  - query head h reads kv head h / (num_q_heads / num_kv_heads);
 *  - a negative slot in a slot mapping means "skip this token".
 *
 * Inputs are read in the dtype the caller stores (fp32 or bf16) and widened to
 * fp64 exactly; all arithmetic is fp64 in the plain loop order below.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_BLOCK 16

enum { ORC_F32 = 0, ORC_BF16 = 1 };
enum { ORC_OK = 0, ORC_BAD_ARG = 1, ORC_BAD_INDEX = 3, ORC_NO_MEM = 5 };

/* Exact widening of one stored element to double. bf16 is the top half of an
 * IEEE binary32, so shifting its 16 bits up gives the float it denotes. */
static double orc_load(const void *base, int64_t idx, int dtype) {
  if (dtype == ORC_F32) return (double)((const float *)base)[idx];
  uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

int orc_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Slot mapping: token j of request i (position p = seq_len - q_len + j) goes to
 * physical block block_tables[i][p / 16], offset p % 16, i.e. slot
 * block * 16 + p % 16.  Writes one int64 slot per query token, in
 * query_start_loc order.  Returns ORC_BAD_INDEX if a request's positions need
 * more table entries than max_blocks or a length is inconsistent. */
int orc_slot_mapping(const int32_t *block_tables, int32_t max_blocks,
                     const int32_t *seq_lens, const int32_t *query_start_loc,
                     int32_t num_seqs, int64_t *slots) {
  for (int32_t i = 0; i < num_seqs; ++i) {
    int32_t q_len = query_start_loc[i + 1] - query_start_loc[i];
    int32_t L = seq_lens[i];
    if (q_len < 0 || L < q_len) return ORC_BAD_INDEX;
    for (int32_t j = 0; j < q_len; ++j) {
      int64_t p = (int64_t)L - q_len + j;
      int64_t logical_block = p / ORC_BLOCK;
      if (logical_block >= max_blocks) return ORC_BAD_INDEX;
      int64_t phys = block_tables[(int64_t)i * max_blocks + logical_block];
      slots[query_start_loc[i] + j] = phys * ORC_BLOCK + p % ORC_BLOCK;
    }
  }
  return ORC_OK;
}

/* KV-slot scatter: for every token t with slot >= 0, copy its K row and V row of
 * each kv head into cache[slot / 16][head][slot % 16][:].  Pure byte copy. */
int orc_write(const void *k, const void *v, const int64_t *slots, int64_t T,
              int32_t num_kv_heads, int32_t head_dim, int32_t elem_bytes,
              int64_t num_blocks, void *k_cache, void *v_cache) {
  const int64_t row_bytes = (int64_t)head_dim * elem_bytes;
  for (int64_t t = 0; t < T; ++t) {
    int64_t s = slots[t];
    if (s < 0) continue;
    int64_t block = s / ORC_BLOCK, off = s % ORC_BLOCK;
    if (block >= num_blocks) return ORC_BAD_INDEX;
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      int64_t src = (t * num_kv_heads + h) * row_bytes;
      int64_t dst = ((block * num_kv_heads + h) * ORC_BLOCK + off) * row_bytes;
      memcpy((char *)k_cache + dst, (const char *)k + src, (size_t)row_bytes);
      memcpy((char *)v_cache + dst, (const char *)v + src, (size_t)row_bytes);
    }
  }
  return ORC_OK;
}

/* Copy-on-write block copy: cache[dst[i]] = cache[src[i]] for K and V, every
 * head and all 16 slots.  All sources are read from a snapshot taken before the
 * first copy, so the result does not depend on the order of the pairs. */
int orc_copy_blocks(const int32_t *src, const int32_t *dst, int64_t n,
                    int64_t block_bytes, int64_t num_blocks, void *k_cache,
                    void *v_cache) {
  if (n == 0) return ORC_OK;
  for (int64_t i = 0; i < n; ++i)
    if (src[i] < 0 || src[i] >= num_blocks || dst[i] < 0 || dst[i] >= num_blocks)
      return ORC_BAD_INDEX;
  char *snap = (char *)malloc((size_t)(2 * n * block_bytes));
  if (!snap) return ORC_NO_MEM;
  for (int64_t i = 0; i < n; ++i) {
    memcpy(snap + (2 * i) * block_bytes, (char *)k_cache + src[i] * block_bytes, (size_t)block_bytes);
    memcpy(snap + (2 * i + 1) * block_bytes, (char *)v_cache + src[i] * block_bytes, (size_t)block_bytes);
  }
  for (int64_t i = 0; i < n; ++i) {
    memcpy((char *)k_cache + dst[i] * block_bytes, snap + (2 * i) * block_bytes, (size_t)block_bytes);
    memcpy((char *)v_cache + dst[i] * block_bytes, snap + (2 * i + 1) * block_bytes, (size_t)block_bytes);
  }
  free(snap);
  return ORC_OK;
}

/* Attention over the paged context, by definition.
 *
 * For each requested query token t (rows[r], or every token when rows == NULL)
 * of request i, at position p = seq_len_i - q_len_i + (t - query_start_loc[i]),
 * and for each query head h with kv head g = h / (num_q_heads / num_kv_heads):
 *   K_u = k_cache[block_tables[i][u / 16]][g][u % 16][:]   (u = 0..p)
 *   s_u = scale * sum_c q[t][h][c] * K_u[c]
 *   w_u = exp(s_u - max_u s_u)
 *   out[r][h][:] = (sum_u w_u * V_u[:]) / (sum_u w_u)
 * Output is fp64 [n_rows][num_q_heads][head_dim]. */
int orc_attention(const void *q, int32_t dtype, const void *k_cache,
                  const void *v_cache, int64_t num_blocks, int32_t num_kv_heads,
                  int32_t head_dim, const int32_t *block_tables,
                  int32_t max_blocks, const int32_t *seq_lens,
                  const int32_t *query_start_loc, int32_t num_seqs,
                  int32_t num_q_heads, float scale, const int64_t *rows,
                  int64_t n_rows, double *out, int32_t n_threads) {
  if (num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0 || head_dim <= 0)
    return ORC_BAD_ARG;
  const int32_t group = num_q_heads / num_kv_heads;
  const int64_t T_q = query_start_loc[num_seqs];
  if (rows == NULL) n_rows = T_q;
  /* validate lengths and every table entry the definition reads */
  for (int32_t i = 0; i < num_seqs; ++i) {
    int32_t q_len = query_start_loc[i + 1] - query_start_loc[i];
    if (q_len < 0 || seq_lens[i] < q_len) return ORC_BAD_INDEX;
    int64_t nb = ((int64_t)seq_lens[i] + ORC_BLOCK - 1) / ORC_BLOCK;
    if (nb > max_blocks) return ORC_BAD_INDEX;
    for (int64_t b = 0; b < nb; ++b) {
      int32_t id = block_tables[(int64_t)i * max_blocks + b];
      if (id < 0 || id >= num_blocks) return ORC_BAD_INDEX;
    }
  }
  for (int64_t r = 0; r < n_rows; ++r) {
    int64_t t = rows ? rows[r] : r;
    if (t < 0 || t >= T_q) return ORC_BAD_ARG;
  }
  const double dscale = (double)scale;
  int failed = 0;
  const int64_t units = n_rows * num_q_heads;
#ifdef _OPENMP
  if (n_threads <= 0) n_threads = omp_get_max_threads();
#pragma omp parallel num_threads(n_threads)
#endif
  {
    /* per-thread logits buffer, grown to the longest context seen */
    double *s = NULL;
    int64_t s_cap = 0;
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int64_t unit = 0; unit < units; ++unit) {
      int64_t r = unit / num_q_heads;
      int32_t h = (int32_t)(unit % num_q_heads);
      int64_t t = rows ? rows[r] : r;
      /* request that owns token t: the last i with query_start_loc[i] <= t and
       * a non-empty query range (binary search over the prefix sums) */
      int32_t lo = 0, hi = num_seqs - 1;
      while (lo < hi) {
        int32_t mid = lo + (hi - lo + 1) / 2;
        if (query_start_loc[mid] <= t) lo = mid; else hi = mid - 1;
      }
      int32_t i = lo;
      int32_t q_len = query_start_loc[i + 1] - query_start_loc[i];
      int64_t p = (int64_t)seq_lens[i] - q_len + (t - query_start_loc[i]);
      int32_t g = h / group;
      int64_t n_keys = p + 1;
      if (n_keys > s_cap) {
        free(s);
        s = (double *)malloc((size_t)n_keys * sizeof(double));
        s_cap = s ? n_keys : 0;
        if (!s) { failed = 1; continue; }
      }
      const int64_t q_base = (t * num_q_heads + h) * head_dim;
      /* pass 1: logits and their maximum */
      double m = -INFINITY;
      for (int64_t u = 0; u < n_keys; ++u) {
        int64_t phys = block_tables[(int64_t)i * max_blocks + u / ORC_BLOCK];
        int64_t k_base = ((phys * num_kv_heads + g) * ORC_BLOCK + u % ORC_BLOCK) * head_dim;
        double dot = 0.0;
        for (int32_t c = 0; c < head_dim; ++c)
          dot += orc_load(q, q_base + c, dtype) * orc_load(k_cache, k_base + c, dtype);
        s[u] = dscale * dot;
        if (s[u] > m) m = s[u];
      }
      /* pass 2: weights, their sum, and the weighted sum of values */
      double *o = out + (r * num_q_heads + h) * head_dim;
      for (int32_t c = 0; c < head_dim; ++c) o[c] = 0.0;
      double denom = 0.0;
      for (int64_t u = 0; u < n_keys; ++u) {
        double w = exp(s[u] - m);
        denom += w;
        int64_t phys = block_tables[(int64_t)i * max_blocks + u / ORC_BLOCK];
        int64_t v_base = ((phys * num_kv_heads + g) * ORC_BLOCK + u % ORC_BLOCK) * head_dim;
        for (int32_t c = 0; c < head_dim; ++c) o[c] += w * orc_load(v_cache, v_base + c, dtype);
      }
      for (int32_t c = 0; c < head_dim; ++c) o[c] /= denom;
    }
    free(s);
  }
  return failed ? ORC_NO_MEM : ORC_OK;
}
