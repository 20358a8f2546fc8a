// block_manager.cpp -- host-side KV block manager (see include/pkv_blocks.h).
//
// Pool of 16-token blocks with a free queue (doubly linked list, allocation from the
// head, release to the tail), reference counts, and a map from chained block hashes
// to cached blocks ("vLLM's PagedAttention" teardown, section "PagedAttention: the KV
// cache is paged, like virtual memory").  A cached block whose count drops to zero
// stays in the map while it waits in the free queue; it is evicted (its hash dropped)
// only when allocation takes it from the head.  Hits compare token ids, so a hash
// collision can never hand out the wrong block.
#include <algorithm>
#include <cstring>
#include <unordered_map>
#include <vector>

#include "pkv_blocks.h"

namespace {

constexpr int64_t kBlock = 16;

// splitmix64 finaliser (S. Vigna): a well-mixed 64-bit function used to chain hashes.
inline uint64_t mix64(uint64_t x) {
  x += 0x9e3779b97f4a7c15ull;
  x = (x ^ (x >> 30)) * 0xbf58476d1ce4e5b9ull;
  x = (x ^ (x >> 27)) * 0x94d049bb133111ebull;
  return x ^ (x >> 31);
}

uint64_t block_hash(uint64_t parent, const int32_t* tokens, uint64_t extra) {
  uint64_t h = mix64(parent ^ 0x5bd1e9955bd1e995ull);
  for (int64_t i = 0; i < kBlock; ++i) h = mix64(h ^ static_cast<uint32_t>(tokens[i]));
  return mix64(h ^ extra);
}

struct Request {
  std::vector<int32_t> blocks;  // logical -> physical
  std::vector<uint64_t> chain;  // chained hashes of the leading full blocks
  int64_t num_tokens = 0;       // tokens the blocks were grown to hold
};

}  // namespace

struct pkv_block_manager {
  int64_t n;
  bool caching;
  std::vector<int32_t> ref;
  std::vector<int64_t> prev, next;  // free-queue links; node n is the sentinel
  std::vector<uint8_t> in_free;
  std::vector<uint8_t> cached;
  std::vector<uint64_t> hash;
  std::vector<std::vector<int32_t>> cached_tokens;
  std::unordered_map<uint64_t, int32_t> by_hash;
  std::unordered_map<int64_t, Request> reqs;
  int64_t num_free = 0;

  explicit pkv_block_manager(int64_t num_blocks, bool enable_cache)
      : n(num_blocks), caching(enable_cache), ref(num_blocks, 0), prev(num_blocks + 1), next(num_blocks + 1),
        in_free(num_blocks, 0), cached(num_blocks, 0), hash(num_blocks, 0), cached_tokens(num_blocks) {
    prev[n] = next[n] = n;
    for (int64_t b = 0; b < n; ++b) push_back(b);
  }

  void push_back(int64_t b) {
    const int64_t t = prev[n];
    next[t] = b;
    prev[b] = t;
    next[b] = n;
    prev[n] = b;
    in_free[b] = 1;
    ++num_free;
  }
  void unlink(int64_t b) {
    next[prev[b]] = next[b];
    prev[next[b]] = prev[b];
    in_free[b] = 0;
    --num_free;
  }
  void evict(int64_t b) {
    if (!cached[b]) return;
    auto it = by_hash.find(hash[b]);
    if (it != by_hash.end() && it->second == b) by_hash.erase(it);
    cached[b] = 0;
    cached_tokens[b].clear();
  }
  // Takes the block at the head of the free queue (evicting its cached hash).
  int32_t pop_front() {
    const int64_t b = next[n];
    unlink(b);
    evict(b);
    ref[b] = 1;
    return static_cast<int32_t>(b);
  }
};

extern "C" {

pkv_block_manager* pkv_bm_create(int64_t num_blocks, int32_t enable_prefix_cache) {
  if (num_blocks <= 0 || num_blocks >= (int64_t(1) << 31)) return nullptr;
  return new pkv_block_manager(num_blocks, enable_prefix_cache != 0);
}

void pkv_bm_destroy(pkv_block_manager* bm) { delete bm; }

int64_t pkv_bm_num_free(const pkv_block_manager* bm) { return bm ? bm->num_free : -3; }

uint64_t pkv_bm_block_hash(uint64_t parent_hash, const int32_t* tokens16, uint64_t extra_key) {
  return block_hash(parent_hash, tokens16, extra_key);
}

int32_t pkv_bm_get_computed_blocks(pkv_block_manager* bm, int64_t req, const int32_t* tokens, int64_t num_tokens) {
  if (!bm || num_tokens < 0 || (num_tokens > 0 && !tokens)) return -3;
  if (bm->reqs.count(req)) return -2;
  Request& r = bm->reqs[req];
  if (!bm->caching) return 0;
  uint64_t parent = 0;
  for (int64_t k = 0; (k + 1) * kBlock <= num_tokens; ++k) {
    const int32_t* blk = tokens + k * kBlock;
    const uint64_t h = block_hash(parent, blk, 0);
    auto it = bm->by_hash.find(h);
    if (it == bm->by_hash.end()) break;
    const int32_t b = it->second;
    if (std::memcmp(bm->cached_tokens[b].data(), blk, kBlock * sizeof(int32_t)) != 0) break;
    if (bm->in_free[b]) bm->unlink(b);  // a cached-but-free block comes back to life
    ++bm->ref[b];
    r.blocks.push_back(b);
    r.chain.push_back(h);
    parent = h;
  }
  r.num_tokens = static_cast<int64_t>(r.blocks.size()) * kBlock;
  return static_cast<int32_t>(r.blocks.size());
}

int32_t pkv_bm_allocate_slots(pkv_block_manager* bm, int64_t req, int64_t total_tokens) {
  if (!bm || total_tokens < 0) return -3;
  auto it = bm->reqs.find(req);
  if (it == bm->reqs.end()) return -2;
  Request& r = it->second;
  const int64_t need = (total_tokens + kBlock - 1) / kBlock - static_cast<int64_t>(r.blocks.size());
  if (need > bm->num_free) return -1;  // None: the pool cannot cover the new tokens
  for (int64_t i = 0; i < need; ++i) r.blocks.push_back(bm->pop_front());
  if (total_tokens > r.num_tokens) r.num_tokens = total_tokens;
  return need > 0 ? static_cast<int32_t>(need) : 0;
}

int32_t pkv_bm_cache_full_blocks(pkv_block_manager* bm, int64_t req, const int32_t* tokens, int64_t num_tokens) {
  if (!bm || num_tokens < 0 || (num_tokens > 0 && !tokens)) return -3;
  auto it = bm->reqs.find(req);
  if (it == bm->reqs.end()) return -2;
  if (!bm->caching) return 0;
  Request& r = it->second;
  int32_t added = 0;
  const int64_t full = num_tokens / kBlock;
  for (int64_t k = static_cast<int64_t>(r.chain.size()); k < full && k < static_cast<int64_t>(r.blocks.size());
       ++k) {
    const int32_t* blk = tokens + k * kBlock;
    const uint64_t h = block_hash(r.chain.empty() ? 0 : r.chain.back(), blk, 0);
    const int32_t b = r.blocks[k];
    if (!bm->by_hash.count(h) && !bm->cached[b]) {
      bm->by_hash[h] = b;
      bm->cached[b] = 1;
      bm->hash[b] = h;
      bm->cached_tokens[b].assign(blk, blk + kBlock);
      ++added;
    }
    r.chain.push_back(h);
  }
  return added;
}

int32_t pkv_bm_block_table(const pkv_block_manager* bm, int64_t req, int32_t* out, int32_t max_out) {
  if (!bm || max_out < 0) return -3;
  auto it = bm->reqs.find(req);
  if (it == bm->reqs.end()) return -2;
  const auto& v = it->second.blocks;
  const int32_t n = static_cast<int32_t>(v.size());
  if (out)
    for (int32_t i = 0; i < n && i < max_out; ++i) out[i] = v[i];
  return n;
}

int32_t pkv_bm_free(pkv_block_manager* bm, int64_t req) {
  if (!bm) return -3;
  auto it = bm->reqs.find(req);
  if (it == bm->reqs.end()) return -2;
  const auto& v = it->second.blocks;
  for (auto b = v.rbegin(); b != v.rend(); ++b)  // tail blocks first: they are evicted first
    if (--bm->ref[*b] == 0) bm->push_back(*b);
  bm->reqs.erase(it);
  return 0;
}

int32_t pkv_bm_fork(pkv_block_manager* bm, int64_t parent, int64_t child) {
  if (!bm) return -3;
  auto it = bm->reqs.find(parent);
  if (it == bm->reqs.end() || bm->reqs.count(child)) return -2;
  Request r = it->second;
  for (int32_t b : r.blocks) ++bm->ref[b];
  bm->reqs[child] = r;
  return 0;
}

int32_t pkv_bm_cow(pkv_block_manager* bm, int64_t req, int32_t logical_block, int32_t* src, int32_t* dst) {
  if (!bm || !src || !dst) return -3;
  auto it = bm->reqs.find(req);
  if (it == bm->reqs.end()) return -2;
  Request& r = it->second;
  if (logical_block < 0 || logical_block >= static_cast<int32_t>(r.blocks.size())) return -3;
  const int32_t old = r.blocks[logical_block];
  if (bm->ref[old] <= 1) return 0;
  if (bm->num_free == 0) return -1;
  const int32_t fresh = bm->pop_front();
  --bm->ref[old];
  r.blocks[logical_block] = fresh;
  // the copy will diverge: its hash chain from this block on is no longer known
  if (static_cast<int32_t>(r.chain.size()) > logical_block) r.chain.resize(logical_block);
  *src = old;
  *dst = fresh;
  return 1;
}

int32_t pkv_bm_prefix_groups(const pkv_block_manager* bm, const int64_t* reqs, int32_t n, int32_t max_prefix_blocks,
                             int32_t max_groups, int32_t* prefix_tables, int32_t* prefix_num_blocks,
                             int32_t* member_start, int32_t* member_seqs) {
  if (!bm || n < 0 || (n > 0 && !reqs) || max_prefix_blocks < 1 || max_groups < 0 || !member_start) return -3;
  if (max_groups > 0 && (!prefix_tables || !prefix_num_blocks || (n > 0 && !member_seqs))) return -3;
  std::vector<const std::vector<int32_t>*> tab(static_cast<size_t>(n));
  for (int32_t k = 0; k < n; ++k) {
    auto it = bm->reqs.find(reqs[k]);
    if (it == bm->reqs.end()) return -2;
    tab[k] = &it->second.blocks;
  }
  // requests by first block, in batch order of each group's first member
  std::unordered_map<int32_t, int32_t> group_of;
  std::vector<std::vector<int32_t>> groups;
  for (int32_t k = 0; k < n; ++k) {
    if (tab[k]->empty()) continue;
    auto ins = group_of.emplace((*tab[k])[0], static_cast<int32_t>(groups.size()));
    if (ins.second) groups.emplace_back();
    groups[ins.first->second].push_back(k);
  }
  int32_t ng = 0, nm = 0;
  member_start[0] = 0;
  for (const auto& members : groups) {
    if (members.size() < 2 || ng == max_groups) continue;
    const std::vector<int32_t>& lead = *tab[members[0]];
    size_t lcp = std::min(lead.size(), static_cast<size_t>(max_prefix_blocks));
    for (size_t m = 1; m < members.size(); ++m) {
      const std::vector<int32_t>& t = *tab[members[m]];
      size_t j = 0;
      while (j < lcp && j < t.size() && t[j] == lead[j]) ++j;
      lcp = j;
    }
    if (lcp == 0) continue;
    for (size_t j = 0; j < static_cast<size_t>(max_prefix_blocks); ++j)
      prefix_tables[static_cast<size_t>(ng) * max_prefix_blocks + j] = j < lcp ? lead[j] : -1;
    prefix_num_blocks[ng] = static_cast<int32_t>(lcp);
    for (int32_t k : members) member_seqs[nm++] = k;
    member_start[++ng] = nm;
  }
  return ng;
}

int32_t pkv_bm_usage(const pkv_block_manager* bm, int64_t* blocks_in_use, int64_t* tokens_held,
                     int64_t* unused_slots) {
  if (!bm || !blocks_in_use || !tokens_held || !unused_slots) return -3;
  int64_t tokens = 0, unused = 0;
  for (const auto& kv : bm->reqs) {
    tokens += kv.second.num_tokens;
    unused += static_cast<int64_t>(kv.second.blocks.size()) * kBlock - kv.second.num_tokens;
  }
  *blocks_in_use = bm->n - bm->num_free;
  *tokens_held = tokens;
  *unused_slots = unused;
  return 0;
}

}  // extern "C"
