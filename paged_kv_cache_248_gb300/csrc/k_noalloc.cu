// k_noalloc.cu -- paged_attention_noalloc: the bf16 tensor-core attention path with
// its scratch memory in a fixed-size static device array instead of a workspace
// allocated on demand.
//
// Who needs this.  paged_attention() grows a device workspace with cudaMalloc the
// first time a batch needs more split-KV scratch than it has.  Some callers cannot
// let a library allocate: a serving process whose pooled or custom allocator must
// account for every byte of device memory (memory taken behind its back can make
// its own later allocations fail at the worst moment), and deployments that reserve
// all device memory at start-up and allow no allocation afterwards.  This entry
// point gives them the same attention with scratch that exists from the moment the
// library is loaded.
//
// The scratch is g_noalloc_scratch below: kNoAllocScratchBytes (16 MiB) of device
// memory that every GPU which loads the library holds until the process exits.  A
// batch whose scratch need is larger is rejected with PKV_ERR_NO_MEMORY before
// anything is launched.  Host code cannot use the array's name as a device pointer,
// so the first call on each device looks its address up with cudaGetSymbolAddress
// (with that device current) and caches it; make that first call before any stream
// capture.  Every call shares the one array and leaves its contents behind; the
// planning kernel re-zeroes the counters and flags each call needs, so nothing has
// to be cleared by the caller.  Calls whose kernels overlap on the GPU (different
// streams, or different host threads) race on the array and must be serialised by
// the caller.  Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <cmath>
#include <mutex>

#include "pkv_internal.cuh"

namespace pkv {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device
constexpr size_t kErrSlotBytes = 256;                       // fallback error word

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_setup_mu;
void* g_scratch_addr[kMaxDev] = {};
int g_sms[kMaxDev] = {};

// Once per device, with that device current: resolve the array's device address.
int setup_device(int dev, void** addr, int* sms) {
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return PKV_ERR_CUDA;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return PKV_ERR_CUDA;
    g_sms[dev] = n;
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  *sms = g_sms[dev];
  return PKV_OK;
}

bool is_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace pkv

using namespace pkv;

extern "C" PKV_API int paged_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                               const pkv_cache_desc* cache, const int32_t* block_tables,
                                               int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                               const int32_t* query_start_loc, int32_t num_seqs,
                                               int32_t num_q_heads, int64_t num_tokens, int32_t max_query_len,
                                               int32_t max_seq_len, float scale, void* out,
                                               uint32_t* error_bits, void* stream) {
  if (!cache || cache->block_size != PKV_BLOCK_SIZE || cache->num_blocks <= 0 || cache->num_kv_heads <= 0)
    return PKV_ERR_INVALID_ARG;
  if (cache->dtype != PKV_BF16 || cache->head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (num_tokens < 0 || num_seqs < 0 || num_q_heads <= 0 || num_q_heads % cache->num_kv_heads != 0)
    return PKV_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (num_seqs == 0 || max_blocks_per_seq <= 0 || max_query_len <= 0 || max_seq_len <= 0) return PKV_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !query_start_loc || !out) return PKV_ERR_INVALID_ARG;
  if (!is_aligned16(q) || !is_aligned16(k_cache) || !is_aligned16(v_cache) || !is_aligned16(out))
    return PKV_ERR_INVALID_ARG;
  const int32_t hkv = cache->num_kv_heads;
  const int32_t group = num_q_heads / hkv;
  if (group > 16) return PKV_ERR_UNSUPPORTED;

  // size check first: a batch that does not fit is refused before any CUDA call
  const int32_t gp = group <= 4 ? 4 : (group <= 8 ? 8 : 16);
  const int64_t max_splits = (static_cast<int64_t>(max_seq_len) + kSplitKeys - 1) / kSplitKeys;
  const int64_t max_dec_items = static_cast<int64_t>(num_seqs) * hkv * max_splits;
  if (max_dec_items >= (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;  // as paged_attention()
  const int64_t max_pre_units = max_prefill_units(num_tokens, num_seqs, gp);
  const size_t need = layout_workspace(nullptr, num_seqs, hkv, gp, cache->head_dim, max_dec_items, max_pre_units,
                                       nullptr);
  if (need > kNoAllocScratchBytes - kErrSlotBytes) return PKV_ERR_NO_MEMORY;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return PKV_ERR_CUDA;
  void* scratch = nullptr;
  int sms = 0;
  int st = setup_device(dev, &scratch, &sms);
  if (st) return st;
  uint32_t* err = error_bits ? error_bits : static_cast<uint32_t*>(scratch);
  Workspace ws;
  layout_workspace(static_cast<uint8_t*>(scratch) + kErrSlotBytes, num_seqs, hkv, gp, cache->head_dim,
                   max_dec_items, max_pre_units, &ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  AttnArgs a{q,        k_cache,    v_cache,       *cache,      block_tables, max_blocks_per_seq, seq_lens,
             query_start_loc, num_seqs, num_q_heads, num_tokens, max_query_len, max_seq_len, scale, out};
  PlanArgs plan{seq_lens, query_start_loc, num_seqs, num_tokens, hkv, max_blocks_per_seq, max_seq_len,
                kSplitKeys, kPrefillTilesPerItem * (kTileKeys / gp), ws.counters, ws.dec_prefix, ws.pre_prefix, ws.unit_bad,
                ws.merge_list, err};
  plan.pre_order = ws.pre_order;
  plan.max_pre_units = max_pre_units;
  plan.rows_q = kTileKeys / gp;
  plan.dec_order = ws.dec_order;
  plan.dec_start = ws.dec_start;
  plan.dec_pos = ws.dec_pos;
  plan.num_sms = sms;
  st = launch_plan(plan, s);
  if (st) return st;
  st = launch_decode_tc(a, ws, sms, err, s);
  if (st) return st;
  if (max_query_len > 1) st = launch_prefill_tc(a, ws, sms, err, s);
  return st;
}
