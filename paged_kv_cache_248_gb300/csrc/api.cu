// api.cu -- the C ABI of libpkv: host-side argument checks, per-device context
// (error word, workspace), tensor-map encoding, launch tracing, and dispatch to
// the kernels.  Every compute step runs on the GPU; nothing here touches tensor data.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdlib>
#include <mutex>
#include <vector>

#include "pkv_internal.cuh"
#include "k_generic.cuh"

namespace pkv {

// ------------------------------------------------------------------ status helpers
int cuda_status(cudaError_t e) { return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA; }

namespace {
std::mutex g_mu;
constexpr int kMaxDevices = 64;
DeviceCtx g_ctx[kMaxDevices];
bool g_ctx_ready[kMaxDevices] = {};
}  // namespace

DeviceCtx* device_ctx(int* status) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    *status = PKV_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_ctx_ready[dev]) {
    DeviceCtx& c = g_ctx[dev];
    c.device = dev;
    if (cudaDeviceGetAttribute(&c.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      *status = PKV_ERR_CUDA;
      return nullptr;
    }
    void* p = nullptr;
    if (cudaMalloc(&p, 256) != cudaSuccess) {
      *status = PKV_ERR_NO_MEMORY;
      return nullptr;
    }
    if (cudaMemset(p, 0, 256) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess) {
      cudaFree(p);
      *status = PKV_ERR_CUDA;
      return nullptr;
    }
    c.err = static_cast<uint32_t*>(p);
    g_ctx_ready[dev] = true;
  }
  return &g_ctx[dev];
}

int ensure_workspace(DeviceCtx* ctx, size_t bytes, cudaStream_t stream) {
  if (ctx->ws_bytes >= bytes) return PKV_OK;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return PKV_ERR_CUDA;
  if (cap != cudaStreamCaptureStatusNone) return PKV_ERR_NO_MEMORY;  // never allocate while capturing
  size_t want = ctx->ws_bytes ? ctx->ws_bytes : (1u << 20);
  while (want < bytes) want *= 2;
  if (ctx->ws) {
    if (cudaFree(ctx->ws) != cudaSuccess) return PKV_ERR_CUDA;  // device-wide sync: no kernel still reads it
    ctx->ws = nullptr;
    ctx->ws_bytes = 0;
  }
  if (cudaMalloc(&ctx->ws, want) != cudaSuccess) {
    ctx->ws = nullptr;
    return PKV_ERR_NO_MEMORY;
  }
  ctx->ws_bytes = want;
  return PKV_OK;
}

size_t layout_workspace(void* base, int32_t num_seqs, int32_t hkv, int32_t group, int32_t head_dim,
                        int64_t max_dec_items, int64_t max_pre_units, Workspace* ws, const CascadeArgs* cas) {
  size_t off = 0;
  auto take = [&](size_t bytes) -> void* {
    void* p = base ? static_cast<char*>(base) + off : nullptr;
    off += (bytes + 255) & ~static_cast<size_t>(255);
    return p;
  };
  Workspace w{};
  w.counters = static_cast<int32_t*>(take(kNumQueueCounters * sizeof(int32_t)));
  w.dec_prefix = static_cast<int32_t*>(take((static_cast<size_t>(num_seqs) + 1) * sizeof(int32_t)));
  w.pre_prefix = static_cast<int32_t*>(take((static_cast<size_t>(num_seqs) + 1) * sizeof(int32_t)));
  w.pre_order = static_cast<int32_t*>(take(static_cast<size_t>(max_pre_units) * 2 * sizeof(int32_t)));
  w.dec_order = static_cast<int32_t*>(take(static_cast<size_t>(num_seqs) * sizeof(int32_t)));
  w.dec_start = static_cast<int32_t*>(take((static_cast<size_t>(num_seqs) + 1) * sizeof(int32_t)));
  w.dec_pos = static_cast<int32_t*>(take(static_cast<size_t>(2 * kDecPosMax) * sizeof(int32_t)));
  w.unit_bad = static_cast<int32_t*>(take(static_cast<size_t>(num_seqs) * hkv * sizeof(int32_t)));
  w.merge_list = static_cast<int32_t*>(take(static_cast<size_t>(num_seqs) * 8 * sizeof(int32_t)));
  w.part_ml = static_cast<float*>(take(static_cast<size_t>(max_dec_items) * group * 2 * sizeof(float)));
  w.part_o = static_cast<float*>(take(static_cast<size_t>(max_dec_items) * group * head_dim * sizeof(float)));
  if (cas && cas->num_groups > 0 && cas->num_members > 0) {
    const size_t nm = static_cast<size_t>(cas->num_members);
    w.cas_np_max = static_cast<int32_t>(cascade_splits(static_cast<int64_t>(cas->max_blocks) * kBlock));
    const size_t slots = nm * hkv * w.cas_np_max;
    w.seq_prefix = static_cast<int32_t*>(take(static_cast<size_t>(num_seqs) * sizeof(int32_t)));
    w.seq_entry = static_cast<int32_t*>(take(static_cast<size_t>(num_seqs) * sizeof(int32_t)));
    w.member_ok = static_cast<int32_t*>(take(nm * sizeof(int32_t)));
    w.cas_prefix = static_cast<int32_t*>(take((static_cast<size_t>(cas->num_groups) + 1) * sizeof(int32_t)));
    w.grp_ok = static_cast<int32_t*>(take(static_cast<size_t>(cas->num_groups) * sizeof(int32_t)));
    w.blk_mark = static_cast<int32_t*>(take(static_cast<size_t>(cas->pool_blocks) * sizeof(int32_t)));
    w.cas_ml = static_cast<float*>(take(slots * group * 2 * sizeof(float)));
    w.cas_o = static_cast<float*>(take(slots * group * head_dim * sizeof(float)));
  }
  if (ws) *ws = w;
  return off;
}

// ------------------------------------------------------------------ tensor maps
namespace {
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

// The maps the last calls of this host thread encoded, by everything that goes into
// one: a step reuses its pools and usually its q buffer, so most launches find their
// map here instead of calling the driver's encoder.
struct MapKey {
  const void* base;
  uint64_t dims[3], strides[2];
  uint32_t box[3], rank;
  bool operator==(const MapKey& o) const {
    return base == o.base && rank == o.rank && dims[0] == o.dims[0] && dims[1] == o.dims[1] &&
           dims[2] == o.dims[2] && strides[0] == o.strides[0] && strides[1] == o.strides[1] &&
           box[0] == o.box[0] && box[1] == o.box[1] && box[2] == o.box[2];
  }
};
constexpr int kMapCacheSlots = 16;
struct MapCache {
  MapKey key[kMapCacheSlots];
  CUtensorMap map[kMapCacheSlots];
  int used = 0, next = 0;
};
thread_local MapCache t_maps;

int encode_tiled(CUtensorMap* map, const MapKey& k) {
  for (int i = 0; i < t_maps.used; ++i) {
    if (t_maps.key[i] == k) {
      *map = t_maps.map[i];
      return PKV_OK;
    }
  }
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return PKV_ERR_CUDA;
  const cuuint64_t dims[3] = {k.dims[0], k.dims[1], k.dims[2]};
  const cuuint64_t strides[2] = {k.strides[0], k.strides[1]};
  const cuuint32_t box[3] = {k.box[0], k.box[1], k.box[2]};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, k.rank, const_cast<void*>(k.base), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return PKV_ERR_INVALID_ARG;
  const int slot = t_maps.next;
  t_maps.key[slot] = k;
  t_maps.map[slot] = *map;
  t_maps.next = (slot + 1) % kMapCacheSlots;
  if (t_maps.used < kMapCacheSlots) ++t_maps.used;
  return PKV_OK;
}
}  // namespace

int encode_tensor_map_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                         uint32_t box_inner, uint32_t box_outer) {
  const MapKey k{base, {inner, outer, 0}, {row_bytes, 0}, {box_inner, box_outer, 0}, 2};
  return encode_tiled(map, k);
}

int encode_tensor_map_3d(CUtensorMap* map, const void* base, const uint64_t dims_in[3], const uint64_t strides_in[2],
                         const uint32_t box_in[3]) {
  const MapKey k{base,
                 {dims_in[0], dims_in[1], dims_in[2]},
                 {strides_in[0], strides_in[1]},
                 {box_in[0], box_in[1], box_in[2]},
                 3};
  return encode_tiled(map, k);
}

bool pdl_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("PKV_PDL");
    return !(v && v[0] == '0' && v[1] == '\0');
  }();
  return on;
}

// Opt-in to more than 48 KB of dynamic shared memory, once per device and kernel.
int set_smem_once(const void* kernel, int bytes, uint64_t* done_mask) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PKV_ERR_CUDA;
  const uint64_t bit = uint64_t(1) << dev;
  if (__atomic_load_n(done_mask, __ATOMIC_ACQUIRE) & bit) return PKV_OK;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess)
    return PKV_ERR_CUDA;
  __atomic_fetch_or(done_mask, bit, __ATOMIC_RELEASE);
  return PKV_OK;
}

// ------------------------------------------------------------------ tracing
namespace {
constexpr int kTraceSlots = 8192;
bool g_trace_on = false;
int g_trace_device = -1;
std::vector<cudaEvent_t> g_ev_start, g_ev_stop;
std::vector<int> g_pending_kind;  // kind per used slot
int64_t g_launches[PKV_TRACE_KINDS] = {};
double g_ms[PKV_TRACE_KINDS] = {};
const char* kTraceNames[PKV_TRACE_KINDS] = {"slot_mapping", "write", "copy_blocks", "plan",
                                            "decode", "prefill", "generic_attention", "merge",
                                            "cascade"};
}  // namespace

TraceScope::TraceScope(int k, cudaStream_t s) : kind(k), stream(s), slot(-1) {
  if (!g_trace_on) return;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev != g_trace_device) return;
  std::lock_guard<std::mutex> lock(g_mu);
  if (static_cast<int>(g_pending_kind.size()) >= kTraceSlots) return;
  slot = static_cast<int>(g_pending_kind.size());
  g_pending_kind.push_back(kind);
  cudaEventRecord(g_ev_start[slot], stream);
}
TraceScope::~TraceScope() {
  if (slot >= 0) cudaEventRecord(g_ev_stop[slot], stream);
}

}  // namespace pkv

using namespace pkv;

// ------------------------------------------------------------------ argument checks
namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_cache(const pkv_cache_desc* c) {
  if (!c) return PKV_ERR_INVALID_ARG;
  if (c->block_size != PKV_BLOCK_SIZE || c->num_blocks <= 0 || c->num_kv_heads <= 0 || c->head_dim <= 0)
    return PKV_ERR_INVALID_ARG;
  if (c->num_blocks > (int64_t(1) << 40)) return PKV_ERR_INVALID_ARG;
  if (c->dtype == PKV_F32 && (c->head_dim == 64 || c->head_dim == 128)) return PKV_OK;
  if (c->dtype == PKV_BF16 && c->head_dim == 128) return PKV_OK;
  return PKV_ERR_UNSUPPORTED;
}

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

}  // namespace

extern "C" {

int pkv_slot_mapping(const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                     const int32_t* query_start_loc, int32_t num_seqs, int64_t num_tokens, int64_t* slot_mapping,
                     void* stream) {
  if (num_tokens < 0 || num_seqs < 0) return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (num_seqs == 0 || max_blocks_per_seq <= 0 || !block_tables || !seq_lens || !query_start_loc ||
      !slot_mapping)
    return PKV_ERR_INVALID_ARG;
  int st = PKV_OK;
  DeviceCtx* ctx = device_ctx(&st);
  if (!ctx) return st;
  return launch_slot_mapping(block_tables, max_blocks_per_seq, seq_lens, query_start_loc, num_seqs, num_tokens,
                             slot_mapping, ctx->err, as_stream(stream));
}

int pkv_write(const void* k, const void* v, const int64_t* slot_mapping, int64_t num_tokens, void* k_cache,
              void* v_cache, const pkv_cache_desc* cache, void* stream) {
  int st = check_cache(cache);
  if (st) return st;
  if (num_tokens < 0) return PKV_ERR_INVALID_ARG;
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PKV_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_INVALID_ARG;
  DeviceCtx* ctx = device_ctx(&st);
  if (!ctx) return st;
  return launch_write(k, v, slot_mapping, num_tokens, k_cache, v_cache, *cache, ctx->err, as_stream(stream));
}

int pkv_copy_blocks(const int32_t* src, const int32_t* dst, int64_t n, void* k_cache, void* v_cache,
                    const pkv_cache_desc* cache, void* stream) {
  int st = check_cache(cache);
  if (st) return st;
  if (n < 0) return PKV_ERR_INVALID_ARG;
  if (n == 0) return PKV_OK;
  if (!src || !dst || !k_cache || !v_cache || !aligned16(k_cache) || !aligned16(v_cache))
    return PKV_ERR_INVALID_ARG;
  DeviceCtx* ctx = device_ctx(&st);
  if (!ctx) return st;
  return launch_copy_blocks(src, dst, n, k_cache, v_cache, *cache, ctx->err, as_stream(stream));
}

}  // extern "C"

namespace {

// The writer CTAs of a planning launch: new tokens' K/V rows into their slots (a warp per
// 64-vector piece of a token's rows, at most two CTAs per SM).
void set_writers(PlanArgs& p, const void* k_new, const void* v_new, const void* k_cache, const void* v_cache,
                 const pkv_cache_desc& cache, int64_t* slots_out, int64_t num_tokens, int num_sms) {
  const int64_t warps_per_cta = 1024 / 32;
  const int elem = cache.dtype == PKV_F32 ? 4 : 2;
  const int64_t pieces = (cache.num_kv_heads * (cache.head_dim * elem / 16) + 63) / 64;
  const int64_t want = (num_tokens * pieces + warps_per_cta - 1) / warps_per_cta;
  p.k_new = static_cast<const uint4*>(k_new);
  p.v_new = static_cast<const uint4*>(v_new);
  p.k_cache = static_cast<uint4*>(const_cast<void*>(k_cache));
  p.v_cache = static_cast<uint4*>(const_cast<void*>(v_cache));
  p.slots_out = slots_out;
  p.num_slots = cache.num_blocks * kBlock;
  p.vec_per_row = cache.head_dim * elem / 16;
  p.write_ctas = static_cast<int32_t>(want < 2 * num_sms ? want : 2 * num_sms);
}

// paged_attention, paged_attention_cascade, paged_attention_step and
// paged_attention_step_cow: `groups` null = no shared prefixes; `k_new` null = no new
// tokens to write first; num_cow > 0 = copy those blocks (as pkv_copy_blocks) before
// anything else.
int attention_impl(const void* q, const void* k_new, const void* v_new, const void* k_cache, const void* v_cache,
                   const pkv_cache_desc* cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                   const int32_t* seq_lens, const int32_t* query_start_loc, int32_t num_seqs, int32_t num_q_heads,
                   int64_t num_tokens, int32_t max_query_len, int32_t max_seq_len, float scale,
                   const pkv_prefix_groups* groups, int64_t* slots_out, void* out, void* stream,
                   const int32_t* cow_src = nullptr, const int32_t* cow_dst = nullptr, int64_t num_cow = 0) {
  int st = check_cache(cache);
  if (st) return st;
  if (num_cow < 0 || (num_cow > 0 && (!cow_src || !cow_dst))) return PKV_ERR_INVALID_ARG;
  const bool write = k_new != nullptr;
  if (write && (!v_new || !aligned16(k_new) || !aligned16(v_new))) return PKV_ERR_INVALID_ARG;
  if (num_tokens < 0 || num_seqs < 0 || num_q_heads <= 0 || num_q_heads % cache->num_kv_heads != 0)
    return PKV_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return PKV_ERR_INVALID_ARG;
  CascadeArgs cas{};
  if (groups) {
    if (groups->num_groups < 0 || groups->num_members < 0) return PKV_ERR_INVALID_ARG;
    if (groups->num_groups > 0 && groups->num_members > 0) {
      if (!groups->prefix_block_tables || !groups->prefix_num_blocks || !groups->member_start ||
          !groups->member_seqs || groups->max_prefix_blocks < 1)
        return PKV_ERR_INVALID_ARG;
      cas = CascadeArgs{groups->prefix_block_tables, groups->max_prefix_blocks, groups->prefix_num_blocks,
                        groups->member_start,        groups->member_seqs,       groups->num_groups,
                        groups->num_members};
    }
  }
  if (num_tokens == 0) {  // nothing to attend; the copies (if any) still happen
    if (num_cow == 0) return PKV_OK;
    if (!k_cache || !v_cache || !aligned16(k_cache) || !aligned16(v_cache)) return PKV_ERR_INVALID_ARG;
    DeviceCtx* ctx = device_ctx(&st);
    if (!ctx) return st;
    return launch_copy_blocks(cow_src, cow_dst, num_cow, const_cast<void*>(k_cache), const_cast<void*>(v_cache),
                              *cache, ctx->err, as_stream(stream));
  }
  if (num_seqs == 0 || max_blocks_per_seq <= 0 || max_query_len <= 0 || max_seq_len <= 0) return PKV_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !query_start_loc || !out)
    return PKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return PKV_ERR_INVALID_ARG;
  if (cache->dtype == PKV_BF16) {  // sizes the tensor-core path cannot index, refused before any CUDA call
    const int32_t group = num_q_heads / cache->num_kv_heads;
    if (group > 16) return PKV_ERR_UNSUPPORTED;
    const int64_t splits = (static_cast<int64_t>(max_seq_len) + kSplitKeys - 1) / kSplitKeys;
    if (static_cast<int64_t>(num_seqs) * cache->num_kv_heads * splits >= (int64_t(1) << 31))
      return PKV_ERR_UNSUPPORTED;
  }
  DeviceCtx* ctx = device_ctx(&st);
  if (!ctx) return st;
  AttnArgs a{q,        k_cache,    v_cache,       *cache,      block_tables, max_blocks_per_seq, seq_lens,
             query_start_loc, num_seqs, num_q_heads, num_tokens, max_query_len, max_seq_len, scale, out};
  cudaStream_t s = as_stream(stream);
  if (num_cow > 0) {
    st = launch_copy_blocks(cow_src, cow_dst, num_cow, const_cast<void*>(k_cache), const_cast<void*>(v_cache), *cache,
                            ctx->err, s);
    if (st) return st;
  }
  if (cache->dtype == PKV_F32) {  // groups do not change results
    if (write && max_query_len == 1) {  // one new token a request: written by the attention launch itself
      const GenericWrite gw{k_new, v_new, slots_out};
      return launch_generic_attention_write(a, gw, ctx->err, s);
    }
    if (write) {  // slot mapping and scatter in the writer CTAs of a launch that plans nothing
      PlanArgs w{seq_lens, query_start_loc, num_seqs, num_tokens, cache->num_kv_heads, max_blocks_per_seq,
                 max_seq_len, kSplitKeys, 0, nullptr, nullptr, nullptr, nullptr, nullptr, ctx->err};
      w.bt = block_tables;
      w.writers_only = 1;
      set_writers(w, k_new, v_new, k_cache, v_cache, *cache, slots_out, num_tokens, ctx->num_sms);
      w.cow_dst = cow_dst;
      w.num_cow = num_cow;
      st = launch_plan(w, s);
      if (st) return st;
    }
    return launch_generic_attention(a, ctx->err, s);
  }
  // bf16, head_dim 128: tensor-core path
  const int32_t hkv = cache->num_kv_heads;
  const int32_t group = num_q_heads / hkv;
  if (group > 16) return PKV_ERR_UNSUPPORTED;
  const int32_t gp = group <= 4 ? 4 : (group <= 8 ? 8 : 16);
  const int64_t max_splits = (static_cast<int64_t>(max_seq_len) + kSplitKeys - 1) / kSplitKeys;
  const int64_t max_dec_items = static_cast<int64_t>(num_seqs) * hkv * max_splits;
  if (max_dec_items >= (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;
  if (cas.num_groups > 0) {
    const int64_t slots = static_cast<int64_t>(cas.num_members) * hkv *
                          cascade_splits(static_cast<int64_t>(cas.max_blocks) * kBlock);
    if (slots * gp >= (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;
  }
  cas.pool_blocks = cache->num_blocks;
  const CascadeArgs* casp = cas.num_groups > 0 ? &cas : nullptr;
  const int64_t max_pre_units = max_prefill_units(num_tokens, num_seqs, gp);
  const size_t need =
      layout_workspace(nullptr, num_seqs, hkv, gp, cache->head_dim, max_dec_items, max_pre_units, nullptr, casp);
  st = ensure_workspace(ctx, need, s);
  if (st) return st;
  Workspace ws;
  layout_workspace(ctx->ws, num_seqs, hkv, gp, cache->head_dim, max_dec_items, max_pre_units, &ws, casp);
  PlanArgs plan{seq_lens, query_start_loc, num_seqs, num_tokens, hkv, max_blocks_per_seq, max_seq_len,
                kSplitKeys, kPrefillTilesPerItem * (kTileKeys / gp), ws.counters, ws.dec_prefix, ws.pre_prefix, ws.unit_bad,
                ws.merge_list, ctx->err};
  plan.bt = block_tables;
  plan.pre_order = ws.pre_order;
  plan.max_pre_units = max_pre_units;
  plan.rows_q = kTileKeys / gp;
  plan.dec_order = ws.dec_order;
  plan.dec_start = ws.dec_start;
  plan.dec_pos = ws.dec_pos;
  plan.num_sms = ctx->num_sms;
  if (write) {
    set_writers(plan, k_new, v_new, k_cache, v_cache, *cache, slots_out, num_tokens, ctx->num_sms);
    plan.cow_dst = cow_dst;
    plan.num_cow = num_cow;
  }
  const int cas_tpi = casp ? cascade_tiles_per_item(cas.num_members, hkv, gp, cas.max_blocks, ctx->num_sms) : 1;
  // with few groups the cascade kernel finds its own items and runs beside the planner
  const int cas_concurrent = casp && cas.num_groups <= kCasConcurrentGroups ? 1 : 0;
  if (casp) {
    plan.cas = cas;
    plan.cas_rows = cas_tpi * (kTileKeys / gp);
    plan.seq_prefix = ws.seq_prefix;
    plan.seq_entry = ws.seq_entry;
    plan.member_ok = ws.member_ok;
    plan.cas_prefix = ws.cas_prefix;
    plan.grp_ok = ws.grp_ok;
    plan.blk_mark = ws.blk_mark;
    plan.num_blocks = cache->num_blocks;
    plan.cas_concurrent = cas_concurrent;
    // a fresh mark value per call (bit 30 set; the multiplier spreads consecutive calls)
    plan.epoch = static_cast<int32_t>(0x40000000u | ((++ctx->calls * 2654435761u) & 0x3FFFFFFFu));
  }
  st = launch_plan(plan, s);
  if (st) return st;
  if (casp) {
    st = launch_cascade_tc(a, cas, ws, ctx->num_sms, cas_tpi, cas_concurrent, ctx->err, s);
    if (st) return st;
  }
  if (max_query_len <= 1) return launch_decode_tc(a, ws, ctx->num_sms, ctx->err, s);
  // decode, then the prefill filling the decode's tail, then the split merge
  st = launch_decode_tc(a, ws, ctx->num_sms, ctx->err, s, kDecodeLaunch);
  if (st) return st;
  st = launch_prefill_tc(a, ws, ctx->num_sms, ctx->err, s, 1);
  if (st) return st;
  return launch_decode_tc(a, ws, ctx->num_sms, ctx->err, s, kMergeLaunch);
}

}  // namespace

extern "C" {

int paged_attention(const void* q, const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                    const int32_t* query_start_loc, int32_t num_seqs, int32_t num_q_heads, int64_t num_tokens,
                    int32_t max_query_len, int32_t max_seq_len, float scale, void* out, void* stream) {
  return attention_impl(q, nullptr, nullptr, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, seq_lens,
                        query_start_loc, num_seqs, num_q_heads, num_tokens, max_query_len, max_seq_len, scale,
                        nullptr, nullptr, out, stream);
}

int paged_attention_cascade(const void* q, const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
                            const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* seq_lens,
                            const int32_t* query_start_loc, int32_t num_seqs, int32_t num_q_heads,
                            int64_t num_tokens, int32_t max_query_len, int32_t max_seq_len, float scale,
                            const pkv_prefix_groups* groups, void* out, void* stream) {
  return attention_impl(q, nullptr, nullptr, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, seq_lens,
                        query_start_loc, num_seqs, num_q_heads, num_tokens, max_query_len, max_seq_len, scale,
                        groups, nullptr, out, stream);
}

int paged_attention_step(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                         const pkv_cache_desc* cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                         const int32_t* seq_lens, const int32_t* query_start_loc, int32_t num_seqs,
                         int32_t num_q_heads, int64_t num_tokens, int32_t max_query_len, int32_t max_seq_len,
                         float scale, const pkv_prefix_groups* groups, int64_t* slot_mapping, void* out,
                         void* stream) {
  if (!k_new || !v_new) return PKV_ERR_INVALID_ARG;
  return attention_impl(q, k_new, v_new, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, seq_lens,
                        query_start_loc, num_seqs, num_q_heads, num_tokens, max_query_len, max_seq_len, scale,
                        groups, slot_mapping, out, stream);
}

int paged_attention_step_cow(const void* q, const void* k_new, const void* v_new, void* k_cache, void* v_cache,
                             const pkv_cache_desc* cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                             const int32_t* seq_lens, const int32_t* query_start_loc, int32_t num_seqs,
                             int32_t num_q_heads, int64_t num_tokens, int32_t max_query_len, int32_t max_seq_len,
                             float scale, const pkv_prefix_groups* groups, const int32_t* cow_src,
                             const int32_t* cow_dst, int64_t num_cow, int64_t* slot_mapping, void* out,
                             void* stream) {
  if (!k_new || !v_new) return PKV_ERR_INVALID_ARG;
  return attention_impl(q, k_new, v_new, k_cache, v_cache, cache, block_tables, max_blocks_per_seq, seq_lens,
                        query_start_loc, num_seqs, num_q_heads, num_tokens, max_query_len, max_seq_len, scale,
                        groups, slot_mapping, out, stream, cow_src, cow_dst, num_cow);
}

int pkv_peek_error_bits(void* stream, uint32_t* bits) {
  if (!bits) return PKV_ERR_INVALID_ARG;
  int st = PKV_OK;
  DeviceCtx* ctx = device_ctx(&st);
  if (!ctx) return st;
  if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return PKV_ERR_CUDA;
  if (cudaMemcpy(bits, ctx->err, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess) return PKV_ERR_CUDA;
  return PKV_OK;
}

int pkv_get_last_error(void* stream) {
  uint32_t bits = 0;
  int st = pkv_peek_error_bits(stream, &bits);
  if (st) return st;
  int dummy = PKV_OK;
  DeviceCtx* ctx = device_ctx(&dummy);
  if (cudaMemset(ctx->err, 0, sizeof(uint32_t)) != cudaSuccess || cudaDeviceSynchronize() != cudaSuccess)
    return PKV_ERR_CUDA;
  if (bits & kErrTimeout) return PKV_ERR_TIMEOUT;
  if (bits) return PKV_ERR_INDEX;
  return PKV_OK;
}

const char* pkv_status_string(int status) {
  switch (status) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_INVALID_ARG: return "PKV_ERR_INVALID_ARG";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED";
    case PKV_ERR_INDEX: return "PKV_ERR_INDEX";
    case PKV_ERR_CUDA: return "PKV_ERR_CUDA";
    case PKV_ERR_NO_MEMORY: return "PKV_ERR_NO_MEMORY";
    case PKV_ERR_TIMEOUT: return "PKV_ERR_TIMEOUT";
    default: return "PKV_ERR_UNKNOWN";
  }
}

int pkv_num_workers(int32_t* workers) {
  if (!workers) return PKV_ERR_INVALID_ARG;
  int st = PKV_OK;
  DeviceCtx* ctx = device_ctx(&st);
  if (!ctx) return st;
  *workers = ctx->num_sms;
  return PKV_OK;
}

void pkv_shutdown(void) {
  std::lock_guard<std::mutex> lock(g_mu);
  int prev = 0;
  cudaGetDevice(&prev);
  for (int d = 0; d < kMaxDevices; ++d) {
    if (!g_ctx_ready[d]) continue;
    cudaSetDevice(d);
    cudaDeviceSynchronize();
    if (g_ctx[d].ws) cudaFree(g_ctx[d].ws);
    if (g_ctx[d].err) cudaFree(g_ctx[d].err);
    g_ctx[d] = DeviceCtx{};
    g_ctx_ready[d] = false;
  }
  cudaSetDevice(prev);
}

int pkv_trace_enable(int on) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (on) {
    if (g_ev_start.empty() || g_trace_device != dev) {
      for (auto e : g_ev_start) cudaEventDestroy(e);
      for (auto e : g_ev_stop) cudaEventDestroy(e);
      g_ev_start.assign(kTraceSlots, nullptr);
      g_ev_stop.assign(kTraceSlots, nullptr);
      for (int i = 0; i < kTraceSlots; ++i) {
        if (cudaEventCreate(&g_ev_start[i]) != cudaSuccess || cudaEventCreate(&g_ev_stop[i]) != cudaSuccess)
          return PKV_ERR_CUDA;
      }
    }
    g_trace_device = dev;
    g_pending_kind.clear();
    for (int k = 0; k < PKV_TRACE_KINDS; ++k) {
      g_launches[k] = 0;
      g_ms[k] = 0.0;
    }
  }
  g_trace_on = on != 0;
  return PKV_OK;
}

int pkv_trace_read(int64_t* launches, double* total_ms) {
  if (!launches || !total_ms) return PKV_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) return PKV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  for (size_t i = 0; i < g_pending_kind.size(); ++i) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, g_ev_start[i], g_ev_stop[i]) != cudaSuccess) return PKV_ERR_CUDA;
    g_launches[g_pending_kind[i]] += 1;
    g_ms[g_pending_kind[i]] += ms;
  }
  g_pending_kind.clear();
  for (int k = 0; k < PKV_TRACE_KINDS; ++k) {
    launches[k] = g_launches[k];
    total_ms[k] = g_ms[k];
    g_launches[k] = 0;
    g_ms[k] = 0.0;
  }
  return PKV_OK;
}

const char* pkv_trace_kind_name(int kind) {
  if (kind < 0 || kind >= PKV_TRACE_KINDS) return "unknown";
  return kTraceNames[kind];
}

int pkv_umma_selftest(const int32_t* params, const void* a_img, const void* b_img, float* d_out, void* stream) {
  if (!params || !a_img || !b_img || !d_out) return PKV_ERR_INVALID_ARG;
  if (!aligned16(a_img) || !aligned16(b_img)) return PKV_ERR_INVALID_ARG;
  int st = PKV_OK;
  DeviceCtx* ctx = device_ctx(&st);
  if (!ctx) return st;
  return run_umma_selftest(params, a_img, b_img, d_out, ctx->err, as_stream(stream));
}

int pkv_tma_selftest(const void* src, int64_t rows, int32_t row0, void* dump, void* stream) {
  if (!src || !dump || !aligned16(src) || !aligned16(dump)) return PKV_ERR_INVALID_ARG;
  int st = PKV_OK;
  DeviceCtx* ctx = device_ctx(&st);
  if (!ctx) return st;
  return run_tma_selftest(src, rows, row0, dump, ctx->err, as_stream(stream));
}

int pkv_wait_selftest(void* stream) {
  int st = PKV_OK;
  DeviceCtx* ctx = device_ctx(&st);
  if (!ctx) return st;
  return run_wait_selftest(ctx->err, as_stream(stream));
}

}  // extern "C"
