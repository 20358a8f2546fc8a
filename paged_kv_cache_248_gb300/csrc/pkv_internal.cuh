// pkv_internal.cuh -- definitions shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "pkv.h"

namespace pkv {

constexpr int kBlock = 16;  // tokens per KV block

// Device error word bits (pkv_peek_error_bits).
enum : uint32_t {
  kErrBlockId = 1u << 0,   // block id outside [0, num_blocks)
  kErrSlot = 1u << 1,      // slot past the pool
  kErrLength = 1u << 2,    // seq_len < q_len, or more blocks than a table row holds
  kErrTimeout = 1u << 3,   // a bounded wait gave up
};

constexpr int kTileKeys = 128;       // keys per tensor-core tile (8 blocks)
constexpr int kPrefillTilesPerItem = 2;  // query tiles of one prefill work item (sharing K/V)
constexpr int kSplitKeys = 2048;     // decode key-split length (a multiple of kTileKeys)
constexpr int kNoSplitKeys = 2048;   // decode contexts up to this length are never split

// Key splits of a decode request of context length L: a function of L alone, so
// a request's result does not depend on the rest of the batch.
__host__ __device__ inline int64_t decode_splits(int64_t L) {
  return L <= kNoSplitKeys ? 1 : (L + kSplitKeys - 1) / kSplitKeys;
}
constexpr int kNumQueueCounters = 8; // work-queue counters in the workspace
constexpr int kMergeCountSlot = 2;   // counters[2]: number of requests in the merge list
constexpr int kDecOrderSlot = 4;     // counters[4]: 1 when the decode items follow dec_order
// A decode batch the planner orders (at most 16 items per SM) also gets a direct map
// from queue position to (request, the request's first position); sized for GPUs of
// up to 256 SMs.
constexpr int kDecOrderMaxItemsPerSm = 16;
constexpr int kDecPosMax = kDecOrderMaxItemsPerSm * 256;

// Shared-prefix (cascade) key splits: a prefix of P tokens is attended in pieces of
// kCascadeSplitKeys keys, a function of P alone.
constexpr int kCascadeSplitKeys = 512;
__host__ __device__ inline int64_t cascade_splits(int64_t P) {
  return (P + kCascadeSplitKeys - 1) / kCascadeSplitKeys;
}

// Trace kinds (pkv_trace_read).
enum TraceKind : int {
  kTraceSlotMap = 0,
  kTraceWrite = 1,
  kTraceCopy = 2,
  kTracePlan = 3,
  kTraceDecode = 4,
  kTracePrefill = 5,
  kTraceGeneric = 6,
  kTraceMerge = 7,
  kTraceCascade = 8,
};

// Programmatic dependent launch.  Every library kernel is launched so that it may
// start while the kernel before it in the stream is still running (launch_k below).
// Each kernel therefore does only on-chip set-up (shared memory, barriers, TMEM,
// tensor-map prefetch) before grid_dep_wait(), which returns once the preceding
// grid has completed and its memory writes are visible; every CTA calls it before
// its first global-memory access and before any early exit, so that a kernel's
// completion always implies its predecessors'.  grid_dep_launch() then lets the
// next kernel's CTAs be scheduled as SMs free up.  Both are no-ops when the kernel
// was launched without the attribute.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void flag_error(uint32_t* err, uint32_t bits) {
  if (err != nullptr) atomicOr(err, bits);
}

template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static __device__ __forceinline__ float to_f32(float x) { return x; }
  static __device__ __forceinline__ float from_f32(float x) { return x; }
};
template <>
struct Elem<__nv_bfloat16> {
  static __device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }
  static __device__ __forceinline__ __nv_bfloat16 from_f32(float x) { return __float2bfloat16_rn(x); }
};

// Binary search: the request owning query token t (last i with qsl[i] <= t).
__device__ __forceinline__ int find_seq(const int32_t* __restrict__ qsl, int num_seqs, int64_t t) {
  int lo = 0, hi = num_seqs - 1;
  while (lo < hi) {
    int mid = lo + (hi - lo + 1) / 2;
    if (static_cast<int64_t>(__ldg(qsl + mid)) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace pkv

// ------------------------------------------------------------------ host side
namespace pkv {

struct DeviceCtx {
  int device = -1;
  int num_sms = 0;
  uint32_t* err = nullptr;     // device error word
  void* ws = nullptr;          // workspace
  size_t ws_bytes = 0;
  uint32_t calls = 0;          // calls with prefix groups so far: seeds each call's block-mark epoch
};

// Per-device context (created on first use on the current device).
DeviceCtx* device_ctx(int* status);
// Ensures the workspace holds at least `bytes`; refuses to grow during capture.
int ensure_workspace(DeviceCtx* ctx, size_t bytes, cudaStream_t stream);

// Tracing: bracket a launch with events when tracing is on.
struct TraceScope {
  int kind;
  cudaStream_t stream;
  int slot;
  TraceScope(int kind, cudaStream_t stream);
  ~TraceScope();
};

int cuda_status(cudaError_t e);

// Launchers implemented in the kernel translation units (return pkv_status).
int launch_slot_mapping(const int32_t* bt, int32_t max_blocks, const int32_t* seq_lens, const int32_t* qsl,
                        int32_t num_seqs, int64_t num_tokens, int64_t* slots, uint32_t* err, cudaStream_t s);
int launch_write(const void* k, const void* v, const int64_t* slots, int64_t T, void* kc, void* vc,
                 const pkv_cache_desc& c, uint32_t* err, cudaStream_t s);
int launch_copy_blocks(const int32_t* src, const int32_t* dst, int64_t n, void* kc, void* vc,
                       const pkv_cache_desc& c, uint32_t* err, cudaStream_t s);

struct AttnArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  pkv_cache_desc cache;
  const int32_t* block_tables;
  int32_t max_blocks;
  const int32_t* seq_lens;
  const int32_t* qsl;
  int32_t num_seqs;
  int32_t num_q_heads;
  int64_t num_tokens;
  int32_t max_query_len;
  int32_t max_seq_len;
  float scale;
  void* out;
};
// prefill_only: skip the rows of requests with exactly one query token.
int launch_generic_attention(const AttnArgs& a, uint32_t* err, cudaStream_t s, bool prefill_only = false);

// Per-call workspace carved from the library-owned device buffer.
struct Workspace {
  int32_t* counters;     // [kNumQueueCounters] work-queue heads
  int32_t* dec_prefix;   // [num_seqs + 1] exclusive prefix of decode items
  int32_t* pre_prefix;   // [num_seqs + 1] exclusive prefix of prefill items
  int32_t* pre_order;    // [2 * max_pre_units] prefill pairs, heaviest first: (pair id in request order, its request)
  int32_t* dec_order;    // [num_seqs] decode requests, largest item first (small batches)
  int32_t* dec_start;    // [num_seqs + 1] exclusive prefix of decode items in that order
  int32_t* dec_pos;      // [2 * kDecPosMax] per queue position of an ordered batch: (request, first position)
  int32_t* unit_bad;     // [num_seqs * hkv] a split saw a bad block id
  int32_t* merge_list;   // [num_seqs][8] decode requests cut into several splits: (request, its first
                         // item, splits, query row, prefix keys, member entry, 0, 0)
  float* part_ml;        // [max_dec_items * GP * 2] split running max and sum
  float* part_o;         // [max_dec_items * head_dim * GP] split accumulators
  // shared-prefix (cascade) state; all null without prefix groups
  int32_t* seq_prefix;   // [num_seqs] prefix tokens attended by the cascade kernel (0: none)
  int32_t* seq_entry;    // [num_seqs] the request's member-list entry (-1: none)
  int32_t* member_ok;    // [num_members] planner scratch (the global membership checks)
  int32_t* cas_prefix;   // [num_groups + 1] exclusive prefix of cascade work items
  int32_t* grp_ok;       // [num_groups] the group may admit members: its prefix ids are valid blocks
                         // that no new token of the call is written into
  int32_t* blk_mark;     // [pool blocks] a block is in some group's prefix iff it holds the call's epoch
  float* cas_ml;         // [num_members * hkv * cas_np_max * GP * 2] prefix partial max and sum
  float* cas_o;          // [num_members * hkv * cas_np_max * GP * head_dim] prefix accumulators
  int32_t cas_np_max;    // key splits of the longest prefix
};

// Shared-prefix groups of one call (the device arrays of pkv_prefix_groups).
struct CascadeArgs {
  const int32_t* tables;   // [num_groups][max_blocks] physical ids of each prefix
  int32_t max_blocks;
  const int32_t* blocks;   // [num_groups] prefix length in blocks
  const int32_t* start;    // [num_groups + 1] CSR offsets into members
  const int32_t* members;  // [num_members] request indices
  int32_t num_groups;
  int32_t num_members;
  int64_t pool_blocks = 0;  // blocks of the K/V pool (sizes the workspace's block marks)
};

// Computes the layout at `base` (nullptr: only the size) and returns the bytes needed;
// `group` is the padded head-group width GP the decode partials are stored with.
// `max_pre_units` bounds the prefill items' query-tile pairs.  With `cas`, also the
// shared-prefix arrays.
size_t layout_workspace(void* base, int32_t num_seqs, int32_t hkv, int32_t group, int32_t head_dim,
                        int64_t max_dec_items, int64_t max_pre_units, Workspace* ws,
                        const CascadeArgs* cas = nullptr);
// Query-tile pairs of the prefill items of a batch: at most one per 2R query tokens plus
// one per request (R = 128 / GP query tokens per tile).
inline int64_t max_prefill_units(int64_t num_tokens, int32_t num_seqs, int32_t gp) {
  return num_tokens / (kPrefillTilesPerItem * (kTileKeys / gp)) + num_seqs;
}

struct PlanArgs {
  const int32_t* seq_lens;
  const int32_t* qsl;
  int32_t num_seqs;
  int64_t num_tokens;
  int32_t hkv;
  int32_t max_blocks;
  int64_t max_seq_len;
  int32_t split_keys;
  int32_t rows_per_tile;  // query tokens per prefill item
  int32_t* counters;
  int32_t* dec_prefix;
  int32_t* pre_prefix;
  int32_t* unit_bad;
  int32_t* merge_list;
  uint32_t* err;
  // shared-prefix groups (cas.num_groups == 0: none)
  const int32_t* bt = nullptr;
  CascadeArgs cas{};
  int32_t cas_rows = 0;  // member requests per cascade item
  int32_t* pre_order = nullptr;  // heaviest-first order of the prefill pairs, two ints per position
  int32_t* dec_order = nullptr;  // largest-item-first order of the decode requests
  int32_t* dec_start = nullptr;
  int32_t* dec_pos = nullptr;
  int32_t num_sms = 0;
  int64_t max_pre_units = 0;
  int32_t rows_q = 0;            // query tokens per prefill tile
  int32_t* seq_prefix = nullptr;
  int32_t* seq_entry = nullptr;
  int32_t* member_ok = nullptr;
  int32_t* cas_prefix = nullptr;
  int32_t* grp_ok = nullptr;
  int32_t* blk_mark = nullptr;
  int64_t num_blocks = 0;
  int32_t epoch = 0;              // this call's block-mark value (bit 30 set, so stale small integers never match)
  int32_t cas_concurrent = 0;     // the cascade kernel runs beside this launch and reads prefix blocks while the
                                  //   writers write: a group is admitted only if no new token lands in its prefix
  // new tokens written by the same launch (k_new null: none): slot mapping and K/V scatter
  const uint4* k_new = nullptr;
  const uint4* v_new = nullptr;
  uint4* k_cache = nullptr;
  uint4* v_cache = nullptr;
  int64_t* slots_out = nullptr;  // optional
  int64_t num_slots = 0;         // num_blocks * 16
  int32_t vec_per_row = 0;       // 16-byte vectors per (token, kv head) row
  int32_t write_ctas = 0;        // CTAs after the planning CTA that do the writes
  // copy-on-write copies launched by the same call just before this launch (num_cow 0:
  // none).  Their kernel waited for everything before it, so the planner need not;
  // the writers wait for the copies and let the kernels after this one launch first
  const int32_t* cow_dst = nullptr;
  int64_t num_cow = 0;
  int32_t writers_only = 0;      // CTA 0 plans nothing (the fp32 path: only the writes)
  int32_t cas_onchip = 0;        // set by launch_plan: the membership checks run in shared memory
  int32_t ord_onchip = 0;        // set by launch_plan: the decode order is built in shared memory
  int32_t ord_offset = 0;        //   at this int offset of the planner's dynamic shared memory
};
// One launch: CTA 0 plans; CTAs 1..write_ctas (if any) map and scatter the new tokens.
int launch_plan(const PlanArgs& p, cudaStream_t s);
// `what`: kDecodeLaunch, kMergeLaunch or both (the split merge, when a context may be
// split, right after the decode kernel unless the caller puts another launch between).
enum : int { kDecodeLaunch = 1, kMergeLaunch = 2 };
int launch_decode_tc(const AttnArgs& a, const Workspace& ws, int num_sms, uint32_t* err, cudaStream_t s,
                     int what = kDecodeLaunch | kMergeLaunch);
// Attends the member decodes of every prefix group to the group's shared prefix,
// writing per-split partials for the merge (after launch_plan, before launch_decode_tc).
// Query tiles per cascade item: pairs (sharing each K/V tile) when they still give
// every SM an item, single tiles otherwise.  A function of the hint sizes only; how
// member rows are grouped into tiles does not change any row's result.
inline int cascade_tiles_per_item(int64_t num_members, int hkv, int gp, int64_t max_prefix_blocks, int num_sms) {
  const int64_t rows = kTileKeys / gp;
  const int64_t pairs = (num_members + 2 * rows - 1) / (2 * rows) * hkv * cascade_splits(max_prefix_blocks * kBlock);
  return pairs >= num_sms ? 2 : 1;
}
// With `concurrent` (at most kCasConcurrentGroups groups) the kernel derives its items
// from the hint alone and waits for the planning launch only before it exits, so the
// two run side by side; otherwise it starts once the planner's item prefix is written.
constexpr int kCasConcurrentGroups = 32;
int launch_cascade_tc(const AttnArgs& a, const CascadeArgs& cas, const Workspace& ws, int num_sms, int tiles_per_item,
                      int concurrent, uint32_t* err, cudaStream_t s);
// `after_decode`: launched right after this call's decode kernel (with the merge after
// it).  It reads nothing the decode writes, so its CTAs start on the SMs the decode's
// CTAs leave, and wait for the decode only before they exit: the launches after it wait
// on it alone.
int launch_prefill_tc(const AttnArgs& a, const Workspace& ws, int num_sms, uint32_t* err, cudaStream_t s,
                      int after_decode = 0);
int encode_tensor_map_3d(CUtensorMap* map, const void* base, const uint64_t dims[3], const uint64_t strides[2],
                         const uint32_t box[3]);

// Whether kernels are launched as programmatic dependents of their predecessor
// (environment PKV_PDL=0 turns it off; read once per process).
bool pdl_enabled();

// Launches `kernel` on `s`, as a programmatic dependent when pdl_enabled().
template <typename... Params, typename... Args>
cudaError_t launch_k(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Params>(args)...);
}

// cudaFuncSetAttribute(kernel, MaxDynamicSharedMemorySize, bytes) on the current
// device the first time only; done_mask holds one bit per device.
int set_smem_once(const void* kernel, int bytes, uint64_t* done_mask);
int encode_tensor_map_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                         uint32_t box_inner, uint32_t box_outer);

int run_umma_selftest(const int32_t* params, const void* a_img, const void* b_img, float* d_out, uint32_t* err,
                      cudaStream_t s);
int run_tma_selftest(const void* src, int64_t rows, int32_t row0, void* dump, uint32_t* err, cudaStream_t s);
int run_wait_selftest(uint32_t* err, cudaStream_t s);

}  // namespace pkv
