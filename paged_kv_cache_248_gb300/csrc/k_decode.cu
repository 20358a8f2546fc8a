// k_decode.cu -- split-KV GQA decode on tcgen05 tensor cores (bf16, head_dim 128).
//
// What it computes ("vLLM's PagedAttention" teardown, section "PagedAttention":
// the kernel is handed a per-request block table and gathers K/V from wherever the
// 16-token blocks live): for a decode request i (one query token at position
// seq_len - 1) and kv head h, the G query heads of h attend to all seq_len keys.
//
// Work decomposition.  Each (request, kv head) is cut into key splits
// (decode_splits: none up to kNoSplitKeys keys, else kSplitKeys-key pieces -- a
// function of the request's own length only), giving
// (request, kv head, split) items handed out by an atomic queue to persistent CTAs,
// one per SM.  A split walks 128-key tiles (8 blocks).  A split that is the whole
// request writes the output directly; otherwise it stores its fp32 partial
// (running max, sum, unnormalised accumulator) and merge_kernel, launched right
// after on the same stream, combines the partials in split order (log-sum-exp
// merge), so results never depend on scheduling.
//
// Per CTA (256 threads):
//   warp 6     scheduler: takes items off the queue ahead of use and resolves the
//              request, its lengths, its query row and the item's block ids (checked
//              against the pool) into a ring in shared memory.
//   warp 0     K producer: only TMA -- the G query rows (one 3-D box per half) and,
//              per tile, 2 boxes per block (two 64-column halves of K, 128-byte
//              swizzle) straight from the block's physical location -- the
//              block-table gather.  kStages tiles in flight.
//   warp 7     V producer: the same for V, into the V half of each stage.  A stage's
//              K is free once its S^T is done and its V once its P V is, so the K
//              of the next tiles (and of the next item) is requested a softmax
//              earlier than if the two waited for each other.
//   warp 1     MMA issuer (one lane): S^T = K Q^T with the 128 keys on M and the
//              query-head group on N = 16, then O^T = V^T P^T with head_dim on M,
//              both accumulating fp32 in TMEM.  V^T is read MN-major from the same
//              swizzled V tile, so no transpose is ever materialised.
//   warps 2-5  softmax: thread r owns TMEM lane r (key r of the tile for S^T, head
//              element r for O^T).  Tile maxima per head by warp shuffles plus a
//              4-warp exchange; exp2 of scaled logits; P^T written as bf16 into an
//              unswizzled MN-major operand; partial O folded into registers with
//              the online-softmax rescale.
// Every wait is bounded; on a timeout the CTA raises an abort flag, reports
// PKV_ERR_TIMEOUT, drains its in-flight copies and MMAs, frees TMEM and exits.
#include "ptx.cuh"
#include "pkv_internal.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 256;                 // 8 warps, see the role list above
constexpr int kStages = 3;
constexpr int kHalfBytes = 16384;             // one 64-column half of a 128-key tile
constexpr int kKBytes = 2 * kHalfBytes;       // K tile: [2 halves][128 keys][128 B]
constexpr int kStageBytes = 2 * kKBytes;      // K + V
constexpr int kQBytes = 4096;                 // Q: [2 halves][16 rows][128 B]
constexpr int kPBytes = 4096;                 // P^T: 128 keys x 16 heads, MN-major, no swizzle
constexpr int kRing = 3;                      // ring of items prepared by the scheduler
constexpr int kAheadTiles = 4;                // key tiles claimed but not yet issued before another claim
constexpr int kMaxIds = kNoSplitKeys / kBlock;  // block ids of one item (the longest item is unsplit)
constexpr uint32_t kTmemCols = 64;            // S^T x2 (cols 0, 16), O^T x2 (cols 32, 48)
constexpr int kBlocksPerTile = kTileKeys / kBlock;
constexpr int kCasStage = 16;                 // prefix-partial floats a softmax thread stages per item

struct alignas(16) ItemInfo {
  int32_t idx;  // decode item index; -1 = queue exhausted
  int32_t seq, head, split;
  int32_t nsplit, key_start, key_end, valid;
  int32_t trow, row_ok, member, centry;  // the request's query row, whether it is addressable,
                                         // whether a shared prefix was attended by the cascade
                                         // kernel, and then the request's member-list entry
};

struct Ctl {
  uint64_t kfull[kStages], kempty[kStages], vfull[kStages], vempty[kStages];
  uint64_t s_full[2], s_free[2], p_full[2], p_free[2], o_full[2], o_free[2];
  uint64_t q_full[2], q_free[2];
  uint64_t item_full[kRing], item_empty[kRing];
  uint64_t drain;
  uint64_t group_bar;  // the four softmax warps' exchange barrier
  ItemInfo ring[kRing];
  int bad[kRing];
  int32_t ids[kRing][kMaxIds];  // physical block ids of each ring item, validated
  float red[2][4][16];
  uint32_t issued_tiles;  // key tiles the producer has issued so far (it alone writes this)
  // a shared-prefix member's prefix partials, copied in at the start of its item and
  // folded at the end: accumulators [split * GP + head][128], max and sum by item parity
  float cas_o[kCasStage][128];
  float cas_ml[2][2 * kCasStage];
  uint32_t tmem_base;
  int abort_flag;
};

constexpr int kSmemBytes = kStages * kStageBytes + 2 * kQBytes + 2 * kPBytes + static_cast<int>(sizeof(Ctl)) + 1024;
static_assert(kSmemBytes <= 232448, "decode shared memory");

struct DecodeParams {
  __nv_bfloat16* out;
  const int32_t* bt;
  const int32_t* seq_lens;
  const int32_t* qsl;
  const int32_t* dec_prefix;
  const int32_t* dec_order;   // when *order_flag: queue position order of the requests
  const int32_t* dec_start;   //   and the items' exclusive prefix in that order
  const int32_t* dec_pos;     //   and per queue position (request, its first position)
  const int32_t* order_flag;
  int32_t* queue;
  int32_t* unit_bad;
  float* part_o;   // [items][128][GP]
  float* part_ml;  // [items][GP][2]
  const int32_t* seq_prefix;  // [num_seqs] keys before this many are the cascade kernel's; null: none
  const int32_t* seq_entry;   // [num_seqs] member-list entry of a shared-prefix member
  const float* cas_o;         // prefix partials [entry][hkv][cas_np_max][GP][128]
  const float* cas_ml;        // [entry][hkv][cas_np_max][GP][2]
  int32_t cas_np_max;
  uint32_t* err;
  int64_t num_blocks;
  int64_t num_tokens;
  int32_t num_seqs, max_blocks, hkv, group, gp, hq, split_keys;
  int32_t kv_evict_first;  // K/V tiles loaded with an L2 evict-first hint (decode-only batches)
  float scale_log2;
};

// Folds one partial (running max m, sum l, accumulator o, per head) into a
// log-sum-exp merge.  (The exponents take the MUFU 2^x: their arguments are <= 0,
// and -inf gives 0.)
template <int GP>
__device__ __forceinline__ void merge_fold(float (&M)[GP], float (&num)[GP], float (&den)[GP], const float (&ml)[2 * GP],
                                           const float (&ov)[GP]) {
#pragma unroll
  for (int g = 0; g < GP; ++g) {
    const float m_new = fmaxf(M[g], ml[2 * g]);
    const float a = ex2_approx(M[g] - m_new);
    const float b = ex2_approx(ml[2 * g] - m_new);
    den[g] = fmaf(den[g], a, ml[2 * g + 1] * b);
    num[g] = fmaf(num[g], a, ov[g] * b);
    M[g] = m_new;
  }
}

__device__ __forceinline__ void raise_abort(Ctl& c, uint32_t* err) {
  *reinterpret_cast<volatile int*>(&c.abort_flag) = 1;
  flag_error(err, kErrTimeout);
}

// Barrier among the four softmax warps (one arrival per warp), bounded like every
// other wait; `phase` counts the syncs this thread has made.
__device__ __forceinline__ bool group_sync(Ctl& c, uint32_t& phase) {
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(&c.group_bar);
  const bool ok = mbar_wait(&c.group_bar, phase & 1, &c.abort_flag);
  ++phase;
  return ok;
}

// Reduce GP per-lane values over the warp for every head at once.  Each halving
// exchange sends half of the remaining values to the partner lane, so after log2(GP)
// exchanges a lane holds one head's partial (head_of_lane), and the remaining lane
// bits are folded with a plain butterfly: GP - 1 + 5 - log2(GP) shuffles in all,
// instead of 5 per head.
template <int GP, bool kMax>
__device__ __forceinline__ float warp_reduce_scatter(float (&v)[GP]) {
  const int lane = threadIdx.x & 31;
  int o = 16;
#pragma unroll
  for (int n = GP; n > 1; n >>= 1, o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int k = 0; k < n / 2; ++k) {
      const float send = upper ? v[k] : v[k + n / 2];
      const float keep = upper ? v[k + n / 2] : v[k];
      const float recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[k] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
  float x = v[0];
#pragma unroll
  for (; o > 0; o >>= 1) {
    const float recv = __shfl_xor_sync(0xffffffffu, x, o);
    x = kMax ? fmaxf(x, recv) : x + recv;
  }
  return x;
}
// The head whose reduction warp_reduce_scatter<GP> leaves in this lane.
template <int GP>
__device__ __forceinline__ int head_of_lane(int lane) {
  int g = 0, o = 16;
#pragma unroll
  for (int n = GP; n > 1; n >>= 1, o >>= 1) g = (g << 1) | ((lane & o) ? 1 : 0);
  return g;
}

// ------------------------------------------------------------------ scheduler warp
// Takes items off the queue ahead of use and resolves everything the other roles need
// from global memory -- the request, its lengths and query row, and the item's block
// ids (validated) -- into a ring in shared memory, so that the TMA producer never
// waits on a global load.  The ring is short on purpose: an item taken off the queue
// early is an item no idle CTA can take at the end.
__device__ void scheduler_warp(const DecodeParams& P, Ctl& c) {
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = &c.abort_flag;
  // the first item's position record is loaded with the item count and the order flag
  // (one round trip); it is used only if the batch turns out to be ordered
  const int2* pos_rec = reinterpret_cast<const int2*>(P.dec_pos);
  const int2 first_rec = blockIdx.x < kDecPosMax ? __ldg(pos_rec + blockIdx.x) : make_int2(0, 0);
  const int total = P.dec_prefix[P.num_seqs];
  // queue positions follow the planner's order of the requests when it made one
  const bool ordered = *P.order_flag != 0;
  const int32_t* starts = ordered ? P.dec_start : P.dec_prefix;
  uint32_t claimed_tiles = 0;  // key tiles of the valid items taken so far
  for (uint32_t it = 0;; ++it) {
    const int slot = it % kRing;
    if (!mbar_wait(&c.item_empty[slot], ((it / kRing) & 1) ^ 1, abort_flag)) {
      if (!*abort_flag && lane == 0) raise_abort(c, P.err);
      break;
    }
    // An item taken off the queue is one no other CTA can take: take the next only when
    // the producer is within kAheadTiles tiles of needing it, so that long items are
    // not held here while other CTAs run dry at the end (short items still fill the
    // ring).  The producer's progress needs nothing from this warp, so the wait ends;
    // it is bounded like every other wait.
    if (it > 0) {
      const volatile uint32_t* issued = &c.issued_tiles;
      if (static_cast<int32_t>(claimed_tiles - *issued) > kAheadTiles) {
        const uint64_t t0 = globaltimer_ns();
        bool waited = true;
        while (static_cast<int32_t>(claimed_tiles - *issued) > kAheadTiles) {
          if (*abort_flag || globaltimer_ns() - t0 > kWaitTimeoutNs) {
            waited = false;
            break;
          }
          __nanosleep(64);
        }
        if (!waited) {
          if (!*abort_flag && lane == 0) raise_abort(c, P.err);
          break;
        }
      }
    }
    // every CTA's first item is its own index; later ones come off the queue after those
    int idx = static_cast<int>(blockIdx.x);
    if (it > 0) {
      if (lane == 0) idx = static_cast<int>(gridDim.x) + atomicAdd(P.queue, 1);
      idx = __shfl_sync(0xffffffffu, idx, 0);
    }
    ItemInfo r{};
    if (idx >= total) {
      if (lane == 0) {
        r.idx = -1;
        c.ring[slot] = r;
        mbar_arrive(&c.item_full[slot]);
      }
      break;
    }
    // the request owning the queue position and its first position: one load in an
    // ordered batch, else the last k with starts[k] <= idx by a 32-way search (each
    // round the 32 lanes probe evenly spaced candidates)
    int i, qbase;
    if (ordered) {
      const int2 e = it == 0 ? first_rec : __ldg(pos_rec + idx);
      i = e.x;
      qbase = e.y;
    } else {
      int lo = 0, hi = P.num_seqs - 1;
      while (hi > lo) {
        const int step = (hi - lo + 32) / 32;
        const int pos = lo + lane * step;
        const bool le = pos <= hi && __ldg(starts + pos) <= idx;
        const unsigned m = __ballot_sync(0xffffffffu, le);  // lane 0 always: starts[lo] <= idx
        lo += (31 - __clz(m)) * step;
        hi = min(hi, lo + step - 1);
      }
      i = lo;
      qbase = __ldg(starts + lo);
    }
    const int base = __ldg(P.dec_prefix + i);  // the request's items in request order
    const int cnt = __ldg(P.dec_prefix + i + 1) - base;
    const int64_t L = __ldg(P.seq_lens + i);
    const int64_t t = __ldg(P.qsl + i), t1 = __ldg(P.qsl + i + 1);
    const int nsplit = cnt / P.hkv;
    const int64_t pre = P.seq_prefix ? __ldg(P.seq_prefix + i) : 0;  // shared-prefix keys, done elsewhere
    r.idx = base + (idx - qbase);  // the item's index in request order: where its partial goes
    r.seq = i;
    r.row_ok = (t >= 0 && t < P.num_tokens && t1 == t + 1) ? 1 : 0;
    r.trow = r.row_ok ? static_cast<int32_t>(t) : 0;
    r.nsplit = 1;
    if (nsplit > 0) {  // always, for a consistent plan
      const int local = idx - qbase;
      r.head = local / nsplit;
      r.split = local % nsplit;
      r.nsplit = nsplit;
      const bool ok = r.row_ok && L >= 1 && (L + kBlock - 1) / kBlock <= P.max_blocks && pre >= 0 && pre < L &&
                      static_cast<int64_t>(nsplit) == decode_splits(L - pre);
      if (ok) {
        r.valid = 1;
        r.member = pre > 0 ? 1 : 0;
        r.centry = pre > 0 ? __ldg(P.seq_entry + i) : 0;
        if (nsplit == 1) {
          r.key_start = static_cast<int32_t>(pre);
          r.key_end = static_cast<int32_t>(L);
        } else {
          r.key_start = static_cast<int32_t>(pre) + r.split * P.split_keys;
          const int64_t split_end = static_cast<int64_t>(r.key_start) + P.split_keys;
          r.key_end = static_cast<int32_t>(L < split_end ? L : split_end);
        }
      }
    }
    int bad = 0;
    if (r.valid) {
      const int nblk = (r.key_end - r.key_start + kBlock - 1) / kBlock;
      const int32_t* row = P.bt + static_cast<int64_t>(i) * P.max_blocks + r.key_start / kBlock;
      for (int b = lane; b < nblk; b += 32) {
        int id = __ldg(row + b);
        if (id < 0 || id >= P.num_blocks) {
          bad = 1;
          id = 0;
        }
        c.ids[slot][b] = id;
      }
    }
    bad = __any_sync(0xffffffffu, bad);
    if (r.valid) claimed_tiles += static_cast<uint32_t>((r.key_end - r.key_start + kTileKeys - 1) / kTileKeys);
    if (lane == 0) {
      if (bad) flag_error(P.err, kErrBlockId);
      c.ring[slot] = r;
      c.bad[slot] = bad;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&c.item_full[slot]);
  }
}

// ------------------------------------------------------------------ producer warp
// Only mbarrier waits and TMA issues.  The K producer (kV false): the G query rows of
// the item (one 3-D box per 64-column half) and, per 128-key tile, two 16 x 64 boxes of
// K per block taken straight from the block's physical location (the block-table
// gather).  The V producer: the same boxes of V.  Each walks the item ring on its own.
template <bool kV>
__device__ void producer_warp(const DecodeParams& P, const CUtensorMap* qmap, const CUtensorMap* kmap,
                              const CUtensorMap* vmap, Ctl& c, uint8_t* stages, uint8_t* qbuf) {
  const int lane = threadIdx.x & 31;
  uint32_t it = 0, tc = 0, qc = 0;
  volatile int* abort_flag = &c.abort_flag;
  const uint64_t pol_q = l2_policy_evict_first();
  const uint64_t pol_kv = l2_policy_evict_first();
  const bool kv_ef = P.kv_evict_first != 0;
  bool ok = true;
  while (ok) {
    const int slot = it % kRing;
    if (!mbar_wait(&c.item_full[slot], (it / kRing) & 1, abort_flag)) {
      ok = false;
      break;
    }
    const ItemInfo info = c.ring[slot];
    ++it;
    if (info.idx < 0) break;
    if (info.valid) {
      if (!kV) {
        const int qb = qc & 1;
        if (!mbar_wait(&c.q_free[qb], ((qc >> 1) & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&c.q_full[qb], 2u * static_cast<uint32_t>(P.gp) * 128u);
          const int32_t y = info.head * P.group;
          tma_load_3d(qbuf + qb * kQBytes, qmap, &c.q_full[qb], 0, y, info.trow, pol_q);
          tma_load_3d(qbuf + qb * kQBytes + 2048, qmap, &c.q_full[qb], 64, y, info.trow, pol_q);
        }
        ++qc;
      }
      const int nt = (info.key_end - info.key_start + kTileKeys - 1) / kTileKeys;
      for (int j = 0; j < nt; ++j) {
        const int st = tc % kStages;
        if (!mbar_wait(kV ? &c.vempty[st] : &c.kempty[st], ((tc / kStages) & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        const int t0 = info.key_start + j * kTileKeys;
        const int nblk = min(kBlocksPerTile, (info.key_end - t0 + kBlock - 1) / kBlock);
        const int id = lane < nblk ? c.ids[slot][j * kBlocksPerTile + lane] : 0;
        uint64_t* bar = kV ? &c.vfull[st] : &c.kfull[st];
        const CUtensorMap* map = kV ? vmap : kmap;
        if (lane == 0) mbar_arrive_expect_tx(bar, static_cast<uint32_t>(nblk) * 4096u);
        __syncwarp();
        if (lane < nblk) {
          uint8_t* s = stages + st * kStageBytes + (kV ? kKBytes : 0) + lane * 2048;
          const int32_t row = (id * P.hkv + info.head) * kBlock;
          if (kv_ef) {  // each tile is read once: let the stream give way to code and tables in L2
            tma_load_2d(s, map, bar, 0, row, pol_kv);
            tma_load_2d(s + kHalfBytes, map, bar, 64, row, pol_kv);
          } else {
            tma_load_2d(s, map, bar, 0, row);
            tma_load_2d(s + kHalfBytes, map, bar, 64, row);
          }
        }
        ++tc;
        if (!kV && lane == 0) *reinterpret_cast<volatile uint32_t*>(&c.issued_tiles) = tc;
      }
      if (!ok) break;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&c.item_empty[slot]);
  }
  if (!ok && !*abort_flag && lane == 0) raise_abort(c, P.err);
  if (*abort_flag) {
    // let copies already issued land before the CTA's shared memory goes away
    const uint32_t first = tc > static_cast<uint32_t>(kStages) ? tc - kStages : 0;
    for (uint32_t cnt = first; cnt < tc; ++cnt)
      mbar_wait(kV ? &c.vfull[cnt % kStages] : &c.kfull[cnt % kStages], (cnt / kStages) & 1, nullptr);
    if (qc > 0) mbar_wait(&c.q_full[(qc - 1) & 1], ((qc - 1) >> 1) & 1, nullptr);
  }
}

// ------------------------------------------------------------------ MMA warp
__device__ void mma_warp(const DecodeParams& P, Ctl& c, uint8_t* stages, uint8_t* qbuf, uint8_t* pbuf,
                         uint32_t tmem) {
  // One thread polls the barriers and issues every MMA, running this whole loop alone:
  // the other lanes wait at the end, so no warp-wide exchange sits between two issues.
  if ((threadIdx.x & 31) == 0) {
    const uint32_t idesc_s = umma_idesc_bf16(128, 16, false, false);
    const uint32_t idesc_o = umma_idesc_bf16(128, 16, true, true);
    volatile int* abort_flag = &c.abort_flag;
    uint32_t it = 0, tc = 0, qc = 0;
    bool issued = false;
    bool ok = true;
    while (ok) {
      const int slot = it % kRing;
      if (!mbar_wait(&c.item_full[slot], (it / kRing) & 1, abort_flag)) {
        ok = false;
        break;
      }
      const ItemInfo info = c.ring[slot];
      ++it;
      if (info.idx < 0) break;
      if (info.valid) {
        const int qb = qc & 1;
        if (!mbar_wait(&c.q_full[qb], (qc >> 1) & 1, abort_flag)) {
          ok = false;
          break;
        }
        const uint64_t qdesc = umma_smem_desc(smem_u32(qbuf + qb * kQBytes), 16, 1024, kLayout128B);
        // Issue S^T(j) as soon as tile j has landed and its TMEM buffer is free, and
        // O^T(j) = V^T P^T as soon as the softmax has written P(j): polled, so that neither
        // kind of MMA waits behind the other (a late tile must not hold back the P V
        // that frees an earlier stage).  The clock is read only while nothing is ready:
        // the wait is bounded from the first poll that finds nothing to issue.
        const int nt = (info.key_end - info.key_start + kTileKeys - 1) / kTileKeys;
        int ns = 0, npv = 0;
        bool idle = false;
        uint64_t t_idle = 0;
        while (npv < nt) {
          bool progress = false;
          if (ns < nt) {
            const uint32_t cnt = tc + ns;
            const int st = cnt % kStages, sb = cnt & 1;
            if (mbar_test(&c.kfull[st], (cnt / kStages) & 1) && mbar_test(&c.s_free[sb], ((cnt >> 1) & 1) ^ 1)) {
              tc_fence_after();
              const uint64_t a = umma_smem_desc(smem_u32(stages + st * kStageBytes), 16, 1024, kLayout128B);
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                umma_f16_ss(tmem + 16 * sb, umma_desc_advance(a, (kk >> 2) * kHalfBytes + (kk & 3) * 32),
                            umma_desc_advance(qdesc, (kk >> 2) * 2048 + (kk & 3) * 32), idesc_s, kk > 0);
              umma_commit(&c.s_full[sb]);
              umma_commit(&c.kempty[st]);  // this K is read by no other MMA
              if (ns == nt - 1) umma_commit(&c.q_free[qb]);
              issued = true;
              ++ns;
              progress = true;
            }
          }
          if (npv < ns) {
            const uint32_t cnt = tc + npv;
            const int st = cnt % kStages, b = cnt & 1;
            const uint32_t ph = (cnt >> 1) & 1;
            if (mbar_test(&c.p_full[b], ph) && mbar_test(&c.o_free[b], ph ^ 1)) {
              tc_fence_after();
              const uint64_t a =
                  umma_smem_desc(smem_u32(stages + st * kStageBytes + kKBytes), kHalfBytes, 1024, kLayout128B);
              const uint64_t bd = umma_smem_desc(smem_u32(pbuf + b * kPBytes), 128, 2048, kLayoutNone);
#pragma unroll
              for (int kk = 0; kk < 8; ++kk)
                umma_f16_ss(tmem + 32 + 16 * b, umma_desc_advance(a, kk * 2048), umma_desc_advance(bd, kk * 256),
                            idesc_o, kk > 0);
              umma_commit(&c.o_full[b]);
              umma_commit(&c.p_free[b]);
              umma_commit(&c.vempty[st]);
              ++npv;
              progress = true;
            }
          }
          if (progress) {
            idle = false;
          } else if (!idle) {
            idle = true;
            t_idle = globaltimer_ns();
          } else if (*abort_flag || globaltimer_ns() - t_idle > kWaitTimeoutNs) {
            ok = false;
            break;
          }
        }
        tc += nt;
        ++qc;
      }
      if (!ok) break;
      mbar_arrive(&c.item_empty[slot]);
    }
    if (!ok && !*abort_flag) raise_abort(c, P.err);
    if (issued) {
      // every MMA issued so far, and the barrier arrivals its commits trigger, must be
      // complete before TMEM is freed and the CTA's shared memory goes away
      umma_commit(&c.drain);
      mbar_wait(&c.drain, 0, nullptr);
    }
  }
  __syncwarp();
}

// ------------------------------------------------------------------ softmax warps
template <int GP>
__device__ void softmax_warps(const DecodeParams& P, Ctl& c, uint8_t* stages, uint8_t* pbuf, uint32_t tmem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wq = warp & 3;                       // TMEM lane quarter this warp may access
  const int r = wq * 32 + lane;                  // key of the tile (S^T) / head element (O^T)
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  const int G = P.group;
  volatile int* abort_flag = &c.abort_flag;
  uint32_t it = 0, tc = 0, gph = 0, nstaged = 0;
  bool ok = true;
  while (ok) {
    const int slot = it % kRing;
    if (!mbar_wait(&c.item_full[slot], (it / kRing) & 1, abort_flag)) {
      ok = false;
      break;
    }
    const ItemInfo info = c.ring[slot];
    ++it;
    if (info.idx < 0) break;
    if (!info.valid) {
      // report once per request and zero what can be addressed
      if (info.split == 0 && info.head == 0 && r == 0) flag_error(P.err, kErrLength);
      const int64_t trow = info.trow;
      if (info.split == 0 && info.row_ok)
        for (int g = 0; g < G; ++g)
          P.out[(trow * P.hq + static_cast<int64_t>(info.head) * G + g) * 128 + r] = __float2bfloat16_rn(0.f);
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.item_empty[slot]);
      continue;
    }

    // a shared-prefix member whose own keys are one split finishes here: the first nst
    // of its prefix partials (written by the cascade kernel) are copied into shared
    // memory now, so that the fold at the end does not wait on global loads.  Each
    // thread copies (and later reads) its own accumulator elements; the max/sum pairs
    // are read by all four warps after the group barrier that follows the copies' wait.
    const bool fold_prefix = info.member && info.nsplit == 1;
    const int64_t cbase = (static_cast<int64_t>(info.centry) * P.hkv + info.head) * P.cas_np_max;
    const int npre = fold_prefix ? static_cast<int>(cascade_splits(info.key_start)) : 0;
    const int nst = npre < kCasStage / GP ? npre : kCasStage / GP;
    // the pairs alternate between two buffers over the items that stage them: another
    // warp may still be reading the previous such item's pairs, but not the one before
    // (that would take it past the previous item's group barriers)
    const int mlb = nstaged & 1;
    if (nst > 0) {
      ++nstaged;
      for (int k = 0; k < nst * GP; ++k) cp_async4(&c.cas_o[k][r], P.cas_o + (cbase * GP + k) * 128 + r);
      if (r < 2 * GP * nst) cp_async4(&c.cas_ml[mlb][r], P.cas_ml + cbase * GP * 2 + r);
      cp_async_commit();
    }

    float m_run[GP], l_run[GP], acc[GP], alpha_prev[GP];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      m_run[g] = -INFINITY;
      l_run[g] = 0.f;
      acc[g] = 0.f;
      alpha_prev[g] = 0.f;
    }
    auto fold = [&](uint32_t cnt, const float (&a)[GP]) -> bool {
      const int b = cnt & 1;
      if (!mbar_wait(&c.o_full[b], (cnt >> 1) & 1, abort_flag)) return false;
      tc_fence_after();
      uint32_t o[16];
      tmem_ld16_sync(tmem + lane_off + 32 + 16 * b, o);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.o_free[b]);
#pragma unroll
      for (int g = 0; g < GP; ++g) acc[g] = fmaf(acc[g], a[g], __uint_as_float(o[g]));
      return true;
    };

    const int nt = (info.key_end - info.key_start + kTileKeys - 1) / kTileKeys;
    for (int j = 0; j < nt && ok; ++j) {
      const int st = tc % kStages, sb = tc & 1;
      const uint32_t ph2 = (tc >> 1) & 1;
      const int t0 = info.key_start + j * kTileKeys;
      // S^T lane r = logits of key t0 + r for every head of the group
      if (!mbar_wait(&c.s_full[sb], ph2, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sraw[16];
      tmem_ld16_sync(tmem + lane_off + 16 * sb, sraw);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.s_free[sb]);
      const bool valid_key = t0 + r < info.key_end;
      float x[GP], tmax[GP];
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        x[g] = valid_key ? __uint_as_float(sraw[g]) * P.scale_log2 : -INFINITY;
        tmax[g] = x[g];
      }
      const float wmax = warp_reduce_scatter<GP, true>(tmax);
      const int rb = gph & 1;
      if ((lane & (32 / GP - 1)) == 0) c.red[rb][wq][head_of_lane<GP>(lane)] = wmax;
      if (!group_sync(c, gph)) {
        ok = false;
        break;
      }
      float alpha[GP], p[GP];
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        const float mt = fmaxf(fmaxf(c.red[rb][0][g], c.red[rb][1][g]), fmaxf(c.red[rb][2][g], c.red[rb][3][g]));
        const float m_new = fmaxf(m_run[g], mt);
        alpha[g] = ex2_approx(m_run[g] - m_new);  // arguments <= 0; -inf gives 0
        p[g] = ex2_approx(x[g] - m_new);
        l_run[g] = fmaf(l_run[g], alpha[g], p[g]);
        m_run[g] = m_new;
      }
      // the tile's V has landed (needed to zero V rows of masked keys; P V is issued
      // only after P, so this wait also orders it after the load)
      if (!mbar_wait(&c.vfull[st], (tc / kStages) & 1, abort_flag)) {
        ok = false;
        break;
      }
      if (!valid_key) {
        // rows are 128 bytes apart: each lane starts at chunk r mod 8, so eight lanes
        // cover all 32 banks instead of sharing four
        uint8_t* vrow = stages + st * kStageBytes + kKBytes + r * 128;
        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c16 = 0; c16 < 8; ++c16) {
          const int off = ((c16 + r) & 7) * 16;
          *reinterpret_cast<uint4*>(vrow + off) = z;
          *reinterpret_cast<uint4*>(vrow + kHalfBytes + off) = z;
        }
      }
      // P^T row r (MN-major, unswizzled): heads 0-7 in one 16-byte chunk, 8-15 in another
      const int pb = tc & 1;
      if (!mbar_wait(&c.p_free[pb], ph2 ^ 1, abort_flag)) {
        ok = false;
        break;
      }
      {
        float p16[16];
#pragma unroll
        for (int g = 0; g < 16; ++g) p16[g] = 0.f;
#pragma unroll
        for (int g = 0; g < GP; ++g) p16[g] = g < G ? p[g] : 0.f;
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          __nv_bfloat162 h2 = __floats2bfloat162_rn(p16[2 * k], p16[2 * k + 1]);
          w[k] = *reinterpret_cast<uint32_t*>(&h2);
        }
        uint8_t* prow = pbuf + pb * kPBytes + (r >> 3) * 128 + (r & 7) * 16;
        *reinterpret_cast<uint4*>(prow) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(prow + 2048) = make_uint4(w[4], w[5], w[6], w[7]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.p_full[pb]);
      if (j > 0 && !fold(tc - 1, alpha_prev)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int g = 0; g < GP; ++g) alpha_prev[g] = alpha[g];
      ++tc;
    }
    if (!ok) break;
    if (!fold(tc - 1, alpha_prev)) {
      ok = false;
      break;
    }

    // total softmax denominators: sum the per-thread partial sums over the 128 keys lanes
    float lt[GP];
    if (nst > 0) cp_async_wait_all();  // the staged prefix partials, before the barrier
    {
#pragma unroll
      for (int g = 0; g < GP; ++g) lt[g] = l_run[g];
      const float wsum = warp_reduce_scatter<GP, false>(lt);
      const int rb = gph & 1;
      if ((lane & (32 / GP - 1)) == 0) c.red[rb][wq][head_of_lane<GP>(lane)] = wsum;
      if (!group_sync(c, gph)) {
        ok = false;
        break;
      }
#pragma unroll
      for (int g = 0; g < GP; ++g) lt[g] = c.red[rb][0][g] + c.red[rb][1][g] + c.red[rb][2][g] + c.red[rb][3][g];
    }
    const bool bad = c.bad[slot] != 0;
    const int64_t trow = info.trow;
    const int64_t unit = static_cast<int64_t>(info.seq) * P.hkv + info.head;
    __nv_bfloat16* orow = P.out + (trow * P.hq + static_cast<int64_t>(info.head) * G) * 128 + r;
    // (the fast division is exact enough for a bf16 result; every denominator is at
    // least 1, the term of the maximum itself)
    if (info.nsplit == 1 && !info.member) {
#pragma unroll
      for (int g = 0; g < GP; ++g)
        if (g < G) orow[g * 128] = __float2bfloat16_rn(bad ? 0.f : __fdividef(acc[g], lt[g]));
    } else if (fold_prefix) {
      // the prefix partials in split order, then this item: the split merge's order
      float M[GP], num[GP], den[GP];
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        M[g] = -INFINITY;
        num[g] = 0.f;
        den[g] = 0.f;
      }
      for (int s = 0; s < nst; ++s) {
        float ml[2 * GP], ov[GP];
#pragma unroll
        for (int k = 0; k < 2 * GP; ++k) ml[k] = c.cas_ml[mlb][s * 2 * GP + k];
#pragma unroll
        for (int g = 0; g < GP; ++g) ov[g] = c.cas_o[s * GP + g][r];
        merge_fold<GP>(M, num, den, ml, ov);
      }
      // the rest straight from global memory, kU splits' loads issued before their folds
      constexpr int kU = GP <= 4 ? 4 : GP == 8 ? 2 : 1;
      for (int s0 = nst; s0 < npre; s0 += kU) {
        float ml[kU][2 * GP], ov[kU][GP];
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          if (s0 + u < npre) {
            const int64_t e = cbase + s0 + u;
#pragma unroll
            for (int k = 0; k < 2 * GP; ++k) ml[u][k] = __ldg(P.cas_ml + e * GP * 2 + k);
#pragma unroll
            for (int g = 0; g < GP; ++g) ov[u][g] = __ldg(P.cas_o + (e * GP + g) * 128 + r);
          }
        }
#pragma unroll
        for (int u = 0; u < kU; ++u)
          if (s0 + u < npre) merge_fold<GP>(M, num, den, ml[u], ov[u]);
      }
      float ml[2 * GP];
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        ml[2 * g] = m_run[g];
        ml[2 * g + 1] = lt[g];
      }
      merge_fold<GP>(M, num, den, ml, acc);
      // (a member's prefix has only valid block ids: the planner admits no member of a
      // group whose prefix names a bad one, so only this item's own tiles can be bad)
#pragma unroll
      for (int g = 0; g < GP; ++g)
        if (g < G) orow[g * 128] = __float2bfloat16_rn(bad ? 0.f : __fdividef(num[g], den[g]));
    } else {
      // partials: accumulators [item][d][GP] (one float4 run per thread), max and sum
      // [item][GP][2]; the merge kernel that runs after this one combines them
      float4* po = reinterpret_cast<float4*>(P.part_o + (static_cast<int64_t>(info.idx) * 128 + r) * GP);
#pragma unroll
      for (int k = 0; k < GP / 4; ++k) po[k] = make_float4(acc[4 * k], acc[4 * k + 1], acc[4 * k + 2], acc[4 * k + 3]);
      float* pml = P.part_ml + static_cast<int64_t>(info.idx) * GP * 2;
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        if (r == g) {
          pml[2 * g] = m_run[g];
          pml[2 * g + 1] = lt[g];
        }
      }
      if (bad && r == 0) P.unit_bad[unit] = 1;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&c.item_empty[slot]);
  }
  if (!ok && !*abort_flag && lane == 0) raise_abort(c, P.err);
}

template <int GP>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const __grid_constant__ CUtensorMap qmap,
                                                             const __grid_constant__ CUtensorMap kmap,
                                                             const __grid_constant__ CUtensorMap vmap,
                                                             const DecodeParams P) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* stages = base;
  uint8_t* qbuf = stages + kStages * kStageBytes;
  uint8_t* pbuf = qbuf + 2 * kQBytes;
  Ctl& c = *reinterpret_cast<Ctl*>(pbuf + 2 * kPBytes);
  const int warp = threadIdx.x >> 5;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&c.kfull[s], 1);
      mbar_init(&c.kempty[s], 1);
      mbar_init(&c.vfull[s], 1);
      mbar_init(&c.vempty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&c.s_full[b], 1);
      mbar_init(&c.s_free[b], 4);
      mbar_init(&c.p_full[b], 4);
      mbar_init(&c.p_free[b], 1);
      mbar_init(&c.o_full[b], 1);
      mbar_init(&c.o_free[b], 4);
      mbar_init(&c.q_full[b], 1);
      mbar_init(&c.q_free[b], 1);
    }
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&c.item_full[s], 1);
      mbar_init(&c.item_empty[s], 7);  // two producers, MMA warp, four softmax warps
    }
    mbar_init(&c.drain, 1);
    mbar_init(&c.group_bar, 4);
    c.abort_flag = 0;
    c.issued_tiles = 0;
    fence_mbar_init();
    tma_prefetch_map(&qmap);
    tma_prefetch_map(&kmap);
    tma_prefetch_map(&vmap);
  }
  // zero Q (padding rows stay zero) and P^T buffers
  for (int i = threadIdx.x; i < (2 * kQBytes + 2 * kPBytes) / 16; i += kThreads)
    reinterpret_cast<uint4*>(qbuf)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 1) tmem_alloc(&c.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c.tmem_base;
  grid_dep_wait();  // the plan (and new tokens) of this call, from the kernels before
  grid_dep_launch();

  if (warp == 0) producer_warp<false>(P, &qmap, &kmap, &vmap, c, stages, qbuf);
  else if (warp == 1) mma_warp(P, c, stages, qbuf, pbuf, tmem);
  else if (warp < 6) softmax_warps<GP>(P, c, stages, pbuf, tmem);
  else if (warp == 6) scheduler_warp(P, c);
  else producer_warp<true>(P, &qmap, &kmap, &vmap, c, stages, qbuf);

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
    tmem_relinquish();
  }
}

// ------------------------------------------------------------------ split merge
// Combines the partials of every (request, kv head) that was cut into several key
// splits -- the planner lists those requests -- by a log-sum-exp merge, one CTA per
// unit.  A shared-prefix member's prefix partials (the cascade kernel's, stored
// [GP][128] per split) come first, then its own key splits: that list is cut into
// kMergeGroups contiguous runs, each folded in order by one group of 128 threads
// (thread d = head element, float4 loads), and the runs' results are folded in run
// order -- a fixed tree, so the result does not depend on scheduling.  Requests of
// one split were written by the decode kernel.
constexpr int kMergeGroups = 4;
struct MergeParams {
  __nv_bfloat16* out;
  const int32_t* counters;
  const int32_t* merge_list;
  const int32_t* dec_prefix;
  const int32_t* qsl;
  const int32_t* unit_bad;
  const float* part_o;
  const float* part_ml;
  const int32_t* seq_prefix;  // null: no shared-prefix groups
  const int32_t* seq_entry;
  const float* cas_o;
  const float* cas_ml;
  int32_t cas_np_max;
  int32_t num_seqs, hkv, group, hq;
};

// Two CTAs per SM where the registers allow it (GP <= 8), so that a batch's (request, kv
// head) units run in one wave rather than two.
template <int GP>
__global__ void __launch_bounds__(128 * kMergeGroups, GP <= 8 ? 2 : 0) merge_kernel(const MergeParams P) {
  __shared__ float xfer[GP][3][128];  // one run's (max, sum, accumulator) handed to run 0
  grid_dep_wait();
  grid_dep_launch();
  const int d = threadIdx.x % 128, run = threadIdx.x / 128;
  // the planner's record of the request (loaded with the list length: a record past
  // the list is never used)
  const int4* recs = reinterpret_cast<const int4*>(P.merge_list);
  int64_t e = blockIdx.x;
  int4 ra = make_int4(0, 0, 0, 0), rb = ra;
  if (e / P.hkv < P.num_seqs) {
    ra = __ldg(recs + 2 * (e / P.hkv));
    rb = __ldg(recs + 2 * (e / P.hkv) + 1);
  }
  const int64_t n_units = static_cast<int64_t>(P.counters[kMergeCountSlot]) * P.hkv;
  for (; e < n_units; e += gridDim.x) {
    if (e != blockIdx.x) {
      ra = __ldg(recs + 2 * (e / P.hkv));
      rb = __ldg(recs + 2 * (e / P.hkv) + 1);
    }
    const int i = ra.x, h = static_cast<int>(e % P.hkv);
    const int64_t u = static_cast<int64_t>(i) * P.hkv + h;
    const int base_i = ra.y, ns = ra.z;
    const int pre = rb.x;
    if (ns <= 1) continue;  // (a member of one split was finished by the decode kernel)
    const bool bad = __ldg(P.unit_bad + u) != 0;
    const int64_t base = base_i + static_cast<int64_t>(h) * ns;
    const int npre = pre > 0 ? static_cast<int>(cascade_splits(pre)) : 0;
    const int64_t cbase = pre > 0 ? (static_cast<int64_t>(rb.y) * P.hkv + h) * P.cas_np_max : 0;
    // this run: entries [e0, e1) of prefix partials then splits
    const int n_all = npre + ns;
    const int per = (n_all + kMergeGroups - 1) / kMergeGroups;
    const int e0 = min(n_all, run * per), e1 = min(n_all, e0 + per);
    float M[GP], num[GP], den[GP];
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      M[g] = -INFINITY;
      num[g] = 0.f;
      den[g] = 0.f;
    }
    for (int k = e0; k < min(e1, npre); ++k) {
      const float* ml_p = P.cas_ml + (cbase + k) * GP * 2;
      const float* o_p = P.cas_o + (cbase + k) * GP * 128 + d;
      float ml[2 * GP], ov[GP];
#pragma unroll
      for (int q = 0; q < 2 * GP; ++q) ml[q] = __ldg(ml_p + q);
#pragma unroll
      for (int g = 0; g < GP; ++g) ov[g] = __ldg(o_p + g * 128);
      merge_fold<GP>(M, num, den, ml, ov);
    }
#pragma unroll 4
    for (int k = max(e0, npre); k < e1; ++k) {
      const int64_t it = base + (k - npre);
      const float4* ml4 = reinterpret_cast<const float4*>(P.part_ml + it * GP * 2);
      const float4* o4 = reinterpret_cast<const float4*>(P.part_o + (it * 128 + d) * GP);
      float ml[2 * GP], ov[GP];
#pragma unroll
      for (int q = 0; q < GP / 2; ++q) {
        const float4 t = __ldg(ml4 + q);
        ml[4 * q] = t.x;
        ml[4 * q + 1] = t.y;
        ml[4 * q + 2] = t.z;
        ml[4 * q + 3] = t.w;
      }
#pragma unroll
      for (int q = 0; q < GP / 4; ++q) {
        const float4 t = __ldg(o4 + q);
        ov[4 * q] = t.x;
        ov[4 * q + 1] = t.y;
        ov[4 * q + 2] = t.z;
        ov[4 * q + 3] = t.w;
      }
      merge_fold<GP>(M, num, den, ml, ov);
    }
    // runs 1.. hand their results to run 0, which folds them in run order (run 0's
    // list is never empty, so its maximum is finite; an empty run folds as nothing)
    for (int k = 1; k < kMergeGroups; ++k) {
      __syncthreads();
      if (run == k) {
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          xfer[g][0][d] = M[g];
          xfer[g][1][d] = den[g];
          xfer[g][2][d] = num[g];
        }
      }
      __syncthreads();
      if (run == 0 && k * per < n_all) {
        float ml[2 * GP], ov[GP];
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          ml[2 * g] = xfer[g][0][d];
          ml[2 * g + 1] = xfer[g][1][d];
          ov[g] = xfer[g][2][d];
        }
        merge_fold<GP>(M, num, den, ml, ov);
      }
    }
    if (run == 0) {
      const int64_t trow = ra.w;
      __nv_bfloat16* orow = P.out + (trow * P.hq + static_cast<int64_t>(h) * P.group) * 128 + d;
#pragma unroll
      for (int g = 0; g < GP; ++g)
        if (g < P.group) orow[g * 128] = __float2bfloat16_rn(bad ? 0.f : __fdividef(num[g], den[g]));
    }
  }
}

// The split merge when no unit folds more than MergeSmall<GP>::kEntries partials (the
// host bounds this from the longest context and prefix): one 128-thread CTA per
// (request, kv head) whose thread d runs all four of merge_kernel's runs for its column
// one after another -- the same folds in the same order, so the same bits -- with every
// partial's load issued before the first fold and no block barrier.
template <int GP>
struct MergeSmall {
  static constexpr int kEntries = GP <= 4 ? 8 : GP == 8 ? 4 : 2;
};
template <int GP>
__global__ void __launch_bounds__(128) merge_small_kernel(const MergeParams P) {
  constexpr int E = MergeSmall<GP>::kEntries;
  grid_dep_wait();
  grid_dep_launch();
  const int d = threadIdx.x;
  const int4* recs = reinterpret_cast<const int4*>(P.merge_list);
  int64_t e = blockIdx.x;
  int4 ra = make_int4(0, 0, 0, 0), rb = ra;
  if (e / P.hkv < P.num_seqs) {
    ra = __ldg(recs + 2 * (e / P.hkv));
    rb = __ldg(recs + 2 * (e / P.hkv) + 1);
  }
  const int64_t n_units = static_cast<int64_t>(P.counters[kMergeCountSlot]) * P.hkv;
  for (; e < n_units; e += gridDim.x) {
    if (e != blockIdx.x) {
      ra = __ldg(recs + 2 * (e / P.hkv));
      rb = __ldg(recs + 2 * (e / P.hkv) + 1);
    }
    const int i = ra.x, h = static_cast<int>(e % P.hkv);
    const int base_i = ra.y, ns = ra.z, pre = rb.x;
    if (ns <= 1) continue;
    const int64_t u = static_cast<int64_t>(i) * P.hkv + h;
    const bool bad = __ldg(P.unit_bad + u) != 0;
    const int64_t base = base_i + static_cast<int64_t>(h) * ns;
    const int npre = pre > 0 ? static_cast<int>(cascade_splits(pre)) : 0;
    const int64_t cbase = pre > 0 ? (static_cast<int64_t>(rb.y) * P.hkv + h) * P.cas_np_max : 0;
    const int n_all = min(npre + ns, E);
    float ml[E][2 * GP], ov[E][GP];
#pragma unroll
    for (int k = 0; k < E; ++k) {
      if (k < n_all && k < npre) {
        const float* ml_p = P.cas_ml + (cbase + k) * GP * 2;
        const float* o_p = P.cas_o + (cbase + k) * GP * 128 + d;
#pragma unroll
        for (int q = 0; q < 2 * GP; ++q) ml[k][q] = __ldg(ml_p + q);
#pragma unroll
        for (int g = 0; g < GP; ++g) ov[k][g] = __ldg(o_p + g * 128);
      } else if (k < n_all) {
        const int64_t it = base + (k - npre);
        const float4* ml4 = reinterpret_cast<const float4*>(P.part_ml + it * GP * 2);
        const float4* o4 = reinterpret_cast<const float4*>(P.part_o + (it * 128 + d) * GP);
#pragma unroll
        for (int q = 0; q < GP / 2; ++q) {
          const float4 t = __ldg(ml4 + q);
          ml[k][4 * q] = t.x;
          ml[k][4 * q + 1] = t.y;
          ml[k][4 * q + 2] = t.z;
          ml[k][4 * q + 3] = t.w;
        }
#pragma unroll
        for (int q = 0; q < GP / 4; ++q) {
          const float4 t = __ldg(o4 + q);
          ov[k][4 * q] = t.x;
          ov[k][4 * q + 1] = t.y;
          ov[k][4 * q + 2] = t.z;
          ov[k][4 * q + 3] = t.w;
        }
      }
    }
    // merge_kernel's runs: run r folds entries [r * per, (r + 1) * per) from nothing, and
    // runs 1.. are then folded into run 0 in order
    const int per = (n_all + kMergeGroups - 1) / kMergeGroups;
    float M[GP], num[GP], den[GP];
#pragma unroll
    for (int r = 0; r < kMergeGroups; ++r) {
      float Mr[GP], nr[GP], dr[GP];
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        Mr[g] = -INFINITY;
        nr[g] = 0.f;
        dr[g] = 0.f;
      }
      const int e0 = min(n_all, r * per), e1 = min(n_all, e0 + per);
#pragma unroll
      for (int k = 0; k < E; ++k)
        if (k >= e0 && k < e1) merge_fold<GP>(Mr, nr, dr, ml[k], ov[k]);
      if (r == 0) {
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          M[g] = Mr[g];
          num[g] = nr[g];
          den[g] = dr[g];
        }
      } else if (r * per < n_all) {
        float mlr[2 * GP];
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          mlr[2 * g] = Mr[g];
          mlr[2 * g + 1] = dr[g];
        }
        merge_fold<GP>(M, num, den, mlr, nr);
      }
    }
    __nv_bfloat16* orow = P.out + (static_cast<int64_t>(ra.w) * P.hq + static_cast<int64_t>(h) * P.group) * 128 + d;
#pragma unroll
    for (int g = 0; g < GP; ++g)
      if (g < P.group) orow[g * 128] = __float2bfloat16_rn(bad ? 0.f : __fdividef(num[g], den[g]));
  }
}

template <int GP>
int launch_gp(const CUtensorMap& qm, const CUtensorMap& km, const CUtensorMap& vm, const DecodeParams& p, int grid,
              const Workspace& ws, bool may_split, int max_entries, int what, cudaStream_t s) {
  const int32_t* counters = ws.counters;
  const int32_t* merge_list = ws.merge_list;
  static uint64_t smem_set = 0;
  const int st = set_smem_once(reinterpret_cast<const void*>(decode_kernel<GP>), kSmemBytes, &smem_set);
  if (st) return st;
  cudaError_t e;
  if (what & kDecodeLaunch) {
    TraceScope trace(kTraceDecode, s);
    e = launch_k(decode_kernel<GP>, dim3(grid), dim3(kThreads), kSmemBytes, s, qm, km, vm, p);
    if (e != cudaSuccess) return cuda_status(e);
  }
  if (!may_split || !(what & kMergeLaunch)) return PKV_OK;  // (no context long enough to be split: nothing to merge)
  MergeParams m{p.out,          counters,  merge_list, p.dec_prefix,  p.qsl,     p.unit_bad,    p.part_o,
                p.part_ml,      p.seq_prefix, ws.seq_entry, ws.cas_o, ws.cas_ml, ws.cas_np_max, p.num_seqs,
                p.hkv,          p.group,   p.hq};
  // the list length is only known on the device: enough CTAs for every unit of a
  // full list, each exiting at once when the list is shorter
  const int64_t n_units = static_cast<int64_t>(p.num_seqs) * p.hkv;
  const int64_t cap = static_cast<int64_t>(grid) * 4;
  const int mgrid = static_cast<int>(n_units < cap ? n_units : cap);
  TraceScope trace(kTraceMerge, s);
  if (max_entries <= MergeSmall<GP>::kEntries) {
    const int64_t scap = static_cast<int64_t>(grid) * 16;
    return cuda_status(launch_k(merge_small_kernel<GP>, dim3(static_cast<unsigned>(n_units < scap ? n_units : scap)),
                                dim3(128), 0, s, m));
  }
  return cuda_status(launch_k(merge_kernel<GP>, dim3(mgrid), dim3(128 * kMergeGroups), 0, s, m));
}

}  // namespace

int launch_decode_tc(const AttnArgs& a, const Workspace& ws, int num_sms, uint32_t* err, cudaStream_t s, int what) {
  const int hkv = a.cache.num_kv_heads;
  const int group = a.num_q_heads / hkv;
  if (group > 16 || a.cache.head_dim != 128 || a.cache.dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
  const uint64_t rows = static_cast<uint64_t>(a.cache.num_blocks) * hkv * kBlock;
  if (rows >= (1ull << 31)) return PKV_ERR_UNSUPPORTED;
  if (a.num_tokens >= (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;
  const int gp = group <= 4 ? 4 : (group <= 8 ? 8 : 16);
  CUtensorMap qm, km, vm;
  int st = encode_tensor_map_2d(&km, a.k_cache, 128, rows, 256, 64, 16);
  if (st) return st;
  st = encode_tensor_map_2d(&vm, a.v_cache, 128, rows, 256, 64, 16);
  if (st) return st;
  // q viewed as [token][head][128]: one box = the GP query heads of a kv head, one token
  const uint64_t qdims[3] = {128, static_cast<uint64_t>(a.num_q_heads), static_cast<uint64_t>(a.num_tokens)};
  const uint64_t qstrides[2] = {256, static_cast<uint64_t>(a.num_q_heads) * 256};
  const uint32_t qbox[3] = {64, static_cast<uint32_t>(gp), 1};
  st = encode_tensor_map_3d(&qm, a.q, qdims, qstrides, qbox);
  if (st) return st;
  DecodeParams p;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.bt = a.block_tables;
  p.seq_lens = a.seq_lens;
  p.qsl = a.qsl;
  p.dec_prefix = ws.dec_prefix;
  p.dec_order = ws.dec_order;
  p.dec_start = ws.dec_start;
  p.dec_pos = ws.dec_pos;
  p.order_flag = ws.counters + kDecOrderSlot;
  p.queue = ws.counters + 0;
  p.unit_bad = ws.unit_bad;
  p.part_o = ws.part_o;
  p.part_ml = ws.part_ml;
  p.seq_prefix = ws.seq_prefix;
  p.seq_entry = ws.seq_entry;
  p.cas_o = ws.cas_o;
  p.cas_ml = ws.cas_ml;
  p.cas_np_max = ws.cas_np_max;
  p.err = err;
  p.num_blocks = a.cache.num_blocks;
  p.num_tokens = a.num_tokens;
  p.num_seqs = a.num_seqs;
  p.max_blocks = a.max_blocks;
  p.hkv = hkv;
  p.group = group;
  p.gp = gp;
  p.hq = a.num_q_heads;
  p.split_keys = kSplitKeys;
  // Measured on GB300 (A/B of the same kernel, CUDA events): an L2 evict-first hint on the K/V
  // tiles speeds decode-only steps (batched decode 91 -> 85 us, shared-prefix step 100 -> 91 us,
  // long-context decode launch 627 -> 613 us) and slows the mixed step's decode launch, which
  // follows 67 MB of new-token writes (2.701 -> 2.742 ms).  So only batches without prefill
  // chunks take the hint.
  p.kv_evict_first = a.max_query_len <= 1 ? 1 : 0;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  // the planner never splits a request longer than the host bound, and none up to kNoSplitKeys
  const bool may_split = a.max_seq_len > kNoSplitKeys;
  // the most partials one unit can fold: its own key splits plus its prefix's splits
  const int max_entries = static_cast<int>(decode_splits(a.max_seq_len)) +
                          (ws.seq_prefix ? ws.cas_np_max : 0);
  if (gp == 4) return launch_gp<4>(qm, km, vm, p, num_sms, ws, may_split, max_entries, what, s);
  if (gp == 8) return launch_gp<8>(qm, km, vm, p, num_sms, ws, may_split, max_entries, what, s);
  return launch_gp<16>(qm, km, vm, p, num_sms, ws, may_split, max_entries, what, s);
}

}  // namespace pkv
