// k_prefill.cu -- causal varlen chunked prefill on tcgen05 tensor cores (bf16, head_dim 128).
//
// What it computes ("vLLM's PagedAttention" teardown, section "Continuous
// batching": a long prompt is split across steps by chunked prefill; a chunk
// attends to its cached prior context and, causally, to itself).  For a request
// with q_len query tokens and context seq_len, query j sits at position
// seq_len - q_len + j and sees keys 0..that position, gathered through the block
// table like the decode path.
//
// Work decomposition.  The G query heads that share a kv head are folded into the
// 128 rows of one MMA tile: R = 128 / GP queries x GP heads (GP = G rounded up to
// 4, 8 or 16), row r <-> (query j0 + r / GP, head r % GP).  An item is a pair of
// query tiles of one (request, kv head) -- tiles 2p + 1 and 2p, the later one as
// tile 0 of the item -- and every K/V tile it loads feeds both: the later tile sees
// the earlier one's keys and at most one tile more.  Items come from an atomic queue
// to persistent CTAs, one per SM, in the planner's order: the heaviest pairs of the
// whole batch first.
//
// Per CTA (320 threads):
//   warp 0     producer: TMA-loads the two Q tiles (3-D boxes over [token][head][dim])
//              and, per 128-key tile, 2 K and 2 V boxes per 16-token block from the
//              block's physical location (the block-table gather), 128-byte swizzle.
//              K tiles go into a 2-slot ring and V tiles into a 3-slot one, each tile's
//              K and V issued together.
//   warp 1     MMA issuer; one thread runs the whole loop, so no warp convergence sits
//              between two MMA bursts.  Per key tile j and query tile w it issues O_w +=
//              P_w(j-1) V(j-1), then S_w(j) = Q_w K(j)^T.  S_w lives in TMEM; the softmax writes
//              P_w as bf16 over the first 64 of S_w's columns and the P V MMA reads its
//              A operand from there.  MMAs issued by one thread complete in order, so
//              S_w(j+1) cannot overwrite P_w(j) before P_w(j) V(j) has read it, and S_w(j)
//              complete means P_w(j-1) V(j-1) is complete too.  While one tile's softmax
//              runs, the tensor core works on the other tile.  P_w(j) arrives in two
//              halves of 64 keys, and each half's P V is issued as soon as it is there.
//   warps 2-5  softmax of query tile 0, warps 6-9 of tile 1: thread r owns row r.  Per
//              key tile it reads its S row from TMEM twice -- for the row maximum, then
//              for the exponents -- so that no whole row is held in registers, applies the
//              causal mask, and keeps a per-row reference maximum; only when a row's
//              maximum grows by more than 2^8 does the warp rescale its O rows in TMEM.
//              Two scores go through each packed fp32x2 FMA and add, and each
//              three-input max.  The softmax warps also release the K and V ring slots
//              (plain arrivals: S_w(j) complete means every earlier MMA is).  The final
//              O / l is stored per row, the whole row loaded from TMEM first.
// All waits are bounded (see ptx.cuh); a timeout raises the CTA abort flag.
//
// Shared-prefix (cascade) mode, kCas = true.  The same pipeline attends the member
// decodes of a prefix group to the group's shared prefix: an item is (group, two
// tiles of R member requests each, kv head, key split of kCascadeSplitKeys prefix
// keys), a tile's 128 rows are (member, head) pairs whose query rows the softmax warps
// gather with plain loads into the swizzled Q tile (members are scattered over the
// batch), every key of the split is visible to every row (all members sit past the
// prefix), and each row leaves its unnormalised accumulator, reference maximum and
// sum as a partial for the split merge instead of a final output.  The prefix's K/V
// are read once per (group, kv head, split, 2R members).
#include "ptx.cuh"
#include "pkv_internal.cuh"

namespace pkv {
namespace {

constexpr int kThreads = 320;
constexpr int kKStages = 2;               // K tiles in flight
constexpr int kVStages = 3;               // V tiles in flight (a V tile is needed later than its K)
constexpr int kHalfBytes = 16384;          // 128 rows x 128 B
constexpr int kTileBytes = 2 * kHalfBytes;  // 128 x 128 bf16, K-major, two 64-column halves
constexpr int kRing = 4;
constexpr uint32_t kTmemCols = 512;         // S_0, S_1 (cols 0, 128; P_w over S_w's first 64), O_0, O_1 (256, 384)
constexpr uint32_t kOCol = 256;
constexpr int kBlocksPerTile = kTileKeys / kBlock;
constexpr float kRescaleThreshold = 8.0f;   // log2 units: rescale O when a row max grows by > 2^8
static_assert(kPrefillTilesPerItem == 2, "an item is a pair of query tiles");

struct alignas(16) PItem {
  int32_t idx;                    // -1: queue exhausted
  int32_t seq, head, split;       // seq: the request (cascade: the prefix group)
  int32_t q_len, ctx, t0, valid;  // t0: the request's first token row
  int32_t ks, pad0, pad1, pad2;   // the item's keys start at ks (cascade: the split's first key)
  int32_t nt[2], kend[2];         // query tile w: keys [ks, kend[w]) in nt[w] tiles (0: no tile w)
  int32_t j0[2], nq[2];           // its first query (cascade: first member entry) and how many
  int32_t qt[2], pad3, pad4;      // its query-tile index (-1: none)
};

struct Ctl {
  // K and V tiles have rings of their own: a K tile is released when the S MMAs of
  // both query tiles have read it, a V tile when both P V MMAs have
  uint64_t kfull[kKStages], kempty[kKStages], vfull[kVStages], vempty[kVStages];
  uint64_t s_full[2], o_full[2], o_free[2];  // per query tile
  uint64_t p_full[2][2];                     // per query tile: P of keys 0-63, then of keys 64-127
  uint64_t q_full[2], q_free[2];
  uint64_t item_full[kRing], item_empty[kRing];
  uint64_t drain;
  PItem ring[kRing];
  int bad[kRing];
  uint32_t tmem_base;
  int abort_flag;
};

constexpr int kSmemBytes = (2 /*Q*/ + kKStages + kVStages) * kTileBytes + static_cast<int>(sizeof(Ctl)) + 1024;
static_assert(kSmemBytes <= 232448, "prefill shared memory");

struct PrefillParams {
  __nv_bfloat16* out;
  const int32_t* bt;
  const int32_t* seq_lens;
  const int32_t* qsl;
  const int32_t* pre_prefix;
  const int32_t* pre_order;  // pairs heaviest first: (id pre_prefix[i] / hkv + pl, request i) per position
  int32_t* queue;
  uint32_t* err;
  int64_t num_blocks;
  int64_t num_tokens;
  int32_t num_seqs, max_blocks, hkv, group, gp, rows_q, hq;
  int32_t out_v8;  // out is 32-byte aligned (every row then is): whole-sector stores
  float scale_log2;
  // shared-prefix mode
  const __nv_bfloat16* q;
  const int32_t* cas_tables;
  const int32_t* cas_blocks;
  const int32_t* cas_start;
  const int32_t* cas_members;
  const int32_t* cas_prefix;  // the planner's item prefix (used without cas_concurrent)
  float* cas_o;
  float* cas_ml;
  int32_t cas_max_blocks, cas_groups, cas_np_max;
  int32_t cas_tiles;       // query tiles per cascade item: 2, or 1 (tile 1 of every item absent)
  int32_t cas_concurrent;  // items from the hint alone, beside the planning launch (groups <= 32)
  int32_t after_decode;    // right after this call's decode kernel, which it need not wait for
};

// Three-input maximum / minimum (one instruction on sm_100 and later).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float r;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}
// (ya, yb) = (xa, xb) * s + t and (a0, a1) += (b0, b1): one packed fp32x2 instruction
// each, rounded like the scalar forms lane by lane.
__device__ __forceinline__ void ffma2(float& ya, float& yb, float xa, float xb, float s, float t) {
  asm("{\n\t.reg .b64 x, y, m, c;\n\t"
      "mov.b64 x, {%2, %3};\n\t"
      "mov.b64 m, {%4, %4};\n\t"
      "mov.b64 c, {%5, %5};\n\t"
      "fma.rn.f32x2 y, x, m, c;\n\t"
      "mov.b64 {%0, %1}, y;\n\t}"
      : "=f"(ya), "=f"(yb)
      : "f"(xa), "f"(xb), "f"(s), "f"(t));
}
__device__ __forceinline__ void fadd2(float& a0, float& a1, float b0, float b1) {
  asm("{\n\t.reg .b64 a, b;\n\t"
      "mov.b64 a, {%0, %1};\n\t"
      "mov.b64 b, {%2, %3};\n\t"
      "add.rn.f32x2 a, a, b;\n\t"
      "mov.b64 {%0, %1}, a;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(b0), "f"(b1));
}

// The extremum of one S row of 128 raw scores from TMEM (taddr: the row's first
// column): the maximum, or for kPos false the minimum (a negative scale turns it into
// the maximum of scale * s).  With kMask, keys from nvis on do not count.  Each
// 32-column piece is loaded while the previous one is reduced.
template <bool kPos, bool kMask>
__device__ __forceinline__ float row_extremum(uint32_t taddr, int nvis) {
  const float hidden = kPos ? -INFINITY : INFINITY;
  float mx[8];  // eight independent running extrema keep the dependency chains short
#pragma unroll
  for (int k = 0; k < 8; ++k) mx[k] = hidden;
  uint32_t a[32], b[32];
  tmem_ld32_issue(taddr, a);
  tmem_ld32_wait(a);
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    uint32_t(&cur)[32] = (h & 1) ? b : a;
    uint32_t(&nxt)[32] = (h & 1) ? a : b;
    if (h < 3) tmem_ld32_issue(taddr + 32 * (h + 1), nxt);
#pragma unroll
    for (int k = 0; k < 32; k += 2) {  // two scores per three-input instruction
      const float xa = (!kMask || 32 * h + k < nvis) ? __uint_as_float(cur[k]) : hidden;
      const float xb = (!kMask || 32 * h + k + 1 < nvis) ? __uint_as_float(cur[k + 1]) : hidden;
      const int c = (k >> 1) & 7;
      mx[c] = kPos ? fmax3(mx[c], xa, xb) : fmin3(mx[c], xa, xb);
    }
    if (h < 3) tmem_ld32_wait(nxt);
  }
  return kPos ? fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])))
              : fminf(fminf(fminf(mx[0], mx[1]), fminf(mx[2], mx[3])), fminf(fminf(mx[4], mx[5]), fminf(mx[6], mx[7])));
}

// The exponents 2^(scale * s - m_ref) of one S row (masked keys: 0, with kMask),
// written back as bf16 P over the row's first 64 columns; returns the row sum.  Each
// 32-column piece is loaded while the previous one is converted, and the 16 P columns
// a piece gives land on columns this thread has already read.  A masked key's scaled
// score is set to -inf before its exponent (an infinite raw score would give NaN at
// scale 0).  Once the P of keys 0-63 is stored, half() runs (the hand-over of that
// half) while the third piece's load is in flight.
template <bool kMask, typename Half>
__device__ __forceinline__ float row_exp_to_p(uint32_t taddr, int nvis, float scale, float m_ref, Half&& half) {
  float ls[4] = {0.f, 0.f, 0.f, 0.f};  // the row sum in four independent parts (two packed pairs)
  uint32_t a[32], b[32];
  tmem_ld32_issue(taddr, a);
  tmem_ld32_wait(a);
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    uint32_t(&cur)[32] = (h & 1) ? b : a;
    uint32_t(&nxt)[32] = (h & 1) ? a : b;
    if (h < 3) tmem_ld32_issue(taddr + 32 * (h + 1), nxt);
    uint32_t pw[16];
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const int k = 32 * h + 2 * q;
      float ya, yb;
      ffma2(ya, yb, __uint_as_float(cur[2 * q]), __uint_as_float(cur[2 * q + 1]), scale, -m_ref);
      const float pa = ex2_approx((!kMask || k < nvis) ? ya : -INFINITY);
      const float pb = ex2_approx((!kMask || k + 1 < nvis) ? yb : -INFINITY);
      if (q & 1) fadd2(ls[2], ls[3], pa, pb);
      else fadd2(ls[0], ls[1], pa, pb);
      __nv_bfloat162 h2 = __floats2bfloat162_rn(pa, pb);
      pw[q] = *reinterpret_cast<uint32_t*>(&h2);
    }
    tmem_st16(taddr + 16 * h, pw);
    if (h == 1) half();
    if (h < 3) tmem_ld32_wait(nxt);
  }
  return (ls[0] + ls[1]) + (ls[2] + ls[3]);
}

// One 32-byte global store (a whole sector) of eight 32-bit words; p is 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&w)[8]) {
  asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
               "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

__device__ __forceinline__ void raise_abort(Ctl& c, uint32_t* err) {
  *reinterpret_cast<volatile int*>(&c.abort_flag) = 1;
  flag_error(err, kErrTimeout);
}

__device__ PItem make_item(const PrefillParams& P, int idx, int total) {
  PItem r{};
  r.qt[0] = r.qt[1] = -1;
  if (idx >= total) {
    r.idx = -1;
    return r;
  }
  // the planner's order of (request, pair) units, heaviest first, with each unit's
  // request; the kv heads of a unit are consecutive items
  const int2 ord = reinterpret_cast<const int2*>(P.pre_order)[idx / P.hkv];
  const int unit = ord.x;
  const int i = ord.y >= 0 && ord.y < P.num_seqs ? ord.y : 0;
  const int base = P.pre_prefix[i];
  const int cnt = P.pre_prefix[i + 1] - base;
  const int npair = cnt / P.hkv;
  const int pl = unit - base / P.hkv;
  r.idx = idx;
  r.seq = i;
  if (npair <= 0 || ord.y != i || pl < 0 || pl >= npair) return r;  // inconsistent plan: invalid item
  const int pair = npair - 1 - pl;  // pl = 0: the request's latest (heaviest) query tiles
  r.head = idx % P.hkv;
  const int64_t q0 = P.qsl[i], q1 = P.qsl[i + 1];
  const int64_t L = P.seq_lens[i];
  const int64_t q_len = q1 - q0;
  r.q_len = static_cast<int32_t>(q_len);
  r.t0 = static_cast<int32_t>(q0);
  // tile 0 of the item is the later query tile of the pair, tile 1 the earlier one
  const int64_t nqt = q_len > 0 ? (q_len + P.rows_q - 1) / P.rows_q : 0;
  const int hi_t = 2 * pair + 1, lo_t = 2 * pair;
  r.qt[0] = hi_t < nqt ? hi_t : lo_t;
  r.qt[1] = hi_t < nqt ? lo_t : -1;
  const bool ok = q_len > 1 && L >= q_len && (L + kBlock - 1) / kBlock <= P.max_blocks && q0 >= 0 &&
                  q1 <= P.num_tokens && (q_len + 2 * P.rows_q - 1) / (2 * P.rows_q) == npair && lo_t < nqt;
  r.valid = ok ? 1 : 0;
  if (ok) {
    r.ctx = static_cast<int32_t>(L - q_len);
    for (int w = 0; w < 2; ++w) {
      if (r.qt[w] < 0) continue;
      r.j0[w] = r.qt[w] * P.rows_q;
      const int64_t left = q_len - r.j0[w];
      r.nq[w] = static_cast<int32_t>(left < P.rows_q ? left : P.rows_q);
      r.kend[w] = r.ctx + r.j0[w] + r.nq[w];  // keys [0, kend) are visible to some row of the tile
      r.nt[w] = (r.kend[w] + kTileKeys - 1) / kTileKeys;
    }
  }
  return r;
}

// Cascade items of one group: its member entries in tiles of cas_tiles * rows_q (the
// planner counts them the same way) x kv heads x key splits of the prefix.
__device__ __forceinline__ int cas_group_items(const PrefillParams& P, int e0, int e1, int pb) {
  if (pb < 1 || pb > P.cas_max_blocks || e1 <= e0) return 0;
  const int rows = P.cas_tiles * P.rows_q;
  return (e1 - e0 + rows - 1) / rows * P.hkv * static_cast<int>(cascade_splits(int64_t(pb) * kBlock));
}

// A cascade item: item `local` of group g (entries e0 .. e1 - 1, pb prefix blocks), as
// (member tile pair, kv head, key split).
__device__ PItem make_cas_item(const PrefillParams& P, int idx, int g, int local, int e0, int e1, int pb) {
  PItem r{};
  r.qt[0] = r.qt[1] = -1;
  if (g < 0) {
    r.idx = -1;
    return r;
  }
  r.idx = idx;
  r.seq = g;
  if (pb < 1 || pb > P.cas_max_blocks || e1 <= e0 || local < 0) return r;  // inconsistent: invalid item
  const int np = static_cast<int>(cascade_splits(int64_t(pb) * kBlock));
  r.split = local % np;
  r.head = (local / np) % P.hkv;
  const int pq = local / np / P.hkv;  // the item's tile group of member entries
  r.ks = r.split * kCascadeSplitKeys;
  const int kend = min(pb * kBlock, r.ks + kCascadeSplitKeys);
  const int nt = (kend - r.ks + kTileKeys - 1) / kTileKeys;
  for (int w = 0; w < 2; ++w) {
    r.qt[w] = P.cas_tiles * pq + w;
    r.j0[w] = e0 + r.qt[w] * P.rows_q;
    r.nq[w] = w < P.cas_tiles ? min(P.rows_q, e1 - r.j0[w]) : 0;
    if (r.nq[w] > 0) {
      r.kend[w] = kend;
      r.nt[w] = nt;
    } else {
      r.nq[w] = 0;
      r.qt[w] = -1;
    }
  }
  r.valid = (r.nq[0] > 0 && r.ks < kend) ? 1 : 0;
  return r;
}

// ------------------------------------------------------------------ producer warp
template <bool kCas>
__device__ void producer_warp(const PrefillParams& P, const CUtensorMap* qmap, const CUtensorMap* kmap,
                              const CUtensorMap* vmap, Ctl& c, uint8_t* qbuf, uint8_t* kbuf, uint8_t* vbuf) {
  const int lane = threadIdx.x & 31;
  // cascade items beside the planner: lane g holds group g's entries, prefix length,
  // item count and the exclusive prefix of the counts
  int ce0 = 0, ce1 = 0, cpb = 0, ccnt = 0, cpfx = 0;
  int total;
  if (kCas && P.cas_concurrent) {
    if (lane < P.cas_groups) {
      ce0 = __ldg(P.cas_start + lane);
      ce1 = __ldg(P.cas_start + lane + 1);
      cpb = __ldg(P.cas_blocks + lane);
      ccnt = cas_group_items(P, ce0, ce1, cpb);
    }
    int incl = ccnt;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += y;
    }
    cpfx = incl - ccnt;
    total = __shfl_sync(0xffffffffu, incl, 31);
  } else {
    total = kCas ? P.cas_prefix[P.cas_groups] : P.pre_prefix[P.num_seqs];
  }
  volatile int* abort_flag = &c.abort_flag;
  uint32_t it = 0, tk = 0, tv = 0;  // items; K and V tiles issued
  uint32_t qc[2] = {0, 0};          // Q tiles loaded per tile slot
  bool ok = true;
  while (ok) {
    const int slot = it % kRing;
    if (!mbar_wait(&c.item_empty[slot], ((it / kRing) & 1) ^ 1, abort_flag)) {
      ok = false;
      break;
    }
    if (kCas) {
      // cascade items are alike, so CTA b takes items b, b + grid, b + 2 grid, ...; the
      // item's group is the last one whose first item is not past it
      const int idx = static_cast<int>(blockIdx.x + it * gridDim.x);
      int g = -1, local = 0, e0 = 0, e1 = 0, pb = 0;
      if (idx < total) {
        if (P.cas_concurrent) {
          const unsigned m = __ballot_sync(0xffffffffu, ccnt > 0 && cpfx <= idx);
          g = m ? 31 - __clz(m) : 0;
          local = idx - __shfl_sync(0xffffffffu, cpfx, g);
          e0 = __shfl_sync(0xffffffffu, ce0, g);
          e1 = __shfl_sync(0xffffffffu, ce1, g);
          pb = __shfl_sync(0xffffffffu, cpb, g);
          if (!m) local = -1;
        } else if (lane == 0) {
          int lo = 0, hi = P.cas_groups - 1;
          while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (P.cas_prefix[mid] <= idx) lo = mid; else hi = mid - 1;
          }
          g = lo;
          local = idx - P.cas_prefix[lo];
          e0 = P.cas_start[lo];
          e1 = P.cas_start[lo + 1];
          pb = P.cas_blocks[lo];
        }
      }
      if (lane == 0) {
        c.ring[slot] = make_cas_item(P, idx, g, local, e0, e1, pb);
        c.bad[slot] = 0;
        mbar_arrive(&c.item_full[slot]);
      }
    } else if (lane == 0) {
      // every CTA's first item is its own index; later ones come off the queue after those
      const int idx = it == 0 ? static_cast<int>(blockIdx.x) : static_cast<int>(gridDim.x) + atomicAdd(P.queue, 1);
      c.ring[slot] = make_item(P, idx, total);
      c.bad[slot] = 0;
      mbar_arrive(&c.item_full[slot]);
    }
    __syncwarp();
    const PItem info = c.ring[slot];
    ++it;
    if (info.idx < 0) break;
    if (!info.valid) continue;
    if (!kCas) {  // (cascade: the softmax warps gather Q)
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        if (!ok) break;
        if (info.nt[w] == 0) continue;
        if (!mbar_wait(&c.q_free[w], (qc[w] & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          uint8_t* q = qbuf + w * kTileBytes;
          mbar_arrive_expect_tx(&c.q_full[w], kTileBytes);
          const int32_t y = info.head * P.group, z = info.t0 + info.j0[w];
          tma_load_3d(q, qmap, &c.q_full[w], 0, y, z, l2_policy_evict_first());
          tma_load_3d(q + kHalfBytes, qmap, &c.q_full[w], 64, y, z, l2_policy_evict_first());
        }
        __syncwarp();
        ++qc[w];
      }
      if (!ok) break;
    }
    const int32_t* btrow = kCas ? P.cas_tables + static_cast<int64_t>(info.seq) * P.cas_max_blocks
                                : P.bt + static_cast<int64_t>(info.seq) * P.max_blocks;
    // per key tile of the item (tile 0's keys cover tile 1's): K, then V, each into
    // its ring once the MMAs that read the ring slot's previous tile are done
    for (int j = 0; j < info.nt[0]; ++j) {
      const int sk = tk % kKStages;
      if (!mbar_wait(&c.kempty[sk], ((tk / kKStages) & 1) ^ 1, abort_flag)) {
        ok = false;
        break;
      }
      const int t0 = info.ks + j * kTileKeys;
      const int nblk = min(kBlocksPerTile, (info.kend[0] - t0 + kBlock - 1) / kBlock);
      int id = 0;
      bool bad = false;
      if (lane < nblk) {
        id = __ldg(btrow + t0 / kBlock + lane);
        if (id < 0 || id >= P.num_blocks) {
          bad = true;
          id = 0;
        }
      }
      if (__any_sync(0xffffffffu, bad)) {
        if (bad) flag_error(P.err, kErrBlockId);
        if (lane == 0) c.bad[slot] = 1;
      }
      __syncwarp();
      const int32_t row = (id * P.hkv + info.head) * kBlock;
      if (lane == 0) mbar_arrive_expect_tx(&c.kfull[sk], static_cast<uint32_t>(nblk) * 4096u);
      __syncwarp();
      if (lane < nblk) {
        uint8_t* d = kbuf + sk * kTileBytes + lane * 2048;
        tma_load_2d(d, kmap, &c.kfull[sk], 0, row);
        tma_load_2d(d + kHalfBytes, kmap, &c.kfull[sk], 64, row);
      }
      ++tk;
      const int sv = tv % kVStages;
      if (!mbar_wait(&c.vempty[sv], ((tv / kVStages) & 1) ^ 1, abort_flag)) {
        ok = false;
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(&c.vfull[sv], static_cast<uint32_t>(nblk) * 4096u);
      __syncwarp();
      if (lane < nblk) {
        uint8_t* d = vbuf + sv * kTileBytes + lane * 2048;
        tma_load_2d(d, vmap, &c.vfull[sv], 0, row);
        tma_load_2d(d + kHalfBytes, vmap, &c.vfull[sv], 64, row);
      }
      ++tv;
    }
  }
  if (!ok && !*abort_flag && lane == 0) raise_abort(c, P.err);
  if (*abort_flag) {
    // let copies already issued land before the CTA's shared memory goes away
    for (uint32_t cnt = tk > static_cast<uint32_t>(kKStages) ? tk - kKStages : 0; cnt < tk; ++cnt)
      mbar_wait(&c.kfull[cnt % kKStages], (cnt / kKStages) & 1, nullptr);
    for (uint32_t cnt = tv > static_cast<uint32_t>(kVStages) ? tv - kVStages : 0; cnt < tv; ++cnt)
      mbar_wait(&c.vfull[cnt % kVStages], (cnt / kVStages) & 1, nullptr);
#pragma unroll
    for (int w = 0; w < 2; ++w)
      if (qc[w] > 0) mbar_wait(&c.q_full[w], (qc[w] - 1) & 1, nullptr);
  }
}

// ------------------------------------------------------------------ MMA warp
__device__ void mma_warp(const PrefillParams& P, Ctl& c, uint8_t* qbuf, uint8_t* kbuf, uint8_t* vbuf, uint32_t tmem) {
  // One thread issues every MMA and runs this whole loop alone: the other lanes wait at
  // the end, so no warp-wide convergence sits between two MMA bursts.
  if ((threadIdx.x & 31) == 0) {
    const uint32_t idesc_s = umma_idesc_bf16(128, 128, false, false);
    const uint32_t idesc_o = umma_idesc_bf16(128, 128, false, true);
    const uint64_t qdesc[2] = {umma_smem_desc(smem_u32(qbuf), 16, 1024, kLayout128B),
                               umma_smem_desc(smem_u32(qbuf + kTileBytes), 16, 1024, kLayout128B)};
    volatile int* abort_flag = &c.abort_flag;
    uint32_t it = 0, tk = 0, tv = 0;
    uint32_t qc0 = 0, qc1 = 0, pc0 = 0, pc1 = 0, ic0 = 0, ic1 = 0;  // per tile slot: Q tiles, P tiles, items
    bool issued = false, ok = true;
    // O_w += P_w V over keys 64 hf .. 64 hf + 63 (acc false: the item's first, O_w = P_w V),
    // V in ring slot sv; P_w is bf16 over S_w's first 64 columns
    auto issue_pv = [&](int w, int sv, bool acc, int hf) {
      const uint64_t bd = umma_smem_desc(smem_u32(vbuf + sv * kTileBytes), kHalfBytes, 1024, kLayout128B);
#pragma unroll
      for (int k4 = 0; k4 < 4; ++k4) {
        const int kk = 4 * hf + k4;
        umma_f16_ts(tmem + kOCol + 128 * w, tmem + 128 * w + 8 * kk, umma_desc_advance(bd, kk * 2048), idesc_o,
                    (acc || kk > 0) ? 1u : 0u);
      }
    };
    // S_w = Q_w K^T, K in ring slot sk
    auto issue_s = [&](int w, int sk) {
      const uint64_t b = umma_smem_desc(smem_u32(kbuf + sk * kTileBytes), 16, 1024, kLayout128B);
#pragma unroll
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
        umma_f16_ss(tmem + 128 * w, umma_desc_advance(qdesc[w], off), umma_desc_advance(b, off), idesc_s, kk > 0);
      }
    };
    while (ok) {
      const int slot = it % kRing;
      if (!mbar_wait(&c.item_full[slot], (it / kRing) & 1, abort_flag)) {
        ok = false;
        break;
      }
      const PItem info = c.ring[slot];
      ++it;
      if (info.idx < 0) break;
      if (info.valid) {
        const int nt0 = info.nt[0], nt1 = info.nt[1];
        ok = (nt0 == 0 || mbar_wait(&c.q_full[0], qc0 & 1, abort_flag)) &&
             (nt1 == 0 || mbar_wait(&c.q_full[1], qc1 & 1, abort_flag));
        // Step j: P_0(j-1) V(j-1), S_0(j), P_1(j-1) V(j-1), S_1(j), each P V in two halves
        // of 64 keys issued as the softmax hands them over.  An MMA issue returns only as
        // the tensor core takes it in, so the MMAs are issued back to back: the waits
        // between bursts are for the halves of P, and the K wait sits right after an MMA
        // burst, where the tensor core still has queued work.  V needs no wait: tile 0's
        // softmax warps hand the first half of P_0(j) over only after they have seen V(j)
        // land and zeroed its rows past the context, and P_1(j) V(j) is issued after
        // P_0(j) V(j).  The K and V ring slots are released
        // by the softmax warps, which learn from their own S and O barriers when the MMAs
        // reading a slot are done; a commit here would hold this thread for a queue slot
        // each time.  The item's first P V restarts O_w, once the previous item's O_w was
        // read out.
        for (int j = 0; j <= nt0 && ok; ++j) {
          const int sk = tk % kKStages, sv = tv % kVStages;  // K(j), V(j-1)
          if (j > 0) {
            if (!mbar_wait(&c.p_full[0][0], pc0 & 1, abort_flag) ||
                (j == 1 && !mbar_wait(&c.o_free[0], (ic0 & 1) ^ 1, abort_flag))) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(0, sv, j > 1, 0);
            if (!mbar_wait(&c.p_full[0][1], pc0 & 1, abort_flag)) {
              ok = false;
              break;
            }
            ++pc0;
            tc_fence_after();
            issue_pv(0, sv, j > 1, 1);
            if (j == nt0) umma_commit(&c.o_full[0]);
          }
          if (j < nt0) {
            if (!mbar_wait(&c.kfull[sk], (tk / kKStages) & 1, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_s(0, sk);
            umma_commit(&c.s_full[0]);
            if (j == nt0 - 1) umma_commit(&c.q_free[0]);
            issued = true;
          }
          if (j > 0 && j - 1 < nt1) {
            if (!mbar_wait(&c.p_full[1][0], pc1 & 1, abort_flag) ||
                (j == 1 && !mbar_wait(&c.o_free[1], (ic1 & 1) ^ 1, abort_flag))) {
              ok = false;
              break;
            }
            tc_fence_after();
            issue_pv(1, sv, j > 1, 0);
            if (!mbar_wait(&c.p_full[1][1], pc1 & 1, abort_flag)) {
              ok = false;
              break;
            }
            ++pc1;
            tc_fence_after();
            issue_pv(1, sv, j > 1, 1);
            if (j == nt1) umma_commit(&c.o_full[1]);
          }
          if (j < nt1) {
            tc_fence_after();
            issue_s(1, sk);
            umma_commit(&c.s_full[1]);
            if (j == nt1 - 1) umma_commit(&c.q_free[1]);
          }
          if (j < nt0) ++tk;
          if (j > 0) ++tv;
        }
        if (nt0 > 0) {
          ++qc0;
          ++ic0;
        }
        if (nt1 > 0) {
          ++qc1;
          ++ic1;
        }
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
template <bool kCas>
__device__ void softmax_warps(const PrefillParams& P, Ctl& c, uint8_t* qbuf, uint8_t* vbuf, uint32_t tmem) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wq = warp & 3;        // TMEM lane quarter this warp may access
  const int w = (warp - 2) >> 2;  // the item's query tile this warpgroup owns
  const int r = wq * 32 + lane;   // tile row
  const uint32_t lane_off = static_cast<uint32_t>(wq * 32) << 16;
  const uint32_t s_col = 128u * w, o_col = kOCol + 128u * w;
  uint8_t* qtile = qbuf + w * kTileBytes;
  volatile int* abort_flag = &c.abort_flag;
  uint32_t it = 0, tc = 0, ic = 0, qc = 0, vc = 0;  // items, S tiles, own items, gathered Q tiles, V tiles
  bool ok = true;
  const int rj = r / P.gp, rg = r % P.gp;  // query offset and head of this row within a tile
  const float scale = P.scale_log2;
  const bool pos_scale = scale >= 0.f;

  while (ok) {
    const int slot = it % kRing;
    if (!mbar_wait(&c.item_full[slot], (it / kRing) & 1, abort_flag)) {
      ok = false;
      break;
    }
    const PItem info = c.ring[slot];
    ++it;
    if (info.idx < 0) break;
    if (!info.valid) {
      if (kCas) {
        if (r == 0 && w == 0) flag_error(P.err, kErrLength);
      } else {
        if (r == 0 && w == 0 && info.head == 0) flag_error(P.err, kErrLength);
        const int64_t q0 = P.qsl[info.seq], q1 = P.qsl[info.seq + 1];
        const int qt = w ? info.qt[1] : info.qt[0];
        const int64_t jj = static_cast<int64_t>(qt) * P.rows_q + rj;
        if (qt >= 0 && q0 >= 0 && q1 <= P.num_tokens && q0 + jj < q1 && rg < P.group) {
          __nv_bfloat16* zrow = P.out + ((q0 + jj) * P.hq + static_cast<int64_t>(info.head) * P.group + rg) * 128;
          for (int k = 0; k < 16; ++k) reinterpret_cast<uint4*>(zrow)[k] = make_uint4(0, 0, 0, 0);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.item_empty[slot]);
      continue;
    }
    // this warpgroup's query tile of the item
    const int nt = w ? info.nt[1] : info.nt[0];
    const int tj0 = w ? info.j0[1] : info.j0[0];
    const int tnq = w ? info.nq[1] : info.nq[0];
    const int tkend = w ? info.kend[1] : info.kend[0];
    if (nt == 0) {  // the item has one query tile only
      vc += info.nt[0];
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.item_empty[slot]);
      continue;
    }
    const int j_row = tj0 + rj;
    const bool row_out = rj < tnq && rg < P.group;  // a real (token, head) row
    __nv_bfloat16* orow = P.out + ((static_cast<int64_t>(info.t0) + j_row) * P.hq +
                                   static_cast<int64_t>(info.head) * P.group + rg) * 128;
    // this row's member entry (cascade) and its query row: a listed request with one new
    // token (the planner decides later which entries the decode kernel folds in)
    const int entry = tj0 + rj;
    int64_t crow = -1;
    if (kCas && rj < tnq) {
      const int i = __ldg(P.cas_members + entry);
      if (i >= 0 && i < P.num_seqs) {
        const int64_t q0 = __ldg(P.qsl + i), q1 = __ldg(P.qsl + i + 1);
        if (q0 >= 0 && q1 == q0 + 1 && q1 <= P.num_tokens) crow = q0;
      }
    }
    const bool cas_live = kCas && crow >= 0;
    if (kCas) {
      // gather the query row of (member, head) into the swizzled K-major Q tile once
      // the previous item's last S = Q K^T of this tile slot has read it
      if (!mbar_wait(&c.q_free[w], (qc & 1) ^ 1, abort_flag)) {
        ok = false;
        break;
      }
      uint4 qv[16];
      if (cas_live && rg < P.group) {
        const int64_t t = crow;
        const uint4* src = reinterpret_cast<const uint4*>(
            P.q + (t * P.hq + static_cast<int64_t>(info.head) * P.group + rg) * 128);
#pragma unroll
        for (int k = 0; k < 16; ++k) qv[k] = __ldg(src + k);
      } else {
#pragma unroll
        for (int k = 0; k < 16; ++k) qv[k] = make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int k = 0; k < 16; ++k)
        *reinterpret_cast<uint4*>(qtile + (k >> 3) * kHalfBytes + r * 128 + (((k & 7) ^ (r & 7)) << 4)) = qv[k];
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.q_full[w]);
      ++qc;
    }
    // causal bound of this row (padding rows borrow the last real query's bound)
    const int pos = info.ctx + min(j_row, info.q_len - 1);
    const int L = info.ctx + info.q_len;
    // V rows from here on are either past the context or not loaded this item: tile
    // 0's warps zero them (tile 0 loads the item's keys) so that 0-weight keys cannot
    // carry non-finite bytes into P V
    const int zero_from = kCas ? info.kend[0] : min(L, ((info.kend[0] + kBlock - 1) / kBlock) * kBlock);
    float m_ref = -INFINITY, l_sum = 0.f;

    for (int j = 0; j < nt && ok; ++j) {
      const uint32_t vt = vc + j;
      const int sv = vt % kVStages;
      const int k0 = info.ks + j * kTileKeys;
      if (!mbar_wait(&c.s_full[w], tc & 1, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // S_w(j) is complete, and so is every MMA issued before it: S_0(j) (issued before
      // S_1(j)) and P_w(j-1) V(j-1) (P_1 V is issued after P_0 V).  So K(j) and V(j-1)
      // are free once the last query tile that reads them gets here: tile 1's group
      // releases the key tiles both tiles read, tile 0's group the one only it reads.
      if (r == 0) {
        if (w == 1 || j >= info.nt[1]) mbar_arrive(&c.kempty[(vc + j) % kKStages]);
        if (j >= 1 && (w == 1 || j - 1 >= info.nt[1])) mbar_arrive(&c.vempty[(vc + j - 1) % kVStages]);
      }
      // keys k0 .. k0 + nvis - 1 are visible to this row (cascade: the whole split).
      // The scores stay unscaled: the tile maximum of scale * s is scale times the
      // maximum of s (the minimum, for a negative scale), and each exponent takes
      // scale * s - m in one fused multiply-add.  Masked keys count for no extremum and
      // their scaled scores become -inf before the exponent.  Tiles every row of the
      // warp sees whole skip the masking.
      const int nvis = kCas ? tkend - k0 : pos - k0 + 1;
      const bool whole = __all_sync(0xffffffffu, nvis >= kTileKeys);
      const uint32_t srow = tmem + lane_off + s_col;
      // first read of S: the row's extremum (a negative scale takes the masked form)
      const float raw = !pos_scale ? row_extremum<false, true>(srow, nvis)
                                   : whole ? row_extremum<true, false>(srow, nvis) : row_extremum<true, true>(srow, nvis);
      // (a fully masked row gives -inf either way: -inf * scale or +inf * a negative scale)
      const float tmax = raw * scale;
      if (j == 0) {
        m_ref = tmax;  // key 0 is visible to every row, so this is finite
      } else {
        // S_w(j) complete means P_w(j-1) V(j-1), issued before it, is complete: O_w
        // holds every tile before j and may be rescaled
        const bool need = tmax > m_ref + kRescaleThreshold;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = need ? tmax : m_ref;
          const float alpha = exp2f(m_ref - m_new);
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {  // rare: 16 columns at a time keeps registers low
            uint32_t v[16];
            tmem_ld16_sync(tmem + lane_off + o_col + 16 * ch, v);
#pragma unroll
            for (int k = 0; k < 16; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * alpha);
            tmem_st16(tmem + lane_off + o_col + 16 * ch, v);
          }
          tmem_st_wait();
          l_sum *= alpha;
          m_ref = m_new;
        }
      }
      // second read of S: the exponents, written as bf16 P over S's first 64 columns.
      // P goes to the MMA warp in two halves (keys 0-63, then 64-127), so that the first
      // half's P V runs while the second half is computed.  Before the first hand-over,
      // V of this key tile has landed (which also orders the producer's bad-block flag)
      // and tile 0's warps have zeroed its rows past the context.
      bool v_ok = true;
      auto first_half = [&]() {
        tmem_st_wait();
        v_ok = mbar_wait(&c.vfull[sv], (vt / kVStages) & 1, abort_flag);
        if (!v_ok) return;
        if (w == 0 && k0 + r >= zero_from) {
          // rows are 128 bytes apart, so every lane's k-th chunk would sit in the same
          // four banks; starting each lane at chunk r mod 8 spreads eight lanes over all 32
          uint8_t* vrow = vbuf + sv * kTileBytes + r * 128;
#pragma unroll
          for (int c16 = 0; c16 < 8; ++c16) {
            const int off = ((c16 + r) & 7) * 16;
            *reinterpret_cast<uint4*>(vrow + off) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(vrow + kHalfBytes + off) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&c.p_full[w][0]);
      };
      l_sum += whole ? row_exp_to_p<false>(srow, nvis, scale, m_ref, first_half)
                     : row_exp_to_p<true>(srow, nvis, scale, m_ref, first_half);
      if (!v_ok) {
        ok = false;
        break;
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&c.p_full[w][1]);
      ++tc;
    }
    if (!ok) break;
    // final O_w of the item; its last P V is complete, so its last V tile is free
    if (!mbar_wait(&c.o_full[w], ic & 1, abort_flag)) {
      ok = false;
      break;
    }
    ++ic;
    tc_fence_after();
    if (r == 0 && (w == 1 || nt - 1 >= info.nt[1])) mbar_arrive(&c.vempty[(vc + nt - 1) % kVStages]);
    vc += info.nt[0];
    const bool bad = c.bad[slot] != 0;
    if (kCas) {
      // the row's partial: accumulator [slot][head][128], then max and sum
      const int64_t cslot = (static_cast<int64_t>(entry) * P.hkv + info.head) * P.cas_np_max + info.split;
      // whole 32-byte sectors per store (workspace rows are 512-byte multiples from a
      // 256-byte aligned base)
      float* dst = P.cas_o + (cslot * P.gp + rg) * 128;
      uint32_t v[4][32];  // the whole row from TMEM before any store
#pragma unroll
      for (int h = 0; h < 4; ++h) tmem_ld32_issue(tmem + lane_off + o_col + 32 * h, v[h]);
#pragma unroll
      for (int h = 0; h < 4; ++h) tmem_ld32_wait(v[h]);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&c.o_free[w]);
        mbar_arrive(&c.item_empty[slot]);
      }
      if (cas_live) {
#pragma unroll
        for (int h = 0; h < 4; ++h)
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint32_t(&w8)[8] = *reinterpret_cast<const uint32_t(*)[8]>(v[h] + 8 * q);
            st_global_v8(dst + 32 * h + 8 * q, w8);
          }
      }
      // (a prefix with a bad block id admits nobody: the planner checks the ids itself)
      if (cas_live) {
        P.cas_ml[(cslot * P.gp + rg) * 2] = m_ref;
        P.cas_ml[(cslot * P.gp + rg) * 2 + 1] = l_sum;
      }
      continue;
    }
    const float inv = bad ? 0.f : 1.f / l_sum;
    // the whole O row is loaded from TMEM before any store: a load issued after stores
    // waits behind them in the memory pipeline
    uint32_t v[4][32];
#pragma unroll
    for (int h = 0; h < 4; ++h) tmem_ld32_issue(tmem + lane_off + o_col + 32 * h, v[h]);
#pragma unroll
    for (int h = 0; h < 4; ++h) tmem_ld32_wait(v[h]);
    // O_w is in registers: the next item's first P V may overwrite it while the rows
    // are stored, and the item slot is no longer read
    tc_fence_before();
    __syncwarp();
    if (lane == 0) {
      mbar_arrive(&c.o_free[w]);
      mbar_arrive(&c.item_empty[slot]);
    }
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      if (row_out && P.out_v8) {
        // whole 32-byte sectors per store (the lanes of a warp write 32 different rows,
        // so 16-byte stores would leave every sector half written)
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t wv[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(v[h][16 * ch + 2 * q]) * inv,
                                                      __uint_as_float(v[h][16 * ch + 2 * q + 1]) * inv);
            wv[q] = *reinterpret_cast<uint32_t*>(&h2);
          }
          st_global_v8(orow + 32 * h + 16 * ch, wv);
        }
      } else if (row_out) {
#pragma unroll
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t wv[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(v[h][8 * ch + 2 * q]) * inv,
                                                      __uint_as_float(v[h][8 * ch + 2 * q + 1]) * inv);
            wv[q] = *reinterpret_cast<uint32_t*>(&h2);
          }
          reinterpret_cast<uint4*>(orow)[4 * h + ch] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
        }
      }
    }
  }
  if (!ok && !*abort_flag && lane == 0) raise_abort(c, P.err);
}

template <bool kCas>
__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ CUtensorMap qmap,
                                                              const __grid_constant__ CUtensorMap kmap,
                                                              const __grid_constant__ CUtensorMap vmap,
                                                              const PrefillParams P) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* base = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* qbuf = base;                          // Q tiles 0 and 1
  uint8_t* kbuf = qbuf + 2 * kTileBytes;         // K ring
  uint8_t* vbuf = kbuf + kKStages * kTileBytes;  // V ring
  Ctl& c = *reinterpret_cast<Ctl*>(vbuf + kVStages * kTileBytes);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&c.kfull[s], 1);
      mbar_init(&c.kempty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&c.vfull[s], 1);
      mbar_init(&c.vempty[s], 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&c.s_full[w], 1);
      mbar_init(&c.p_full[w][0], 4);
      mbar_init(&c.p_full[w][1], 4);
      mbar_init(&c.o_full[w], 1);
      mbar_init(&c.o_free[w], 4);
      mbar_init(&c.q_full[w], kCas ? 4 : 1);  // cascade: the tile's four softmax warps gather Q
      mbar_init(&c.q_free[w], 1);
    }
    for (int s = 0; s < kRing; ++s) {
      mbar_init(&c.item_full[s], 1);
      mbar_init(&c.item_empty[s], 9);  // the MMA warp and the eight softmax warps
    }
    mbar_init(&c.drain, 1);
    c.abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_map(&qmap);
    tma_prefetch_map(&kmap);
    tma_prefetch_map(&vmap);
  }
  if (warp == 1) tmem_alloc(&c.tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = c.tmem_base;
  // the plan, the new tokens and the earlier kernels of this call; a cascade beside the
  // planner reads nothing those write (the planner admits no member of a group whose
  // prefix a new token lands in) and waits for them only before it exits
  // (likewise a prefill launched right after the decode kernel: it reads only the
  // planner's lists, the cache and q, and writes rows of out the decode does not)
  const bool beside = kCas ? P.cas_concurrent != 0 : P.after_decode != 0;
  if (!beside) grid_dep_wait();
  grid_dep_launch();
  if (warp == 0) producer_warp<kCas>(P, &qmap, &kmap, &vmap, c, qbuf, kbuf, vbuf);
  else if (warp == 1) mma_warp(P, c, qbuf, kbuf, vbuf, tmem);
  else softmax_warps<kCas>(P, c, qbuf, vbuf, tmem);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
    tmem_relinquish();
  }
  // the grid ends after its predecessor (the planning launch, or the decode kernel): the
  // kernels after it wait on this one only
  if (beside && threadIdx.x == 0) grid_dep_wait();
}

}  // namespace

int launch_prefill_tc(const AttnArgs& a, const Workspace& ws, int num_sms, uint32_t* err, cudaStream_t s,
                      int after_decode) {
  const int hkv = a.cache.num_kv_heads;
  const int group = a.num_q_heads / hkv;
  if (group > 16 || a.cache.head_dim != 128 || a.cache.dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
  const int gp = group <= 4 ? 4 : (group <= 8 ? 8 : 16);
  const uint64_t rows = static_cast<uint64_t>(a.cache.num_blocks) * hkv * kBlock;
  if (rows >= (1ull << 31) || a.num_tokens >= (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;
  CUtensorMap qm, km, vm;
  int st = encode_tensor_map_2d(&km, a.k_cache, 128, rows, 256, 64, 16);
  if (st) return st;
  st = encode_tensor_map_2d(&vm, a.v_cache, 128, rows, 256, 64, 16);
  if (st) return st;
  const uint64_t qdims[3] = {128, static_cast<uint64_t>(a.num_q_heads), static_cast<uint64_t>(a.num_tokens)};
  const uint64_t qstrides[2] = {256, static_cast<uint64_t>(a.num_q_heads) * 256};
  const uint32_t qbox[3] = {64, static_cast<uint32_t>(gp), static_cast<uint32_t>(kTileKeys / gp)};
  st = encode_tensor_map_3d(&qm, a.q, qdims, qstrides, qbox);
  if (st) return st;
  PrefillParams p{};
  p.after_decode = after_decode != 0 ? 1 : 0;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.out_v8 = (reinterpret_cast<uintptr_t>(a.out) & 31u) == 0 ? 1 : 0;
  p.bt = a.block_tables;
  p.seq_lens = a.seq_lens;
  p.qsl = a.qsl;
  p.pre_prefix = ws.pre_prefix;
  p.pre_order = ws.pre_order;
  p.queue = ws.counters + 1;
  p.err = err;
  p.num_blocks = a.cache.num_blocks;
  p.num_tokens = a.num_tokens;
  p.num_seqs = a.num_seqs;
  p.max_blocks = a.max_blocks;
  p.hkv = hkv;
  p.group = group;
  p.gp = gp;
  p.rows_q = kTileKeys / gp;
  p.hq = a.num_q_heads;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  static uint64_t smem_set = 0;
  st = set_smem_once(reinterpret_cast<const void*>(prefill_kernel<false>), kSmemBytes, &smem_set);
  if (st) return st;
  TraceScope trace(kTracePrefill, s);
  return cuda_status(launch_k(prefill_kernel<false>, dim3(num_sms), dim3(kThreads), kSmemBytes, s, qm, km, vm, p));
}

int launch_cascade_tc(const AttnArgs& a, const CascadeArgs& cas, const Workspace& ws, int num_sms, int tiles_per_item,
                      int concurrent, uint32_t* err, cudaStream_t s) {
  const int hkv = a.cache.num_kv_heads;
  const int group = a.num_q_heads / hkv;
  if (group > 16 || a.cache.head_dim != 128 || a.cache.dtype != PKV_BF16) return PKV_ERR_UNSUPPORTED;
  if (cas.num_groups <= 0 || cas.num_members <= 0 || !ws.cas_o) return PKV_OK;
  const int gp = group <= 4 ? 4 : (group <= 8 ? 8 : 16);
  const uint64_t rows = static_cast<uint64_t>(a.cache.num_blocks) * hkv * kBlock;
  if (rows >= (1ull << 31) || a.num_tokens >= (int64_t(1) << 31)) return PKV_ERR_UNSUPPORTED;
  CUtensorMap km, vm;
  int st = encode_tensor_map_2d(&km, a.k_cache, 128, rows, 256, 64, 16);
  if (st) return st;
  st = encode_tensor_map_2d(&vm, a.v_cache, 128, rows, 256, 64, 16);
  if (st) return st;
  PrefillParams p{};
  p.bt = a.block_tables;
  p.seq_lens = a.seq_lens;
  p.qsl = a.qsl;
  p.err = err;
  p.num_blocks = a.cache.num_blocks;
  p.num_tokens = a.num_tokens;
  p.num_seqs = a.num_seqs;
  p.max_blocks = a.max_blocks;
  p.hkv = hkv;
  p.group = group;
  p.gp = gp;
  p.rows_q = kTileKeys / gp;
  p.hq = a.num_q_heads;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.cas_tables = cas.tables;
  p.cas_blocks = cas.blocks;
  p.cas_start = cas.start;
  p.cas_members = cas.members;
  p.cas_prefix = ws.cas_prefix;
  p.cas_o = ws.cas_o;
  p.cas_ml = ws.cas_ml;
  p.cas_concurrent = concurrent != 0 && cas.num_groups <= kCasConcurrentGroups ? 1 : 0;
  p.cas_max_blocks = cas.max_blocks;
  p.cas_groups = cas.num_groups;
  p.cas_np_max = ws.cas_np_max;
  p.cas_tiles = tiles_per_item;
  static uint64_t smem_set = 0;
  st = set_smem_once(reinterpret_cast<const void*>(prefill_kernel<true>), kSmemBytes, &smem_set);
  if (st) return st;
  TraceScope trace(kTraceCascade, s);
  // at most ceil(members / rows) + groups member tiles: CTAs past the items would only
  // hold an SM until the planner ends
  const int64_t tile_rows = static_cast<int64_t>(tiles_per_item) * p.rows_q;
  const int64_t items = ((cas.num_members + tile_rows - 1) / tile_rows + cas.num_groups) * hkv *
                        cascade_splits(static_cast<int64_t>(cas.max_blocks) * kBlock);
  const int grid = static_cast<int>(items < num_sms ? items : num_sms);
  // the Q tensor map is unused in this mode (Q rows are gathered); K's stands in
  return cuda_status(launch_k(prefill_kernel<true>, dim3(grid), dim3(kThreads), kSmemBytes, s, km, km, vm, p));
}

}  // namespace pkv
