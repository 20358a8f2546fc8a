// k_plan.cu -- device-side planning of one paged_attention call.
//
// One CTA scans the batch ("Continuous batching": every request is a pair of
// computed / total tokens, and one step mixes decodes and prefill chunks) and
// writes two work lists as exclusive prefix sums over the requests:
//   decode items  -- requests with exactly one query token: num_kv_heads x
//                    decode_splits(seq_len) (kv head, key split) items;
//   prefill items -- requests with more query tokens: num_kv_heads x
//                    ceil(q_len / rows_per_tile) (kv head, query rows) items, an item
//                    being the prefill kernel's pair of query tiles.
// Split boundaries depend only on a request's own length and a library constant,
// so a request's result does not depend on what else is in the batch.  It also
// zeroes the work-queue counters and the per-(request, kv head) bad-block flags
// used by the split merge, and lists the requests whose splits need merging.  Lengths that contradict the host
// bounds become a single item that reports the error and zeroes its output.
//
// Shared-prefix groups (paged_attention_cascade) are checked here first.  A listed
// request becomes a member of its group only if it is listed once, is a decode whose
// context goes past the prefix, and its block table starts with the prefix's block
// ids.  A member's decode items then cover only the keys after the prefix, it goes
// to the split merge when those keys are cut into several splits, and
// the cascade kernel gets ceil(members / rows) x kv heads x cascade_splits(P) items
// (rows: the member requests of one item)
// per group.  Anything else listed is attended the ordinary way.
#include "pkv_internal.cuh"

namespace pkv {
namespace {

constexpr int kPlanThreads = 1024;
constexpr int kPlanSmemMax = 196 * 1024;  // dynamic shared memory the plan launch may ask for

__device__ __forceinline__ int warp_inclusive_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  return v;
}

// Block-wide exclusive scan of three counters at once.
__device__ void block_scan3(const int (&v)[3], int (&ex)[3], int (&tot)[3]) {
  __shared__ int ws[3][32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  int inc[3];
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    inc[k] = warp_inclusive_scan(v[k]);
    if (lane == 31) ws[k][warp] = inc[k];
  }
  __syncthreads();
  if (warp == 0) {
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      int x = lane < nwarps ? ws[k][lane] : 0;
      ws[k][lane] = warp_inclusive_scan(x);
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < 3; ++k) {
    ex[k] = (warp ? ws[k][warp - 1] : 0) + inc[k] - v[k];
    tot[k] = ws[k][nwarps - 1];
  }
  __syncthreads();
}

// Shared-prefix membership: fills seq_prefix / seq_entry and the cascade item prefix
// over groups (member_ok is its scratch).  Called by the whole block.
__device__ void plan_cascade(const PlanArgs& p) {
  __shared__ int s_ok;
  const CascadeArgs& g = p.cas;
  const int tid = threadIdx.x, nthr = blockDim.x;
  for (int i = tid; i < p.num_seqs; i += nthr) {
    p.seq_prefix[i] = 0;
    p.seq_entry[i] = -1;
  }
  if (tid == 0) s_ok = g.start[0] == 0 && g.start[g.num_groups] == g.num_members;
  __syncthreads();
  for (int k = tid; k < g.num_groups; k += nthr)
    if (g.start[k] > g.start[k + 1]) s_ok = 0;  // CSR offsets must not decrease
  __syncthreads();
  const bool csr_ok = s_ok != 0;
  // each request may be claimed by one entry; a second claim marks it listed twice
  if (csr_ok) {
    for (int k = tid; k < g.num_members; k += nthr) {
      const int i = g.members[k];
      if (i >= 0 && i < p.num_seqs && atomicCAS(&p.seq_entry[i], -1, k) != -1) atomicExch(&p.seq_prefix[i], -1);
    }
  }
  __syncthreads();
  // the group of entry k: last gi with start[gi] <= k
  auto group_of = [&](int k) {
    int lo = 0, hi = g.num_groups - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (g.start[mid] <= k) lo = mid; else hi = mid - 1;
    }
    return lo;
  };
  // per entry, the conditions on the request; member_ok[k] holds the prefix length in
  // blocks while the tables are compared (0: rejected)
  for (int k = tid; k < g.num_members; k += nthr) {
    const int i = g.members[k];
    int pb_ok = 0;
    if (csr_ok && i >= 0 && i < p.num_seqs && p.seq_entry[i] == k && p.seq_prefix[i] == 0) {
      const int gk = group_of(k);
      const int pb = p.grp_ok[gk] ? g.blocks[gk] : 0;
      const int64_t q0 = p.qsl[i], q1 = p.qsl[i + 1], L = p.seq_lens[i];
      if (pb >= 1 && pb <= g.max_blocks && q0 >= 0 && q1 == q0 + 1 && q1 <= p.num_tokens && L <= p.max_seq_len &&
          (L + kBlock - 1) / kBlock <= p.max_blocks && L > static_cast<int64_t>(pb) * kBlock)
        pb_ok = pb;
    }
    p.member_ok[k] = pb_ok;
  }
  __syncthreads();
  // the member's table must start with the prefix's block ids: (entry, 16-id chunk)
  // pairs spread over the block; a mismatch anywhere rejects the entry
  constexpr int kChunk = 16;
  const int chunks = (g.max_blocks + kChunk - 1) / kChunk;
  const int64_t work = static_cast<int64_t>(g.num_members) * chunks;
  for (int64_t wi = tid; wi < work; wi += nthr) {
    const int k = static_cast<int>(wi / chunks), j0 = static_cast<int>(wi % chunks) * kChunk;
    const int pb = *reinterpret_cast<volatile int32_t*>(p.member_ok + k);
    if (j0 >= pb) continue;
    const int32_t* own = p.bt + static_cast<int64_t>(g.members[k]) * p.max_blocks;
    const int32_t* pre = g.tables + static_cast<int64_t>(group_of(k)) * g.max_blocks;
    const int j1 = min(pb, j0 + kChunk);
    int diff = 0;
    if (j1 - j0 == kChunk && ((reinterpret_cast<uintptr_t>(own + j0) | reinterpret_cast<uintptr_t>(pre + j0)) & 15) == 0) {
      // a whole chunk of both rows in four 16-byte loads each: the warp's lanes read 32
      // different rows, so fewer, wider requests matter
#pragma unroll
      for (int q = 0; q < kChunk / 4; ++q) {
        const int4 a = __ldg(reinterpret_cast<const int4*>(own + j0) + q);
        const int4 b = __ldg(reinterpret_cast<const int4*>(pre + j0) + q);
        diff |= (a.x != b.x) | (a.y != b.y) | (a.z != b.z) | (a.w != b.w);
      }
    } else {
      for (int j = j0; j < j1; ++j) diff |= __ldg(own + j) != __ldg(pre + j);
    }
    if (diff) *reinterpret_cast<volatile int32_t*>(p.member_ok + k) = 0;
  }
  __syncthreads();
  for (int k = tid; k < g.num_members; k += nthr) {
    const int i = g.members[k];
    const int pb = p.member_ok[k];
    if (pb > 0) {
      p.seq_prefix[i] = pb * kBlock;
    } else if (csr_ok && i >= 0 && i < p.num_seqs && p.seq_entry[i] == k && p.seq_prefix[i] == 0) {
      p.seq_entry[i] = -1;  // claimed but not a member
    }
  }
  __syncthreads();
  for (int i = tid; i < p.num_seqs; i += nthr) {
    if (p.seq_prefix[i] < 0) {  // listed twice: not a member anywhere
      p.seq_prefix[i] = 0;
      p.seq_entry[i] = -1;
    }
  }
  // cascade items per group: member tiles x kv heads x prefix key splits
  int carry = 0;
  for (int base = 0; base < g.num_groups; base += nthr) {
    const int gi = base + tid;
    int nu = 0;
    if (gi < g.num_groups && csr_ok) {
      const int pb = g.blocks[gi];
      const int cnt = g.start[gi + 1] - g.start[gi];
      if (pb >= 1 && pb <= g.max_blocks && cnt > 0)
        nu = ((cnt + p.cas_rows - 1) / p.cas_rows) * p.hkv * static_cast<int>(cascade_splits(int64_t(pb) * kBlock));
    }
    const int v[3] = {nu, 0, 0};
    int ex[3], tot[3];
    block_scan3(v, ex, tot);
    if (gi < g.num_groups) p.cas_prefix[gi] = carry + ex[0];
    carry += tot[0];
  }
  if (tid == 0) p.cas_prefix[g.num_groups] = carry;
  __syncthreads();
}

// Which groups may admit members (grp_ok).  A group whose prefix names a block outside
// the pool admits nobody: its members attend their whole context in the decode kernel,
// which reports the bad id for them.  When the cascade kernel runs beside this launch
// (cas_concurrent) it reads the prefix blocks while the writer CTAs may still be
// writing this call's new tokens, so then a new token that lands in any group's prefix
// block, a copy-on-write copy of the same call that lands in one, or a
// query_start_loc that decreases (which the writers would map differently) admits
// nobody anywhere: a correct, slower fallback for inputs a serving loop does not
// produce, since shared prefix blocks are full and never written.  Every group's
// prefix blocks are marked with the call's epoch in the workspace, then a thread per
// request checks the blocks its new tokens go to, as the writers compute them, and the
// copies' destinations are checked the same way.  Called by the whole block; returns
// synchronised.
__device__ void prefix_block_checks(const PlanArgs& p) {
  __shared__ int s_conflict;
  const CascadeArgs& g = p.cas;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const bool marks = p.cas_concurrent && (p.k_new != nullptr || p.num_cow > 0);
  if (tid == 0) s_conflict = 0;
  for (int gi = tid; gi < g.num_groups; gi += nthr) p.grp_ok[gi] = 1;
  __syncthreads();
  const int64_t n_ids = static_cast<int64_t>(g.num_groups) * g.max_blocks;
  for (int64_t x = tid; x < n_ids; x += nthr) {
    const int gi = static_cast<int>(x / g.max_blocks), j = static_cast<int>(x % g.max_blocks);
    if (j >= __ldg(g.blocks + gi)) continue;  // (a length outside [1, max_blocks] admits nobody anyway)
    const int32_t b = __ldg(g.tables + x);
    if (b < 0 || b >= p.num_blocks) p.grp_ok[gi] = 0;
    else if (marks) p.blk_mark[b] = p.epoch;
  }
  __syncthreads();
  if (marks) {
    // a thread per request: its loads overlap those of the other requests
    for (int i = tid; p.k_new != nullptr && i < p.num_seqs; i += nthr) {
      const int64_t q0 = __ldg(p.qsl + i), q1 = __ldg(p.qsl + i + 1), L = __ldg(p.seq_lens + i);
      if (q1 < q0) {
        s_conflict = 1;
        continue;
      }
      // new tokens at positions L - (q1 - q0) .. L - 1, those the writers store: pos >= 0
      // and pos / 16 < max_blocks
      const int64_t first = L - (q1 - q0) > 0 ? L - (q1 - q0) : 0, last = L - 1;
      if (q1 == q0 || last < first) continue;
      const int64_t lb1 = last / kBlock < p.max_blocks - 1 ? last / kBlock : p.max_blocks - 1;
      const int32_t* row = p.bt + static_cast<int64_t>(i) * p.max_blocks;
      bool hit = false;
#pragma unroll 4
      for (int64_t lb = first / kBlock; lb <= lb1; ++lb) {
        const int32_t b = __ldg(row + lb);
        hit |= b >= 0 && b < p.num_blocks && p.blk_mark[b] == p.epoch;
      }
      if (hit) s_conflict = 1;
    }
    // a copy-on-write destination in a prefix (the copies may still be running)
    for (int64_t x = tid; x < p.num_cow; x += nthr) {
      const int32_t b = __ldg(p.cow_dst + x);
      if (b >= 0 && b < p.num_blocks && p.blk_mark[b] == p.epoch) s_conflict = 1;
    }
    __syncthreads();
    if (s_conflict)
      for (int gi = tid; gi < g.num_groups; gi += nthr) p.grp_ok[gi] = 0;
  }
  __syncthreads();
}

// The same membership decisions with every intermediate state in shared memory (`sm`,
// the launch's dynamic buffer), for batches within the limits below.  One pass over
// (entry, 16-id chunk) pairs makes every check at once -- the chunk-0 thread of an
// entry claims the request and checks its lengths, every thread compares its chunk of
// the request's table with the prefix's -- so the planner waits on three rounds of
// global loads (the group offsets; each entry's request; that request's lengths and
// table rows) instead of one or more per phase.  Leaves each request's prefix tokens
// and member entry in shared memory for the rest of the plan and writes the global
// copies the other kernels read.  Called by the whole block.
constexpr int kCasOnchipSeqs = 8192;
constexpr int kCasOnchipMembers = 8192;
constexpr int kCasOnchipGroups = 1024;
constexpr int kCasOnchipBlocks = 512;  // longest prefix table compared in this pass
__host__ __device__ constexpr int64_t cas_onchip_ints(int64_t n, int64_t m, int64_t g) { return 2 * n + 2 * m + 2 * g + 1; }
__device__ void plan_cascade_onchip(const PlanArgs& p, int32_t* sm, int32_t*& s_prefix, int32_t*& s_entry) {
  __shared__ int s_csr_ok;
  constexpr int kChunk = 16;
  const CascadeArgs& g = p.cas;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int n = p.num_seqs, M = g.num_members, G = g.num_groups;
  s_entry = sm;                    // [n]: claiming entry; -1 none; -2 listed more than once
  s_prefix = s_entry + n;          // [n]: prefix tokens of a member, else 0
  int32_t* s_pb = s_prefix + n;    // [M]: the entry's prefix blocks if its lengths pass, else 0
  int32_t* s_diff = s_pb + M;      // [M]: some chunk of the table differs from the prefix
  int32_t* s_start = s_diff + M;   // [G + 1]
  int32_t* s_blocks = s_start + G + 1;  // [G]
  for (int i = tid; i < n; i += nthr) s_entry[i] = -1;
  for (int k = tid; k < M; k += nthr) s_diff[k] = 0;
  for (int k = tid; k <= G; k += nthr) s_start[k] = __ldg(g.start + k);
  for (int k = tid; k < G; k += nthr) s_blocks[k] = p.grp_ok[k] ? __ldg(g.blocks + k) : 0;  // 0: admits nobody
  if (tid == 0) s_csr_ok = 1;
  __syncthreads();
  if (tid == 0 && !(s_start[0] == 0 && s_start[G] == M)) s_csr_ok = 0;
  for (int k = tid; k < G; k += nthr)
    if (s_start[k] > s_start[k + 1]) s_csr_ok = 0;  // CSR offsets must not decrease
  __syncthreads();
  const bool csr_ok = s_csr_ok != 0;
  const int chunks = (g.max_blocks + kChunk - 1) / kChunk;
  const int64_t work = csr_ok ? static_cast<int64_t>(M) * chunks : 0;
  for (int64_t wi = tid; wi < work; wi += nthr) {
    const int k = static_cast<int>(wi / chunks), j0 = static_cast<int>(wi % chunks) * kChunk;
    const int i = __ldg(g.members + k);
    const bool i_ok = i >= 0 && i < n;
    int lo = 0, hi = G - 1;  // the entry's group: last gi with start[gi] <= k
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_start[mid] <= k) lo = mid; else hi = mid - 1;
    }
    const int pb = s_blocks[lo];
    const bool pb_ok = pb >= 1 && pb <= g.max_blocks && pb <= p.max_blocks;  // (also keeps the reads in the rows)
    if (j0 == 0) {  // the entry's own checks, once
      int keep = 0;
      if (i_ok) {
        if (atomicCAS(&s_entry[i], -1, k) != -1) atomicExch(&s_entry[i], -2);  // a second claim: listed twice
        const int64_t q0 = __ldg(p.qsl + i), q1 = __ldg(p.qsl + i + 1), L = __ldg(p.seq_lens + i);
        if (pb_ok && q0 >= 0 && q1 == q0 + 1 && q1 <= p.num_tokens && L <= p.max_seq_len &&
            (L + kBlock - 1) / kBlock <= p.max_blocks && L > static_cast<int64_t>(pb) * kBlock)
          keep = pb;
      }
      s_pb[k] = keep;
    }
    if (i_ok && pb_ok && j0 < pb) {  // this chunk of the request's table against the prefix's
      const int32_t* own = p.bt + static_cast<int64_t>(i) * p.max_blocks;
      const int32_t* pre = g.tables + static_cast<int64_t>(lo) * g.max_blocks;
      const int j1 = min(pb, j0 + kChunk);
      int diff = 0;
      if (j1 - j0 == kChunk && ((reinterpret_cast<uintptr_t>(own + j0) | reinterpret_cast<uintptr_t>(pre + j0)) & 15) == 0) {
#pragma unroll
        for (int q = 0; q < kChunk / 4; ++q) {
          const int4 a = __ldg(reinterpret_cast<const int4*>(own + j0) + q);
          const int4 b = __ldg(reinterpret_cast<const int4*>(pre + j0) + q);
          diff |= (a.x != b.x) | (a.y != b.y) | (a.z != b.z) | (a.w != b.w);
        }
      } else {
        for (int j = j0; j < j1; ++j) diff |= __ldg(own + j) != __ldg(pre + j);
      }
      if (diff) s_diff[k] = 1;
    }
  }
  __syncthreads();
  // a request is a member iff exactly one entry claimed it and that entry passed
  for (int i = tid; i < n; i += nthr) {
    const int k = s_entry[i];
    const int pb = (k >= 0 && !s_diff[k]) ? s_pb[k] : 0;
    s_prefix[i] = pb * kBlock;
    s_entry[i] = pb > 0 ? k : -1;
    p.seq_prefix[i] = pb * kBlock;
    p.seq_entry[i] = pb > 0 ? k : -1;
  }
  __syncthreads();
  // cascade items per group: member tiles x kv heads x prefix key splits
  int carry = 0;
  for (int base = 0; base < G; base += nthr) {
    const int gi = base + tid;
    int nu = 0;
    if (gi < G && csr_ok) {
      const int pb = s_blocks[gi];
      const int cnt = s_start[gi + 1] - s_start[gi];
      if (pb >= 1 && pb <= g.max_blocks && cnt > 0)
        nu = ((cnt + p.cas_rows - 1) / p.cas_rows) * p.hkv * static_cast<int>(cascade_splits(int64_t(pb) * kBlock));
    }
    const int v[3] = {nu, 0, 0};
    int ex[3], tot[3];
    block_scan3(v, ex, tot);
    if (gi < G) p.cas_prefix[gi] = carry + ex[0];
    carry += tot[0];
  }
  if (tid == 0) p.cas_prefix[G] = carry;
  __syncthreads();
}

// The writer CTAs of a fused step: a warp per 64-vector piece of a new token's rows
// computes the token's slot (as slot_mapping_kernel does) and copies the piece of
// its K and V rows into it (as write_kernel does), with the same error flags.  The
// attention kernels launched after this one see the rows.
//
// Latency, not bandwidth, bounds this part: a step's few new tokens each wait on a
// chain of dependent loads.  The chain is kept short: the CTA stages query_start_loc
// in shared memory with one round of coalesced loads (batches up to kWriterQslMax
// requests; larger ones search global memory), and every lane loads its part of the
// piece before the slot is known, so those loads overlap the two dependent loads the
// slot needs (the request's length, then its table entry).
constexpr int kWriterQslMax = 8192;
constexpr int kWriterPiece = 64;  // 16-byte vectors of a (token) row a warp moves: two per lane, K and V
__device__ void write_new_tokens(const PlanArgs& p, int32_t* s_qsl) {
  const int lane = threadIdx.x & 31;
  const bool staged = p.num_seqs <= kWriterQslMax;  // (the launch then gives s_qsl num_seqs + 1 ints)
  if (staged) {
    for (int i = threadIdx.x; i <= p.num_seqs; i += blockDim.x) s_qsl[i] = __ldg(p.qsl + i);
    __syncthreads();
  }
  const int64_t nwarps = static_cast<int64_t>(gridDim.x - 1) * (blockDim.x >> 5);
  const int per_tok = p.hkv * p.vec_per_row;  // 16-byte vectors of a token's K (or V) row
  const int pieces = (per_tok + kWriterPiece - 1) / kWriterPiece;
  const int64_t units = p.num_tokens * pieces;
  for (int64_t u = static_cast<int64_t>(blockIdx.x - 1) * (blockDim.x >> 5) + (threadIdx.x >> 5); u < units;
       u += nwarps) {
    const int64_t t = u / pieces;
    const int r0 = static_cast<int>(u - t * pieces) * kWriterPiece + lane;  // this lane's vectors: r0, r0 + 32
    const uint4* ks = p.k_new + t * per_tok;
    const uint4* vs = p.v_new + t * per_tok;
    uint4 ka = make_uint4(0, 0, 0, 0), kb = ka, va = ka, vb = ka;
    if (r0 < per_tok) {
      ka = __ldcs(ks + r0);
      va = __ldcs(vs + r0);
    }
    if (r0 + 32 < per_tok) {
      kb = __ldcs(ks + r0 + 32);
      vb = __ldcs(vs + r0 + 32);
    }
    int64_t slot = -1;
    if (lane == 0) {
      int i;
      int64_t q0, q1;
      if (staged) {
        int lo = 0, hi = p.num_seqs - 1;
        while (lo < hi) {
          const int mid = lo + (hi - lo + 1) / 2;
          if (static_cast<int64_t>(s_qsl[mid]) <= t) lo = mid; else hi = mid - 1;
        }
        i = lo;
        q0 = s_qsl[i];
        q1 = s_qsl[i + 1];
      } else {
        i = find_seq(p.qsl, p.num_seqs, t);
        q0 = __ldg(p.qsl + i);
        q1 = __ldg(p.qsl + i + 1);
      }
      const int64_t pos = static_cast<int64_t>(__ldg(p.seq_lens + i)) - (q1 - q0) + (t - q0);
      const bool first = r0 == 0;  // errors and the slot are reported once per token
      if (t < q0 || t >= q1 || pos < 0 || pos / kBlock >= p.max_blocks) {
        if (first) flag_error(p.err, kErrLength);
      } else {
        const int32_t b = __ldg(p.bt + static_cast<int64_t>(i) * p.max_blocks + pos / kBlock);
        if (b < 0) {
          if (first) flag_error(p.err, kErrBlockId);
        } else {
          slot = static_cast<int64_t>(b) * kBlock + pos % kBlock;
        }
      }
      if (first && p.slots_out) p.slots_out[t] = slot;
      if (slot >= p.num_slots) {
        if (first) flag_error(p.err, kErrSlot);
        slot = -1;
      }
    }
    slot = __shfl_sync(0xffffffffu, slot, 0);
    if (slot < 0) continue;
    // vector r = (kv head h, column c) goes to ((block * hkv + h) * 16 + off) * vpr + c
    const int vpr = p.vec_per_row;
    const int64_t base = ((slot / kBlock) * p.hkv * kBlock + slot % kBlock) * vpr;
    if (r0 < per_tok) {
      const int h = r0 / vpr;
      const int64_t d = base + static_cast<int64_t>(h) * kBlock * vpr + (r0 - h * vpr);
      p.k_cache[d] = ka;
      p.v_cache[d] = va;
    }
    if (r0 + 32 < per_tok) {
      const int h = (r0 + 32) / vpr;
      const int64_t d = base + static_cast<int64_t>(h) * kBlock * vpr + (r0 + 32 - h * vpr);
      p.k_cache[d] = kb;
      p.v_cache[d] = vb;
    }
  }
}

// Key tiles of the later query tile of prefill pair `pl` of a request (pl = 0: its
// heaviest pair): the pair's cost, the same count the prefill kernel derives.
__device__ __forceinline__ int pair_key_tiles(int64_t ctx, int64_t q_len, int rows_q, int pl) {
  const int64_t nqt = (q_len + rows_q - 1) / rows_q;
  const int64_t npair = (nqt + 1) / 2;
  const int64_t pair = npair - 1 - pl;
  const int64_t hi = 2 * pair + 1;
  const int64_t t0 = hi < nqt ? hi : 2 * pair;
  const int64_t j0 = t0 * rows_q;
  const int64_t nq = q_len - j0 < rows_q ? q_len - j0 : rows_q;
  const int64_t kend = ctx + j0 + nq;
  return kend > 0 ? static_cast<int>((kend + kTileKeys - 1) / kTileKeys) : 0;
}

// The prefill pairs (request, pair) of the whole batch ordered heaviest first -- a
// counting sort on the pair's key-tile count (clamped to the bucket range) -- so that
// the pairs handed out last are the lightest and the CTAs run out of work together.
// Ids are the pairs' positions in request order (pre_prefix / hkv + pl).  Pairs of
// equal cost land in any order: which CTA runs a pair changes no result.
constexpr int kOrderBuckets = kPlanThreads;
__device__ void order_prefill_pairs(const PlanArgs& p) {
  __shared__ int bucket[kOrderBuckets];
  const int tid = threadIdx.x;
  bucket[tid] = 0;
  __syncthreads();
  auto for_each_pair = [&](auto&& fn) {
    for (int i = tid; i < p.num_seqs; i += blockDim.x) {
      const int64_t q0 = p.qsl[i], q1 = p.qsl[i + 1];
      const int64_t q_len = q1 - q0;
      if (!(q0 >= 0 && q1 >= q0 && q1 <= p.num_tokens) || q_len <= 1) continue;
      const int64_t ctx = static_cast<int64_t>(p.seq_lens[i]) - q_len;
      const int base = p.pre_prefix[i] / p.hkv;
      const int npair = (p.pre_prefix[i + 1] - p.pre_prefix[i]) / p.hkv;
      for (int pl = 0; pl < npair; ++pl) {
        const int key = min(pair_key_tiles(ctx, q_len, p.rows_q, pl), kOrderBuckets - 1);
        fn(kOrderBuckets - 1 - key, base + pl, i);  // heavier pairs in lower buckets
      }
    }
  };
  for_each_pair([&](int b, int, int) { atomicAdd(&bucket[b], 1); });
  __syncthreads();
  {
    const int v[3] = {bucket[tid], 0, 0};
    int ex[3], tot[3];
    block_scan3(v, ex, tot);
    bucket[tid] = ex[0];  // first position of the bucket
  }
  __syncthreads();
  // each position gets the pair's id and its request, so that a CTA taking the pair
  // needs no search for the request
  for_each_pair([&](int b, int id, int i) {
    const int pos = atomicAdd(&bucket[b], 1);
    if (pos < p.max_pre_units) reinterpret_cast<int2*>(p.pre_order)[pos] = make_int2(id, i);
  });
}

// A small decode batch -- at most kDecOrderMaxItemsPerSm items per SM, where the last
// items decide when the kernel ends -- is handed out largest item first: the decode
// requests sorted by the key tiles of their largest item (an unsplit request's whole
// context, else one split), with the items' prefix in that order, and for every queue
// position the request and its first position, so that the decode kernel finds an
// item's request with one load.  The decode kernel keeps storing partials by the
// request-order item index.  Larger batches keep request order.
constexpr int kDecOrderBuckets = 32;
__device__ void order_decode_requests(const PlanArgs& p, int total, const int32_t* seq_prefix) {
  __shared__ int bucket[kDecOrderBuckets];
  const int tid = threadIdx.x;
  if (tid < kDecOrderBuckets) bucket[tid] = 0;
  __syncthreads();
  auto for_each_request = [&](auto&& fn) {
    for (int i = tid; i < p.num_seqs; i += blockDim.x) {
      const int nd = p.dec_prefix[i + 1] - p.dec_prefix[i];
      if (nd <= 0) continue;
      const int ns = nd / p.hkv;
      const bool cascade = p.cas.num_groups > 0 && p.cas.num_members > 0;
      const int64_t keys = static_cast<int64_t>(p.seq_lens[i]) - (cascade ? seq_prefix[i] : 0);
      const int64_t tiles = ns > 1 ? p.split_keys / kTileKeys : (keys + kTileKeys - 1) / kTileKeys;
      const int key = static_cast<int>(tiles < kDecOrderBuckets - 1 ? (tiles > 0 ? tiles : 0) : kDecOrderBuckets - 1);
      fn(kDecOrderBuckets - 1 - key, i);  // larger items in lower buckets
    }
  };
  for_each_request([&](int b, int) { atomicAdd(&bucket[b], 1); });
  __syncthreads();
  if (tid < 32) {  // exclusive prefix over the buckets, one warp
    const int v = bucket[tid];
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, inc, o);
      if (tid >= o) inc += n;
    }
    bucket[tid] = inc - v;
  }
  __syncthreads();
  for_each_request([&](int b, int i) { p.dec_order[atomicAdd(&bucket[b], 1)] = i; });
  __syncthreads();
  const int nreq = bucket[kDecOrderBuckets - 1];  // every decode request has a place
  // the items' exclusive prefix in that order; positions past the last request hold the
  // total, so a search over all num_seqs positions never lands there
  int carry = 0;
  for (int base = 0; base < p.num_seqs; base += blockDim.x) {
    const int k = base + tid;
    int v3[3] = {0, 0, 0};
    int i = -1;
    if (k < nreq) {
      i = p.dec_order[k];
      v3[0] = p.dec_prefix[i + 1] - p.dec_prefix[i];
    }
    int ex[3], tot[3];
    block_scan3(v3, ex, tot);
    const int start = carry + ex[0];
    if (k < p.num_seqs) p.dec_start[k] = start;
    for (int m = 0; m < v3[0]; ++m) reinterpret_cast<int2*>(p.dec_pos)[start + m] = make_int2(i, start);
    carry += tot[0];
  }
  if (tid == 0) {
    p.dec_start[p.num_seqs] = total;
    p.counters[kDecOrderSlot] = 1;
  }
}

// The same order built entirely in shared memory, for batches of at most kOrdOnchipSeqs
// requests: the main loop leaves each request's decode item count and bucket in
// s_nd / s_key, and only the position table goes to global memory (the decode
// kernel reads nothing else of an ordered batch).
constexpr int kOrdOnchipSeqs = 4096;
__device__ void order_decode_onchip(const PlanArgs& p, const int32_t* s_nd, const int32_t* s_key, int32_t* s_order) {
  __shared__ int bucket[kDecOrderBuckets];
  const int tid = threadIdx.x;
  if (tid < kDecOrderBuckets) bucket[tid] = 0;
  __syncthreads();
  for (int i = tid; i < p.num_seqs; i += blockDim.x)
    if (s_nd[i] > 0) atomicAdd(&bucket[s_key[i]], 1);
  __syncthreads();
  if (tid < 32) {  // exclusive prefix over the buckets, one warp
    const int v = bucket[tid];
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, inc, o);
      if (tid >= o) inc += n;
    }
    bucket[tid] = inc - v;
  }
  __syncthreads();
  for (int i = tid; i < p.num_seqs; i += blockDim.x)
    if (s_nd[i] > 0) s_order[atomicAdd(&bucket[s_key[i]], 1)] = i;
  __syncthreads();
  const int nreq = bucket[kDecOrderBuckets - 1];  // every decode request has a place
  int carry = 0;
  for (int base = 0; base < nreq; base += blockDim.x) {
    const int k = base + tid;
    const int i = k < nreq ? s_order[k] : -1;
    int v3[3] = {k < nreq ? s_nd[i] : 0, 0, 0};
    int ex[3], tot[3];
    block_scan3(v3, ex, tot);
    const int start = carry + ex[0];
    for (int m = 0; m < v3[0]; ++m) reinterpret_cast<int2*>(p.dec_pos)[start + m] = make_int2(i, start);
    carry += tot[0];
  }
  if (tid == 0) p.counters[kDecOrderSlot] = 1;
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs p) {
  extern __shared__ int32_t plan_smem[];  // writers: query_start_loc; planner: on-chip membership
  // the previous step's kernels read the workspace this rewrites and the cache the
  // writers write: wait for them.  After this call's own copy-on-write launch, which
  // waited for them before it let this one start, only the writers wait (for the
  // copies); the kernels after this one may then start before the copies end
  if (p.num_cow > 0) {
    grid_dep_launch();
    if (blockIdx.x > 0) grid_dep_wait();
  } else {
    grid_dep_wait();
    grid_dep_launch();
  }
  if (blockIdx.x > 0) {  // writer CTAs never join the planner's block barriers
    write_new_tokens(p, plan_smem);
    return;
  }
  if (p.writers_only) return;
  const int64_t n_units = static_cast<int64_t>(p.num_seqs) * p.hkv;
  for (int64_t u = threadIdx.x; u < n_units; u += blockDim.x) {
    p.unit_bad[u] = 0;
  }
  if (threadIdx.x < kNumQueueCounters) p.counters[threadIdx.x] = 0;
  const bool cascade = p.cas.num_groups > 0 && p.cas.num_members > 0;
  const int32_t* seq_pre = p.seq_prefix;  // each request's prefix tokens and member entry
  const int32_t* seq_ent = p.seq_entry;
  if (cascade) {
    prefix_block_checks(p);
    if (p.cas_onchip) {
      int32_t *sp = nullptr, *se = nullptr;
      plan_cascade_onchip(p, plan_smem, sp, se);
      seq_pre = sp;
      seq_ent = se;
    } else {
      plan_cascade(p);
    }
  }
  __syncthreads();
  // on-chip ordering state after the membership region: items and bucket per request
  int32_t* s_nd = nullptr;
  int32_t* s_key = nullptr;
  if (p.ord_onchip) {
    s_nd = plan_smem + p.ord_offset;
    s_key = s_nd + p.num_seqs;
  }
  int carry_d = 0, carry_p = 0, carry_m = 0;
  for (int base = 0; base < p.num_seqs; base += blockDim.x) {
    const int i = base + threadIdx.x;
    int nd = 0, np = 0, nm = 0, key = 0;
    if (i < p.num_seqs) {
      const int64_t q0 = p.qsl[i], q1 = p.qsl[i + 1];
      const int64_t L = p.seq_lens[i];
      const int64_t q_len = q1 - q0;
      const bool rows_ok = q0 >= 0 && q1 >= q0 && q1 <= p.num_tokens;
      if (!rows_ok) {
        flag_error(p.err, kErrLength);  // rows cannot be addressed: no item
      } else if (q_len == 1) {
        const bool ok = L >= 1 && L <= p.max_seq_len && (L + kBlock - 1) / kBlock <= p.max_blocks;
        const int P = cascade ? seq_pre[i] : 0;  // keys the cascade kernel attends
        const int ns = ok ? static_cast<int>(decode_splits(L - P)) : 1;
        nd = p.hkv * ns;
        // the request's bucket for a largest-first order: key tiles of its largest item
        const int64_t tiles = ns > 1 ? p.split_keys / kTileKeys : (L - P + kTileKeys - 1) / kTileKeys;
        key = kDecOrderBuckets - 1 - static_cast<int>(tiles < kDecOrderBuckets - 1 ? (tiles > 0 ? tiles : 0)
                                                                                   : kDecOrderBuckets - 1);
        nm = ns > 1 ? 1 : 0;  // its partials need the split merge (a member of one split
                              // folds its prefix partials in the decode kernel)
      } else if (q_len > 1) {
        np = p.hkv * static_cast<int>((q_len + p.rows_per_tile - 1) / p.rows_per_tile);
      }
    }
    const int v[3] = {nd, np, nm};
    int ex[3], tot[3];
    block_scan3(v, ex, tot);
    if (i < p.num_seqs && s_nd) {
      s_nd[i] = nd;
      s_key[i] = key;
    }
    if (i < p.num_seqs) {
      p.dec_prefix[i] = carry_d + ex[0];
      p.pre_prefix[i] = carry_p + ex[1];
      if (nm) {  // everything the split merge needs about the request, in one 32-byte record
        int4* m = reinterpret_cast<int4*>(p.merge_list) + 2 * static_cast<int64_t>(carry_m + ex[2]);
        m[0] = make_int4(i, carry_d + ex[0], nd / p.hkv, static_cast<int>(p.qsl[i]));
        m[1] = make_int4(cascade ? seq_pre[i] : 0, cascade ? seq_ent[i] : -1, 0, 0);
      }
    }
    carry_d += tot[0];
    carry_p += tot[1];
    carry_m += tot[2];
  }
  if (threadIdx.x == 0) {
    p.dec_prefix[p.num_seqs] = carry_d;
    p.pre_prefix[p.num_seqs] = carry_p;
  }
  // (carry_p and carry_d are the same in every thread)
  if (carry_p > 0 && p.pre_order) order_prefill_pairs(p);
  if (carry_d > 0 && p.dec_order && carry_d <= kDecOrderMaxItemsPerSm * p.num_sms && carry_d <= kDecPosMax) {
    if (p.ord_onchip) order_decode_onchip(p, s_nd, s_key, s_key + p.num_seqs);
    else order_decode_requests(p, carry_d, seq_pre);
  }
  if (threadIdx.x == 0) {
    p.counters[kMergeCountSlot] = carry_m;
  }
}

}  // namespace

int launch_plan(const PlanArgs& p, cudaStream_t s) {
  const int writers = p.k_new ? p.write_ctas : 0;
  // dynamic shared memory: query_start_loc for the writers, the membership state for
  // the planner (on chip when the batch is within the limits), whichever is larger
  PlanArgs q = p;
  size_t smem = 0;
  if (writers > 0 && p.num_seqs <= kWriterQslMax) smem = (static_cast<size_t>(p.num_seqs) + 1) * sizeof(int32_t);
  const bool cascade = p.cas.num_groups > 0 && p.cas.num_members > 0;
  q.cas_onchip = cascade && p.num_seqs <= kCasOnchipSeqs && p.cas.num_members <= kCasOnchipMembers &&
                 p.cas.num_groups <= kCasOnchipGroups && p.cas.max_blocks <= kCasOnchipBlocks;
  q.ord_onchip = p.dec_order != nullptr && p.num_seqs <= kOrdOnchipSeqs;
  // the planner's layout: membership region, then ordering region (each dropped to its
  // global-memory form if the two would not fit)
  auto planner_ints = [&]() {
    int64_t ints = q.cas_onchip ? cas_onchip_ints(p.num_seqs, p.cas.num_members, p.cas.num_groups) : 0;
    q.ord_offset = static_cast<int32_t>(ints);
    return ints + (q.ord_onchip ? 3 * static_cast<int64_t>(p.num_seqs) : 0);  // items, bucket, order
  };
  if (planner_ints() * 4 > kPlanSmemMax) q.ord_onchip = 0;
  if (planner_ints() * 4 > kPlanSmemMax) q.cas_onchip = 0;
  const size_t need = static_cast<size_t>(planner_ints()) * sizeof(int32_t);
  smem = need > smem ? need : smem;
  static uint64_t smem_set = 0;
  const int st = set_smem_once(reinterpret_cast<const void*>(plan_kernel), kPlanSmemMax, &smem_set);
  if (st) return st;
  TraceScope trace(kTracePlan, s);
  return cuda_status(launch_k(plan_kernel, dim3(1 + writers), dim3(kPlanThreads), smem, s, q));
}

}  // namespace pkv
