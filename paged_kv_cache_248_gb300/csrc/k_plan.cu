// k_plan.cu -- device-side planning of one paged_attention call.
//
// One CTA scans the batch ("Continuous batching": every request is a pair of
// computed / total tokens, and one step mixes decodes and prefill chunks) and
// writes two work lists as exclusive prefix sums over the requests:
//   decode items  -- requests with exactly one query token: num_kv_heads x
//                    decode_splits(seq_len) (kv head, key split) items;
//   prefill items -- requests with more query tokens: num_kv_heads x
//                    ceil(q_len / rows_per_tile) (kv head, query tile) items.
// Split boundaries depend only on a request's own length and a library constant,
// so a request's result does not depend on what else is in the batch.  It also
// zeroes the work-queue counters and the per-(request, kv head) bad-block flags
// used by the split merge, and lists the requests whose splits need merging.  Lengths that contradict the host
// bounds become a single item that reports the error and zeroes its output.
//
// Shared-prefix groups (paged_attention_cascade) are checked here first.  A listed
// request becomes a member of its group only if it is listed once, is a decode whose
// context goes past the prefix, and its block table starts with the prefix's block
// ids (one warp compares a member's row, 32 ids per load).  A member's decode items
// then cover only the keys after the prefix, it always goes to the split merge, and
// the cascade kernel gets ceil(members / rows) x kv heads x cascade_splits(P) items
// per group.  Anything else listed is attended the ordinary way.
#include "pkv_internal.cuh"

namespace pkv {
namespace {

constexpr int kPlanThreads = 1024;

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

// Shared-prefix membership: fills seq_prefix / seq_entry / member_ok and the
// cascade item prefix over groups.  Called by the whole block.
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
  const int warp = tid >> 5, lane = tid & 31, nwarps = nthr >> 5;
  for (int k = warp; k < g.num_members; k += nwarps) {  // warp-uniform per entry
    const int i = g.members[k];
    int ok = 0, P = 0;
    if (csr_ok && i >= 0 && i < p.num_seqs && p.seq_entry[i] == k && p.seq_prefix[i] == 0) {
      int lo = 0, hi = g.num_groups - 1;  // the group of entry k: last gi with start[gi] <= k
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (g.start[mid] <= k) lo = mid; else hi = mid - 1;
      }
      const int pb = g.blocks[lo];
      const int64_t q0 = p.qsl[i], q1 = p.qsl[i + 1], L = p.seq_lens[i];
      if (pb >= 1 && pb <= g.max_blocks && q0 >= 0 && q1 == q0 + 1 && q1 <= p.num_tokens && L <= p.max_seq_len &&
          (L + kBlock - 1) / kBlock <= p.max_blocks && L > static_cast<int64_t>(pb) * kBlock) {
        const int32_t* own = p.bt + static_cast<int64_t>(i) * p.max_blocks;
        const int32_t* pre = g.tables + static_cast<int64_t>(lo) * g.max_blocks;
        int diff = 0;
        for (int j = lane; j < pb; j += 32) diff |= __ldg(own + j) != __ldg(pre + j);
        ok = !__any_sync(0xffffffffu, diff);
        P = pb * kBlock;
      }
    }
    if (lane == 0) {
      p.member_ok[k] = ok;
      if (ok) p.seq_prefix[i] = P;
      else if (csr_ok && i >= 0 && i < p.num_seqs && p.seq_entry[i] == k && p.seq_prefix[i] == 0)
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

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs p) {
  const int64_t n_units = static_cast<int64_t>(p.num_seqs) * p.hkv;
  for (int64_t u = threadIdx.x; u < n_units; u += blockDim.x) {
    p.unit_bad[u] = 0;
  }
  if (threadIdx.x < kNumQueueCounters) p.counters[threadIdx.x] = 0;
  const bool cascade = p.cas.num_groups > 0 && p.cas.num_members > 0;
  if (cascade) plan_cascade(p);
  __syncthreads();
  int carry_d = 0, carry_p = 0, carry_m = 0;
  for (int base = 0; base < p.num_seqs; base += blockDim.x) {
    const int i = base + threadIdx.x;
    int nd = 0, np = 0, nm = 0;
    if (i < p.num_seqs) {
      const int64_t q0 = p.qsl[i], q1 = p.qsl[i + 1];
      const int64_t L = p.seq_lens[i];
      const int64_t q_len = q1 - q0;
      const bool rows_ok = q0 >= 0 && q1 >= q0 && q1 <= p.num_tokens;
      if (!rows_ok) {
        flag_error(p.err, kErrLength);  // rows cannot be addressed: no item
      } else if (q_len == 1) {
        const bool ok = L >= 1 && L <= p.max_seq_len && (L + kBlock - 1) / kBlock <= p.max_blocks;
        const int P = cascade ? p.seq_prefix[i] : 0;  // keys the cascade kernel attends
        const int ns = ok ? static_cast<int>(decode_splits(L - P)) : 1;
        nd = p.hkv * ns;
        nm = (ns > 1 || P > 0) ? 1 : 0;  // its partials need the split merge
      } else if (q_len > 1) {
        np = p.hkv * static_cast<int>((q_len + p.rows_per_tile - 1) / p.rows_per_tile);
      }
    }
    const int v[3] = {nd, np, nm};
    int ex[3], tot[3];
    block_scan3(v, ex, tot);
    if (i < p.num_seqs) {
      p.dec_prefix[i] = carry_d + ex[0];
      p.pre_prefix[i] = carry_p + ex[1];
      if (nm) p.merge_list[carry_m + ex[2]] = i;
    }
    carry_d += tot[0];
    carry_p += tot[1];
    carry_m += tot[2];
  }
  if (threadIdx.x == 0) {
    p.dec_prefix[p.num_seqs] = carry_d;
    p.pre_prefix[p.num_seqs] = carry_p;
    p.counters[kMergeCountSlot] = carry_m;
  }
}

}  // namespace

int launch_plan(const PlanArgs& p, cudaStream_t s) {
  TraceScope trace(kTracePlan, s);
  plan_kernel<<<1, kPlanThreads, 0, s>>>(p);
  return cuda_status(cudaGetLastError());
}

}  // namespace pkv
