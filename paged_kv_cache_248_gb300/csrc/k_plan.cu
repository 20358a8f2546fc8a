// k_plan.cu -- device-side planning of one paged_attention call.
//
// One CTA scans the batch ("Continuous batching": every request is a pair of
// computed / total tokens, and one step mixes decodes and prefill chunks) and
// writes two work lists as exclusive prefix sums over the requests:
//   decode items  -- requests with exactly one query token: num_kv_heads x
//                    ceil(seq_len / split_keys) (kv head, key split) items;
//   prefill items -- requests with more query tokens: num_kv_heads x
//                    ceil(q_len / rows_per_tile) (kv head, query tile) items.
// Split boundaries depend only on a request's own length and a library constant,
// so a request's result does not depend on what else is in the batch.  It also
// zeroes the work-queue counters and the per-(request, kv head) bad-block flags
// used by the split merge.  Lengths that contradict the host
// bounds become a single item that reports the error and zeroes its output.
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

// Block-wide exclusive scan of two counters at once.
__device__ void block_scan2(int a, int b, int& ex_a, int& ex_b, int& tot_a, int& tot_b) {
  __shared__ int wa[32], wb[32];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const int ia = warp_inclusive_scan(a), ib = warp_inclusive_scan(b);
  if (lane == 31) {
    wa[warp] = ia;
    wb[warp] = ib;
  }
  __syncthreads();
  if (warp == 0) {
    int x = lane < nwarps ? wa[lane] : 0;
    int y = lane < nwarps ? wb[lane] : 0;
    x = warp_inclusive_scan(x);
    y = warp_inclusive_scan(y);
    wa[lane] = x;
    wb[lane] = y;
  }
  __syncthreads();
  ex_a = (warp ? wa[warp - 1] : 0) + ia - a;
  ex_b = (warp ? wb[warp - 1] : 0) + ib - b;
  tot_a = wa[nwarps - 1];
  tot_b = wb[nwarps - 1];
  __syncthreads();
}

__global__ void __launch_bounds__(kPlanThreads) plan_kernel(PlanArgs p) {
  const int64_t n_units = static_cast<int64_t>(p.num_seqs) * p.hkv;
  for (int64_t u = threadIdx.x; u < n_units; u += blockDim.x) {
    p.unit_bad[u] = 0;
  }
  if (threadIdx.x < kNumQueueCounters) p.counters[threadIdx.x] = 0;
  int carry_d = 0, carry_p = 0;
  for (int base = 0; base < p.num_seqs; base += blockDim.x) {
    const int i = base + threadIdx.x;
    int nd = 0, np = 0;
    if (i < p.num_seqs) {
      const int64_t q0 = p.qsl[i], q1 = p.qsl[i + 1];
      const int64_t L = p.seq_lens[i];
      const int64_t q_len = q1 - q0;
      const bool rows_ok = q0 >= 0 && q1 >= q0 && q1 <= p.num_tokens;
      if (!rows_ok) {
        flag_error(p.err, kErrLength);  // rows cannot be addressed: no item
      } else if (q_len == 1) {
        const bool ok = L >= 1 && L <= p.max_seq_len && (L + kBlock - 1) / kBlock <= p.max_blocks;
        nd = p.hkv * (ok ? static_cast<int>((L + p.split_keys - 1) / p.split_keys) : 1);
      } else if (q_len > 1) {
        np = p.hkv * static_cast<int>((q_len + p.rows_per_tile - 1) / p.rows_per_tile);
      }
    }
    int ed, ep, td, tp;
    block_scan2(nd, np, ed, ep, td, tp);
    if (i < p.num_seqs) {
      p.dec_prefix[i] = carry_d + ed;
      p.pre_prefix[i] = carry_p + ep;
    }
    carry_d += td;
    carry_p += tp;
  }
  if (threadIdx.x == 0) {
    p.dec_prefix[p.num_seqs] = carry_d;
    p.pre_prefix[p.num_seqs] = carry_p;
  }
}

}  // namespace

int launch_plan(const PlanArgs& p, cudaStream_t s) {
  TraceScope trace(kTracePlan, s);
  plan_kernel<<<1, kPlanThreads, 0, s>>>(p);
  return cuda_status(cudaGetLastError());
}

}  // namespace pkv
