// k_generic.cu -- CUDA-core paged attention for any query row (decode or prefill).
//
// One CTA per (query token, kv head, chunk of up to 8 query heads of that kv head's
// group).  The CTA walks the token's visible keys (positions 0..p, p = seq_len -
// q_len + j; "vLLM's PagedAttention" teardown, sections "PagedAttention" and
// "Continuous batching"), gathering each key's row through the block table.  Each
// warp takes every fourth key and keeps its own online-softmax state (running
// maximum, running sum, rescaled accumulator, all fp32); the four states are merged
// at the end.  Lane l owns head_dim/32 consecutive elements, so every K/V row read is
// one coalesced warp access.  This path serves the fp32 caches, where tensor cores
// would not keep the 1e-4 accuracy the fp32 inputs call for.
//
// Fused form (kWrite), for a step whose requests each bring one new token: before it
// attends, every CTA stores its kv head's K and V rows of its own token into the
// token's slot (the slot mapping of the teardown's "PagedAttention" section), with the
// error checks and slot report of the writer path, then reads the cache coherently
// (L2) so that its own rows are seen.  CTAs of the same token write the same bytes,
// and no CTA reads a row another token's CTA writes: a one-token request's only new
// row is its own query's.  So one launch replaces the writer launch and this one.
#include <cmath>

#include "k_generic.cuh"

namespace pkv {
namespace {

constexpr int kGenThreads = 128;
constexpr int kGenWarps = kGenThreads / 32;
constexpr int kHeadChunk = 8;
constexpr float kLog2e = 1.4426950408889634f;

// A K or V element: through the read-only path, or (kCoherent, after this kernel's own
// stores to the cache) from L2.
template <bool kCoherent>
__device__ __forceinline__ float ld_kv(const float* p) {
  return kCoherent ? __ldcg(p) : __ldg(p);
}
template <bool kCoherent>
__device__ __forceinline__ float ld_kv(const __nv_bfloat16* p) {
  return __bfloat162float(__ldg(p));  // (the fused form is built for fp32 caches only)
}

template <typename T, int D, bool kWrite>
__global__ void __launch_bounds__(kGenThreads) generic_attention_kernel(
    const T* __restrict__ q, const T* kc, const T* vc, int64_t num_blocks, int hkv,
    const int32_t* __restrict__ bt, int32_t max_blocks, const int32_t* __restrict__ seq_lens,
    const int32_t* __restrict__ qsl, int num_seqs, int hq, float scale_log2, T* __restrict__ out, uint32_t* err,
    int prefill_only, const T* __restrict__ k_new, const T* __restrict__ v_new, int64_t* __restrict__ slots_out) {
  static_assert(!kWrite || sizeof(T) == 4, "the fused form serves the fp32 caches");
  constexpr int E = D / 32;
  __shared__ int bad;
  __shared__ float sm_m[kGenWarps][kHeadChunk];
  __shared__ float sm_l[kGenWarps][kHeadChunk];
  __shared__ float sm_o[kGenWarps][kHeadChunk][D];
  grid_dep_wait();
  grid_dep_launch();

  const int group = hq / hkv;
  const int nchunks = (group + kHeadChunk - 1) / kHeadChunk;
  int64_t bid = blockIdx.x;
  const int chunk = static_cast<int>(bid % nchunks);
  bid /= nchunks;
  const int g = static_cast<int>(bid % hkv);
  const int64_t t = bid / hkv;
  const int h0 = g * group + chunk * kHeadChunk;
  const int nh = min(kHeadChunk, group - chunk * kHeadChunk);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  const int i = find_seq(qsl, num_seqs, t);
  const int64_t q0 = __ldg(qsl + i), q1 = __ldg(qsl + i + 1);
  const int64_t L = __ldg(seq_lens + i);
  const int64_t p = L - (q1 - q0) + (t - q0);
  if (prefill_only && q1 - q0 == 1 && t == q0) return;  // decode rows belong to the decode kernel
  if (threadIdx.x == 0) bad = 0;
  if (kWrite) {
    // this token's slot, with the writer path's checks (errors and the slot reported by
    // one CTA of the token); a request with more than one new token breaks the launch's
    // premise, so its rows are flagged and zeroed instead
    const bool reporter = g == 0 && chunk == 0 && threadIdx.x == 0;
    int64_t slot = -1;
    if (t < q0 || t >= q1 || p < 0 || p / kBlock >= max_blocks || q1 - q0 != 1) {
      if (reporter) flag_error(err, kErrLength);
      if (threadIdx.x == 0) bad = 1;
    } else {
      const int32_t b = __ldg(bt + static_cast<int64_t>(i) * max_blocks + p / kBlock);
      if (b < 0) {
        if (reporter) flag_error(err, kErrBlockId);
      } else {
        slot = static_cast<int64_t>(b) * kBlock + p % kBlock;
      }
    }
    if (reporter && slots_out) slots_out[t] = slot;
    if (slot >= num_blocks * kBlock) {
      if (reporter) flag_error(err, kErrSlot);
      slot = -1;
    }
    constexpr int kVecs = D * static_cast<int>(sizeof(T)) / 16;  // 16-byte pieces of one kv head's row
    if (slot >= 0 && threadIdx.x < kVecs) {
      const int64_t src = (t * hkv + g) * kVecs + threadIdx.x;
      const int64_t dst = (((slot / kBlock) * hkv + g) * kBlock + slot % kBlock) * kVecs + threadIdx.x;
      reinterpret_cast<uint4*>(const_cast<T*>(kc))[dst] = __ldg(reinterpret_cast<const uint4*>(k_new) + src);
      reinterpret_cast<uint4*>(const_cast<T*>(vc))[dst] = __ldg(reinterpret_cast<const uint4*>(v_new) + src);
    }
  }
  __syncthreads();
  const bool len_ok = t >= q0 && t < q1 && p >= 0 && (L + kBlock - 1) / kBlock <= max_blocks;
  if (!len_ok && threadIdx.x == 0) {
    flag_error(err, kErrLength);
    bad = 1;
  }

  float qr[kHeadChunk][E];
#pragma unroll
  for (int hh = 0; hh < kHeadChunk; ++hh)
#pragma unroll
    for (int e = 0; e < E; ++e)
      qr[hh][e] = hh < nh ? Elem<T>::to_f32(q[(t * hq + h0 + hh) * D + lane * E + e]) : 0.f;

  float m[kHeadChunk], l[kHeadChunk], o[kHeadChunk][E];
#pragma unroll
  for (int hh = 0; hh < kHeadChunk; ++hh) {
    m[hh] = -INFINITY;
    l[hh] = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) o[hh][e] = 0.f;
  }

  const int64_t nkeys = len_ok ? p + 1 : 0;
  const int32_t* row = bt + static_cast<int64_t>(i) * max_blocks;
  for (int64_t u = warp; u < nkeys; u += kGenWarps) {
    const int32_t b = __ldg(row + u / kBlock);
    if (b < 0 || b >= num_blocks) {
      if (lane == 0) {
        flag_error(err, kErrBlockId);
        bad = 1;
      }
      break;
    }
    const int64_t off = ((static_cast<int64_t>(b) * hkv + g) * kBlock + u % kBlock) * D + lane * E;
    float kf[E], vf[E];
#pragma unroll
    for (int e = 0; e < E; ++e) {
      kf[e] = ld_kv<kWrite>(kc + off + e);
      vf[e] = ld_kv<kWrite>(vc + off + e);
    }
#pragma unroll
    for (int hh = 0; hh < kHeadChunk; ++hh) {
      if (hh >= nh) break;
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < E; ++e) dot = fmaf(qr[hh][e], kf[e], dot);
#pragma unroll
      for (int sh = 16; sh > 0; sh >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, sh);
      const float s = dot * scale_log2;
      const float m_new = fmaxf(m[hh], s);
      const float alpha = exp2f(m[hh] - m_new);
      const float pr = exp2f(s - m_new);
      l[hh] = l[hh] * alpha + pr;
#pragma unroll
      for (int e = 0; e < E; ++e) o[hh][e] = fmaf(o[hh][e], alpha, pr * vf[e]);
      m[hh] = m_new;
    }
  }

#pragma unroll
  for (int hh = 0; hh < kHeadChunk; ++hh) {
    if (lane == 0) {
      sm_m[warp][hh] = m[hh];
      sm_l[warp][hh] = l[hh];
    }
#pragma unroll
    for (int e = 0; e < E; ++e) sm_o[warp][hh][lane * E + e] = o[hh][e];
  }
  __syncthreads();
  const bool zero = bad != 0;
  for (int idx = threadIdx.x; idx < nh * D; idx += kGenThreads) {
    const int hh = idx / D, c = idx % D;
    float res = 0.f;
    if (!zero) {
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kGenWarps; ++w) M = fmaxf(M, sm_m[w][hh]);
      float den = 0.f, num = 0.f;
#pragma unroll
      for (int w = 0; w < kGenWarps; ++w) {
        const float f = exp2f(sm_m[w][hh] - M);  // warps that saw no key have m = -inf -> f = 0
        den = fmaf(sm_l[w][hh], f, den);
        num = fmaf(sm_o[w][hh][c], f, num);
      }
      res = num / den;
    }
    out[(t * hq + h0 + hh) * D + c] = Elem<T>::from_f32(res);
  }
}

template <typename T, int D, bool kWrite>
int launch_typed(const AttnArgs& a, uint32_t* err, cudaStream_t s, bool prefill_only, const GenericWrite* w) {
  const int hkv = a.cache.num_kv_heads;
  const int group = a.num_q_heads / hkv;
  const int nchunks = (group + kHeadChunk - 1) / kHeadChunk;
  const int64_t blocks = a.num_tokens * hkv * nchunks;
  if (blocks > 0x7fffffffLL) return PKV_ERR_INVALID_ARG;
  return cuda_status(launch_k(generic_attention_kernel<T, D, kWrite>, dim3(static_cast<unsigned>(blocks)),
                              dim3(kGenThreads), 0, s, static_cast<const T*>(a.q), static_cast<const T*>(a.k_cache),
                              static_cast<const T*>(a.v_cache), a.cache.num_blocks, hkv, a.block_tables,
                              a.max_blocks, a.seq_lens, a.qsl, a.num_seqs, a.num_q_heads, a.scale * kLog2e,
                              static_cast<T*>(a.out), err, prefill_only ? 1 : 0,
                              static_cast<const T*>(w ? w->k_new : nullptr), static_cast<const T*>(w ? w->v_new : nullptr),
                              w ? w->slots_out : nullptr));
}

}  // namespace

int launch_generic_attention(const AttnArgs& a, uint32_t* err, cudaStream_t s, bool prefill_only) {
  if (a.num_tokens == 0) return PKV_OK;
  TraceScope trace(kTraceGeneric, s);
  const int d = a.cache.head_dim;
  if (a.cache.dtype == PKV_F32) {
    if (d == 64) return launch_typed<float, 64, false>(a, err, s, prefill_only, nullptr);
    if (d == 128) return launch_typed<float, 128, false>(a, err, s, prefill_only, nullptr);
  } else if (a.cache.dtype == PKV_BF16) {
    if (d == 128) return launch_typed<__nv_bfloat16, 128, false>(a, err, s, prefill_only, nullptr);
  }
  return PKV_ERR_UNSUPPORTED;
}

int launch_generic_attention_write(const AttnArgs& a, const GenericWrite& w, uint32_t* err, cudaStream_t s) {
  if (a.num_tokens == 0) return PKV_OK;
  TraceScope trace(kTraceGeneric, s);
  const int d = a.cache.head_dim;
  if (a.cache.dtype == PKV_F32) {
    if (d == 64) return launch_typed<float, 64, true>(a, err, s, false, &w);
    if (d == 128) return launch_typed<float, 128, true>(a, err, s, false, &w);
  }
  return PKV_ERR_UNSUPPORTED;
}

}  // namespace pkv
