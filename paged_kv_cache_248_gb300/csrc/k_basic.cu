// k_basic.cu -- slot mapping, KV-slot scatter and copy-on-write block copy.
//
// These are the byte-moving steps of the paged KV cache ("vLLM's PagedAttention"
// teardown, section "PagedAttention: the KV cache is paged, like virtual memory";
// "The 1960s Operating System Trick ..." page, Technical Details, Copy-on-Write).
// All three are HBM/latency bound: 16-byte vector loads and stores, grids sized in
// multiples of the SM count, no shared-memory staging (nothing is reused).
#include "pkv_internal.cuh"

namespace pkv {
namespace {

// One thread per new token: p = seq_len - q_len + j, slot = table[p / 16] * 16 + p % 16.
__global__ void __launch_bounds__(256) slot_mapping_kernel(const int32_t* __restrict__ bt, int32_t max_blocks,
                                                           const int32_t* __restrict__ seq_lens,
                                                           const int32_t* __restrict__ qsl, int32_t num_seqs,
                                                           int64_t num_tokens, int64_t* __restrict__ slots,
                                                           uint32_t* err) {
  grid_dep_wait();
  grid_dep_launch();
  const int64_t t = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (t >= num_tokens) return;
  const int i = find_seq(qsl, num_seqs, t);
  const int64_t q0 = __ldg(qsl + i), q1 = __ldg(qsl + i + 1);
  const int64_t p = static_cast<int64_t>(__ldg(seq_lens + i)) - (q1 - q0) + (t - q0);
  int64_t slot = -1;
  if (t < q0 || t >= q1 || p < 0 || p / kBlock >= max_blocks) {
    flag_error(err, kErrLength);
  } else {
    const int32_t b = __ldg(bt + static_cast<int64_t>(i) * max_blocks + p / kBlock);
    if (b < 0) flag_error(err, kErrBlockId);
    else slot = static_cast<int64_t>(b) * kBlock + p % kBlock;
  }
  slots[t] = slot;
}

// One thread per 16-byte vector of a token's K row (and the same vector of its V row).
__global__ void __launch_bounds__(256) write_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                                    const int64_t* __restrict__ slots, int64_t num_tokens,
                                                    int32_t hkv, int32_t vec_per_row, int64_t num_slots,
                                                    uint4* __restrict__ kc, uint4* __restrict__ vc, uint32_t* err) {
  grid_dep_wait();
  grid_dep_launch();
  const int64_t per_tok = static_cast<int64_t>(hkv) * vec_per_row;
  const int64_t total = num_tokens * per_tok;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int64_t t = idx / per_tok;
    const int64_t r = idx - t * per_tok;  // h * vec_per_row + c
    const int64_t s = __ldg(slots + t);
    if (s < 0) continue;
    if (s >= num_slots) {
      if (r == 0) flag_error(err, kErrSlot);
      continue;
    }
    const int64_t h = r / vec_per_row, c = r - h * vec_per_row;
    const int64_t dst = (((s / kBlock) * hkv + h) * kBlock + (s % kBlock)) * vec_per_row + c;
    const uint4 kv = __ldcs(k + idx);
    const uint4 vv = __ldcs(v + idx);
    kc[dst] = kv;
    vc[dst] = vv;
  }
}

// One CTA per (pair, slice): copies a slice of the K block and of the V block.
constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;
__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(const int32_t* __restrict__ src,
                                                                   const int32_t* __restrict__ dst, int64_t n,
                                                                   int64_t num_blocks, int64_t vec_per_block,
                                                                   int32_t slices, uint4* kc, uint4* vc,
                                                                   uint32_t* err) {
  grid_dep_wait();
  grid_dep_launch();
  const int64_t pair = blockIdx.x / slices;
  const int32_t slice = blockIdx.x % slices;
  if (pair >= n) return;
  const int64_t s = __ldg(src + pair), d = __ldg(dst + pair);
  if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
    if (threadIdx.x == 0 && slice == 0) flag_error(err, kErrBlockId);
    return;
  }
  const int64_t per_slice = (vec_per_block + slices - 1) / slices;
  const int64_t begin = slice * per_slice;
  const int64_t end = begin + per_slice < vec_per_block ? begin + per_slice : vec_per_block;
  const uint4* ks = kc + s * vec_per_block;
  const uint4* vs = vc + s * vec_per_block;
  uint4* kd = kc + d * vec_per_block;
  uint4* vd = vc + d * vec_per_block;
  for (int64_t c0 = begin + threadIdx.x; c0 < end; c0 += kCopyThreads * kCopyUnroll) {
    uint4 a[kCopyUnroll], b[kCopyUnroll];
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t c = c0 + static_cast<int64_t>(u) * kCopyThreads;
      if (c < end) {
        a[u] = ks[c];
        b[u] = vs[c];
      }
    }
#pragma unroll
    for (int u = 0; u < kCopyUnroll; ++u) {
      const int64_t c = c0 + static_cast<int64_t>(u) * kCopyThreads;
      if (c < end) {
        kd[c] = a[u];
        vd[c] = b[u];
      }
    }
  }
}

}  // namespace

int launch_slot_mapping(const int32_t* bt, int32_t max_blocks, const int32_t* seq_lens, const int32_t* qsl,
                        int32_t num_seqs, int64_t num_tokens, int64_t* slots, uint32_t* err, cudaStream_t s) {
  if (num_tokens == 0) return PKV_OK;
  TraceScope trace(kTraceSlotMap, s);
  const int threads = 256;
  const int64_t blocks = (num_tokens + threads - 1) / threads;
  return cuda_status(launch_k(slot_mapping_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, s, bt,
                              max_blocks, seq_lens, qsl, num_seqs, num_tokens, slots, err));
}

int launch_write(const void* k, const void* v, const int64_t* slots, int64_t T, void* kc, void* vc,
                 const pkv_cache_desc& c, uint32_t* err, cudaStream_t s) {
  if (T == 0) return PKV_OK;
  int status = PKV_OK;
  DeviceCtx* ctx = device_ctx(&status);
  if (!ctx) return status;
  TraceScope trace(kTraceWrite, s);
  const int elem = c.dtype == PKV_F32 ? 4 : 2;
  const int32_t vec_per_row = c.head_dim * elem / 16;
  const int64_t total = T * c.num_kv_heads * vec_per_row;
  const int threads = 256;
  int64_t blocks = (total + threads - 1) / threads;
  const int64_t cap = static_cast<int64_t>(ctx->num_sms) * 16;
  if (blocks > cap) blocks = cap;
  return cuda_status(launch_k(write_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, s,
                              static_cast<const uint4*>(k), static_cast<const uint4*>(v), slots, T, c.num_kv_heads,
                              vec_per_row, c.num_blocks * kBlock, static_cast<uint4*>(kc),
                              static_cast<uint4*>(vc), err));
}

int launch_copy_blocks(const int32_t* src, const int32_t* dst, int64_t n, void* kc, void* vc,
                       const pkv_cache_desc& c, uint32_t* err, cudaStream_t s) {
  if (n == 0) return PKV_OK;
  int status = PKV_OK;
  DeviceCtx* ctx = device_ctx(&status);
  if (!ctx) return status;
  TraceScope trace(kTraceCopy, s);
  const int elem = c.dtype == PKV_F32 ? 4 : 2;
  const int64_t vec_per_block = static_cast<int64_t>(c.num_kv_heads) * kBlock * c.head_dim * elem / 16;
  // enough CTAs to cover every SM a few times even for few pairs
  int32_t slices = 1;
  while (n * slices < 4LL * ctx->num_sms && vec_per_block / (slices * 2) >= kCopyThreads) slices *= 2;
  const int64_t blocks = n * slices;
  if (blocks > 0x7fffffffLL) return PKV_ERR_INVALID_ARG;
  return cuda_status(launch_k(copy_blocks_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kCopyThreads), 0, s,
                              src, dst, n, c.num_blocks, vec_per_block, slices, static_cast<uint4*>(kc),
                              static_cast<uint4*>(vc), err));
}

}  // namespace pkv
