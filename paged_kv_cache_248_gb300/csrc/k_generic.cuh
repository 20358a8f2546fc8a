// k_generic.cuh -- the fused form of the CUDA-core attention path (fp32 caches).
#pragma once
#include "pkv_internal.cuh"

namespace pkv {

// A step whose requests each bring one new token, on an fp32 cache: each CTA of the
// attention launch first stores its token's K and V rows ([T, Hkv, head_dim], like
// pkv_write) into the token's slot and reports the slot in slots_out (may be null), with
// the writer path's error checks, so that no separate write launch is needed.
struct GenericWrite {
  const void* k_new;
  const void* v_new;
  int64_t* slots_out;
};
int launch_generic_attention_write(const AttnArgs& a, const GenericWrite& w, uint32_t* err, cudaStream_t s);

}  // namespace pkv
