// route.cuh -- router top-k for one token, computed by one warp.
//
// A router directs each token to its most relevant experts (AWS ML Blog "Efficiently
// serve dozens of fine-tuned models with vLLM on Amazon SageMaker AI and Amazon
// Bedrock", section "Implementing multi-LoRA inference for MoE models in vLLM").
// Experts are chosen by raw fp32 logit, descending, ties to the lower index; the
// weight of expert j is exp(l_j - l_max) / sum over the chosen k, which equals the
// softmax over all E experts renormalised over the chosen k.
#pragma once

#include <cstdint>

#include "common.cuh"

namespace moe {

// Lane i owns experts i, i+32, ... (E <= 1024 -> 32 per lane).  Lane 0 writes the k
// ids and weights of the token to ids[0..k) and wts[0..k) (any address space).
__device__ __forceinline__ void route_token(const float* __restrict__ l, int E, int k, int lane, int32_t* ids,
                                            float* wts) {
  uint32_t taken = 0;   // bit s: expert lane + 32*s already chosen
  float vals[MOE_LORA_MAX_TOPK];
  int chosen[MOE_LORA_MAX_TOPK];
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
    for (int s = 0, ex = lane; ex < E; ++s, ex += 32) {
      if (taken & (1u << s)) continue;
      const float v = l[ex];
      if (bi == 0x7fffffff || v > bv || (v == bv && ex < bi)) {
        bv = v;
        bi = ex;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (oi != 0x7fffffff && (bi == 0x7fffffff || ov > bv || (ov == bv && oi < bi))) {
        bv = ov;
        bi = oi;
      }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    vals[j] = bv;
    chosen[j] = bi;
  }
  if (lane == 0) {
    const float mx = vals[0];
    float z = 0.f;
    for (int j = 0; j < k; ++j) z += expf(vals[j] - mx);
    const float inv = 1.0f / z;
    for (int j = 0; j < k; ++j) {
      ids[j] = chosen[j];
      wts[j] = expf(vals[j] - mx) * inv;
    }
  }
}

}  // namespace moe
