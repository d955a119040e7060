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

static_assert(MOE_LORA_MAX_TOPK <= 32, "lane j of the routing warp keeps the j-th choice");

// Lane i owns experts i, i+32, ... (SLOTS per lane, E <= 32 * SLOTS).  With REGS its
// logits are read into registers once and the k selection passes run on registers;
// without (the widest routers) every pass re-reads them, which keeps the register
// count of the kernels around it low.  Lane j keeps the j-th choice (k <= 32).  Lanes
// j < k write the ids and weights of the token to ids[j] and wts[j] (any address space).
template <int SLOTS, bool REGS = true>
__device__ __forceinline__ void route_token_n(const float* __restrict__ l, int E, int k, int lane, int32_t* ids,
                                              float* wts) {
  float lv[REGS ? SLOTS : 1];
  if constexpr (REGS) {
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      const int ex = lane + 32 * s;
      lv[s] = ex < E ? l[ex] : 0.f;
    }
  }
  uint32_t taken = 0;   // bit s: expert lane + 32*s already chosen
  float my_v = 0.f;     // lane j: the j-th chosen logit and expert
  int my_e = 0;
  for (int j = 0; j < k; ++j) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      const int ex = lane + 32 * s;
      if (ex >= E || (taken & (1u << s))) continue;
      const float v = REGS ? lv[s] : l[ex];
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
    if (lane == j) {
      my_v = bv;
      my_e = bi;
    }
  }
  // every lane forms the same sum, in choice order
  const float mx = __shfl_sync(0xffffffffu, my_v, 0);
  float z = 0.f;
  for (int j = 0; j < k; ++j) z += expf(__shfl_sync(0xffffffffu, my_v, j) - mx);
  const float inv = 1.0f / z;
  if (lane < k) {
    ids[lane] = my_e;
    wts[lane] = expf(my_v - mx) * inv;
  }
}

// route_token_n with the fewest register slots that hold E experts (warp-uniform E).
__device__ __forceinline__ void route_token(const float* __restrict__ l, int E, int k, int lane, int32_t* ids,
                                            float* wts) {
  if (E <= 32) route_token_n<1>(l, E, k, lane, ids, wts);
  else if (E <= 64) route_token_n<2>(l, E, k, lane, ids, wts);
  else if (E <= 128) route_token_n<4>(l, E, k, lane, ids, wts);
  else if (E <= 256) route_token_n<8>(l, E, k, lane, ids, wts);
  else route_token_n<(MOE_LORA_MAX_EXPERTS + 31) / 32, false>(l, E, k, lane, ids, wts);
}

}  // namespace moe
