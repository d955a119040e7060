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
    // this lane's best remaining expert (ties: the lower index, i.e. the lower slot)
    float bv = 0.f;
    int bi = 0x7fffffff;
#pragma unroll
    for (int s = 0; s < SLOTS; ++s) {
      const int ex = lane + 32 * s;
      if (ex >= E || (taken & (1u << s))) continue;
      const float v = REGS ? lv[s] : l[ex];
      if (bi == 0x7fffffff || v > bv) {
        bv = v;
        bi = ex;
      }
    }
    // the warp's best: the largest logit by an order-preserving integer image (-0 and
    // +0 made equal, as the float comparison has them), then the lowest expert index
    // among the lanes holding it
    const float z0 = bv + 0.0f;
    const uint32_t u = __float_as_uint(z0);
    const uint32_t key = bi == 0x7fffffff ? 0u : ((u & 0x80000000u) ? ~u : (u | 0x80000000u));
    const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
    const int win = static_cast<int>(__reduce_min_sync(0xffffffffu, key == kmax && bi != 0x7fffffff
                                                                         ? static_cast<uint32_t>(bi)
                                                                         : 0xffffffffu));
    const float wv = __shfl_sync(0xffffffffu, bv, win & 31);
    if ((win & 31) == lane) taken |= 1u << (win >> 5);
    if (lane == j) {
      my_v = wv;
      my_e = win;
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
