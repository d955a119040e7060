// route.cu -- router top-k with softmax weights renormalised over the chosen experts.
//
// A router directs each token to its most relevant experts (AWS ML Blog "Efficiently
// serve dozens of fine-tuned models with vLLM on Amazon SageMaker AI and Amazon
// Bedrock", section "Implementing multi-LoRA inference for MoE models in vLLM").
// Experts are chosen by raw fp32 logit, descending, ties to the lower index; the
// weight of expert j is exp(l_j - l_max) / sum over the chosen k, which equals the
// softmax over all E experts renormalised over the chosen k.
#include "common.cuh"

namespace moe {
namespace {

// One warp per token.  Lane i owns experts i, i+32, ... (E <= 1024 -> 32 per lane).
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int64_t T, int E, int k,
                                                    int32_t* __restrict__ ids, float* __restrict__ wts) {
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* l = logits + t * E;
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
      ids[t * k + j] = chosen[j];
      wts[t * k + j] = expf(vals[j] - mx) * inv;
    }
  }
}

}  // namespace

cudaError_t launch_route(const float* logits, int64_t T, int E, int k, int32_t* ids, float* w, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int warps = 8;
  const int64_t blocks = (T + warps - 1) / warps;
  route_kernel<<<static_cast<unsigned>(blocks), warps * 32, 0, s>>>(logits, T, E, k, ids, w);
  return cudaGetLastError();
}

}  // namespace moe
