// route.cu -- router top-k with softmax weights renormalised over the chosen experts
// (the per-token rule is in route.cuh).
#include "route.cuh"

namespace moe {
namespace {

// One warp per token.
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int64_t T, int E, int k,
                                                    int32_t* __restrict__ ids, float* __restrict__ wts) {
  const int lane = threadIdx.x & 31;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (t >= T) return;
  route_token(logits + t * E, E, k, lane, ids + t * k, wts + t * k);
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
