// shrink_rows.cu -- the LoRA shrink of short adapter runs on CUDA cores.
//
// S_run = X_run * A[a,e]^T for runs of a few token rows (weight-streaming blocks of
// 16-64 rows; a decode run holds one or two).  The work is a skinny matrix-vector
// product, read-bound on A, so it is split over the hidden dimension: one CTA per
// (run, 256-wide K slice), each warp taking rank rows with its lanes across the slice
// and a warp-shuffle reduction per dot product.  The pages tune the skinny shrink
// with Split-K (AWS ML Blog "Efficiently serve dozens of fine-tuned models with vLLM
// on Amazon SageMaker AI and Amazon Bedrock", section "Kernel optimizations").  The
// fp32 slice partials are added in slice order by the CTA that completes the run's
// count, so the result does not depend on which CTA finishes first.  The output is the
// same S tile the tensor-core shrink writes: [run][block_m][r_pad] bf16, rows outside
// the run zero, ranks past the adapter's zero.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kRanksPerWarp = 64 / kWarps;   // rank <= 64

__device__ __forceinline__ void unpack8(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__global__ void __launch_bounds__(kThreads) shrink_rows_kernel(const ShrinkRowsLaunch a) {
  __shared__ __align__(16) uint16_t s_x[64][kShrinkSlice];   // the run's token rows of this slice
  __shared__ int s_last;
  // token rows come from the previous kernel (gather or gate_up); the GEMM after this
  // one may launch now and stream its base weights
  pdl_wait();
  pdl_trigger();
  const int run = static_cast<int>(blockIdx.x) / a.slices;
  const int ks = static_cast<int>(blockIdx.x) - run * a.slices;
  if (run >= a.totals[2]) return;
  const int b = a.runs[4 * run + 0], ad = a.runs[4 * run + 1];
  const int beg = a.runs[4 * run + 2], end = a.runs[4 * run + 3];
  const int e = a.block_expert[b];
  const int r = a.ranks[ad];
  const int nrows = end - beg;   // <= block_m <= 64
  const int k0 = ks * kShrinkSlice;
  const int kl = min(kShrinkSlice, a.K - k0);   // multiple of 64
  const int v8 = kl / 8;
  for (int idx = threadIdx.x; idx < nrows * v8; idx += kThreads) {
    const int i = idx / v8, c = idx - i * v8;
    reinterpret_cast<uint4*>(s_x[i])[c] =
        __ldg(reinterpret_cast<const uint4*>(a.xs + static_cast<size_t>(beg + i) * a.K + k0) + c);
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool act = lane < v8;
  // this warp's rank rows j = warp + kWarps * t: all loads in flight at once
  const uint16_t* Ab = a.A + (static_cast<size_t>(ad) * a.E + e) * a.r_max * a.K + k0;
  float av[kRanksPerWarp][8];
#pragma unroll
  for (int t = 0; t < kRanksPerWarp; ++t) {
    const int j = warp + kWarps * t;
    uint4 raw = make_uint4(0u, 0u, 0u, 0u);
    if (act && j < r) raw = __ldg(reinterpret_cast<const uint4*>(Ab + static_cast<size_t>(j) * a.K) + lane);
    unpack8(raw, av[t]);
  }
  __syncthreads();
  float* part = a.s_part + (static_cast<size_t>(ks) * a.max_runs + run) * a.block_m * a.r_pad;
  for (int i = 0; i < nrows; ++i) {
    float xv[8];
    unpack8(act ? reinterpret_cast<const uint4*>(s_x[i])[lane] : make_uint4(0u, 0u, 0u, 0u), xv);
    float acc[kRanksPerWarp];
#pragma unroll
    for (int t = 0; t < kRanksPerWarp; ++t) {
      float s = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q) s = fmaf(av[t][q], xv[q], s);
      acc[t] = s;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
#pragma unroll
      for (int t = 0; t < kRanksPerWarp; ++t) acc[t] += __shfl_xor_sync(0xffffffffu, acc[t], off);
    if (lane == 0) {
#pragma unroll
      for (int t = 0; t < kRanksPerWarp; ++t) {
        const int j = warp + kWarps * t;
        if (j < r) part[static_cast<size_t>(i) * a.r_pad + j] = acc[t];
      }
    }
  }
  // the CTA that completes the run's slice count adds the slices in order
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(a.s_cnt + 4 * run, 1) == a.slices - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  uint16_t* S = a.s_out + static_cast<size_t>(run) * a.block_m * a.r_pad;
  const int rb = beg - b * a.block_m;
  for (int idx = threadIdx.x; idx < a.block_m * a.r_pad; idx += kThreads) {
    const int row = idx / a.r_pad, j = idx - row * a.r_pad;
    const int i = row - rb;
    float v = 0.f;
    if (i >= 0 && i < nrows && j < r) {
      for (int sp = 0; sp < a.slices; ++sp)
        v += __ldcg(a.s_part + ((static_cast<size_t>(sp) * a.max_runs + run) * a.block_m + i) * a.r_pad + j);
    }
    __nv_bfloat16 h = __float2bfloat16_rn(v);
    S[idx] = *reinterpret_cast<uint16_t*>(&h);
  }
}

}  // namespace

cudaError_t launch_shrink_rows(const ShrinkRowsLaunch& a, int64_t max_runs, bool pdl, cudaStream_t s) {
  const int64_t grid = max_runs * a.slices;
  if (grid <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, shrink_rows_kernel, a);
}

}  // namespace moe
