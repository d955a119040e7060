// rows.cu -- row gather into sorted order and the final fp32 -> bf16 conversion.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

// x_sorted[row] = x[sorted_p[row] / k] for real rows, zero for padding rows; one warp
// per row, 16-byte vectors.  The same launch zeroes the fp32 combine accumulator and
// the call's device status word, so the forward needs no memset nodes.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ sorted_p,
                                                          const int32_t* __restrict__ totals, int64_t max_rows, int vec_per_row,
                                                          int k, int P, uint4* __restrict__ xs, float4* __restrict__ acc,
                                                          int64_t n_acc4, int32_t* __restrict__ status,
                                                          int32_t* __restrict__ ctr, int n_ctr,
                                                          float4* __restrict__ g_acc, int g_cols4) {
  pdl_trigger();   // the next kernel waits for this grid before reading what it writes
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = tid; i < n_acc4; i += nthr) acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (tid == 0) *status = 0;
  for (int64_t i = tid; i < n_ctr; i += nthr) ctr[i] = 0;
  if (g_acc) {
    const int64_t n_g4 = static_cast<int64_t>(totals[0]) * g_cols4;
    for (int64_t i = tid; i < n_g4; i += nthr) g_acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= max_rows || row >= totals[0]) return;
  const int p = sorted_p[row];
  uint4* dst = xs + row * vec_per_row;
  if (p >= P) {
    for (int v = lane; v < vec_per_row; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
  } else {
    const uint4* src = x + static_cast<int64_t>(p / k) * vec_per_row;
    for (int v = lane; v < vec_per_row; v += 32) dst[v] = __ldg(src + v);
  }
}

__global__ void __launch_bounds__(256) finalize_kernel(const float4* __restrict__ acc, uint2* __restrict__ out, int64_t n4) {
  pdl_wait();   // out_acc is complete once the down GEMM has finished
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 v = acc[i];
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
    __nv_bfloat162 b = __floats2bfloat162_rn(v.z, v.w);
    out[i] = make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
  }
}

}  // namespace

cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* sorted_p, const int32_t* totals, int64_t max_rows,
                               int H, int k, int P, uint16_t* x_sorted, float* out_acc, int64_t n_acc,
                               int32_t* status, int32_t* ctr, int n_ctr, float* g_acc, int g_cols, cudaStream_t s) {
  const int rows_per_cta = 8;
  int64_t grid = (max_rows + rows_per_cta - 1) / rows_per_cta;
  // enough threads for the zeroing too (about 16 float4 per thread, at most 8 CTAs per SM)
  const int64_t zero4 = n_acc / 4 + (g_acc ? max_rows * (g_cols / 4) : 0);
  int64_t zgrid = (zero4 / 16 + 255) / 256;
  if (zgrid > 152 * 8) zgrid = 152 * 8;
  if (grid < zgrid) grid = zgrid;
  if (grid < 1) grid = 1;
  gather_rows_kernel<<<static_cast<unsigned>(grid), rows_per_cta * 32, 0, s>>>(
      reinterpret_cast<const uint4*>(x), sorted_p, totals, max_rows, H / 8, k, P, reinterpret_cast<uint4*>(x_sorted),
      reinterpret_cast<float4*>(out_acc), n_acc / 4, status, ctr, n_ctr, reinterpret_cast<float4*>(g_acc), g_cols / 4);
  return cudaGetLastError();
}

namespace {
// h[row][i] = bf16(silu(g[row][i]) * g[row][I + i]) for rows < totals[0]; 4 features per thread.
__global__ void __launch_bounds__(256) silu_rows_kernel(const float4* __restrict__ g, const int32_t* __restrict__ totals,
                                                        int I4, uint2* __restrict__ h) {
  pdl_wait();      // the gate_up partial sums are complete
  pdl_trigger();
  const int64_t n = static_cast<int64_t>(totals[0]) * I4;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = i / I4, c = i % I4;
    const float4 a = g[row * 2 * I4 + c], b = g[row * 2 * I4 + I4 + c];
    auto silu = [](float z) { return z / (1.0f + __expf(-z)); };
    __nv_bfloat162 lo = __floats2bfloat162_rn(silu(a.x) * b.x, silu(a.y) * b.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(silu(a.z) * b.z, silu(a.w) * b.w);
    h[i] = make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
  }
}
}  // namespace

cudaError_t launch_silu_rows(const float* g_acc, const int32_t* totals, int64_t max_rows, int I, uint16_t* h,
                             bool pdl, cudaStream_t s) {
  int64_t grid = (max_rows * (I / 4) + 255) / 256;
  if (grid > 152 * 8) grid = 152 * 8;
  if (grid < 1) grid = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, silu_rows_kernel, reinterpret_cast<const float4*>(g_acc), totals, I / 4,
                            reinterpret_cast<uint2*>(h));
}

cudaError_t launch_finalize(const float* acc, uint16_t* out, int64_t n, bool pdl, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int64_t n4 = n / 4;
  int64_t grid = (n4 + 255) / 256;
  if (grid > 152 * 8) grid = 152 * 8;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, finalize_kernel, reinterpret_cast<const float4*>(acc),
                            reinterpret_cast<uint2*>(out), n4);
}

}  // namespace moe
