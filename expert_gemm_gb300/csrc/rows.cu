// rows.cu -- row gather into sorted order, the SiLU pass after a K-split gate_up,
// and the weighted top-k combine.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

// One warp per sorted row: lane 0 records pair_row[p] = row (for the combine and the
// token-order copy), and with copy_rows the real rows get x[sorted_p[row] / k] (16-byte
// vectors).  Padding rows are left as they are: every product treats token rows
// independently (a padding row only feeds its own accumulator row or column, whose
// output nothing reads) and the shrinks select S = 0 outside each adapter run.  The
// same launch zeroes the call's device status word and the GEMMs' tile counters, so the
// forward needs no memset nodes.
// The group table of the block-diagonal shrink, built by one CTA: each 128-row unit's
// rank chunks (sum over the runs that reach it of ceil(rank / 16)), then a unit-order
// scan of ceil(chunks / gch) groups per unit and one table entry per group.
__device__ void build_shrink_plan(const ShrinkPlanArgs& pl, const int32_t* __restrict__ totals) {
  __shared__ int32_t s_warp[32];
  __shared__ int32_t s_carry;
  const int tid = threadIdx.x, nt = blockDim.x, lane = tid & 31, warp = tid >> 5, nw = nt >> 5;
  const int upb = pl.block_m / 128;   // units per block
  const int nb = totals[1] * upb, nr = totals[2];
  for (int b = tid; b < nb; b += nt) pl.block_chunks[b] = 0;
  __syncthreads();
  // eight runs' loads in flight per thread before their atomics
  constexpr int kBatch = 8;
  for (int j0 = tid; j0 < nr; j0 += kBatch * nt) {
    int rb[kBatch], ra[kBatch], rs[kBatch], re[kBatch];   // block, adapter, first row, end row
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      const int j = j0 + q * nt;
      const bool in = j < nr;
      rb[q] = in ? pl.runs[4 * j] : -1;
      ra[q] = in ? pl.runs[4 * j + 1] : 0;
      rs[q] = in ? pl.runs[4 * j + 2] : 0;
      re[q] = in ? pl.runs[4 * j + 3] : 0;
    }
#pragma unroll
    for (int q = 0; q < kBatch; ++q) {
      if (rb[q] < 0) continue;
      const int n = (pl.ranks[ra[q]] + kRankChunk - 1) / kRankChunk;
      for (int h = 0; h < upb; ++h) {   // the units the run's rows reach
        const int u0 = rb[q] * pl.block_m + 128 * h;
        if (rs[q] < u0 + 128 && re[q] > u0) atomicAdd(pl.block_chunks + rb[q] * upb + h, n);
      }
    }
  }
  if (tid == 0) s_carry = 0;
  __syncthreads();   // the block's atomics are complete and visible to the block
  for (int base = 0; base < nb; base += nt) {
    const int b = base + tid;
    const int g = b < nb ? (__ldcg(pl.block_chunks + b) + pl.gch - 1) / pl.gch : 0;
    int x = g;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = lane < nw ? s_warp[lane] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, off);
        if (lane >= off) w += y;
      }
      if (lane < nw) s_warp[lane] = w;
    }
    __syncthreads();
    const int first = s_carry + (warp > 0 ? s_warp[warp - 1] : 0) + x - g;
    for (int i = 0; i < g; ++i) {
      pl.plan_block[first + i] = b;
      pl.plan_c0[first + i] = i * pl.gch;
    }
    __syncthreads();   // every thread has read s_carry and s_warp
    if (tid == 0) s_carry += s_warp[nw - 1];
    __syncthreads();
  }
  if (tid == 0) *pl.plan_count = s_carry;
}

// COPY: also copy each pair's token row (row order); without, only the row map, the
// counters and the group table (its own instantiation: the copy loop's registers would
// halve the CTAs an SM holds for the map-only pass).
template <bool COPY>
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ sorted_p,
                                                          const int32_t* __restrict__ totals, int64_t max_rows, int vec_per_row,
                                                          int k, int P, uint4* __restrict__ xs,
                                                          int32_t* __restrict__ pair_row, int32_t* __restrict__ status,
                                                          int32_t* __restrict__ ctr, int n_ctr,
                                                          const __grid_constant__ ShrinkPlanArgs plan, int plan_ctas) {
  // Launched as a programmatic dependent of whatever precedes the forward (the align):
  // its launch overlaps that kernel's tail, its reads wait for it.
  pdl_wait();
  pdl_trigger();   // the next kernel waits for this grid before reading what it writes
  const int64_t tid = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t nthr = static_cast<int64_t>(gridDim.x) * blockDim.x;
  if (tid == 0) *status = 0;
  for (int64_t i = tid; i < n_ctr; i += nthr) ctr[i] = 0;
  if (static_cast<int>(blockIdx.x) < plan_ctas) {   // the first CTA: the shrink's group table
    build_shrink_plan(plan, totals);
    return;
  }
  const int lane = threadIdx.x & 31;
  const int64_t row = static_cast<int64_t>(blockIdx.x - plan_ctas) * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= max_rows || row >= totals[0]) return;
  const int p = sorted_p[row];
  uint4* dst = xs + row * vec_per_row;
  if (p < P) {
    if (lane == 0) pair_row[p] = static_cast<int32_t>(row);
    if constexpr (!COPY) return;
    const uint4* src = x + static_cast<int64_t>(p / k) * vec_per_row;
    // every load of a lane in flight before its first store: one memory round trip for
    // rows of up to 512 vectors (H <= 4096), then one per further 512 (decode step
    // 281.4 -> 279.0 us against four loads in flight; 79 registers halve the CTAs an SM
    // holds, which costs the 32768-row gather of the T = 4096 sweep layer 0.3 us)
    constexpr int kVec = 16;
    for (int v0 = 0; v0 < vec_per_row; v0 += 32 * kVec) {
      uint4 buf[kVec];
#pragma unroll
      for (int u = 0; u < kVec; ++u) {
        const int v = v0 + lane + 32 * u;
        if (v < vec_per_row) buf[u] = __ldg(src + v);
      }
#pragma unroll
      for (int u = 0; u < kVec; ++u) {
        const int v = v0 + lane + 32 * u;
        if (v < vec_per_row) dst[v] = buf[u];
      }
    }
  }
}

// Token order: one warp per token reads x[t] once and writes it to the sorted row of
// each of its pairs (the sorted order puts a token's k copies far apart, so the row
// order would read x from DRAM k times).  A pair's row is trusted only if the sorted
// order holds the pair there.
__global__ void __launch_bounds__(256) copy_tokens_kernel(const uint4* __restrict__ x, const int32_t* __restrict__ pair_row,
                                                          const int32_t* __restrict__ sorted_p,
                                                          const int32_t* __restrict__ totals, int64_t T, int k,
                                                          int vec_per_row, uint4* __restrict__ xs) {
  __shared__ int32_t s_rows[8][MOE_LORA_MAX_TOPK];   // 256 threads: 8 warps
  pdl_wait();      // pair_row of this call is complete
  pdl_trigger();
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int64_t t = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + wib;
  if (t >= T) return;
  int r = -1;
  if (lane < k) {
    const int64_t p = t * k + lane;
    r = pair_row[p];
    if (r < 0 || r >= totals[0] || sorted_p[r] != p) r = -1;
  }
  // the token's rows, gathered while all lanes are converged; the copy loops below
  // run a lane-dependent number of steps and read them from shared memory
  const unsigned valid = __ballot_sync(0xffffffffu, r >= 0);
  if (r >= 0) s_rows[wib][__popc(valid & ((1u << lane) - 1u))] = r;
  __syncwarp();
  const int n = __popc(valid);
  const uint4* src = x + t * vec_per_row;
  int v = lane;
  for (; v + 96 < vec_per_row; v += 128) {   // four loads in flight per lane
    const uint4 a = __ldg(src + v), b = __ldg(src + v + 32), c = __ldg(src + v + 64), d = __ldg(src + v + 96);
    for (int j = 0; j < n; ++j) {
      uint4* dst = xs + static_cast<int64_t>(s_rows[wib][j]) * vec_per_row;
      dst[v] = a;
      dst[v + 32] = b;
      dst[v + 64] = c;
      dst[v + 96] = d;
    }
  }
  for (; v < vec_per_row; v += 32) {
    const uint4 a = __ldg(src + v);
    for (int j = 0; j < n; ++j) xs[static_cast<int64_t>(s_rows[wib][j]) * vec_per_row + v] = a;
  }
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& v, float* f) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

// Columns c, c + 32, ... (U groups of 8) of token t: the sum over its n valid pairs in
// ascending order of w_j * d_j, d_j the pair's row (bf16) or the sum of its K-split
// fp32 partials in split order.
template <bool SPLIT, int U>
__device__ __forceinline__ void combine_cols(const void* __restrict__ y, int ksplit, int64_t part_rows, int H8,
                                             const int32_t* rows, const float* ws, int n, int c, int64_t t,
                                             uint4* __restrict__ out) {
  float acc[U][8];
#pragma unroll
  for (int u = 0; u < U; ++u)
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[u][q] = 0.f;
  for (int j0 = 0; j0 < n; j0 += 4) {
    float d[U][4][8];
#pragma unroll
    for (int u = 0; u < U; ++u) {
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
#pragma unroll
        for (int q = 0; q < 8; ++q) d[u][q4][q] = 0.f;
        if (j0 + q4 < n) {
          const int64_t rr = rows[j0 + q4];
          const int cc = c + 32 * u;
          if constexpr (!SPLIT) {
            unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(y) + rr * H8 + cc), d[u][q4]);
          } else {
            for (int sp = 0; sp < ksplit; ++sp) {
              const float4* src = reinterpret_cast<const float4*>(y) + ((sp * part_rows + rr) * H8 + cc) * 2;
              const float4 a = __ldcg(src), b = __ldcg(src + 1);
              d[u][q4][0] += a.x; d[u][q4][1] += a.y; d[u][q4][2] += a.z; d[u][q4][3] += a.w;
              d[u][q4][4] += b.x; d[u][q4][5] += b.y; d[u][q4][6] += b.z; d[u][q4][7] += b.w;
            }
          }
        }
      }
    }
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      if (j0 + q4 < n) {
        const float w = ws[j0 + q4];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[u][q] += w * d[u][q4][q];
      }
    }
  }
#pragma unroll
  for (int u = 0; u < U; ++u)
    out[t * H8 + c + 32 * u] = make_uint4(pack2(acc[u][0], acc[u][1]), pack2(acc[u][2], acc[u][3]),
                                          pack2(acc[u][4], acc[u][5]), pack2(acc[u][6], acc[u][7]));
}

// One warp per (token, column slab): lanes j < k look up the token's pairs -- a pair's
// row is trusted only if the sorted order really holds the pair there (the row record
// of a dropped pair is stale), so dropped pairs add nothing -- then every lane
// combines 8 columns at a time over the slab.  Large batches give a warp a whole token
// (ns = 1); small ones split the columns so that enough warps stream.  Pairs in
// ascending j, splits in ascending order: the result does not depend on which CTA of
// the GEMM finished first.
constexpr int kCombineThreads = 256;
template <bool SPLIT>
__device__ __forceinline__ void combine_body(const void* __restrict__ y, int ksplit, int64_t part_rows,
                                             const int32_t* __restrict__ pair_row,
                                             const int32_t* __restrict__ sorted_p,
                                             const int32_t* __restrict__ totals, const float* __restrict__ topk_w,
                                             int64_t T, int k, int H8, int ns, uint4* __restrict__ out) {
  __shared__ int32_t s_row[kCombineThreads / 32][MOE_LORA_MAX_TOPK];
  __shared__ float s_w[kCombineThreads / 32][MOE_LORA_MAX_TOPK];
  // The pair lookups read what the gather, align and route wrote: those finished before
  // the down GEMM could start (each kernel of the chain lets its dependent launch only
  // after its own wait), so only the expert rows below wait for the down GEMM.
  const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * (kCombineThreads / 32) + wib;
  if (gw >= T * ns) return;
  const int64_t t = gw / ns;
  const int slab = static_cast<int>(gw - t * ns);
  int r = -1;
  float w = 0.f;
  if (lane < k) {
    const int64_t p = t * k + lane;
    r = pair_row[p];
    if (r < 0 || r >= totals[0] || sorted_p[r] != p) r = -1;
    else w = topk_w[p];
  }
  // compact the valid pairs, keeping ascending j
  const unsigned valid = __ballot_sync(0xffffffffu, r >= 0);
  if (r >= 0) {
    const int slot = __popc(valid & ((1u << lane) - 1u));
    s_row[wib][slot] = r;
    s_w[wib][slot] = w;
  }
  __syncwarp();
  pdl_wait();   // the down GEMM's rows are complete
  const int n = __popc(valid);
  const int per = (H8 + ns - 1) / ns;
  const int c_end = min(H8, (slab + 1) * per);
  // (one column group per step: two per step, more loads in flight, measured slower)
  for (int c = slab * per + lane; c < c_end; c += 32)
    combine_cols<SPLIT, 1>(y, ksplit, part_rows, H8, s_row[wib], s_w[wib], n, c, t, out);
}

// Over bf16 rows: at most 40 registers a thread, so 6 CTAs (48 warps) share an SM.
// Each warp has only its token's few row loads in flight, so the loads in flight per
// SM, i.e. the resident warps, set the combine's bandwidth (prefill 179 -> 122 us
// against 4 CTAs at 57 registers; 8 CTAs spill).
__global__ void __launch_bounds__(kCombineThreads, 6)
    combine_rows_kernel(const void* __restrict__ y, int ksplit, int64_t part_rows, const int32_t* __restrict__ pair_row,
                        const int32_t* __restrict__ sorted_p, const int32_t* __restrict__ totals,
                        const float* __restrict__ topk_w, int64_t T, int k, int H8, int ns, uint4* __restrict__ out) {
  combine_body<false>(y, ksplit, part_rows, pair_row, sorted_p, totals, topk_w, T, k, H8, ns, out);
}
// Over fp32 K-split partials (their sums need more registers; capped, it would spill).
__global__ void __launch_bounds__(kCombineThreads)
    combine_parts_kernel(const void* __restrict__ y, int ksplit, int64_t part_rows, const int32_t* __restrict__ pair_row,
                         const int32_t* __restrict__ sorted_p, const int32_t* __restrict__ totals,
                         const float* __restrict__ topk_w, int64_t T, int k, int H8, int ns, uint4* __restrict__ out) {
  combine_body<true>(y, ksplit, part_rows, pair_row, sorted_p, totals, topk_w, T, k, H8, ns, out);
}

}  // namespace

cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* sorted_p, const int32_t* totals, int64_t max_rows,
                               int H, int k, int P, uint16_t* x_sorted, int32_t* pair_row, int32_t* status,
                               int32_t* ctr, int n_ctr, const ShrinkPlanArgs* plan, cudaStream_t s) {
  const int rows_per_cta = 8;
  const int plan_ctas = plan ? 1 : 0;
  int64_t grid = (max_rows + rows_per_cta - 1) / rows_per_cta + plan_ctas;
  if (grid < 1) grid = 1;
  ShrinkPlanArgs pl{};
  if (plan) pl = *plan;
  // When x is larger than half the 129 MB L2, its k re-reads in sorted-row order come
  // from DRAM: copy in token order then (x read once).  Otherwise one row-order pass.
  const bool token_order = gather_token_order(P / k, H);
  cudaError_t err;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(rows_per_cta * 32, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    auto kern = token_order ? gather_rows_kernel<false> : gather_rows_kernel<true>;
    err = cudaLaunchKernelEx(&cfg, kern, reinterpret_cast<const uint4*>(x), sorted_p, totals, max_rows, H / 8, k, P,
                             reinterpret_cast<uint4*>(x_sorted), pair_row, status, ctr, n_ctr, pl, plan_ctas);
  }
  if (err != cudaSuccess || !token_order) return err;
  const int64_t T = P / k;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((T + 7) / 8), 1, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, copy_tokens_kernel, reinterpret_cast<const uint4*>(x),
                            static_cast<const int32_t*>(pair_row), sorted_p, totals, T, k, H / 8,
                            reinterpret_cast<uint4*>(x_sorted));
}

namespace {
// h[row][i] = bf16(silu(g[row][i]) * g[row][I + i]) for rows < totals[0], g the sum of the
// K splits' partials in split order; 4 features per thread.
__global__ void __launch_bounds__(256) silu_rows_kernel(const float4* __restrict__ g, int ksplit, int64_t part_rows,
                                                        const int32_t* __restrict__ totals, int I4,
                                                        uint2* __restrict__ h) {
  pdl_wait();      // the gate_up partial sums are complete
  pdl_trigger();
  const int64_t n = static_cast<int64_t>(totals[0]) * I4;
  const int64_t split_stride = part_rows * 2 * I4;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t row = i / I4, c = i % I4;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
    for (int sp = 0; sp < ksplit; ++sp) {
      const float4* src = g + sp * split_stride + row * 2 * I4;
      const float4 ga = __ldcg(src + c), gb = __ldcg(src + I4 + c);
      a.x += ga.x; a.y += ga.y; a.z += ga.z; a.w += ga.w;
      b.x += gb.x; b.y += gb.y; b.z += gb.z; b.w += gb.w;
    }
    auto silu = [](float z) { return __fdividef(z, 1.0f + __expf(-z)); };
    h[i] = make_uint2(pack2(silu(a.x) * b.x, silu(a.y) * b.y), pack2(silu(a.z) * b.z, silu(a.w) * b.w));
  }
}
}  // namespace

cudaError_t launch_silu_rows(const float* g_part, int ksplit, int64_t part_rows, const int32_t* totals,
                             int64_t max_rows, int I, uint16_t* h, bool pdl, cudaStream_t s) {
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
  return cudaLaunchKernelEx(&cfg, silu_rows_kernel, reinterpret_cast<const float4*>(g_part), ksplit, part_rows, totals,
                            I / 4, reinterpret_cast<uint2*>(h));
}

cudaError_t launch_combine(const void* y, int ksplit, int64_t part_rows, const int32_t* pair_row,
                           const int32_t* sorted_p, const int32_t* totals, const float* topk_w, int64_t T, int k,
                           int H, uint16_t* out, bool pdl, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  const int H8 = H / 8;
  // column slabs per token: at least ~16 warps per SM (152 SMs) when T is small,
  // each slab at least one 32-lane sweep of columns
  const int64_t want_warps = 152 * 16;
  int64_t ns = T >= want_warps ? 1 : (want_warps + T - 1) / T;
  const int64_t max_ns = (H8 + 31) / 32;
  if (ns > max_ns) ns = max_ns;
  const int64_t warps = T * ns;
  const int64_t blocks = (warps + kCombineThreads / 32 - 1) / (kCombineThreads / 32);
  if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(kCombineThreads, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  uint4* o = reinterpret_cast<uint4*>(out);
  const int nsi = static_cast<int>(ns);
  if (ksplit > 1)
    return cudaLaunchKernelEx(&cfg, combine_parts_kernel, y, ksplit, part_rows, pair_row, sorted_p, totals, topk_w, T,
                              k, H8, nsi, o);
  return cudaLaunchKernelEx(&cfg, combine_rows_kernel, y, ksplit, part_rows, pair_row, sorted_p, totals, topk_w, T,
                            k, H8, nsi, o);
}

}  // namespace moe
