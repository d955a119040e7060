// align.cu -- align-and-sort of the (expert, adapter) compound sparsity.
//
// The pages give the problem, not a layout: default fused-MoE configurations ignore
// the extra grid dimension of the LoRA index and the compound sparsity of many
// adapters (AWS ML Blog "Efficiently serve dozens of fine-tuned models with vLLM on
// Amazon SageMaker AI and Amazon Bedrock", section "Tuning kernel configurations for
// Amazon SageMaker AI and Amazon Bedrock"; agentlenshq.com "vLLM MoE 모델을 위한
// Multi-LoRA 서빙", section "MoE 모델을 위한 Multi-LoRA 서빙").  This library's layout
// (see moe_lora.h): valid pairs sorted by (expert, adapter, pair), each expert padded
// to a multiple of block_m rows, plus per-block adapter runs.
//
// A stable counting sort in three launches:
//   1. chunk:   each CTA sorts its chunk of pair keys (bucket << log2(CH) | local index)
//               with a bitonic network (registers and warp shuffles for short
//               distances, shared memory for long ones) and writes per-bucket counts;
//   2. scan:    one CTA turns counts into per-(chunk, bucket) offsets, expert starts
//               (padded), bucket starts, runs, block experts, padding sentinels;
//   3. scatter: each CTA places its pairs; rank inside the chunk = index - first index
//               of the bucket in the sorted chunk, so equal keys keep pair order.
// Integer work only; the result is bit-identical to the sequential definition.
#include "common.cuh"
#include "route.cuh"

namespace moe {
namespace {

constexpr uint32_t kInvalidKey = 0xFFFFFFFFu;

__device__ __forceinline__ int lower_bound_u32(const uint32_t* a, int lo, int hi, uint32_t key) {
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] < key) lo = mid + 1;
    else hi = mid;
  }
  return lo;
}

// Compare-exchange of a pair held by one thread: ascending unless desc.
__device__ __forceinline__ void cmp_swap(uint32_t& x, uint32_t& y, bool desc) {
  if ((x > y) != desc) {
    const uint32_t t = x;
    x = y;
    y = t;
  }
}

// Ascending bitonic sort of n (a power of two, n <= 4 * blockDim.x) keys in shared
// memory, all threads of the CTA; ends with a barrier.  Thread t holds keys
// [4t, 4t + 4) in registers.  Compare-exchanges at distance 1 and 2 stay inside the
// thread, distances 4..64 go between the lanes of a warp by shuffles, and only
// distances of 128 and more pass through shared memory (15 barrier stages for 4096
// keys instead of 78).  Every thread runs every stage, so the shuffles see full warps.
__device__ void bitonic_sort(uint32_t* keys, int n) {
  const int t = threadIdx.x;
  const int i0 = 4 * t;   // first key of this thread
  uint32_t v[4];
  __syncthreads();        // the keys every thread wrote
#pragma unroll
  for (int q = 0; q < 4; ++q) v[q] = i0 + q < n ? keys[i0 + q] : 0xFFFFFFFFu;
  for (int size = 2; size <= n; size <<= 1) {
    int s = size >> 1;
    if (s >= 128) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (i0 + q < n) keys[i0 + q] = v[q];
      for (; s >= 128; s >>= 1) {
        __syncthreads();
        for (int i = t; i < n / 2; i += blockDim.x) {
          const int lo = 2 * i - (i & (s - 1));
          const int hi = lo + s;
          uint32_t x = keys[lo], y = keys[hi];
          cmp_swap(x, y, (lo & size) != 0);
          keys[lo] = x;
          keys[hi] = y;
        }
      }
      __syncthreads();
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (i0 + q < n) v[q] = keys[i0 + q];
    }
    // distances 4..64: the partner of key i0 + q is key q of lane ^ (s / 4)
    for (; s >= 4; s >>= 1) {
      const bool desc = (i0 & size) != 0, upper = (i0 & s) != 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t p = __shfl_xor_sync(0xffffffffu, v[q], s >> 2);
        // the lower key of an ascending pair keeps the smaller one, and so on
        v[q] = (upper != desc) ? (v[q] > p ? v[q] : p) : (v[q] < p ? v[q] : p);
      }
    }
    // distances 2 and 1 (size 2 has only distance 1; there bit 1 of the key index
    // decides the direction)
    if (s == 2) {
      const bool desc = (i0 & size) != 0;
      cmp_swap(v[0], v[2], desc);
      cmp_swap(v[1], v[3], desc);
      s = 1;
    }
    cmp_swap(v[0], v[1], (i0 & size) != 0);
    cmp_swap(v[2], v[3], ((i0 + 2) & size) != 0);
  }
#pragma unroll
  for (int q = 0; q < 4; ++q)
    if (i0 + q < n) keys[i0 + q] = v[q];
  __syncthreads();
}

// Ascending sort of n <= blockDim.x keys in shared memory by rank counting: key i goes
// to the number of keys below it (equal keys -- only the invalid marker repeats -- in
// index order).  One pass over the keys per thread, two barriers; for the few keys of
// a decode batch this replaces the bitonic network's chain of dependent exchange
// stages.  Ends with a barrier.
constexpr int kRankSortMax = 512;
__device__ void rank_sort(uint32_t* keys, int n) {
  const int t = threadIdx.x;
  __syncthreads();   // the keys every thread wrote
  uint32_t mine = 0;
  int rank = 0;
  if (t < n) {
    mine = keys[t];
    for (int j = 0; j < n; ++j) {
      const uint32_t o = keys[j];   // the same word for the whole warp: a broadcast read
      rank += (o < mine) || (o == mine && j < t);
    }
  }
  __syncthreads();
  if (t < n) keys[rank] = mine;
  __syncthreads();
}

// Phase 1 for one chunk: keys of its pairs sorted in keys[] (shared), per-bucket
// counts of the chunk and its invalid-pair count written to global scratch.  ids: the
// expert ids [P] (global, or shared when the same CTA has just routed them).
__device__ void chunk_phase(const AlignLaunch& a, const int32_t* ids, uint32_t* keys, int chunk, bool store_keys) {
  __shared__ int32_t s_invalid;
  const int CH = 1 << a.ch_log2;
  const int64_t p0 = static_cast<int64_t>(chunk) << a.ch_log2;
  const int LB = a.L + 1;
  const int NB = a.E * LB;
  if (threadIdx.x == 0) s_invalid = 0;
  for (int b = threadIdx.x; b < NB; b += blockDim.x) a.counts[static_cast<int64_t>(chunk) * NB + b] = 0;
  __syncthreads();
  int inval = 0;
  for (int i = threadIdx.x; i < CH; i += blockDim.x) {
    const int64_t p = p0 + i;
    uint32_t key = kInvalidKey;
    if (p < a.P) {
      const int e = ids[p];
      const int ad = a.lora_ids[p / a.k];
      if (e >= 0 && e < a.E && ad >= -1 && ad < a.L)
        key = (static_cast<uint32_t>(e * LB + ad + 1) << a.ch_log2) | static_cast<uint32_t>(i);
      else
        ++inval;
    }
    keys[i] = key;
  }
  if (inval) atomicAdd(&s_invalid, inval);
  bitonic_sort(keys, CH);
  for (int i = threadIdx.x; i < CH; i += blockDim.x) {
    const uint32_t key = keys[i];
    if (store_keys) a.chunk_keys[p0 + i] = key;
    if (key == kInvalidKey) continue;
    const uint32_t bkt = key >> a.ch_log2;
    const bool last = (i == CH - 1) || (keys[i + 1] >> a.ch_log2) != bkt;
    if (last) {
      const int first = lower_bound_u32(keys, 0, i, bkt << a.ch_log2);
      a.counts[static_cast<int64_t>(chunk) * NB + bkt] = i - first + 1;
    }
  }
  if (threadIdx.x == 0) a.chunk_invalid[chunk] = s_invalid;
}

__global__ void __launch_bounds__(1024) align_chunk_kernel(AlignLaunch a) {
  extern __shared__ uint32_t keys[];
  chunk_phase(a, a.topk_ids, keys, blockIdx.x, true);
}

// Block-wide exclusive scan over n values produced by getv(i); put(i, prefix) receives
// each exclusive prefix.  Returns the total (same value in every thread).
template <class GetV, class Put>
__device__ int block_exclusive_scan(int n, GetV getv, Put put, int32_t* s_warp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
  int carry = 0;
  for (int base = 0; base < n; base += blockDim.x) {
    const int i = base + tid;
    const int v = i < n ? getv(i) : 0;
    int x = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, off);
      if (lane >= off) x += y;
    }
    if (lane == 31) s_warp[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = lane < nwarps ? s_warp[lane] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, off);
        if (lane >= off) w += y;
      }
      if (lane < nwarps) s_warp[lane] = w;
    }
    __syncthreads();
    const int excl = carry + (warp > 0 ? s_warp[warp - 1] : 0) + x - v;
    if (i < n) put(i, excl);
    carry += s_warp[nwarps - 1];
    __syncthreads();
  }
  return carry;
}

// Phase 2 (one CTA): bucket offsets, padded expert starts, runs, block experts,
// padding sentinels, totals and block -> first-run index.
__device__ void scan_phase(const AlignLaunch& a) {
  __shared__ int32_t s_warp[32];
  __shared__ int32_t s_rows, s_runs;
  const int LB = a.L + 1;
  const int NB = a.E * LB;
  const int BM = a.BM;
  const int tid = threadIdx.x, nt = blockDim.x;
  const moe_lora_align_buf& o = a.out;

  // The loops below read kBatch values before writing any: loads and stores go to
  // global scratch through the same struct, so the compiler would otherwise wait for
  // each load in turn.
  constexpr int kBatch = 8;
  // 1. bucket totals; counts[c][b] becomes the offset of chunk c inside bucket b
  for (int b = tid; b < NB; b += nt) {
    int run = 0;
    for (int c0 = 0; c0 < a.nchunks; c0 += kBatch) {
      int v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        v[u] = c0 + u < a.nchunks ? a.counts[static_cast<int64_t>(c0 + u) * NB + b] : 0;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (c0 + u < a.nchunks) a.counts[static_cast<int64_t>(c0 + u) * NB + b] = run;
        run += v[u];
      }
    }
    a.bucket_total[b] = run;
  }
  __syncthreads();
  // 2. pairs per expert
  for (int e = tid; e < a.E; e += nt) {
    int n = 0;
    for (int j0 = 0; j0 < LB; j0 += kBatch) {
      int v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) v[u] = j0 + u < LB ? a.bucket_total[e * LB + j0 + u] : 0;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) n += v[u];
    }
    a.expert_n[e] = n;
  }
  __syncthreads();
  // 3. padded expert starts
  const int rows = block_exclusive_scan(
      a.E, [&](int e) { return (a.expert_n[e] + BM - 1) / BM * BM; },
      [&](int e, int pre) { o.expert_begin[e] = pre; }, s_warp);
  if (tid == 0) {
    o.expert_begin[a.E] = rows;
    s_rows = rows;
  }
  __syncthreads();
  // 4. bucket starts: expert start + earlier adapters of the same expert
  for (int e = tid; e < a.E; e += nt) {
    int base = o.expert_begin[e];
    for (int j0 = 0; j0 < LB; j0 += kBatch) {
      int v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) v[u] = j0 + u < LB ? a.bucket_total[e * LB + j0 + u] : 0;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (j0 + u < LB) a.bucket_base[e * LB + j0 + u] = base;
        base += v[u];
      }
    }
  }
  __syncthreads();
  // 5. runs: a bucket of adapter >= 0 splits at block boundaries
  auto nruns_of = [&](int b) -> int {
    const int tot = a.bucket_total[b];
    if (tot == 0 || (b % LB) == 0) return 0;
    const int s = a.bucket_base[b];
    return (s + tot - 1) / BM - s / BM + 1;
  };
  const int nruns = block_exclusive_scan(NB, nruns_of, [&](int b, int pre) { a.run_base[b] = pre; }, s_warp);
  if (tid == 0) s_runs = nruns;
  __syncthreads();
  // 6. write runs; 7. block experts; 8. padding sentinels
  for (int b = tid; b < NB; b += nt) {
    const int cnt = nruns_of(b);
    if (!cnt) continue;
    const int s = a.bucket_base[b], end = s + a.bucket_total[b];
    const int adapter = (b % LB) - 1;
    const int r0 = a.run_base[b];
    for (int i = 0; i < cnt; ++i) {
      const int blk = s / BM + i;
      int* r = o.runs + 4 * static_cast<int64_t>(r0 + i);
      r[0] = blk;
      r[1] = adapter;
      r[2] = max(s, blk * BM);
      r[3] = min(end, (blk + 1) * BM);
    }
  }
  for (int e = tid; e < a.E; e += nt) {
    const int s = o.expert_begin[e], end = o.expert_begin[e + 1];
    for (int blk = s / BM; blk < end / BM; ++blk) o.block_expert[blk] = e;
    for (int r = s + a.expert_n[e]; r < end; ++r) o.sorted_p[r] = static_cast<int32_t>(a.P);
  }
  if (tid == 0) {
    int dropped = 0;
    for (int c = 0; c < a.nchunks; ++c) dropped += a.chunk_invalid[c];
    o.totals[0] = s_rows;
    o.totals[1] = s_rows / BM;
    o.totals[2] = s_runs;
    o.totals[3] = dropped;
  }
  __syncthreads();
  // 9. first run of each block (runs are in block order)
  const int nblocks = s_rows / BM;
  for (int blk = tid; blk <= nblocks; blk += nt) {
    int lo = 0, hi = s_runs;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (o.runs[4 * static_cast<int64_t>(mid)] < blk) lo = mid + 1;
      else hi = mid;
    }
    o.block_runs[blk] = lo;
  }
}

__global__ void __launch_bounds__(1024) align_scan_kernel(AlignLaunch a) { scan_phase(a); }

// Phase 2 with the per-bucket arrays in shared memory (E * (L+1) <= kScanSmemBuckets):
// the same results as scan_phase, but every pass after the first reads and writes
// shared memory instead of making a round trip to L2, and each block's first run comes
// from one pass over the runs instead of a binary search per block.  The bucket bases
// and the per-chunk offsets still go to global memory for the scatter.
constexpr int kScanSmemBuckets = 16384;
__global__ void __launch_bounds__(1024) align_scan_smem_kernel(AlignLaunch a) {
  extern __shared__ int32_t s_buf[];
  __shared__ int32_t s_warp[32];
  __shared__ int32_t s_rows, s_runs;
  const int LB = a.L + 1;
  const int NB = a.E * LB;
  const int BM = a.BM;
  const int tid = threadIdx.x, nt = blockDim.x;
  const moe_lora_align_buf& o = a.out;
  int32_t* s_tot = s_buf;            // [NB] pairs per bucket
  int32_t* s_base = s_buf + NB;      // [NB] first sorted row of each bucket
  int32_t* s_rb = s_buf + 2 * NB;    // [NB] first run of each bucket
  int32_t* s_en = s_buf + 3 * NB;    // [E] pairs per expert
  // 1. bucket totals; counts[c][b] becomes the offset of chunk c inside bucket b (all of
  //    a thread's loads are issued before its stores)
  constexpr int kBatch = 8;
  for (int b = tid; b < NB; b += nt) {
    int run = 0;
    for (int c0 = 0; c0 < a.nchunks; c0 += kBatch) {
      int v[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u)
        v[u] = c0 + u < a.nchunks ? a.counts[static_cast<int64_t>(c0 + u) * NB + b] : 0;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        if (c0 + u < a.nchunks) a.counts[static_cast<int64_t>(c0 + u) * NB + b] = run;
        run += v[u];
      }
    }
    s_tot[b] = run;
  }
  __syncthreads();
  // 2. pairs per expert
  for (int e = tid; e < a.E; e += nt) {
    int n = 0;
    for (int j = 0; j < LB; ++j) n += s_tot[e * LB + j];
    s_en[e] = n;
  }
  __syncthreads();
  // 3. padded expert starts
  const int rows = block_exclusive_scan(
      a.E, [&](int e) { return (s_en[e] + BM - 1) / BM * BM; }, [&](int e, int pre) { o.expert_begin[e] = pre; },
      s_warp);
  if (tid == 0) {
    o.expert_begin[a.E] = rows;
    s_rows = rows;
  }
  __syncthreads();
  // 4. bucket starts: expert start + earlier adapters of the same expert
  for (int e = tid; e < a.E; e += nt) {
    int base = o.expert_begin[e];
    for (int j = 0; j < LB; ++j) {
      s_base[e * LB + j] = base;
      a.bucket_base[e * LB + j] = base;
      base += s_tot[e * LB + j];
    }
  }
  __syncthreads();
  // 5. runs: a bucket of adapter >= 0 splits at block boundaries
  auto nruns_of = [&](int b) -> int {
    const int tot = s_tot[b];
    if (tot == 0 || (b % LB) == 0) return 0;
    const int st = s_base[b];
    return (st + tot - 1) / BM - st / BM + 1;
  };
  const int nruns = block_exclusive_scan(NB, nruns_of, [&](int b, int pre) { s_rb[b] = pre; }, s_warp);
  if (tid == 0) s_runs = nruns;
  __syncthreads();
  // 6. write runs; 7. block experts; 8. padding sentinels
  for (int b = tid; b < NB; b += nt) {
    const int cnt = nruns_of(b);
    if (!cnt) continue;
    const int st = s_base[b], end = st + s_tot[b];
    const int adapter = (b % LB) - 1;
    const int r0 = s_rb[b];
    for (int i = 0; i < cnt; ++i) {
      const int blk = st / BM + i;
      int* r = o.runs + 4 * static_cast<int64_t>(r0 + i);
      r[0] = blk;
      r[1] = adapter;
      r[2] = max(st, blk * BM);
      r[3] = min(end, (blk + 1) * BM);
    }
  }
  for (int e = tid; e < a.E; e += nt) {
    const int st = o.expert_begin[e], end = o.expert_begin[e + 1];
    for (int blk = st / BM; blk < end / BM; ++blk) o.block_expert[blk] = e;
    for (int r = st + s_en[e]; r < end; ++r) o.sorted_p[r] = static_cast<int32_t>(a.P);
  }
  if (tid == 0) {
    int dropped = 0;
    for (int c = 0; c < a.nchunks; ++c) dropped += a.chunk_invalid[c];
    o.totals[0] = s_rows;
    o.totals[1] = s_rows / BM;
    o.totals[2] = s_runs;
    o.totals[3] = dropped;
  }
  __syncthreads();   // the runs written above are visible to the whole CTA
  // 9. first run of each block: run i owns the blocks after the previous run's block up
  //    to its own (blocks without runs point at the next run); blocks after the last
  //    run point past the end
  const int nblocks = s_rows / BM;
  for (int i = tid; i < s_runs; i += nt) {
    const int blk = o.runs[4 * static_cast<int64_t>(i)];
    const int prev = i == 0 ? -1 : o.runs[4 * static_cast<int64_t>(i - 1)];
    for (int q = prev + 1; q <= blk; ++q) o.block_runs[q] = i;
  }
  const int last = s_runs > 0 ? o.runs[4 * static_cast<int64_t>(s_runs - 1)] : -1;
  for (int q = last + 1 + tid; q <= nblocks; q += nt) o.block_runs[q] = s_runs;
}

// Phase 3 for one chunk whose sorted keys are in keys[] (shared): place each pair.
__device__ void scatter_phase(const AlignLaunch& a, const uint32_t* keys, int chunk) {
  const int CH = 1 << a.ch_log2;
  const int64_t p0 = static_cast<int64_t>(chunk) << a.ch_log2;
  const int NB = a.E * (a.L + 1);
  for (int i = threadIdx.x; i < CH; i += blockDim.x) {
    const uint32_t key = keys[i];
    if (key == kInvalidKey) continue;
    const uint32_t bkt = key >> a.ch_log2;
    const int local = static_cast<int>(key & static_cast<uint32_t>(CH - 1));
    const int first = lower_bound_u32(keys, 0, i, bkt << a.ch_log2);
    const int pos = a.bucket_base[bkt] + a.counts[static_cast<int64_t>(chunk) * NB + bkt] + (i - first);
    a.out.sorted_p[pos] = static_cast<int32_t>(p0 + local);
  }
}

__global__ void __launch_bounds__(1024) align_scatter_kernel(AlignLaunch a) {
  extern __shared__ uint32_t keys[];
  const int CH = 1 << a.ch_log2;
  const int64_t p0 = static_cast<int64_t>(blockIdx.x) << a.ch_log2;
  for (int i = threadIdx.x; i < CH; i += blockDim.x) keys[i] = a.chunk_keys[p0 + i];
  __syncthreads();
  scatter_phase(a, keys, blockIdx.x);
}

// Batches that fit one chunk (P <= 4096) in one CTA.  After the sort the whole layout
// comes from the sorted keys in shared memory, with work proportional to the pairs,
// experts and blocks rather than to the E * (L+1) buckets, and no scratch round trips
// through global memory (the decode front end is latency, not bandwidth).
//
// small_keys: the keys of the P pairs sorted in keys[CH]; returns the invalid-pair count.
// lora: the tokens' adapter ids (a.lora_ids, or a shared copy of them).
__device__ int small_keys(const AlignLaunch& a, const int32_t* ids, const int32_t* lora, uint32_t* keys) {
  __shared__ int32_t s_invalid;
  const int CH = 1 << a.ch_log2;
  const int LB = a.L + 1;
  if (threadIdx.x == 0) s_invalid = 0;
  __syncthreads();
  int inval = 0;
  for (int i = threadIdx.x; i < CH; i += blockDim.x) {
    uint32_t key = kInvalidKey;
    if (i < a.P) {
      const int e = ids[i];
      const int ad = lora[i / a.k];
      if (e >= 0 && e < a.E && ad >= -1 && ad < a.L)
        key = (static_cast<uint32_t>(e * LB + ad + 1) << a.ch_log2) | static_cast<uint32_t>(i);
      else
        ++inval;
    }
    keys[i] = key;
  }
  if (inval) atomicAdd(&s_invalid, inval);
  if (CH <= static_cast<int>(blockDim.x) && CH <= kRankSortMax) rank_sort(keys, CH);
  else bitonic_sort(keys, CH);
  return s_invalid;
}

// small_layout: the align outputs from the nv valid sorted keys (keys[0, nv), invalid
// keys sort last).  s_runblk: shared scratch of nv ints (block of each run).
__device__ void small_layout(const AlignLaunch& a, const uint32_t* keys, int n_invalid, int32_t* s_runblk) {
  __shared__ int32_t s_cnt[MOE_LORA_MAX_EXPERTS];      // pairs per expert
  __shared__ int32_t s_first[MOE_LORA_MAX_EXPERTS];    // sorted position of its first pair
  __shared__ int32_t s_begin[MOE_LORA_MAX_EXPERTS + 1];  // padded first row
  __shared__ int32_t s_warp[32];
  const int tid = threadIdx.x, nt = blockDim.x;
  const int LB = a.L + 1, BM = a.BM, lg = a.ch_log2;
  const int nv = static_cast<int>(a.P) - n_invalid;
  const moe_lora_align_buf& o = a.out;
  for (int e = tid; e < a.E; e += nt) s_cnt[e] = 0;
  __syncthreads();
  for (int i = tid; i < nv; i += nt) {
    const int e = static_cast<int>(keys[i] >> lg) / LB;
    if (i == 0 || static_cast<int>(keys[i - 1] >> lg) / LB != e) s_first[e] = i;
    atomicAdd(&s_cnt[e], 1);
  }
  __syncthreads();
  // each expert padded to a multiple of BM rows; experts without pairs get none
  const int rows = block_exclusive_scan(
      a.E, [&](int e) { return (s_cnt[e] + BM - 1) / BM * BM; },
      [&](int e, int pre) {
        s_begin[e] = pre;
        o.expert_begin[e] = pre;
      },
      s_warp);
  if (tid == 0) {
    s_begin[a.E] = rows;
    o.expert_begin[a.E] = rows;
  }
  __syncthreads();
  // sorted pair i: bucket, adapter, row; a run (one adapter >= 0 inside one block)
  // starts where the bucket changes or a block begins, and ends before the next start
  auto bucket = [&](int i) { return static_cast<int>(keys[i] >> lg); };
  auto row_of = [&](int i) {
    const int e = bucket(i) / LB;
    return s_begin[e] + (i - s_first[e]);
  };
  auto starts = [&](int i) -> int {
    if (bucket(i) % LB == 0) return 0;   // adapter -1: no run
    return i == 0 || bucket(i - 1) != bucket(i) || row_of(i) % BM == 0;
  };
  const int nruns = block_exclusive_scan(
      nv, starts,
      [&](int i, int pre) {
        const int r = row_of(i), b = bucket(i), ad = b % LB - 1;
        o.sorted_p[r] = static_cast<int32_t>(keys[i] & ((1u << lg) - 1u));
        if (ad < 0) return;
        const bool st = starts(i);
        const int run = pre + (st ? 1 : 0) - 1;
        int32_t* q = o.runs + 4 * static_cast<int64_t>(run);
        if (st) {
          q[0] = r / BM;
          q[1] = ad;
          q[2] = r;
          s_runblk[run] = r / BM;
        }
        if (i == nv - 1 || bucket(i + 1) != b || row_of(i + 1) % BM == 0) q[3] = r + 1;
      },
      s_warp);
  // padding sentinels and block experts
  for (int e = tid; e < a.E; e += nt) {
    for (int r = s_begin[e] + s_cnt[e]; r < s_begin[e + 1]; ++r) o.sorted_p[r] = static_cast<int32_t>(a.P);
    for (int blk = s_begin[e] / BM; blk < s_begin[e + 1] / BM; ++blk) o.block_expert[blk] = e;
  }
  if (tid == 0) {
    o.totals[0] = rows;
    o.totals[1] = rows / BM;
    o.totals[2] = nruns;
    o.totals[3] = n_invalid;
  }
  __syncthreads();
  // first run of each block (runs are in block order)
  const int nblocks = rows / BM;
  for (int blk = tid; blk <= nblocks; blk += nt) {
    int lo = 0, hi = nruns;
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s_runblk[mid] < blk) lo = mid + 1;
      else hi = mid;
    }
    o.block_runs[blk] = lo;
  }
}

__global__ void __launch_bounds__(1024) align_small_kernel(AlignLaunch a) {
  extern __shared__ uint32_t keys[];
  int32_t* s_runblk = reinterpret_cast<int32_t*>(keys + (1 << a.ch_log2));
  const int inval = small_keys(a, a.topk_ids, a.lora_ids, keys);
  small_layout(a, keys, inval, s_runblk);
}

constexpr int kRouteAlignLoraTokens = 32;   // adapter ids staged in shared memory up to this T

// Route and align in one CTA (one chunk): each warp routes tokens into shared memory,
// the expert ids are copied out to topk_ids, and the align phases read them from
// shared memory.  One launch for the whole routing front of a decode step.
__global__ void __launch_bounds__(1024) route_align_small_kernel(AlignLaunch a, const float* __restrict__ logits,
                                                                 float* __restrict__ topk_w,
                                                                 int32_t* __restrict__ topk_ids) {
  extern __shared__ uint32_t keys[];
  __shared__ int32_t s_lora[kRouteAlignLoraTokens];
  int32_t* s_ids = reinterpret_cast<int32_t*>(keys + (1 << a.ch_log2));
  const int T = static_cast<int>(a.P / a.k);
  const int lane = threadIdx.x & 31;
  // the adapter ids are fetched while the warps route, not after: the two input reads
  // (from DRAM, or host memory over the link) overlap instead of following each other
  const bool stage_lora = T <= kRouteAlignLoraTokens;
  if (stage_lora && static_cast<int>(threadIdx.x) < T) s_lora[threadIdx.x] = a.lora_ids[threadIdx.x];
  for (int t = threadIdx.x >> 5; t < T; t += blockDim.x >> 5)
    route_token(logits + static_cast<int64_t>(t) * a.E, a.E, a.k, lane, s_ids + t * a.k, topk_w + t * a.k);
  __syncthreads();
  for (int p = threadIdx.x; p < a.P; p += blockDim.x) topk_ids[p] = s_ids[p];
  // ends with a barrier: s_ids is free again
  const int inval = small_keys(a, s_ids, stage_lora ? s_lora : a.lora_ids, keys);
  small_layout(a, keys, inval, s_ids);
}

}  // namespace

cudaError_t launch_align(const AlignLaunch& a, cudaStream_t s) {
  const int CH = 1 << a.ch_log2;
  const int threads = CH < 1024 ? CH : 1024;
  const size_t smem = static_cast<size_t>(CH) * sizeof(uint32_t);
  if (a.nchunks == 1) {
    align_small_kernel<<<1, 1024, smem + static_cast<size_t>(a.P) * sizeof(int32_t), s>>>(a);
    return cudaGetLastError();
  }
  if (a.nchunks > 0) {
    align_chunk_kernel<<<a.nchunks, threads, smem, s>>>(a);
    cudaError_t err = cudaGetLastError();
    if (err != cudaSuccess) return err;
  }
  const int64_t nb_buckets = static_cast<int64_t>(a.E) * (a.L + 1);
  if (nb_buckets <= kScanSmemBuckets) {
    const size_t smem = static_cast<size_t>(3 * nb_buckets + a.E) * sizeof(int32_t);
    static bool attr_set = false;   // one device model per process
    if (!attr_set) {
      const cudaError_t e2 = cudaFuncSetAttribute(align_scan_smem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  static_cast<int>((3 * kScanSmemBuckets + MOE_LORA_MAX_EXPERTS) *
                                                                   sizeof(int32_t)));
      if (e2 != cudaSuccess) return e2;
      attr_set = true;
    }
    align_scan_smem_kernel<<<1, 1024, smem, s>>>(a);
  } else {
    align_scan_kernel<<<1, 1024, 0, s>>>(a);
  }
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  if (a.nchunks > 0) {
    align_scatter_kernel<<<a.nchunks, threads, smem, s>>>(a);
    err = cudaGetLastError();
  }
  return err;
}

cudaError_t launch_route_align_small(const AlignLaunch& a, const float* logits, float* topk_w, int32_t* topk_ids,
                                     cudaStream_t s) {
  const size_t smem = (static_cast<size_t>(1) << a.ch_log2) * sizeof(uint32_t) + static_cast<size_t>(a.P) * 4;
  route_align_small_kernel<<<1, 1024, smem, s>>>(a, logits, topk_w, topk_ids);
  return cudaGetLastError();
}

}  // namespace moe
