// moe_lora.cu -- the C ABI (include/moe_lora.h): host-side validation, workspace
// layout, TMA tensor-map encoding and the launch sequence of the MoE-LoRA layer.
//
// Launch sequence of moe_lora_forward (all on the caller's stream):
//   gather    x rows into sorted (expert, adapter, pair) order; zero padding rows
//   shrink    S_gu per adapter run = x_block A_gu[a,e]^T          (tcgen05)
//   gate_up   h = silu(gate) * up, gate/up = x W_gu[e]^T + S_gu B_gu[a,e]   (tcgen05)
//   shrink    S_dn per adapter run = h_block A_dn[a,e]^T          (tcgen05)
//   down      y[row] = h W_dn[e]^T + S_dn B_dn[a,e]                (tcgen05)
//   combine   out[t] = bf16(sum_j w[t,j] y[row of (t,j)]), fixed order
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <new>

#include "common.cuh"
#include "ptx.cuh"

namespace {

thread_local char g_err[512] = "";

// Test hook: limit of the gate_up epilogue's accumulator wait (0 = the default limit).
std::atomic<uint64_t> g_acc_wait_ns{0};

int fail(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(MOE_LORA_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define MOE_CUDA(call)                                  \
  do {                                                  \
    cudaError_t e_ = (call);                            \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
  } while (0)

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

int get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_encode) return fail(MOE_LORA_ECUDA, "cuTensorMapEncodeTiled is not available from the driver");
  return MOE_LORA_OK;
}

// The kernels are compiled for sm_103a only.
int check_device() {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  int maj = 0, min = 0;
  cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&min, cudaDevAttrComputeCapabilityMinor, dev);
  if (maj != 10 || min != 3)
    return fail(MOE_LORA_EUNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a", dev, maj, min);
  return MOE_LORA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t up256(size_t n) { return (n + 255) & ~size_t(255); }

int validate_dims(const moe_lora_dims* d) {
  if (!d) return fail(MOE_LORA_EINVAL, "dims is NULL");
  if (d->T < 0) return fail(MOE_LORA_EINVAL, "T = %lld < 0", (long long)d->T);
  if (d->H <= 0 || d->H % 64) return fail(MOE_LORA_EINVAL, "H = %d must be a positive multiple of 64", d->H);
  if (d->I <= 0 || d->I % 64) return fail(MOE_LORA_EINVAL, "I = %d must be a positive multiple of 64", d->I);
  if (d->E < 1 || d->E > MOE_LORA_MAX_EXPERTS) return fail(MOE_LORA_EUNSUPPORTED, "E = %d outside [1, %d]", d->E, MOE_LORA_MAX_EXPERTS);
  if (d->k < 1 || d->k > d->E || d->k > MOE_LORA_MAX_TOPK)
    return fail(MOE_LORA_EINVAL, "k = %d outside [1, min(E, %d)]", d->k, MOE_LORA_MAX_TOPK);
  if (d->L < 0 || d->L > MOE_LORA_MAX_ADAPTERS) return fail(MOE_LORA_EUNSUPPORTED, "L = %d outside [0, %d]", d->L, MOE_LORA_MAX_ADAPTERS);
  if (d->block_m != 16 && d->block_m != 32 && d->block_m != 64 && d->block_m != 128 && d->block_m != 256)
    return fail(MOE_LORA_EUNSUPPORTED, "block_m = %d not in {16, 32, 64, 128, 256}", d->block_m);
  if (d->T * (int64_t)d->k >= (int64_t(1) << 30)) return fail(MOE_LORA_EUNSUPPORTED, "T*k too large");
  if (d->L > 0) {
    if (d->r_max < 8 || d->r_max > MOE_LORA_MAX_RANK || d->r_max % 8)
      return fail(MOE_LORA_EUNSUPPORTED, "r_max = %d must be a multiple of 8 in [8, %d]", d->r_max, MOE_LORA_MAX_RANK);
    if (!d->ranks) return fail(MOE_LORA_EINVAL, "ranks is NULL with L = %d", d->L);
    for (int a = 0; a < d->L; ++a)
      if (d->ranks[a] < 1 || d->ranks[a] > d->r_max)
        return fail(MOE_LORA_EINVAL, "ranks[%d] = %d outside [1, r_max = %d]", a, d->ranks[a], d->r_max);
  }
  return MOE_LORA_OK;
}

// ---- compiled-in tile table
// The pages tune the fused MoE-LoRA kernels per shape, with tables of tile sizes
// picked by problem size (AWS ML Blog "Efficiently serve dozens of fine-tuned models
// with vLLM on Amazon SageMaker AI and Amazon Bedrock", section "Tuning kernel
// configurations for Amazon SageMaker AI and Amazon Bedrock"; agentlenshq.com "vLLM
// MoE 모델을 위한 Multi-LoRA 서빙", section "Amazon 전용 튜닝").  Here the table is
// compiled in.  A shape's class is its pairs per expert T*k/E -- how many token rows
// each streamed weight tile serves -- and the class fixes the token tile (= align
// block) and, for the weight-streaming kernels, the targets of the K-split rules,
// which then weigh the tile counts against H, I and the SM count.  Rows were set from
// GB300 sweeps over the workloads' shapes: 256-row blocks (CTA pairs, 2-SM MMA) win
// once experts see thousands of tokens (3200 pairs per expert: 3.88 vs 4.13 ms).
// Between 768 and 2047 pairs per expert they win only where the adapter runs are long
// (pairs per (expert, adapter-or-none bucket) T*k / (E*(L+1)) >= 20): a 256-row block of
// short runs carries twice the LoRA expand chunks of a 128-row one.  Measured, 128 vs
// 256 rows: the wide layer (32 adapters) at 768 / 1024 pairs per expert 1.445 / 1.791
// vs 1.398 / 1.736 ms, at 512 1.075 vs 1.094 ms; the sweep layer (64 adapters) at 512 /
// 1024 pairs per expert 1.34 / 2.05 vs 1.80 / 2.48 ms.  16-row tiles (two CTAs an SM)
// beat 32-row ones up to 24 pairs per expert on every layer measured (µs, 16 vs 32 rows:
// sweep layer at 16 / 24 pairs 332 / 388 vs 345 / 400, decode layer at 16 pairs 342 vs
// 357, dense MLP at 16 tokens 182 vs 187).  An expert whose weights exceed the L2 is
// streamed from DRAM once per block of it, so there the smallest tile that holds the
// expert's pairs wins: a 786 MB dense MLP at 32 tokens 187 us on 32 rows against 249 on
// 16 and 241 on 64, at 64 tokens 246 us on 64 rows against 264 on 32 and 290 on 128.
struct TileClass {
  double ppe_above;       // the class holds shapes whose T*k/E exceeds this
  int block_m;            // token tile: < 128 weight-streaming, >= 128 token-tiled
  int gu_tiles_per_cta;   // weight-streaming gate_up: split K until about this many tiles per CTA
  int dn_tiles_per_cta;   // weight-streaming down: the same
  int shrink_min_ktiles;  // weight-streaming shrink: split K only from this many 64-wide K-tiles
  int shrink_max_splits;
  int shrink_cores;       // 1: the shrinks run on CUDA cores (short runs, split over K), else tcgen05
};
constexpr TileClass kTileTable[] = {
    {-1.0, 16, 2, 3, 64, 8, 1},    // up to 24 pairs per expert (decode batches; down split 2
                                   //   ways on the decode layer: 283.9 -> 281.9 us against 3)
    {24.0, 32, 2, 6, 64, 8, 1},    // no class of its own (row 64 shares its bound): experts
                                   //   larger than the L2 with 17 .. 32 pairs
    {24.0, 64, 2, 6, 64, 8, 1},    // 24 .. 95
    {95.0, 128, 1, 1, 0, 1, 0},    // 95 .. 2047: token-tiled, compute-bound, no K split
    {2047.0, 256, 1, 1, 0, 1, 0},  // more than 2047: 256-token blocks on CTA pairs
};
constexpr int kTableRows = sizeof(kTileTable) / sizeof(kTileTable[0]);

// Row of the shape class of (T, k, E, L, H, I); H or I <= 0: expert size unknown.
constexpr double kLongRunsPpe = 768.0;     // from here 256-row blocks can win ...
constexpr double kLongRunsPerBucket = 20.0; // ... when the runs are this long
constexpr double kL2Bytes = 129e6;                 // GB300 L2
constexpr double kLargeExpertMaxPpe = 128.0;       // the large-expert rule up to one 128-row block
int class_row(int64_t T, int32_t k, int32_t E, int32_t L, int64_t H, int64_t I) {
  if (E <= 0 || k <= 0 || T <= 0) return 0;
  const double ppe = (double)T * k / E;
  // an expert's weights (gate_up 2*I*H, down H*I, bf16) larger than the L2
  if (H > 0 && I > 0 && 3.0 * H * I * 2.0 > kL2Bytes && ppe <= kLargeExpertMaxPpe) {
    int row = 0;
    while (row + 1 < kTableRows && kTileTable[row].block_m < ppe) ++row;
    return row;
  }
  int row = 0;
  for (int i = 0; i < kTableRows; ++i)
    if (ppe > kTileTable[i].ppe_above) row = i;
  if (kTileTable[row].block_m == 128 && row + 1 < kTableRows && ppe >= kLongRunsPpe &&
      ppe / ((L > 0 ? L : 0) + 1) >= kLongRunsPerBucket)
    ++row;
  return row;
}

// Row whose constants a launch with this token tile uses (256 takes the 128 row).
int block_row(int block_m) {
  int row = 0;
  for (int i = 0; i < kTableRows; ++i)
    if (kTileTable[i].block_m <= block_m) row = i;
  return row;
}

// block_m == 0 asks for the table's choice; every entry point works on a resolved copy.
int resolve(const moe_lora_dims* in, moe_lora_dims* out) {
  if (!in) return fail(MOE_LORA_EINVAL, "dims is NULL");
  *out = *in;
  if (out->block_m == 0) out->block_m = kTileTable[class_row(out->T, out->k, out->E, out->L, out->H, out->I)].block_m;
  return MOE_LORA_OK;
}
#define MOE_RESOLVE(d)                           \
  moe_lora_dims d##_resolved;                    \
  do {                                           \
    int st_ = resolve(d, &d##_resolved);         \
    if (st_ != MOE_LORA_OK) return st_;          \
  } while (0);                                   \
  d = &d##_resolved

struct Caps {
  int64_t rows, blocks, runs;
};
Caps capacity(const moe_lora_dims* d) {
  const int64_t P = d->T * d->k, BM = d->block_m;
  int64_t rows = P + (P < d->E ? P : d->E) * (BM - 1);
  rows = (rows + BM - 1) / BM * BM;
  const int64_t blocks = rows / BM;
  int64_t runs = blocks + (int64_t)d->E * d->L;
  if (runs > P) runs = P;
  if (d->L == 0) runs = 0;
  return {rows, blocks, runs};
}

int r_pad_of(const moe_lora_dims* d) { return d->L > 0 ? (d->r_max + 15) / 16 * 16 : 16; }

// ---- align scratch layout
struct AlignLayout {
  int ch_log2, nchunks;
  size_t keys, counts, invalid, btotal, bbase, rbase, expn, bytes;
};
AlignLayout align_layout(const moe_lora_dims* d) {
  AlignLayout l{};
  const int64_t P = d->T * d->k;
  int lg = 5;
  while ((int64_t(1) << lg) < P && lg < 12) ++lg;
  l.ch_log2 = lg;
  l.nchunks = (int)((P + (int64_t(1) << lg) - 1) >> lg);
  const size_t NB = (size_t)d->E * (d->L + 1);
  size_t off = 0;
  l.keys = off;    off += up256((size_t)l.nchunks << lg << 2);
  l.counts = off;  off += up256((size_t)l.nchunks * NB * 4);
  l.invalid = off; off += up256((size_t)l.nchunks * 4);
  l.btotal = off;  off += up256(NB * 4);
  l.bbase = off;   off += up256(NB * 4);
  l.rbase = off;   off += up256(NB * 4);
  l.expn = off;    off += up256((size_t)d->E * 4);
  l.bytes = off;
  return l;
}

// ---- forward scratch layout
struct FwdLayout {
  size_t xs, hs, sgu, sdn, y, prow, ctr, gpart, pgu, pdn, plan, bytes;
  int n_ctr, ks_gu, ks_dn;
};
constexpr int kNumGemmCounters = 4;   // tile counters: shrink_gu, gate_up, shrink_dn, down
constexpr int kPlanSMs = 152;         // SM count the K-split heuristics plan for (GB300)
// Whether the shrinks run on CUDA cores (shrink_rows) rather than as tcgen05 tiles, and
// over how many K slices.  The tensor-core shrink is a chain of dependent TMA round
// trips per run; behind a long base-weight stream (the GEMM after it starts streaming
// at once) it is hidden, and a CUDA-core shrink only takes SMs from that stream
// (measured: decode 0.285 -> 0.299 ms, dense_decode 0.193 -> 0.201 ms).  When the
// stream is short -- gate_up's weights of at most min(E, T*k) experts under ~128 MB --
// and the runs are a handful (at most one per 8 SMs: a single token's experts), the
// shrink is the critical path and a run's tile chain is long; split over K on CUDA
// cores it is shorter (one token over 128 experts: 65 -> 61 us).  With tens of short
// runs the tensor-core tiles already spread over the SMs (the 64-token test layer:
// 46 us against 48 on CUDA cores).
constexpr double kShrinkCoresMaxStreamBytes = 128.0 * 1024 * 1024;
bool shrink_on_cores(const moe_lora_dims* d, const Caps& cap) {
  if (d->L <= 0 || d->block_m >= 128 || kTileTable[block_row(d->block_m)].shrink_cores == 0) return false;
  if (cap.runs <= 0 || cap.runs * 8 > kPlanSMs) return false;
  const double experts = (double)(d->T * d->k < d->E ? d->T * d->k : d->E);
  return experts * 2.0 * d->I * d->H * 2.0 <= kShrinkCoresMaxStreamBytes;
}
int shrink_slices(int K) { return (K + moe::kShrinkSlice - 1) / moe::kShrinkSlice; }
int shrink_ksplit(const moe_lora_dims* d, const Caps& cap, int K);
// The tcgen05 shrink of token-tiled blocks can run block-diagonal tiles (several
// adapter runs side by side in N, from a group table the gather launch builds): each
// stage then brings up to 32 KB of A rows instead of one run's 2-8 KB.  On 128-row
// blocks a block gives one to a few such tiles against one per run, so they pay once
// the blocks alone fill the SMs twice over (sweep T = 4096: 319 blocks, shrinks 227/96
// -> 193/80 us); with fewer blocks (wide at 128 rows: 64) the long K loops of too few
// tiles leave SMs idle (shrinks 41/77 -> 68/161 us) and the per-run tiles stay.  On the
// 128-row halves of 256-row blocks, whose runs are long, they lose (wide: 42/79 -> 51/113
// us with 8-chunk groups, 65/145 with 4; prefill 122/114 -> 138/132 us): there the
// per-run half tiles stay, and the block-diagonal form runs only when the test hook
// asks for it.
std::atomic<int> g_shrink_tiles{0};   // test hook: 0 by shape, 1 block-diagonal, 2 per run
bool block_diag_space(const moe_lora_dims* d) { return d->L > 0 && (d->block_m == 128 || d->block_m == 256); }
bool block_diag_shrink(const moe_lora_dims* d, const Caps& cap) {
  if (!block_diag_space(d)) return false;
  const int mode = g_shrink_tiles.load(std::memory_order_relaxed);
  if (mode != 0) return mode == 1;
  if (d->block_m == 256) return false;
  return cap.blocks >= 2 * kPlanSMs;
}
// Rank chunks per block-diagonal group: 16 (N = 256) on 128-row blocks; 8 on the halves
// of 256-row blocks, whose blocks are fewer (at least 4: the group table's capacity).
int shrink_group_chunks(const moe_lora_dims* d) { return d->block_m == 256 ? 8 : 16; }
int gate_up_ksplit(const moe_lora_dims* d, const Caps& cap);
int down_ksplit(const moe_lora_dims* d, const Caps& cap);
// Batches of a few pairs (at most 32: one to four tokens of top-8) on 16-token tiles run
// gate_up and down with a 6-deep ring, one CTA per SM: their tiles are fewer than the
// CTAs, and a tile's latency, not two CTAs sharing an SM, sets the pace.  Measured 3 vs
// 6 stages: sweep T = 1 55.3 -> 51.7 us; the decode layer (64 pairs) 282 -> 288 us and
// sweep T = 16 (128 pairs) 165.5 -> 173.0 us, so larger batches keep 3.
constexpr int64_t kDeepRingPairs = 32;
bool deep_ring(const moe_lora_dims* d) { return d->block_m == 16 && d->T * d->k <= kDeepRingPairs; }
FwdLayout fwd_layout(const moe_lora_dims* d) {
  const Caps c = capacity(d);
  FwdLayout l{};
  l.ks_gu = gate_up_ksplit(d, c);
  l.ks_dn = down_ksplit(d, c);
  size_t off = 0;
  const size_t s_tile = (size_t)d->block_m * r_pad_of(d) * 2;
  l.xs = off;  off += up256((size_t)c.rows * d->H * 2);
  l.hs = off;  off += up256((size_t)c.rows * d->I * 2);
  l.sgu = off; off += up256((size_t)c.runs * s_tile);
  l.sdn = off; off += up256((size_t)c.runs * s_tile);
  // down outputs per sorted row: bf16, or fp32 partials per K split
  l.y = off;   off += up256(l.ks_dn > 1 ? (size_t)l.ks_dn * c.rows * d->H * 4 : (size_t)c.rows * d->H * 2);
  l.prow = off; off += up256((size_t)d->T * d->k * 4);
  l.ctr = off; off += up256((size_t)(kNumGemmCounters + 2 * 4 * c.runs) * 4);
  // fp32 partial gate/up pre-activations of a K-split (weight-streaming) gate_up
  l.gpart = off; off += l.ks_gu > 1 ? up256((size_t)l.ks_gu * c.rows * 2 * d->I * 4) : 0;
  // fp32 partial S of K-split shrinks, and their per-(run, warp) arrival counters
  const size_t s_part = (size_t)c.runs * d->block_m * r_pad_of(d) * 4;
  const bool cores = shrink_on_cores(d, c);
  l.pgu = off; off += up256((size_t)(cores ? shrink_slices(d->H) : shrink_ksplit(d, c, d->H)) * s_part);
  l.pdn = off; off += up256((size_t)(cores ? shrink_slices(d->I) : shrink_ksplit(d, c, d->I)) * s_part);
  // group table of the block-diagonal shrink (128-row blocks): [groups] block, [groups]
  // first chunk, [blocks] chunk counts, the group count; groups <= runs + blocks
  l.plan = off;
  if (block_diag_space(d)) {
    const size_t upb = (size_t)d->block_m / 128;   // 128-row units per block
    off += up256((2 * upb * (size_t)(c.runs + c.blocks) + upb * (size_t)c.blocks + 1) * 4);
  }
  l.n_ctr = kNumGemmCounters + 2 * 4 * (int)c.runs;
  l.bytes = off;
  return l;
}

// ---- tensor maps
int encode(CUtensorMap* m, const void* ptr, int rank, const uint64_t* dims, const uint64_t* strides,
           const uint32_t* box, CUtensorMapSwizzle sw, const char* what) {
  cuuint64_t gd[5];
  cuuint64_t gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i < rank - 1; ++i) gs[i] = strides[i];
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(ptr), gd, gs, bx, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(MOE_LORA_ECUDA, "cuTensorMapEncodeTiled(%s) failed with %d", what, (int)r);
  return MOE_LORA_OK;
}

#define MOE_TRY(x)                         \
  do {                                     \
    int st_ = (x);                         \
    if (st_ != MOE_LORA_OK) return st_;    \
  } while (0)

int check_ptr(const void* p, const char* name, bool need16) {
  if (!p) return fail(MOE_LORA_EINVAL, "%s is NULL", name);
  if (need16 && !aligned16(p)) return fail(MOE_LORA_EALIGN, "%s is not 16-byte aligned", name);
  return MOE_LORA_OK;
}

int check_align_buf(const moe_lora_align_buf* b) {
  if (!b) return fail(MOE_LORA_EINVAL, "align buffer struct is NULL");
  MOE_TRY(check_ptr(b->sorted_p, "sorted_p", false));
  MOE_TRY(check_ptr(b->expert_begin, "expert_begin", false));
  MOE_TRY(check_ptr(b->block_expert, "block_expert", false));
  MOE_TRY(check_ptr(b->block_runs, "block_runs", false));
  MOE_TRY(check_ptr(b->runs, "runs", false));
  MOE_TRY(check_ptr(b->totals, "totals", false));
  return MOE_LORA_OK;
}

// K splits of a weight-streaming GEMM (n_ft feature tiles per block, reduction K):
// enough tiles for about `per_cta` per persistent CTA, so the CTAs finish together;
// each split keeps at least 8 K-tiles, at most 4 splits.  Token-tiled (compute-bound)
// shapes keep one.
int weight_stream_ksplit(const moe_lora_dims* d, const Caps& cap, int n_ft, int K, int per_cta) {
  if (d->block_m >= 128 || per_cta <= 1) return 1;
  const int64_t P = d->T * d->k;
  int64_t est_blocks = cap.blocks;
  if (est_blocks > d->E) est_blocks = d->E;
  if (est_blocks > P) est_blocks = P;
  const int64_t tiles = (int64_t)n_ft * (est_blocks > 0 ? est_blocks : 1);
  int64_t ks = ((int64_t)per_cta * kPlanSMs + tiles - 1) / tiles;
  const int64_t nk = K / 64;
  const int64_t ks_max = nk / 8 < 4 ? (nk / 8 > 1 ? nk / 8 : 1) : 4;
  if (ks > ks_max) ks = ks_max;
  return ks < 1 ? 1 : (int)ks;
}
int down_ksplit(const moe_lora_dims* d, const Caps& cap) {
  return weight_stream_ksplit(d, cap, (d->H + 255) / 256, d->I, kTileTable[block_row(d->block_m)].dn_tiles_per_cta);
}
// gate_up splits only when its tiles are too few to spread over the SMs: a split adds
// an fp32 round trip of the pre-activations and a SiLU pass.
int gate_up_ksplit(const moe_lora_dims* d, const Caps& cap) {
  return weight_stream_ksplit(d, cap, (d->I + 127) / 128, d->H, kTileTable[block_row(d->block_m)].gu_tiles_per_cta);
}
// The weight-streaming shrink splits K only for long reductions whose runs cannot fill
// the SMs -- a run's tile otherwise walks all of K alone.  Measured: splitting short
// reductions only adds per-tile overhead and keeps the SMs from the next kernel
// (decode: 57 runs of 45 K-tiles; a single token's 8 runs of 32 K-tiles: 67 -> 70 us
// split 4 ways).  About one tile per SM, each split at least 16 K-tiles, or 8 when the
// runs are a handful (at most one per 8 SMs; dense_decode: 0.197 -> 0.193 ms).
int shrink_ksplit(const moe_lora_dims* d, const Caps& cap, int K) {
  const TileClass& tc = kTileTable[block_row(d->block_m)];
  const int64_t nk = K / 64;
  const bool few = cap.runs > 0 && cap.runs * 8 <= kPlanSMs;
  if (d->block_m >= 128 || d->L == 0 || cap.runs <= 0 || tc.shrink_min_ktiles <= 0 || nk < tc.shrink_min_ktiles ||
      cap.runs >= kPlanSMs)
    return 1;
  int64_t ks = ((int64_t)kPlanSMs + cap.runs - 1) / cap.runs;
  const int64_t per = few ? 8 : 16;
  const int64_t ks_max = nk / per < tc.shrink_max_splits ? nk / per : tc.shrink_max_splits;
  if (ks > ks_max) ks = ks_max;
  return ks < 1 ? 1 : (int)ks;
}

int do_route(const float* logits, int64_t T, int32_t E, int32_t k, int32_t* ids, float* w, cudaStream_t s) {
  if (T < 0 || E < 1 || E > MOE_LORA_MAX_EXPERTS || k < 1 || k > E || k > MOE_LORA_MAX_TOPK)
    return fail(MOE_LORA_EINVAL, "route: T=%lld E=%d k=%d out of range", (long long)T, E, k);
  if (T == 0) return MOE_LORA_OK;
  MOE_TRY(check_ptr(logits, "logits", false));
  MOE_TRY(check_ptr(ids, "topk_ids", false));
  MOE_TRY(check_ptr(w, "topk_w", false));
  MOE_TRY(check_device());
  cudaError_t e = moe::launch_route(logits, T, E, k, ids, w, s);
  if (e != cudaSuccess) return cuda_fail(e, "route kernel launch");
  return MOE_LORA_OK;
}

moe::AlignLaunch align_launch(const moe_lora_dims* d, const AlignLayout& l, const int32_t* topk_ids,
                              const int32_t* lora_ids, const moe_lora_align_buf* out, void* ws) {
  uint8_t* base = static_cast<uint8_t*>(ws);
  moe::AlignLaunch a{};
  a.topk_ids = topk_ids;
  a.lora_ids = lora_ids;
  a.P = d->T * d->k;
  a.k = d->k;
  a.E = d->E;
  a.L = d->L;
  a.BM = d->block_m;
  a.ch_log2 = l.ch_log2;
  a.nchunks = l.nchunks;
  a.chunk_keys = reinterpret_cast<uint32_t*>(base + l.keys);
  a.counts = reinterpret_cast<int32_t*>(base + l.counts);
  a.chunk_invalid = reinterpret_cast<int32_t*>(base + l.invalid);
  a.bucket_total = reinterpret_cast<int32_t*>(base + l.btotal);
  a.bucket_base = reinterpret_cast<int32_t*>(base + l.bbase);
  a.run_base = reinterpret_cast<int32_t*>(base + l.rbase);
  a.expert_n = reinterpret_cast<int32_t*>(base + l.expn);
  a.out = *out;
  return a;
}

int do_align(const moe_lora_dims* d, const int32_t* topk_ids, const int32_t* lora_ids, const moe_lora_align_buf* out,
             void* ws, size_t ws_bytes, cudaStream_t s) {
  MOE_RESOLVE(d);
  MOE_TRY(validate_dims(d));
  MOE_TRY(check_align_buf(out));
  const AlignLayout l = align_layout(d);
  if (d->T > 0) {
    MOE_TRY(check_ptr(topk_ids, "topk_ids", false));
    MOE_TRY(check_ptr(lora_ids, "lora_ids", false));
  }
  MOE_TRY(check_ptr(ws, "workspace", true));
  if (ws_bytes < l.bytes) return fail(MOE_LORA_EWORKSPACE, "align workspace %zu < %zu bytes", ws_bytes, l.bytes);
  MOE_TRY(check_device());
  cudaError_t e = moe::launch_align(align_launch(d, l, topk_ids, lora_ids, out, ws), s);
  if (e != cudaSuccess) return cuda_fail(e, "align kernel launch");
  return MOE_LORA_OK;
}

// Route then align.  Batches of one align chunk (T*k <= 4096) take a single launch;
// larger ones the route kernel and the align kernels.
// Route and align share one single-CTA launch only for a few tokens: in one CTA the
// router costs ~400 issue cycles per token (measured: 3 us at T = 16, 57 us at T = 256
// with E = 128, k = 8), while the route kernel gives every token its own warp across
// the GPU.  Larger one-chunk batches take the route kernel, then the one-CTA align.
constexpr int64_t kFusedRouteTokens = 32;
bool fused_route_align(const moe_lora_dims* d, const AlignLayout& l) {
  return l.nchunks == 1 && d->T <= kFusedRouteTokens;
}

int do_route_align(const moe_lora_dims* d, const float* logits, const int32_t* lora_ids, int32_t* topk_ids,
                   float* topk_w, const moe_lora_align_buf* out, void* ws, size_t ws_bytes, cudaStream_t s) {
  MOE_RESOLVE(d);
  MOE_TRY(validate_dims(d));
  const AlignLayout l = align_layout(d);
  if (!fused_route_align(d, l)) {
    MOE_TRY(do_route(logits, d->T, d->E, d->k, topk_ids, topk_w, s));
    return do_align(d, topk_ids, lora_ids, out, ws, ws_bytes, s);
  }
  MOE_TRY(check_align_buf(out));
  MOE_TRY(check_ptr(logits, "logits", false));
  MOE_TRY(check_ptr(lora_ids, "lora_ids", false));
  MOE_TRY(check_ptr(topk_ids, "topk_ids", false));
  MOE_TRY(check_ptr(topk_w, "topk_w", false));
  MOE_TRY(check_ptr(ws, "workspace", true));
  if (ws_bytes < l.bytes) return fail(MOE_LORA_EWORKSPACE, "align workspace %zu < %zu bytes", ws_bytes, l.bytes);
  MOE_TRY(check_device());
  cudaError_t e = moe::launch_route_align_small(align_launch(d, l, topk_ids, lora_ids, out, ws), logits, topk_w,
                                                topk_ids, s);
  if (e != cudaSuccess) return cuda_fail(e, "route_align kernel launch");
  return MOE_LORA_OK;
}

int do_forward(const moe_lora_dims* d, const uint16_t* x, const float* topk_w, const moe_lora_align_buf* al,
               const uint16_t* W_gu, const uint16_t* W_dn, const uint16_t* A_gu, const uint16_t* B_gu,
               const uint16_t* A_dn, const uint16_t* B_dn, uint16_t* out, void* ws, size_t ws_bytes,
               int32_t* dev_status, cudaStream_t s, void* const* ev) {
  MOE_RESOLVE(d);
  MOE_TRY(validate_dims(d));
  MOE_TRY(check_align_buf(al));
  MOE_TRY(check_ptr(dev_status, "dev_status", false));
  const FwdLayout l = fwd_layout(d);
  const Caps cap = capacity(d);
  if (d->T == 0) {
    MOE_TRY(check_device());
    MOE_CUDA(cudaMemsetAsync(dev_status, 0, sizeof(int32_t), s));
    return MOE_LORA_OK;
  }
  MOE_TRY(check_ptr(x, "x", true));
  MOE_TRY(check_ptr(topk_w, "topk_w", false));
  MOE_TRY(check_ptr(W_gu, "W_gu", true));
  MOE_TRY(check_ptr(W_dn, "W_dn", true));
  MOE_TRY(check_ptr(out, "out", true));
  MOE_TRY(check_ptr(ws, "workspace", true));
  if (d->L > 0) {
    MOE_TRY(check_ptr(A_gu, "A_gu", true));
    MOE_TRY(check_ptr(B_gu, "B_gu", true));
    MOE_TRY(check_ptr(A_dn, "A_dn", true));
    MOE_TRY(check_ptr(B_dn, "B_dn", true));
  }
  if (ws_bytes < l.bytes) return fail(MOE_LORA_EWORKSPACE, "forward workspace %zu < %zu bytes", ws_bytes, l.bytes);
  MOE_TRY(check_device());
  MOE_TRY(get_encoder());

  uint8_t* base = static_cast<uint8_t*>(ws);
  uint16_t* xs = reinterpret_cast<uint16_t*>(base + l.xs);
  uint16_t* hs = reinterpret_cast<uint16_t*>(base + l.hs);
  uint16_t* sgu = reinterpret_cast<uint16_t*>(base + l.sgu);
  uint16_t* sdn = reinterpret_cast<uint16_t*>(base + l.sdn);
  void* y = base + l.y;
  int32_t* prow = reinterpret_cast<int32_t*>(base + l.prow);
  int32_t* ctr = reinterpret_cast<int32_t*>(base + l.ctr);
  const int ks_gu = l.ks_gu;
  float* gpart = ks_gu > 1 ? reinterpret_cast<float*>(base + l.gpart) : nullptr;
  const int BT = d->block_m;
  const uint64_t H = d->H, I = d->I, E = d->E, LE = (uint64_t)d->L * d->E, R = d->r_max;
  const uint64_t rows = cap.rows, RP = r_pad_of(d);
  const uint64_t nruns = cap.runs > 0 ? cap.runs : 1;

  // tensor maps (dims innermost first; strides in bytes for dims 1..rank-1)
  moe::GemmMaps m_sgu{}, m_gu{}, m_sdn{}, m_dn{};
  // K width of each launch's stages and the matching swizzle (64 -> 128-byte, 32 -> 64-byte)
  const uint32_t bk_gu = (uint32_t)moe::gemm_bk(moe::kGateUp, BT), bk_dn = (uint32_t)moe::gemm_bk(moe::kDown, BT);
  const uint32_t bk_sh = (uint32_t)moe::gemm_bk(moe::kShrink, BT);
  auto swz = [](uint32_t bk) { return bk == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B; };
  // token rows one CTA of a gate_up / down launch stages: 256-row blocks run on CTA
  // pairs, each CTA taking its 128 rows
  const uint32_t tok_rows = BT == 256 ? 128u : (uint32_t)BT;
  // token rows a shrink tile stages: 256-row blocks are shrunk in 128-row halves
  const uint32_t sh_rows = BT == 256 ? 128u : (uint32_t)BT;
  {
    const uint64_t dm[4] = {H, I, 2, E}, st[3] = {H * 2, I * H * 2, 2 * I * H * 2};
    const uint32_t bx[4] = {bk_gu, 128, 1, 1};
    MOE_TRY(encode(&m_gu.w, W_gu, 4, dm, st, bx, swz(bk_gu), "W_gu"));
  }
  {
    const uint64_t dm[3] = {I, H, E}, st[2] = {I * 2, H * I * 2};
    const uint32_t bx[3] = {bk_dn, 128, 1};
    MOE_TRY(encode(&m_dn.w, W_dn, 3, dm, st, bx, swz(bk_dn), "W_dn"));
  }
  {
    const uint64_t dm[2] = {H, rows}, st[1] = {H * 2};
    const uint32_t bx[2] = {bk_gu, tok_rows};
    MOE_TRY(encode(&m_gu.tok, xs, 2, dm, st, bx, swz(bk_gu), "x_sorted"));
    const uint32_t bxs[2] = {bk_sh, sh_rows};
    MOE_TRY(encode(&m_sgu.tok, xs, 2, dm, st, bxs, swz(bk_sh), "x_sorted"));
  }
  {
    const uint64_t dm[2] = {I, rows}, st[1] = {I * 2};
    const uint32_t bx[2] = {bk_dn, tok_rows};
    MOE_TRY(encode(&m_dn.tok, hs, 2, dm, st, bx, swz(bk_dn), "h_sorted"));
    const uint32_t bxs[2] = {bk_sh, sh_rows};
    MOE_TRY(encode(&m_sdn.tok, hs, 2, dm, st, bxs, swz(bk_sh), "h_sorted"));
  }
  if (d->L > 0) {
    // A: one map per rank class, boxes of 16, 32, 48, 64 rows (a stage loads an
    // adapter's ranks in one TMA; rows past r_max read as zero)
    for (int c = 0; c < 4; ++c) {
      const uint32_t rows = 16u * (uint32_t)(c + 1);
      {
        const uint64_t dm[3] = {H, R, LE}, st[2] = {H * 2, R * H * 2};
        const uint32_t bx[3] = {64, rows, 1};
        MOE_TRY(encode(c == 0 ? &m_sgu.w : &m_sgu.w_rank[c - 1], A_gu, 3, dm, st, bx, CU_TENSOR_MAP_SWIZZLE_128B,
                       "A_gu"));
      }
      {
        const uint64_t dm[3] = {I, R, LE}, st[2] = {I * 2, R * I * 2};
        const uint32_t bx[3] = {64, rows, 1};
        MOE_TRY(encode(c == 0 ? &m_sdn.w : &m_sdn.w_rank[c - 1], A_dn, 3, dm, st, bx, CU_TENSOR_MAP_SWIZZLE_128B,
                       "A_dn"));
      }
    }
    // B, rank-major: one box is 16 rank rows of the tile's weight columns, landing as
    // 64-column atoms of 16 rows x 128 bytes (the MN-major 128-byte-swizzle operand
    // layout).  Dims: 64 columns, rank, 64-column atom, [gate|up,] adapter x expert.
    // Columns past I (or H) fall outside the atom dimension and read as zero.
    const uint32_t atoms = BT == 256 ? 2u : 4u;   // CTA pairs load their 128 columns each
    {
      const uint64_t dm[5] = {64, R, I / 64, 2, LE}, st[4] = {2 * I * 2, 128, I * 2, R * 2 * I * 2};
      const uint32_t bx[5] = {64, 16, 2, atoms / 2, 1};
      MOE_TRY(encode(&m_gu.lw, B_gu, 5, dm, st, bx, CU_TENSOR_MAP_SWIZZLE_128B, "B_gu"));
    }
    {
      const uint64_t dm[4] = {64, R, H / 64, LE}, st[3] = {H * 2, 128, R * H * 2};
      const uint32_t bx[4] = {64, 16, atoms, 1};
      MOE_TRY(encode(&m_dn.lw, B_dn, 4, dm, st, bx, CU_TENSOR_MAP_SWIZZLE_128B, "B_dn"));
    }
    {
      const uint64_t dm[3] = {RP, (uint64_t)BT, nruns}, st[2] = {RP * 2, (uint64_t)BT * RP * 2};
      const uint32_t bx[3] = {16, tok_rows, 1};
      MOE_TRY(encode(&m_gu.ls, sgu, 3, dm, st, bx, CU_TENSOR_MAP_SWIZZLE_32B, "S_gu"));
      MOE_TRY(encode(&m_dn.ls, sdn, 3, dm, st, bx, CU_TENSOR_MAP_SWIZZLE_32B, "S_dn"));
    }
  } else {
    // No adapter runs exist, so these maps are never loaded through; keep them valid.
    m_gu.lw = m_gu.ls = m_gu.w;
    m_dn.lw = m_dn.ls = m_dn.w;
  }
  m_sgu.lw = m_sgu.ls = m_sgu.out = m_sgu.w;
  m_sdn.lw = m_sdn.ls = m_sdn.out = m_sdn.w;
  // output rows of the CTA-pair gate_up / down epilogues (TMA stores of 32 rows x 64 columns)
  m_gu.out = m_gu.w;
  m_dn.out = m_dn.w;
  if (BT == 256) {
    const uint32_t bx[2] = {64, 32};
    {
      const uint64_t dm[2] = {I, rows}, st[1] = {I * 2};
      MOE_TRY(encode(&m_gu.out, hs, 2, dm, st, bx, CU_TENSOR_MAP_SWIZZLE_128B, "h_sorted (store)"));
    }
    if (l.ks_dn == 1) {
      const uint64_t dm[2] = {H, rows}, st[1] = {H * 2};
      MOE_TRY(encode(&m_dn.out, y, 2, dm, st, bx, CU_TENSOR_MAP_SWIZZLE_128B, "y (store)"));
    }
  }

  moe::GemmParams p{};
  p.block_expert = al->block_expert;
  p.expert_begin = al->expert_begin;
  p.block_runs = al->block_runs;
  p.runs = al->runs;
  p.totals = al->totals;
  p.sorted_p = al->sorted_p;
  p.part_rows = cap.rows;
  p.status = dev_status;
  p.acc_wait_ns = moe::kWaitTimeoutNs;
  p.E = d->E;
  p.k = d->k;
  p.P = (int32_t)(d->T * d->k);
  p.r_pad = (int32_t)RP;
  p.ksplit = 1;
  p.lora_after_pdl = 0;
  p.max_runs = (int32_t)cap.runs;
  for (int a = 0; a < d->L; ++a) p.ranks[a] = d->ranks[a];
  const bool bdiag = block_diag_shrink(d, cap);
  moe::ShrinkPlanArgs plan{};
  if (bdiag) {
    int32_t* pb = reinterpret_cast<int32_t*>(base + l.plan);
    const int64_t upb = BT / 128;
    const int64_t G = upb * (cap.runs + cap.blocks);
    plan.block_runs = al->block_runs;
    plan.runs = al->runs;
    plan.plan_block = pb;
    plan.plan_c0 = pb + G;
    plan.block_chunks = pb + 2 * G;
    plan.plan_count = pb + 2 * G + upb * cap.blocks;
    plan.block_m = BT;
    plan.gch = shrink_group_chunks(d);
    for (int a = 0; a < d->L; ++a) plan.ranks[a] = d->ranks[a];
    p.plan_block = plan.plan_block;
    p.plan_c0 = plan.plan_c0;
    p.plan_count = plan.plan_count;
    p.shrink_gch = plan.gch;
  }

  auto mark = [&](int i) -> cudaError_t {
    return ev ? cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), s) : cudaSuccess;
  };
  // Each kernel after the gather is launched as a programmatic dependent of the one
  // before it: it may start (prologue, weight streaming) while its predecessor
  // finishes, and waits on the device exactly where it reads that predecessor's
  // output.  Stage events, when given, sit between launches.
  const bool lora = d->L > 0;
  MOE_CUDA(mark(0));
  MOE_CUDA(moe::launch_gather_rows(x, al->sorted_p, al->totals, cap.rows, d->H, d->k, p.P, xs, prow, dev_status, ctr,
                                   l.n_ctr, bdiag ? &plan : nullptr, s));
  MOE_CUDA(mark(1 + MOE_LORA_STAGE_GATHER));

  const bool cores = shrink_on_cores(d, cap);
  // the shrink on CUDA cores: same inputs, same S tiles
  auto shrink_rows = [&](const uint16_t* rows_in, const uint16_t* A, int K, uint16_t* s_out, size_t part_off,
                         int32_t* cnt) -> cudaError_t {
    moe::ShrinkRowsLaunch r{};
    r.xs = rows_in;
    r.A = A;
    r.runs = al->runs;
    r.block_expert = al->block_expert;
    r.totals = al->totals;
    r.s_part = reinterpret_cast<float*>(base + part_off);
    r.s_cnt = cnt;
    r.s_out = s_out;
    r.K = K;
    r.E = d->E;
    r.r_max = d->r_max;
    r.r_pad = (int32_t)RP;
    r.block_m = BT;
    r.slices = shrink_slices(K);
    r.max_runs = (int32_t)cap.runs;
    for (int a = 0; a < d->L; ++a) r.ranks[a] = d->ranks[a];
    return moe::launch_shrink_rows(r, cap.runs, true, s);
  };
  if (lora) {
    moe::GemmParams q = p;
    q.K = d->H;
    q.s_out = sgu;
    q.tile_ctr = ctr + 0;
    q.ksplit = shrink_ksplit(d, cap, d->H);
    q.s_part = reinterpret_cast<float*>(base + l.pgu);
    q.s_cnt = ctr + kNumGemmCounters;
    if (cores) MOE_CUDA(shrink_rows(xs, A_gu, d->H, sgu, l.pgu, q.s_cnt));
    else MOE_CUDA(moe::launch_gemm(moe::kShrink, BT, m_sgu, q, cap.blocks, cap.runs, true, s, bdiag));
  }
  MOE_CUDA(mark(1 + MOE_LORA_STAGE_SHRINK_GU));
  {
    moe::GemmParams q = p;
    q.K = d->H;
    q.n_feat = d->I;
    q.h_out = hs;
    q.lora_after_pdl = lora;
    q.tile_ctr = ctr + 1;
    q.n_ft = (d->I + 127) / 128;
    const uint64_t lim = g_acc_wait_ns.load(std::memory_order_relaxed);
    if (lim != 0 && lim < moe::kWaitTimeoutNs) q.acc_wait_ns = lim;
    q.ksplit = ks_gu;
    q.g_part = gpart;
    MOE_CUDA(moe::launch_gemm(moe::kGateUp, BT, m_gu, q, cap.blocks, cap.runs, true, s, false, deep_ring(d)));
    if (ks_gu > 1) MOE_CUDA(moe::launch_silu_rows(gpart, ks_gu, cap.rows, al->totals, cap.rows, d->I, hs, true, s));
  }
  MOE_CUDA(mark(1 + MOE_LORA_STAGE_GATE_UP));
  if (lora) {
    moe::GemmParams q = p;
    q.K = d->I;
    q.s_out = sdn;
    q.tile_ctr = ctr + 2;
    q.ksplit = shrink_ksplit(d, cap, d->I);
    q.s_part = reinterpret_cast<float*>(base + l.pdn);
    q.s_cnt = ctr + kNumGemmCounters + 4 * cap.runs;
    if (cores) MOE_CUDA(shrink_rows(hs, A_dn, d->I, sdn, l.pdn, q.s_cnt));
    else MOE_CUDA(moe::launch_gemm(moe::kShrink, BT, m_sdn, q, cap.blocks, cap.runs, true, s, bdiag));
  }
  MOE_CUDA(mark(1 + MOE_LORA_STAGE_SHRINK_DN));
  {
    moe::GemmParams q = p;
    q.K = d->I;
    q.n_feat = d->H;
    q.y_out = y;
    q.lora_after_pdl = lora;
    q.ksplit = l.ks_dn;
    q.tile_ctr = ctr + 3;
    q.n_ft = (d->H + 255) / 256;
    MOE_CUDA(moe::launch_gemm(moe::kDown, BT, m_dn, q, cap.blocks, cap.runs, true, s, false, deep_ring(d)));
  }
  MOE_CUDA(mark(1 + MOE_LORA_STAGE_DOWN));
  MOE_CUDA(moe::launch_combine(y, l.ks_dn, cap.rows, prow, al->sorted_p, al->totals, topk_w, d->T, d->k, d->H, out,
                               true, s));
  MOE_CUDA(mark(1 + MOE_LORA_STAGE_COMBINE));
  return MOE_LORA_OK;
}

// ---- layer_host workspace: [align | forward | inputs | route out | align arrays | out | status]
struct LayerLayout {
  size_t align, fwd, logits, lora, x, ids, w, sp, eb, be, br, runs, out, status, bytes;
};
LayerLayout layer_layout(const moe_lora_dims* d) {
  const AlignLayout a = align_layout(d);
  const FwdLayout f = fwd_layout(d);
  const Caps c = capacity(d);
  LayerLayout l{};
  size_t off = 0;
  l.align = off;  off += up256(a.bytes);
  l.fwd = off;    off += up256(f.bytes);
  l.logits = off; off += up256((size_t)d->T * d->E * 4);
  l.lora = off;   off += up256((size_t)d->T * 4);
  l.x = off;      off += up256((size_t)d->T * d->H * 2);
  l.ids = off;    off += up256((size_t)d->T * d->k * 4);
  l.w = off;      off += up256((size_t)d->T * d->k * 4);
  l.sp = off;     off += up256((size_t)c.rows * 4);
  l.eb = off;     off += up256((size_t)(d->E + 1) * 4);
  l.be = off;     off += up256((size_t)c.blocks * 4);
  l.br = off;     off += up256((size_t)(c.blocks + 1) * 4);
  l.runs = off;   off += up256((size_t)c.runs * 16);
  l.out = off;    off += up256((size_t)d->T * d->H * 2);
  l.status = off; off += up256(8 * 4);   // {status, unused[3], totals[4]}
  l.bytes = off;
  return l;
}

}  // namespace

extern "C" {

int moe_lora_version(void) { return 304; }

int moe_lora_debug_set_acc_wait_ns(uint64_t ns) {
  g_acc_wait_ns.store(ns, std::memory_order_relaxed);
  return MOE_LORA_OK;
}

int moe_lora_debug_set_shrink_tiles(int32_t mode) {
  if (mode < 0 || mode > 2) return fail(MOE_LORA_EINVAL, "shrink tile mode %d not in {0, 1, 2}", mode);
  g_shrink_tiles.store(mode, std::memory_order_relaxed);
  return MOE_LORA_OK;
}

const char* moe_lora_status_string(int status) {
  switch (status) {
    case MOE_LORA_OK: return "ok";
    case MOE_LORA_EINVAL: return "invalid argument";
    case MOE_LORA_EALIGN: return "pointer not 16-byte aligned";
    case MOE_LORA_EWORKSPACE: return "workspace too small";
    case MOE_LORA_EUNSUPPORTED: return "unsupported shape or device";
    case MOE_LORA_ECUDA: return "CUDA error";
    case MOE_LORA_EDEVICE: return "device reported an error";
    default: return "unknown status";
  }
}

const char* moe_lora_last_error(void) { return g_err; }

int32_t moe_lora_pick_block_m(int64_t T, int32_t k, int32_t E, int32_t L, int32_t H, int32_t I) {
  return kTileTable[class_row(T, k, E, L, H, I)].block_m;
}

int moe_lora_plan_query(const moe_lora_dims* d, moe_lora_plan* out) {
  MOE_RESOLVE(d);
  MOE_TRY(validate_dims(d));
  if (!out) return fail(MOE_LORA_EINVAL, "plan is NULL");
  const Caps cap = capacity(d);
  const FwdLayout l = fwd_layout(d);
  moe_lora_plan p{};
  p.block_m = d->block_m;
  p.table_row = block_row(d->block_m);
  p.weight_streaming = d->block_m < 128;
  const bool lora = d->L > 0;
  const bool cores = shrink_on_cores(d, cap);
  p.shrink_on_cores = cores ? 1 : 0;
  p.shrink_block_diag = block_diag_shrink(d, cap) ? 1 : 0;
  p.ksplit[0] = lora ? (cores ? shrink_slices(d->H) : shrink_ksplit(d, cap, d->H)) : 0;
  p.ksplit[1] = l.ks_gu;
  p.ksplit[2] = lora ? (cores ? shrink_slices(d->I) : shrink_ksplit(d, cap, d->I)) : 0;
  p.ksplit[3] = l.ks_dn;
  const int modes[4] = {moe::kShrink, moe::kGateUp, moe::kShrink, moe::kDown};
  for (int g = 0; g < 4; ++g)
    if (!moe::gemm_stage_shape(modes[g], d->block_m, &p.k_tile[g], &p.stages[g], deep_ring(d)))
      return fail(MOE_LORA_EUNSUPPORTED, "no GEMM compiled for block_m = %d", d->block_m);
  if (cores) {   // one K slice per CTA, no pipeline
    p.k_tile[0] = p.k_tile[2] = moe::kShrinkSlice;
    p.stages[0] = p.stages[2] = 1;
  }
  const int64_t P = d->T * d->k;
  const AlignLayout al = align_layout(d);
  p.launches_route_align = P == 0 ? 1 : fused_route_align(d, al) ? 1 : al.nchunks == 1 ? 2 : 4;
  // gather (+ its token-order copy when x outgrows L2), shrinks, gate_up (+ SiLU pass
  // after a K split), down, combine
  p.launches_forward =
      d->T == 0 ? 0 : 4 + (moe::gather_token_order(d->T, d->H) ? 1 : 0) + (lora ? 2 : 0) + (l.ks_gu > 1 ? 1 : 0);
  *out = p;
  return MOE_LORA_OK;
}

int moe_lora_align_capacity(const moe_lora_dims* d, int64_t* max_rows, int64_t* max_blocks, int64_t* max_runs) {
  MOE_RESOLVE(d);
  MOE_TRY(validate_dims(d));
  const Caps c = capacity(d);
  if (max_rows) *max_rows = c.rows;
  if (max_blocks) *max_blocks = c.blocks;
  if (max_runs) *max_runs = c.runs;
  return MOE_LORA_OK;
}

int moe_lora_workspace_size(const moe_lora_dims* d, size_t* align_bytes, size_t* forward_bytes) {
  MOE_RESOLVE(d);
  MOE_TRY(validate_dims(d));
  if (align_bytes) *align_bytes = align_layout(d).bytes;
  if (forward_bytes) *forward_bytes = fwd_layout(d).bytes;
  return MOE_LORA_OK;
}

int moe_lora_layer_workspace_size(const moe_lora_dims* d, size_t* bytes) {
  MOE_RESOLVE(d);
  MOE_TRY(validate_dims(d));
  if (!bytes) return fail(MOE_LORA_EINVAL, "bytes is NULL");
  *bytes = layer_layout(d).bytes;
  return MOE_LORA_OK;
}

int moe_lora_route(const float* logits, int64_t T, int32_t E, int32_t k, int32_t* topk_ids, float* topk_w,
                   void* stream) {
  return do_route(logits, T, E, k, topk_ids, topk_w, static_cast<cudaStream_t>(stream));
}

int moe_lora_align(const moe_lora_dims* d, const int32_t* topk_ids, const int32_t* lora_ids,
                   const moe_lora_align_buf* out, void* workspace, size_t workspace_bytes, void* stream) {
  return do_align(d, topk_ids, lora_ids, out, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

int moe_lora_route_align(const moe_lora_dims* d, const float* logits, const int32_t* lora_ids, int32_t* topk_ids,
                         float* topk_w, const moe_lora_align_buf* out, void* workspace, size_t workspace_bytes,
                         void* stream) {
  return do_route_align(d, logits, lora_ids, topk_ids, topk_w, out, workspace, workspace_bytes,
                        static_cast<cudaStream_t>(stream));
}

int moe_lora_forward(const moe_lora_dims* d, const uint16_t* x, const float* topk_w,
                     const moe_lora_align_buf* aligned, const uint16_t* W_gu, const uint16_t* W_dn,
                     const uint16_t* A_gu, const uint16_t* B_gu, const uint16_t* A_dn, const uint16_t* B_dn,
                     uint16_t* out, void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream,
                     void* const* stage_events) {
  return do_forward(d, x, topk_w, aligned, W_gu, W_dn, A_gu, B_gu, A_dn, B_dn, out, workspace, workspace_bytes,
                    dev_status, static_cast<cudaStream_t>(stream), stage_events);
}

}  // extern "C"

namespace {
// Host buffers the kernels read or write in place instead of through a copy: pinned and
// mapped (cudaHostAlloc, cudaHostRegister) at the same address on both sides, as pinned
// memory is under unified addressing on a coherent CPU-GPU link, and 16-byte aligned
// (the kernels touch them in 16-byte vectors).  Both ends of the range are checked, so
// a buffer registered only in part takes the copy.  Up to kInPlaceMaxBytes: a copy node
// costs a few microseconds whatever its size, while a kernel reading or writing through
// the link runs longer the more it moves; past a few MB the copy engines win.
constexpr size_t kInPlaceMaxBytes = 4u << 20;
// x in place up to 1 MB of gather reads: measured through the captured layer, a
// 16-token decode batch (369 KB of reads) gained 2 us over the copy.
constexpr size_t kInPlaceMaxGatherBytes = 1u << 20;
bool in_place(const void* p, size_t bytes) {
  if (!p || bytes == 0 || bytes > kInPlaceMaxBytes || !aligned16(p)) return false;
  const char* ends[2] = {static_cast<const char*>(p), static_cast<const char*>(p) + bytes - 1};
  for (const char* q : ends) {
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, q) != cudaSuccess) {
      (void)cudaGetLastError();   // an unknown pointer is not an error of this call
      return false;
    }
    if (a.type != cudaMemoryTypeHost || a.devicePointer != static_cast<const void*>(q)) return false;
  }
  return true;
}

// Which host buffers of a layer call the kernels touch in place.  Decided before any
// stream capture (the pointer queries are not stream work).
struct InPlace {
  bool logits = false, lora = false, x = false, out = false;
};
InPlace in_place_of(const moe_lora_dims* d, const float* logits_host, const int32_t* lora_ids_host,
                    const uint16_t* x_host, const uint16_t* out_host) {
  InPlace ip;
  if (d->T <= 0) return ip;
  const size_t T = (size_t)d->T;
  ip.logits = in_place(logits_host, T * d->E * 4);
  ip.lora = in_place(lora_ids_host, T * 4);
  // the gather reads a token's row once per pair: k times its bytes over the link
  ip.x = T * d->H * 2 * d->k <= kInPlaceMaxGatherBytes && in_place(x_host, T * d->H * 2);
  ip.out = in_place(out_host, T * d->H * 2);
  return ip;
}

// Enqueues the layer_host sequence on s without synchronising: inputs in (copied, or
// read in place), route+align, forward, out back (written in place, or copied) and one
// copy of the 32-byte record {status, unused[3], totals[4]} into status8_dst (host int32[8]).
int layer_enqueue(const moe_lora_dims* d, const float* logits_host, const int32_t* lora_ids_host,
                  const uint16_t* x_host, const uint16_t* W_gu, const uint16_t* W_dn, const uint16_t* A_gu,
                  const uint16_t* B_gu, const uint16_t* A_dn, const uint16_t* B_dn, uint16_t* out_host,
                  void* workspace, size_t workspace_bytes, int32_t* status8_dst, const InPlace& ip,
                  cudaStream_t s) {
  MOE_TRY(validate_dims(d));
  const LayerLayout l = layer_layout(d);
  MOE_TRY(check_ptr(workspace, "workspace", true));
  if (workspace_bytes < l.bytes) return fail(MOE_LORA_EWORKSPACE, "layer workspace %zu < %zu bytes", workspace_bytes, l.bytes);
  if (d->T > 0) {
    MOE_TRY(check_ptr(logits_host, "logits_host", false));
    MOE_TRY(check_ptr(lora_ids_host, "lora_ids_host", false));
    MOE_TRY(check_ptr(x_host, "x_host", false));
    MOE_TRY(check_ptr(out_host, "out_host", false));
  }
  uint8_t* b = static_cast<uint8_t*>(workspace);
  float* logits = reinterpret_cast<float*>(b + l.logits);
  int32_t* lora = reinterpret_cast<int32_t*>(b + l.lora);
  uint16_t* x = reinterpret_cast<uint16_t*>(b + l.x);
  int32_t* ids = reinterpret_cast<int32_t*>(b + l.ids);
  float* w = reinterpret_cast<float*>(b + l.w);
  uint16_t* out = reinterpret_cast<uint16_t*>(b + l.out);
  int32_t* status = reinterpret_cast<int32_t*>(b + l.status);   // [0] status, [4..7] align totals
  moe_lora_align_buf al{reinterpret_cast<int32_t*>(b + l.sp), reinterpret_cast<int32_t*>(b + l.eb),
                        reinterpret_cast<int32_t*>(b + l.be), reinterpret_cast<int32_t*>(b + l.br),
                        reinterpret_cast<int32_t*>(b + l.runs), status + 4};
  const size_t T = (size_t)d->T;
  if (T > 0) {
    const size_t lb = T * d->E * 4, rb = T * 4, xb = T * d->H * 2;
    const float* lg = logits;
    const int32_t* lr = lora;
    const uint16_t* xi = x;
    if (ip.logits) lg = logits_host;
    else MOE_CUDA(cudaMemcpyAsync(logits, logits_host, lb, cudaMemcpyHostToDevice, s));
    if (ip.lora) lr = lora_ids_host;
    else MOE_CUDA(cudaMemcpyAsync(lora, lora_ids_host, rb, cudaMemcpyHostToDevice, s));
    if (ip.x) xi = x_host;
    else MOE_CUDA(cudaMemcpyAsync(x, x_host, xb, cudaMemcpyHostToDevice, s));
    uint16_t* o = ip.out ? out_host : out;
    MOE_TRY(do_route_align(d, lg, lr, ids, w, &al, b + l.align, l.fwd - l.align, s));
    MOE_TRY(do_forward(d, xi, w, &al, W_gu, W_dn, A_gu, B_gu, A_dn, B_dn, o, b + l.fwd, l.logits - l.fwd, status, s,
                       nullptr));
    if (o == out) MOE_CUDA(cudaMemcpyAsync(out_host, out, xb, cudaMemcpyDeviceToHost, s));
  } else {
    MOE_TRY(do_align(d, ids, lora, &al, b + l.align, l.fwd - l.align, s));
    MOE_TRY(do_forward(d, x, w, &al, W_gu, W_dn, A_gu, B_gu, A_dn, B_dn, out, b + l.fwd, l.logits - l.fwd, status, s,
                       nullptr));
  }
  MOE_CUDA(cudaMemcpyAsync(status8_dst, status, 32, cudaMemcpyDeviceToHost, s));
  return MOE_LORA_OK;
}
}  // namespace

struct moe_lora_graph {
  cudaGraphExec_t exec = nullptr;
  int32_t* status_host = nullptr;   // {status, unused[3], totals[4]}, copied in by each run
};

extern "C" {

int moe_lora_layer_host(const moe_lora_dims* d, const float* logits_host, const int32_t* lora_ids_host,
                        const uint16_t* x_host, const uint16_t* W_gu, const uint16_t* W_dn, const uint16_t* A_gu,
                        const uint16_t* B_gu, const uint16_t* A_dn, const uint16_t* B_dn, uint16_t* out_host,
                        void* workspace, size_t workspace_bytes, int64_t* dropped, void* stream) {
  MOE_RESOLVE(d);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t rec[8] = {0, 0, 0, 0, 0, 0, 0, 0};   // {status, unused[3], totals[4]}
  MOE_TRY(validate_dims(d));
  const InPlace ip = in_place_of(d, logits_host, lora_ids_host, x_host, out_host);
  MOE_TRY(layer_enqueue(d, logits_host, lora_ids_host, x_host, W_gu, W_dn, A_gu, B_gu, A_dn, B_dn, out_host,
                        workspace, workspace_bytes, rec, ip, s));
  MOE_CUDA(cudaStreamSynchronize(s));
  if (dropped) *dropped = rec[4 + 3];
  if (rec[0] != 0) return fail(MOE_LORA_EDEVICE, "device status 0x%x", rec[0]);
  return MOE_LORA_OK;
}

int moe_lora_layer_graph_create(const moe_lora_dims* d, const float* logits_host, const int32_t* lora_ids_host,
                                const uint16_t* x_host, const uint16_t* W_gu, const uint16_t* W_dn,
                                const uint16_t* A_gu, const uint16_t* B_gu, const uint16_t* A_dn,
                                const uint16_t* B_dn, uint16_t* out_host, int32_t* status_host, void* workspace,
                                size_t workspace_bytes, void* stream, moe_lora_graph** graph) {
  MOE_RESOLVE(d);
  if (!graph) return fail(MOE_LORA_EINVAL, "graph is NULL");
  *graph = nullptr;
  MOE_TRY(check_ptr(status_host, "status_host", false));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (!s) return fail(MOE_LORA_EINVAL, "graph capture needs a non-default stream");
  // one eager run: validation, the in-place decisions and the kernels' one-time
  // set-up happen outside the capture
  MOE_TRY(validate_dims(d));
  const InPlace ip = in_place_of(d, logits_host, lora_ids_host, x_host, out_host);
  MOE_TRY(layer_enqueue(d, logits_host, lora_ids_host, x_host, W_gu, W_dn, A_gu, B_gu, A_dn, B_dn, out_host,
                        workspace, workspace_bytes, status_host, ip, s));
  MOE_CUDA(cudaStreamSynchronize(s));
  if (status_host[0] != 0) return fail(MOE_LORA_EDEVICE, "device status 0x%x", status_host[0]);
  cudaGraph_t g = nullptr;
  MOE_CUDA(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
  const int st = layer_enqueue(d, logits_host, lora_ids_host, x_host, W_gu, W_dn, A_gu, B_gu, A_dn, B_dn, out_host,
                               workspace, workspace_bytes, status_host, ip, s);
  const cudaError_t ce = cudaStreamEndCapture(s, &g);
  if (st != MOE_LORA_OK) {
    if (g) cudaGraphDestroy(g);
    return st;
  }
  if (ce != cudaSuccess) return cuda_fail(ce, "cudaStreamEndCapture");
  cudaGraphExec_t exec = nullptr;
  const cudaError_t ie = cudaGraphInstantiate(&exec, g, 0);
  cudaGraphDestroy(g);
  if (ie != cudaSuccess) return cuda_fail(ie, "cudaGraphInstantiate");
  moe_lora_graph* h = new (std::nothrow) moe_lora_graph;
  if (!h) {
    cudaGraphExecDestroy(exec);
    return fail(MOE_LORA_EINVAL, "out of host memory");
  }
  h->exec = exec;
  h->status_host = status_host;
  *graph = h;
  return MOE_LORA_OK;
}

int moe_lora_layer_graph_run(moe_lora_graph* graph, void* stream, int64_t* dropped) {
  if (!graph || !graph->exec) return fail(MOE_LORA_EINVAL, "graph is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  MOE_CUDA(cudaGraphLaunch(graph->exec, s));
  MOE_CUDA(cudaStreamSynchronize(s));
  if (dropped) *dropped = graph->status_host[4 + 3];
  if (graph->status_host[0] != 0) return fail(MOE_LORA_EDEVICE, "device status 0x%x", graph->status_host[0]);
  return MOE_LORA_OK;
}

int moe_lora_layer_graph_destroy(moe_lora_graph* graph) {
  if (!graph) return MOE_LORA_OK;
  cudaError_t e = graph->exec ? cudaGraphExecDestroy(graph->exec) : cudaSuccess;
  delete graph;
  if (e != cudaSuccess) return cuda_fail(e, "cudaGraphExecDestroy");
  return MOE_LORA_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// moe_lora_align_static: align with its scratch in a static device array, for
// callers that cannot allocate device memory when they call.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_static_scratch[MOE_LORA_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
struct StaticScratchEntry {
  void* ptr = nullptr;
  unsigned long long ctx_id = 0;   // driver id of the context the address belongs to
};
StaticScratchEntry g_static[kMaxDevices];

PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_id = nullptr;
std::once_flag g_ctx_once;

// Unique id of the calling thread's current context (0 if there is none yet).  A
// context created after a cudaDeviceReset, or another context on the same device,
// loads the module anew and the array may sit elsewhere, so the cache is keyed on it.
unsigned long long current_ctx_id() {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(fn);
  });
  if (!g_ctx_current || !g_ctx_id) return 0;
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  unsigned long long id = 0;
  if (g_ctx_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of g_static_scratch in the current device's current context.  (In
// host code the array's name is only a host-side stand-in.)  The address is looked up
// once per (device, context): the first call on a device, and the first call after
// its context was replaced, do the look-up.
int static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(MOE_LORA_EUNSUPPORTED, "device ordinal %d >= %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_static_mu);
  StaticScratchEntry& ent = g_static[dev];
  const unsigned long long id = current_ctx_id();
  if (!ent.ptr || id == 0 || id != ent.ctx_id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);   // creates the context if needed
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    if (!p) return fail(MOE_LORA_ECUDA, "cudaGetSymbolAddress(static scratch) returned NULL");
    ent.ptr = p;
    ent.ctx_id = current_ctx_id();
  }
  *out = ent.ptr;
  return MOE_LORA_OK;
}

}  // namespace

extern "C" int moe_lora_align_static(const moe_lora_dims* d, const int32_t* topk_ids, const int32_t* lora_ids,
                                     const moe_lora_align_buf* out, void* stream) {
  MOE_RESOLVE(d);
  MOE_TRY(validate_dims(d));
  const size_t need = align_layout(d).bytes;
  if (need > MOE_LORA_STATIC_SCRATCH_BYTES)
    return fail(MOE_LORA_EWORKSPACE, "align needs %zu bytes of scratch; the static scratch holds %u", need,
                MOE_LORA_STATIC_SCRATCH_BYTES);
  MOE_TRY(check_device());
  void* scratch = nullptr;
  MOE_TRY(static_scratch(&scratch));
  return do_align(d, topk_ids, lora_ids, out, scratch, MOE_LORA_STATIC_SCRATCH_BYTES,
                  static_cast<cudaStream_t>(stream));
}
