// gemm_tc.cuh -- grouped expert GEMM on the 5th-generation tensor core (tcgen05 + TMEM),
// fed by TMA, for the three GEMM-shaped steps of the MoE-LoRA layer:
//
//   kShrink : S_run = X_block * A[a,e]^T           LoRA shrink of gate_up or down
//   kGateUp : g = X W_gu[e]^T (+ S_run B_gu[a,e] per adapter run), h = silu(g_gate) * g_up
//   kDown   : d = H W_dn[e]^T (+ S_run B_dn[a,e] per adapter run), stored per sorted row
//
// The LoRA expand is not a separate kernel: every adapter run of a token block adds
// ceil(rank/16) extra K-steps (packed BK/16 per pipeline stage) to the same TMEM
// accumulator, with the run's S tile (rows outside the run are zero) as the
// token-side operand and B[a,e] as the weight-side operand.  SiLU gating happens in
// the epilogue that drains TMEM; the down epilogue stores each real row's output with
// plain stores and a separate pass combines a token's k rows in a fixed order (no
// atomics anywhere, so repeated calls give identical bytes).  This is the pages'
// fusion of the LoRA add into the expand kernel (AWS ML Blog "Efficiently serve
// dozens of fine-tuned models with vLLM on Amazon SageMaker AI and Amazon Bedrock",
// section "Kernel optimizations") taken one step further: base GEMM, expand and
// epilogue share one accumulator.
//
// Two tile orientations (template SWAP):
//   SWAP = false (token blocks of 128 or 256 rows): MMA M = 128 tokens per accumulator
//          (MT = BT/128 accumulators), N = 256 weight rows (gate_up: 128 gate + 128 up
//          rows of the same features; down: 256 features); 256-row gate_up / down tiles
//          run on CTA pairs (M = 256), the shrink of 256-row blocks takes one 128-row
//          half per tile.  The shrink's N is the rank rows of one adapter run, or (BD)
//          of a group of runs side by side.
//   SWAP = true  (token blocks of 16/32/64 rows, few tokens per expert): MMA M = 128
//          weight rows, N = BT tokens; two accumulators (gate/up, or two feature halves).
//          Weights stream through the tensor core at full tile height however few
//          tokens an expert has.
//
// Persistent CTAs (one per SM, or as many as fit): each CTA takes tiles from a
// global counter until none are left, so per-CTA set-up is paid once, the TMA ring
// runs on from one tile into the next, and with two TMEM accumulator buffers the
// epilogue of one tile overlaps the MMAs of the next.  Warp roles (224 threads):
//   warp 0    TMA producer;
//   warp 1    TMEM owner and MMA issuer;
//   warps 2-5 epilogue (warp w drains TMEM lanes 32*(w%4) .. +31);
//   warp 6    tile scheduler: takes the next tile id, decodes it with all 32 lanes
//             (the block's adapter runs are looked up in parallel) and publishes it
//             through a small shared ring to the other roles.  It claims tile i + 1
//             when the producer is a few stages from the end of tile i, so the
//             decode's chain of dependent loads is off the producer's path while the
//             claim stays late enough for the dynamic balance across CTAs.  In a CTA
//             pair the even CTA's scheduler claims and hands each id to the odd CTA's
//             through shared::cluster, so both take the same tiles.
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {

template <int MODE, bool SWAP, int BT, bool BD = false, bool DEEP = false>
struct GemmCfg {
  static constexpr bool kLora = MODE != kShrink;
  // BD: the block-diagonal shrink of 128-row token blocks: a tile is one group of up to
  // 16 rank chunks of the block's adapter runs, N = their ranks side by side, so a
  // stage brings up to 32 KB of A rows (the HBM stream) per 16 KB of token rows.  Its
  // tiles come from the group table the gather launch builds.
  static constexpr bool BDIAG = BD;
  static_assert(!BD || (MODE == kShrink && !SWAP && (BT == 128 || BT == 256)),
                "block-diagonal tiles: the shrink of token-tiled blocks");
  // DEEP: the 16-token weight-streaming gate_up / down with a 6-deep ring (one CTA per
  // SM), for batches of a few pairs whose tiles are fewer than the CTAs
  static_assert(!DEEP || (SWAP && BT == 16 && MODE != kShrink), "deep ring: 16-token weight-streaming GEMMs");
  // 256-token blocks of gate_up / down run on a CTA pair (a cluster of 2): one 2-SM
  // MMA of M = 256 tokens x N = 256 weight rows per K-step; each CTA stages its own
  // 128 token rows and half of the weight rows, and holds its tokens' accumulator.
  static constexpr bool CTA2 = !SWAP && BT == 256 && MODE != kShrink;
  // The shrink of 256-row blocks takes a run's block in 128-row halves, one tile each:
  // most runs sit in one half, and an M = 256 tile would spend half its MMAs and token
  // loads on rows outside the run.  A half the run does not reach is a tile without
  // K-steps that writes the half's S rows as zeros.
  static constexpr bool HALF = MODE == kShrink && !SWAP && BT == 256;
  static constexpr int TROWS = CTA2 || HALF ? 128 : BT;   // token rows staged by this CTA
  static constexpr int BK = gemm_bk(MODE, BT);        // K elements per stage
  static constexpr int ROWB = BK * 2;                 // bytes of one staged row = swizzle span
  static constexpr uint32_t SW = BK == 64 ? kSw128 : kSw64;
  static constexpr uint32_t SBO = 8 * ROWB;           // bytes between 8-row core groups
  static constexpr int CPS = BK / kRankChunk;         // LoRA rank chunks per stage
  // weight-side rows staged per K-tile (a shrink's A: rank <= 64 rows, so the weight-
  // streaming shrink issues M = 64 MMAs over them)
  static constexpr int WROWS = MODE == kShrink ? (BDIAG ? 256 : 64) : (CTA2 ? 128 : 256);
  static constexpr int WM = SWAP ? (MODE == kShrink ? 64 : 128) : 0;   // MMA M of weight-streaming tiles
  static constexpr int W_BYTES = WROWS * ROWB;
  static constexpr int T_BYTES = TROWS * ROWB;
  static constexpr int STAGE_BYTES = W_BYTES + T_BYTES;
  // (16-token weight-streaming tiles: 3 stages, so two CTAs share an SM and a GEMM CTA
  // fits beside a shrink CTA -- measured faster on the decode shapes; 32/64: 5)
  // (weight-streaming shrink: 10-16 KB stages, 8 deep, 6 for 64-token tiles)
  static constexpr int STAGES = MODE == kShrink ? (SWAP ? (BT <= 32 ? 8 : 6) : 4)
                                : SWAP           ? (BT <= 16 ? (DEEP ? 6 : 3) : 5)
                                : CTA2           ? 6   // + 16 KB of output staging
                                                 : (192 * 1024) / STAGE_BYTES;
  // accumulators: non-swapped MT tiles of M=128 tokens x N; swapped NH tiles of 128 x BT
  static constexpr int NH = MODE == kShrink ? 1 : 2;
  static constexpr int MT = SWAP ? 1 : TROWS / 128;
  static constexpr int NACC = MODE == kShrink && !BDIAG ? 64 : 256;   // columns of one non-swapped accumulator
  static constexpr int ACC_COLS = SWAP ? NH * BT : MT * NACC;
  static constexpr int NBUF = 2 * ACC_COLS <= 512 ? 2 : 1;  // TMEM accumulator buffers
  static constexpr int TMEM_NEED = NBUF * ACC_COLS;
  static constexpr int TMEM_COLS =
      TMEM_NEED <= 32 ? 32 : TMEM_NEED <= 64 ? 64 : TMEM_NEED <= 128 ? 128 : TMEM_NEED <= 256 ? 256 : 512;
  static constexpr int SD = 4;                              // tile-id ring depth
  // CTA pairs stage their bf16 output rows in shared memory and write them with TMA
  // stores: per epilogue warp one buffer of 32 rows x 64 columns (4 KB).  (A second
  // buffer per warp costs a pipeline stage: 5 stages with two, 6 with one; the sixth
  // stage is worth more -- prefill 3.81 -> 3.76 ms.)
  static constexpr bool TMA_STORE = CTA2;
  static constexpr int OUT_BYTES = TMA_STORE ? 4 * 4096 : 0;
  static constexpr int SMEM_BYTES =
      STAGES * STAGE_BYTES + OUT_BYTES + 1024 /*align slack*/ + 4096 /*barriers, tile ring*/;
  static_assert(!SWAP || (BT == 16 || BT == 32 || BT == 64), "swapped tiles take 16/32/64 tokens");
  static_assert(SWAP || BT == 128 || BT == 256, "token-tiled blocks are 128 or 256 rows");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
  static_assert(W_BYTES % 1024 == 0 && T_BYTES % 1024 == 0, "stage regions keep 1024-byte alignment");
  static_assert(STAGES >= 2 && STAGES <= 8, "pipeline depth");
  static_assert(!kLora || CPS * (WROWS + TROWS) * 32 <= STAGE_BYTES, "LoRA chunks of a stage fit its slot");
};

// One unit of work.  kShrink: one adapter run.  kGateUp / kDown: one (K split, token
// block, feature tile), feature tile fastest, K split slowest.  Weight-streaming gate_up
// and down split K when their tiles are too few for the SMs; every split stores its own
// fp32 partial sums, added in split order by the pass after the kernel.
// The producer decodes each tile once and publishes it in the shared ring, so the
// MMA and epilogue warps never wait on the global routing metadata.
constexpr int kMaxBlockRuns = 256;   // runs of one block <= its rows <= 256
struct TileHdr {
  int tau;                // tile id; >= the live count ends the CTA's loop
  int b, e, row0, f0;
  int run0, nruns;        // adapter runs of the block (last K split only)
  int kb0, nk;            // base K-tiles of this split
  int n_it;               // pipeline stages of this tile
  int srun, sa, snch;     // kShrink: run, adapter, rank chunks
  int ks;                 // K split of this tile
};
// Block-diagonal shrink: the part of one adapter run inside a tile's chunk group.
struct ShrinkSeg {
  int32_t run;        // run index (its S tile)
  int16_t ad;         // adapter
  int16_t beg, end;   // the run's rows inside the block
  int16_t rank;       // the adapter's rank
  uint8_t cl;         // first chunk of the run in this tile
  uint8_t n;          // chunks of the run in this tile
  uint8_t pos;        // tile-local chunk of chunk cl (its A rows and accumulator columns)
  uint8_t other;      // 256-row blocks: the run has no rows in the other half, whose S rows
                      //   of these chunks this tile writes as zeros
};
static_assert(sizeof(ShrinkSeg) == 16, "segment layout");
static_assert(kShrinkGroupChunks * sizeof(ShrinkSeg) <= kMaxBlockRuns, "segments fit the run-chunk array");
struct Tile {
  TileHdr h;                               // copied to registers by every reader
  alignas(16) uint8_t nch[kMaxBlockRuns];  // rank chunks of each adapter run of the block
                                           //   (block-diagonal shrink: ShrinkSeg[16] instead)
  int16_t ad[kMaxBlockRuns];               // adapter of each run (the producer's LoRA loads)
};
__device__ __forceinline__ ShrinkSeg* tile_segs(uint8_t* nch) { return reinterpret_cast<ShrinkSeg*>(nch); }
__device__ __forceinline__ const ShrinkSeg* tile_segs(const uint8_t* nch) {
  return reinterpret_cast<const ShrinkSeg*>(nch);
}

struct GemmBars {
  uint64_t full[8];          // stage loaded (TMA transaction bytes)
  uint64_t empty[8];         // stage consumed (MMA commit)
  uint64_t acc_full[2];      // accumulator buffer ready for the epilogue (MMA commit)
  uint64_t acc_empty[2];     // accumulator buffer drained (one arrive per epilogue warp)
  uint64_t sched_full[4];    // tile id published (producer)
  uint64_t sched_empty[4];   // tile id read (MMA thread + one arrive per epilogue warp)
  uint64_t sched_req;        // the producer is near the end of its tile: claim the next
  uint64_t tau_full[4];      // CTA pairs: the even CTA has written the pair's next tile id here
  int32_t tau_val[4];
  uint64_t drain;            // all MMAs of this CTA finished (teardown)
  uint32_t tmem_base;
  int32_t abort;
  Tile tiles[4];             // the tile ring (published with sched_full)
};
constexpr int kBarBytes = 4096;
static_assert(sizeof(GemmBars) <= kBarBytes, "barrier block");

__device__ __forceinline__ void record_timeout(GemmBars* bars, int32_t* status) {
  atomicOr(status, MOE_LORA_DEV_TIMEOUT);
  *reinterpret_cast<volatile int32_t*>(&bars->abort) = 1;
}
__device__ __forceinline__ bool aborted(GemmBars* bars) {
  return *reinterpret_cast<volatile int32_t*>(&bars->abort) != 0;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}
// silu(z) = z / (1 + e^-z) with the fast approximate divide (a few ulp; the result is
// rounded to bf16): the epilogue's instruction count competes with the MMA issuer.
__device__ __forceinline__ float silu_f(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

template <int MODE, bool SWAP, int BT, bool BD>
__device__ __forceinline__ int live_tiles(const GemmParams& prm) {
  if constexpr (BD) return *prm.plan_count;
  else if constexpr (MODE == kShrink) return prm.totals[2] * prm.ksplit * (GemmCfg<MODE, SWAP, BT>::HALF ? 2 : 1);
  else return prm.totals[1] * prm.n_ft * prm.ksplit;
}

// Called by all 32 lanes of the scheduler warp with the same tau; every lane returns
// the same header, and lane j writes the chunk count and adapter of runs j, j + 32, ...
template <int MODE, bool SWAP, int BT, bool BD>
__device__ __forceinline__ TileHdr decode_tile(int tau, const GemmParams& prm, uint8_t* nch_out, int16_t* ad_out,
                                               int workers, int lane) {
  using C = GemmCfg<MODE, SWAP, BT, BD>;
  TileHdr t;
  t.tau = tau;
  const int nk_all = prm.K / C::BK;
  t.run0 = 0;
  t.nruns = 0;
  t.f0 = 0;
  t.srun = t.sa = t.snch = 0;
  if constexpr (C::BDIAG) {
    // group tau: chunks [c0, c0 + gch) of the runs that reach one 128-row unit (a block,
    // or a half of a 256-row block), in run order.  The lanes take 32 runs at a time:
    // each its chunk count if it reaches the unit, a warp scan places its chunks, and
    // the runs overlapping the group become the tile's segments.
    constexpr int UPB = BT / 128;
    const int u = prm.plan_block[tau];
    const int c0 = prm.plan_c0[tau];
    const int gch = prm.shrink_gch;
    const int b = u / UPB, half = u - b * UPB;
    const int rb = prm.block_runs[b], re = prm.block_runs[b + 1];
    t.b = b;
    t.e = prm.block_expert[b];
    t.row0 = b * BT + 128 * half;
    // the other half's rows, relative to this unit's first row
    const int oth_lo = half == 0 ? 128 : -128, oth_hi = oth_lo + 128;
    t.ks = 0;
    t.kb0 = 0;
    t.nk = nk_all;
    t.n_it = nk_all;
    t.run0 = rb;
    ShrinkSeg* seg = tile_segs(nch_out);
    int carry = 0, nseg = 0, nch = 0;
    for (int r0 = rb; r0 < re && carry < c0 + gch; r0 += 32) {
      const int j = r0 + lane;
      int a = 0, n = 0, beg = 0, end = 0;
      if (j < re) {
        a = prm.runs[4 * j + 1];
        beg = prm.runs[4 * j + 2] - t.row0;
        end = prm.runs[4 * j + 3] - t.row0;
        if (beg < 128 && end > 0) n = (prm.ranks[a] + kRankChunk - 1) / kRankChunk;   // reaches the unit
      }
      int incl = n;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      const int cs = carry + incl - n;   // the block-local chunk where run j starts
      const int lo = cs > c0 ? cs : c0;
      const int hi = cs + n < c0 + gch ? cs + n : c0 + gch;
      const bool take = j < re && lo < hi;
      const uint32_t m = __ballot_sync(0xffffffffu, take);
      if (take) {
        ShrinkSeg sg;
        sg.run = j;
        sg.ad = static_cast<int16_t>(a);
        sg.beg = static_cast<int16_t>(beg);
        sg.end = static_cast<int16_t>(end);
        sg.rank = static_cast<int16_t>(prm.ranks[a]);
        sg.cl = static_cast<uint8_t>(lo - cs);
        sg.n = static_cast<uint8_t>(hi - lo);
        sg.pos = static_cast<uint8_t>(lo - c0);
        sg.other = UPB == 2 && !(beg < oth_hi && end > oth_lo);
        seg[nseg + __popc(m & ((1u << lane) - 1u))] = sg;
      }
      nseg += __popc(m);
      nch += __reduce_add_sync(0xffffffffu, take ? hi - lo : 0);
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    t.nruns = nseg;
    t.snch = nch;
    return t;
  } else if constexpr (C::HALF) {
    // run tau / 2, half tau % 2 of its 256-row block (no K split on token-tiled blocks)
    t.srun = tau >> 1;
    t.ks = 0;
    t.b = prm.runs[4 * t.srun + 0];
    t.sa = prm.runs[4 * t.srun + 1];
    const int beg = prm.runs[4 * t.srun + 2], end = prm.runs[4 * t.srun + 3];
    t.snch = (prm.ranks[t.sa] + kRankChunk - 1) / kRankChunk;
    t.kb0 = 0;
    t.nk = nk_all;
    t.e = prm.block_expert[t.b];
    t.row0 = t.b * BT + 128 * (tau & 1);
    t.n_it = beg < t.row0 + 128 && end > t.row0 ? nk_all : 0;   // 0: the half is zeros only
    return t;
  } else if constexpr (MODE == kShrink) {
    // the K splits of one run are consecutive tiles
    t.srun = tau / prm.ksplit;
    t.ks = tau % prm.ksplit;
    t.b = prm.runs[4 * t.srun + 0];
    t.sa = prm.runs[4 * t.srun + 1];
    t.snch = (prm.ranks[t.sa] + kRankChunk - 1) / kRankChunk;
    t.kb0 = t.ks * nk_all / prm.ksplit;
    t.nk = (t.ks + 1) * nk_all / prm.ksplit - t.kb0;
    t.n_it = t.nk;
  } else {
    // Order: K split slowest; then expert by expert; inside an expert, groups of G
    // feature tiles, and inside a group block-major.  The blocks of one expert then
    // share each group's weight tiles while they are resident in L2 (an expert's whole
    // weight matrix can exceed L2); G * (the expert's blocks) ~ the concurrent workers.
    // One block per expert (decode) gives G = n_ft: feature tile fastest.
    const int nb = prm.totals[1];
    const int per_split = nb * prm.n_ft;
    const int ks = tau / per_split;
    const int rest = tau - ks * per_split;
    const int e = prm.block_expert[rest / prm.n_ft];   // an expert's tiles are its blocks' tiles
    const int blk0 = prm.expert_begin[e] / BT;
    const int nbe = prm.expert_begin[e + 1] / BT - blk0;
    const int local = rest - blk0 * prm.n_ft;
    int G = workers / nbe;
    if (G < 1) G = 1;
    if (G > prm.n_ft) G = prm.n_ft;
    const int full = (prm.n_ft / G) * G;           // feature tiles in whole groups
    int ft, bl;
    if (local < full * nbe) {
      const int g = local / (G * nbe), r = local - g * (G * nbe);
      bl = r / G;
      ft = g * G + (r - bl * G);
    } else {
      const int Gl = prm.n_ft - full, r = local - full * nbe;
      bl = r / Gl;
      ft = full + (r - bl * Gl);
    }
    t.b = blk0 + bl;
    t.ks = ks;
    t.f0 = ft * (MODE == kGateUp ? 128 : 256);
    // The LoRA K-steps ride on the last K split: its tiles come last in the tile order,
    // so they reach the S tiles after the shrink kernel before has finished.
    if (ks == prm.ksplit - 1) {
      t.run0 = prm.block_runs[t.b];
      t.nruns = prm.block_runs[t.b + 1] - t.run0;
    }
    t.kb0 = ks * nk_all / prm.ksplit;
    t.nk = (ks + 1) * nk_all / prm.ksplit - t.kb0;
    int chunks = 0;
    for (int r = lane; r < t.nruns; r += 32) {
      const int a = prm.runs[4 * (t.run0 + r) + 1];
      const int nch = (prm.ranks[a] + kRankChunk - 1) / kRankChunk;
      nch_out[r] = static_cast<uint8_t>(nch);
      ad_out[r] = static_cast<int16_t>(a);
      chunks += nch;
    }
    chunks = __reduce_add_sync(0xffffffffu, chunks);
    // the runs' rank chunks fill the LoRA stages back to back, CPS per stage
    t.n_it = t.nk + (chunks + C::CPS - 1) / C::CPS;
    t.snch = chunks;
    t.e = e;   // block t.b is one of expert e's blocks
    t.row0 = t.b * BT;
    return t;
  }
  t.e = prm.block_expert[t.b];
  t.row0 = t.b * BT;
  return t;
}

// Tile of ring slot i (stays valid until the slot is released); null if the wait gave up.
__device__ __forceinline__ const Tile* sched_read(GemmBars* bars, int i, int32_t* status) {
  const int slot = i & 3;
  if (!mbar_wait(&bars->sched_full[slot], (i >> 2) & 1)) {
    record_timeout(bars, status);
    return nullptr;
  }
  return &bars->tiles[slot];
}

// Output staging of the CTA-pair epilogues: epilogue warp q owns one 4 KB buffer of
// 32 rows x 128 bytes (64 bf16 columns) in the 128-byte-swizzled layout of a TMA box
// {64, 32}; lane i writes row i.  Before the buffer is reused, the store issued from
// it must have read it.
__device__ __forceinline__ uint8_t* stage_out_buffer(uint8_t* out_stage, int q, int lane, int n_out) {
  if (n_out >= 1) {
    if (lane == 0) bulk_wait_read<0>();   // the previous store has read the buffer
    __syncwarp();
  }
  return out_stage + q * 4096;
}
// 16-byte chunks j and j + 1 of row `lane` (chunk j holds columns 8j .. 8j + 7).
__device__ __forceinline__ void put_row_chunks(uint8_t* buf, int lane, int j, const uint32_t (&pk)[8]) {
  uint8_t* row = buf + lane * 128;
  *reinterpret_cast<uint4*>(row + ((j ^ (lane & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  *reinterpret_cast<uint4*>(row + (((j + 1) ^ (lane & 7)) << 4)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
}
// Makes the warp's staged rows visible to the async proxy and stores them at (col, row).
__device__ __forceinline__ void store_out_chunk(const CUtensorMap* map, const uint8_t* buf, int lane, int col,
                                                int row, int& n_out) {
  fence_proxy_async_smem();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(map, buf, col, row);
    bulk_commit();
  }
  ++n_out;
}

constexpr int kGemmThreads = 224;
constexpr int kSchedWarp = 6;
// The producer asks for the next tile this many stages before the end of its tile.
constexpr int kClaimAhead = 6;

template <int MODE, bool SWAP, int BT, bool BD, bool DEEP>
__global__ void __launch_bounds__(kGemmThreads, 1)
    moe_gemm_kernel(const __grid_constant__ GemmMaps maps, const __grid_constant__ GemmParams prm) {
  using C = GemmCfg<MODE, SWAP, BT, BD, DEEP>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = C::CTA2 ? cluster_ctarank() : 0u;   // 0: issues the pair's MMAs

  // Ordering with the previous kernel of the stream (programmatic dependent launch):
  // the shrink reads token rows written by it, so it waits before anything else and
  // then lets its dependent (the GEMM that consumes its S tiles) start; the GEMMs
  // wait at the start unless their only input from the previous kernel is the S tiles
  // of the LoRA K-steps, in which case the producer waits just before loading them.
  if constexpr (MODE == kShrink) {
    pdl_wait();
    pdl_trigger();
  } else {
    if (!prm.lora_after_pdl) pdl_wait();
    pdl_trigger();
  }
  // The routing metadata comes from align, complete before the previous kernel began.
  const int n_live = live_tiles<MODE, SWAP, BT, BD>(prm);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* out_stage = smem + C::STAGES * C::STAGE_BYTES;   // 1024-aligned (C::OUT_BYTES)
  GemmBars* bars = reinterpret_cast<GemmBars*>(out_stage + C::OUT_BYTES);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int j = 0; j < 2; ++j) {
      mbar_init(&bars->acc_full[j], 1);
      mbar_init(&bars->acc_empty[j], C::CTA2 ? 8 : 4);   // a pair: both CTAs' epilogue warps
    }
    for (int j = 0; j < C::SD; ++j) {
      mbar_init(&bars->sched_full[j], 1);
      mbar_init(&bars->sched_empty[j], 1 + 1 + 4);   // producer, MMA issuer, epilogue warps
    }
    mbar_init(&bars->sched_req, 1);
    for (int j = 0; j < 4; ++j) mbar_init(&bars->tau_full[j], 1);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    if constexpr (C::CTA2) {
      tmem_alloc_pair(&bars->tmem_base, C::TMEM_COLS);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&bars->tmem_base, C::TMEM_COLS);
      tmem_relinquish();
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if constexpr (C::CTA2) cluster_sync();   // the peer's barriers exist before any remote arrival
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&maps.w);
      tma_prefetch_desc(&maps.tok);
      if constexpr (MODE == kShrink)
        for (int j = 0; j < 3; ++j) tma_prefetch_desc(&maps.w_rank[j]);
      if constexpr (C::kLora) {
        tma_prefetch_desc(&maps.lw);
        tma_prefetch_desc(&maps.ls);
      }
      bool waited_pdl = false;
      int gs = 0;        // stages issued by this CTA (continues across tiles)
      int pst = 0;       // gs % STAGES
      uint32_t pph = 0;  // (gs / STAGES) & 1
      for (int i = 0;; ++i) {
        const Tile* tp = sched_read(bars, i, prm.status);
        if (!tp) break;
        const int slot = i & 3;
        const TileHdr t = tp->h;   // registers; the slot (runs' adapters and chunks) is released after the tile
        if (t.tau >= n_live) {
          mbar_arrive(&bars->sched_empty[slot]);
          break;
        }
        const int claim_at = t.n_it > kClaimAhead ? t.n_it - kClaimAhead : 0;
        bool claimed = false;
        int lr = 0, lc = 0;   // LoRA run and first rank chunk of the next LoRA stage
        bool ok = true;
        for (int it = 0; it < t.n_it; ++it) {
          const int s = pst;
          const uint32_t ph = pph;
          if (it == claim_at) {
            mbar_arrive(&bars->sched_req);
            claimed = true;
          }
          if (aborted(bars)) {
            ok = false;
            break;
          }
          if (!(C::CTA2 ? mbar_wait_cluster(&bars->empty[s], ph ^ 1) : mbar_wait(&bars->empty[s], ph ^ 1))) {
            record_timeout(bars, prm.status);
            ok = false;
            break;
          }
          uint8_t* wdst = smem + s * C::STAGE_BYTES;
          uint8_t* tdst = wdst + C::W_BYTES;
          uint64_t* fb = &bars->full[s];
          // a pair's loads all complete on the even CTA's barrier, which expects both halves
          const uint32_t fb_pair = C::CTA2 ? mapa_shared(fb, 0) : 0u;
          if (C::CTA2 && it < t.nk) {
            const int k0 = (t.kb0 + it) * C::BK;
            if (rank == 0) mbar_arrive_expect_tx(fb, 2 * (C::W_BYTES + C::T_BYTES));
            if constexpr (MODE == kGateUp)
              tma_load_4d_pair(wdst, &maps.w, fb_pair, k0, t.f0, static_cast<int>(rank), t.e);  // gate | up rows
            else
              tma_load_3d_pair(wdst, &maps.w, fb_pair, k0, t.f0 + 128 * static_cast<int>(rank), t.e);
            tma_load_2d_pair(tdst, &maps.tok, fb_pair, k0, t.row0 + 128 * static_cast<int>(rank));
          } else if (it < t.nk) {
            const int k0 = (t.kb0 + it) * C::BK;
            if constexpr (MODE == kGateUp) {
              mbar_arrive_expect_tx(fb, C::W_BYTES + C::T_BYTES);
              tma_load_4d(wdst, &maps.w, fb, k0, t.f0, 0, t.e);                  // gate rows
              tma_load_4d(wdst + 128 * C::ROWB, &maps.w, fb, k0, t.f0, 1, t.e);  // up rows
            } else if constexpr (MODE == kDown) {
              mbar_arrive_expect_tx(fb, C::W_BYTES + C::T_BYTES);
              tma_load_3d(wdst, &maps.w, fb, k0, t.f0, t.e);
              tma_load_3d(wdst + 128 * C::ROWB, &maps.w, fb, k0, t.f0 + 128, t.e);
            } else if constexpr (C::BDIAG) {
              // each segment's rank rows in one box, at its tile-local chunk
              const ShrinkSeg* seg = tile_segs(bars->tiles[slot].nch);
              mbar_arrive_expect_tx(fb, t.snch * kRankChunk * C::ROWB + C::T_BYTES);
              for (int sgi = 0; sgi < t.nruns; ++sgi) {
                const ShrinkSeg sg = seg[sgi];
                tma_load_3d(wdst + sg.pos * kRankChunk * C::ROWB, sg.n <= 1 ? &maps.w : &maps.w_rank[sg.n - 2], fb,
                            k0, sg.cl * kRankChunk, sg.ad * prm.E + t.e);
              }
            } else {
              // the adapter's rank rows in one box: the producer thread's issue loop, not
              // the bytes, paces the shrink's stages
              const int ae = t.sa * prm.E + t.e;
              mbar_arrive_expect_tx(fb, t.snch * kRankChunk * C::ROWB + C::T_BYTES);
              tma_load_3d(wdst, t.snch <= 1 ? &maps.w : &maps.w_rank[t.snch - 2], fb, k0, 0, ae);
            }
            tma_load_2d(tdst, &maps.tok, fb, k0, t.row0);
          } else if constexpr (C::kLora) {
            if (!waited_pdl && prm.lora_after_pdl) {   // S tiles come from the previous kernel
              pdl_wait();
              waited_pdl = true;
            }
            // up to CPS rank chunks, continuing across run boundaries; chunk j of the
            // stage: run lr, chunk lc of that run
            const Tile& tl = bars->tiles[slot];
            const int left = t.snch - (it - t.nk) * C::CPS;
            const int nc = left < C::CPS ? left : C::CPS;
            if constexpr (C::CTA2) {
              if (rank == 0) mbar_arrive_expect_tx(fb, 2 * nc * (C::WROWS * 32 + C::TROWS * 32));
            } else {
              mbar_arrive_expect_tx(fb, nc * (C::WROWS * 32 + C::TROWS * 32));
            }
            for (int j = 0; j < nc; ++j) {
              const int run = t.run0 + lr;
              const int ae = tl.ad[lr] * prm.E + t.e;
              const int c = lc;
              uint8_t* wc = wdst + j * (C::WROWS * 32);
              uint8_t* tc = tdst + j * (C::TROWS * 32);
              // weight side: 16 rank rows of B (rank-major) as 64-column atoms; one box
              // holds the tile's columns (gate_up: gate then up), a pair CTA's half
              if constexpr (C::CTA2) {
                const int rk = static_cast<int>(rank);
                if constexpr (MODE == kGateUp)
                  tma_load_5d_pair(wc, &maps.lw, fb_pair, 0, c * kRankChunk, t.f0 / 64, rk, ae);
                else
                  tma_load_4d_pair(wc, &maps.lw, fb_pair, 0, c * kRankChunk, (t.f0 + 128 * rk) / 64, ae);
                tma_load_3d_pair(tc, &maps.ls, fb_pair, c * kRankChunk, 128 * rk, run);
              } else {
                if constexpr (MODE == kGateUp)
                  tma_load_5d(wc, &maps.lw, fb, 0, c * kRankChunk, t.f0 / 64, 0, ae);
                else
                  tma_load_4d(wc, &maps.lw, fb, 0, c * kRankChunk, t.f0 / 64, ae);
                tma_load_3d(tc, &maps.ls, fb, c * kRankChunk, 0, run);
              }
              if (++lc == tl.nch[lr]) {
                lc = 0;
                ++lr;
              }
            }
          }
          ++gs;
          if (++pst == C::STAGES) {
            pst = 0;
            pph ^= 1;
          }
        }
        if (!claimed) mbar_arrive(&bars->sched_req);   // the scheduler waits for one request per tile
        mbar_arrive(&bars->sched_empty[slot]);
        if (!ok) break;
      }
      // Leave no copy in flight after an abort: wait (bounded) for the last stages issued.
      // (In a pair the even CTA's barriers count both CTAs' copies; the odd CTA stays
      // resident until the closing cluster barrier, after the even CTA has drained.)
      if (aborted(bars) && rank == 0) {
        for (int g = gs - C::STAGES < 0 ? 0 : gs - C::STAGES; g < gs; ++g)
          (void)mbar_wait_cluster(&bars->full[g % C::STAGES], (g / C::STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (C::CTA2 && lane == 0 && rank != 0) {
      // The odd CTA of a pair issues no MMA (the even CTA's 2-SM MMAs fill its TMEM);
      // it only hands its ring slots back.
      for (int i = 0;; ++i) {
        const Tile* tp = sched_read(bars, i, prm.status);
        if (!tp) break;
        const int tau = tp->h.tau;
        mbar_arrive(&bars->sched_empty[i & 3]);
        if (tau >= n_live) break;
      }
    } else if (lane == 0) {
      // pair (2-SM) or single-CTA MMA, and commits that reach both CTAs of a pair
      auto mma = [&](uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accum) {
        if constexpr (C::CTA2) tc_mma_pair(d, a, b, idesc, accum);
        else tc_mma(d, a, b, idesc, accum);
      };
      auto commit = [&](uint64_t* bar) {
        if constexpr (C::CTA2) tc_commit_pair(bar, 0x3);
        else tc_commit(bar);
      };
      constexpr int kM = C::CTA2 ? 256 : 128;
      // stage-0 descriptors: base K-steps (128/64-byte swizzle rows); LoRA K-steps: S
      // K-major in 32-byte rows, B MN-major (64-column atoms of 16 rank rows, 2 KB apart)
      const uint32_t sbase = smem_u32(smem);
      const uint64_t dW = smem_desc(sbase, C::SBO, C::SW), dT = smem_desc(sbase + C::W_BYTES, C::SBO, C::SW);
      const uint64_t dWl = smem_desc_mn128(sbase, 2048), dTl = smem_desc(sbase + C::W_BYTES, 256, kSw32);
      int st = 0;          // stage of the next K-step (continues across tiles)
      uint32_t sph = 0;    // its phase parity
      for (int i = 0;; ++i) {
        const Tile* tp = sched_read(bars, i, prm.status);
        if (!tp) break;
        const TileHdr t = tp->h;   // registers; the slot (run chunk counts) is released after the tile
        if (t.tau >= n_live || aborted(bars)) {
          mbar_arrive(&bars->sched_empty[i & 3]);
          break;
        }
        const int ab = i % C::NBUF;
        const uint32_t eph = ((i / C::NBUF) & 1) ^ 1;
        if (!(C::CTA2 ? mbar_wait_cluster(&bars->acc_empty[ab], eph) : mbar_wait(&bars->acc_empty[ab], eph))) {
          record_timeout(bars, prm.status);
          break;
        }
        tc_fence_after_sync();
        const uint32_t acc_base = tmem + ab * C::ACC_COLS;
        // instruction descriptors of this tile's base and LoRA K-steps
        const uint32_t id_base = SWAP ? idesc_bf16_f32(C::WM, BT)
                                      : idesc_bf16_f32(kM, MODE == kShrink ? t.snch * kRankChunk : 256);
        constexpr uint32_t id_lora =
            SWAP ? (idesc_bf16_f32(128, BT) | kIdescAMn) : (idesc_bf16_f32(kM, 256) | kIdescBMn);
        uint32_t acc = 0;
        bool ok = true;
        // The hot loop issues from one thread: descriptors are the stage-0 ones plus
        // constant offsets (16-byte units), stage and phase advance by increment, and
        // no flag is polled (every wait is bounded, and a failed one ends the loop).
        for (int it = 0; it < t.n_it; ++it) {
          if (!(C::CTA2 ? mbar_wait_cluster(&bars->full[st], sph) : mbar_wait(&bars->full[st], sph))) {
            record_timeout(bars, prm.status);
            ok = false;
            break;
          }
          tc_fence_after_sync();
          const uint64_t so = static_cast<uint64_t>(st) * (C::STAGE_BYTES >> 4);
          if (it < t.nk) {
#pragma unroll
            for (int kk = 0; kk < C::BK / 16; ++kk) {
              const uint64_t ko = so + static_cast<uint64_t>(kk * 2);   // 32 bytes of K per step
              if constexpr (!SWAP) {
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt)
                  mma(acc_base + mt * C::NACC, dT + ko + static_cast<uint64_t>(mt * 8 * C::ROWB), dW + ko, id_base,
                      acc);
              } else {
#pragma unroll
                for (int h = 0; h < C::NH; ++h)
                  tc_mma(acc_base + h * BT, dW + ko + static_cast<uint64_t>(h * 8 * C::ROWB), dT + ko, id_base, acc);
              }
              acc = 1;
            }
          } else if constexpr (C::kLora) {
            // up to CPS rank chunks, of one or several runs (each chunk: its own S and B)
            const int left = t.snch - (it - t.nk) * C::CPS;
            const int nc = left < C::CPS ? left : C::CPS;
            for (int c = 0; c < nc; ++c) {
              const uint64_t wo = so + static_cast<uint64_t>(c * (C::WROWS * 2));   // WROWS x 32 bytes
              const uint64_t to = so + static_cast<uint64_t>(c * (C::TROWS * 2));
              if constexpr (!SWAP) {
#pragma unroll
                for (int mt = 0; mt < C::MT; ++mt)
                  mma(acc_base + mt * C::NACC, dTl + to + static_cast<uint64_t>(mt * 256), dWl + wo, id_lora, 1);
              } else {
#pragma unroll
                for (int h = 0; h < C::NH; ++h)
                  tc_mma(acc_base + h * BT, dWl + wo + static_cast<uint64_t>(h * 256), dTl + to, id_lora, 1);
              }
            }
          }
          commit(&bars->empty[st]);
          if (++st == C::STAGES) {
            st = 0;
            sph ^= 1;
          }
        }
        commit(&bars->acc_full[ab]);   // also after an abort, so the epilogue is released
        mbar_arrive(&bars->sched_empty[i & 3]);
        if (!ok) break;
      }
      commit(&bars->drain);   // arrives once every MMA issued above has completed
    }
  } else if (warp == kSchedWarp) {
    // ------------------------------------------------------------ tile scheduler
    // n_live = no more work.  Both CTAs of a pair must take the same tiles: the even
    // CTA claims each from the counter and writes its id into the odd CTA's ring, whose
    // scheduler waits for it.  (A fixed stride of tiles per pair let slow pairs fall
    // behind the feature group whose weights the others kept in L2.)
    const int workers = C::CTA2 ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);
    for (int i = 0;; ++i) {
      const int slot = i & 3;
      int tau = n_live;
      if (lane == 0) {
        // tile i > 0 once the producer has asked for it; the slot once its last tile is
        // done (the odd CTA of a pair follows the even CTA's claims instead)
        bool ok = i == 0 || (C::CTA2 && rank != 0) || mbar_wait(&bars->sched_req, (i - 1) & 1);
        ok = ok && mbar_wait(&bars->sched_empty[slot], ((i >> 2) & 1) ^ 1);
        if (!ok) {
          record_timeout(bars, prm.status);
          tau = -1;
        } else if constexpr (C::CTA2) {
          if (rank == 0) {
            tau = aborted(bars) ? n_live : atomicAdd(prm.tile_ctr, 1);
            st_shared_cluster_u32(mapa_shared(&bars->tau_val[slot], 1), static_cast<uint32_t>(tau));
            mbar_arrive_cluster(mapa_shared(&bars->tau_full[slot], 1));   // release: the id is visible
          } else if (mbar_wait_cluster(&bars->tau_full[slot], (i >> 2) & 1)) {
            tau = *reinterpret_cast<volatile int32_t*>(&bars->tau_val[slot]);
          } else {
            record_timeout(bars, prm.status);
            tau = -1;
          }
        } else if (!aborted(bars)) {
          tau = atomicAdd(prm.tile_ctr, 1);
        }
      }
      tau = __shfl_sync(0xffffffffu, tau, 0);
      if (tau < 0) break;   // a wait gave up: the readers' own bounded waits end their loops
      TileHdr t;
      t.tau = n_live;
      if (tau < n_live) t = decode_tile<MODE, SWAP, BT, BD>(tau, prm, bars->tiles[slot].nch, bars->tiles[slot].ad,
                                                        workers, lane);
      __syncwarp();   // every lane's run entries are written before lane 0 publishes
      if (lane == 0) {
        bars->tiles[slot].h = t;
        mbar_arrive(&bars->sched_full[slot]);   // release: the tile fields are visible to the readers
      }
      if (tau >= n_live) break;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int m = q * 32 + lane;     // accumulator row (TMEM lane) of this thread
    int n_out = 0;                   // TMA stores issued by this warp (CTA pairs)
    for (int i = 0;; ++i) {
      const Tile* tp = sched_read(bars, i, prm.status);
      if (!tp) break;
      const TileHdr t = tp->h;   // registers; the slot is released after this tile's epilogue
      if (t.tau >= n_live) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->sched_empty[i & 3]);
        break;
      }
      const int ab = i % C::NBUF;
      const uint32_t fph = (i / C::NBUF) & 1;
      const bool got = C::CTA2 ? mbar_wait_cluster(&bars->acc_full[ab], fph)
                               : mbar_wait_for(&bars->acc_full[ab], fph, prm.acc_wait_ns);
      if (!got) record_timeout(bars, prm.status);
      tc_fence_after_sync();
      const bool ok = got && !aborted(bars);
      const uint32_t tq = tmem + ab * C::ACC_COLS + (static_cast<uint32_t>(q * 32) << 16);
      // first token row of this CTA's accumulator (a pair's odd CTA holds rows 128..255)
      const int row0 = t.row0 + 128 * static_cast<int>(rank), f0 = t.f0;
      if (ok) {
        uint32_t v[16], u[16];
        if constexpr (C::BDIAG) {
          // each segment's chunks: the run's rank columns of row m, zero outside the run
          // (256-row blocks: this half's rows of the run's S tile, and the other half's
          // as zeros when the run has none there)
          const ShrinkSeg* seg = tile_segs(tp->nch);
          const int hoff = row0 - t.b * BT;
          for (int sgi = 0; sgi < t.nruns; ++sgi) {
            const ShrinkSeg sg = seg[sgi];
            const bool in_run = m >= sg.beg && m < sg.end;
            uint16_t* srow = prm.s_out + (static_cast<size_t>(sg.run) * BT + hoff + m) * prm.r_pad;
            uint16_t* sother = prm.s_out + (static_cast<size_t>(sg.run) * BT + (BT - 128 - hoff) + m) * prm.r_pad;
            for (int c = 0; c < sg.n; ++c) {
              tmem_ld16(tq + (sg.pos + c) * kRankChunk, v);
              tmem_ld_wait();
              const int col0 = (sg.cl + c) * kRankChunk;   // rank column of the run
              uint32_t pk[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) {
                const int c2 = col0 + 2 * j;
                const float a0 = (in_run && c2 < sg.rank) ? __uint_as_float(v[2 * j]) : 0.f;
                const float a1 = (in_run && c2 + 1 < sg.rank) ? __uint_as_float(v[2 * j + 1]) : 0.f;
                pk[j] = pack_bf16x2(a0, a1);
              }
              uint4* dst = reinterpret_cast<uint4*>(srow + col0);
              dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
              dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
              if (sg.other) {
                uint4* zd = reinterpret_cast<uint4*>(sother + col0);
                zd[0] = make_uint4(0, 0, 0, 0);
                zd[1] = make_uint4(0, 0, 0, 0);
              }
            }
          }
        } else if constexpr (MODE == kShrink) {
          const int beg = prm.runs[4 * t.srun + 2] - row0;
          const int end = prm.runs[4 * t.srun + 3] - row0;
          const int r_a = prm.ranks[t.sa];
          // (a half tile of a 256-row block writes rows row0 - b*BT .. + 127 of the run's S tile)
          uint16_t* srun = prm.s_out + (static_cast<size_t>(t.srun) * BT + (row0 - t.b * BT)) * prm.r_pad;
          // weight-streaming (M = 64 accumulator): rank row mr sits in lane mr % 16 of
          // TMEM lane quarter mr / 16
          const int mr = lane < 16 ? 16 * q + lane : (1 << 30);
          if constexpr (!SWAP) {
            // row mt*128 + m of the token block; columns are ranks
            for (int mt = 0; mt < C::MT; ++mt) {
              const int row = mt * 128 + m;
              const bool in_run = row >= beg && row < end;
              for (int c = 0; c < prm.r_pad; c += 16) {
                if (c < t.snch * kRankChunk) {
                  tmem_ld16(tq + mt * C::NACC + c, v);
                  tmem_ld_wait();
                } else {
#pragma unroll
                  for (int j = 0; j < 16; ++j) v[j] = 0;
                }
                uint32_t pk[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                  const int c0 = c + 2 * j;
                  const float a0 = (in_run && c0 < r_a) ? __uint_as_float(v[2 * j]) : 0.f;
                  const float a1 = (in_run && c0 + 1 < r_a) ? __uint_as_float(v[2 * j + 1]) : 0.f;
                  pk[j] = pack_bf16x2(a0, a1);
                }
                uint4* dst = reinterpret_cast<uint4*>(srun + static_cast<size_t>(row) * prm.r_pad + c);
                dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
              }
            }
          } else if (prm.ksplit == 1) {
            // rank row mr; columns are the BT tokens of the block
            for (int n0 = 0; n0 < BT; n0 += 16) {
              tmem_ld16(tq + n0, v);
              tmem_ld_wait();
              if (mr < prm.r_pad) {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  const int n = n0 + j;
                  const float val = (n >= beg && n < end && mr < r_a) ? __uint_as_float(v[j]) : 0.f;
                  __nv_bfloat16 hv = __float2bfloat16_rn(val);
                  srun[static_cast<size_t>(n) * prm.r_pad + mr] = *reinterpret_cast<uint16_t*>(&hv);
                }
              }
            }
          } else {
            // K split: each epilogue warp owns 16 rank rows.  It stores this split's
            // fp32 partial S for them, then counts itself in on a per-(run, warp)
            // arrival counter; the warp that completes the count (no waiting) sums
            // all splits' partials and writes those rows of the bf16 S tile.
            // Partials: [split][run][BT][r_pad]; counters: [run][4].
            if (q * 16 < prm.r_pad) {
              const size_t part = (static_cast<size_t>(t.ks) * prm.max_runs + t.srun) * BT * prm.r_pad;
              for (int n0 = 0; n0 < BT; n0 += 16) {
                tmem_ld16(tq + n0, v);
                tmem_ld_wait();
                if (mr < prm.r_pad) {
#pragma unroll
                  for (int j = 0; j < 16; ++j)
                    prm.s_part[part + static_cast<size_t>(n0 + j) * prm.r_pad + mr] = __uint_as_float(v[j]);
                }
              }
              __threadfence();
              __syncwarp();
              int last = 0;
              if (lane == 0) last = atomicAdd(prm.s_cnt + 4 * t.srun + q, 1) == prm.ksplit - 1;
              last = __shfl_sync(0xffffffffu, last, 0);
              if (last) {
                __threadfence();
                if (mr < prm.r_pad) {
                  for (int n = 0; n < BT; ++n) {
                    float sum = 0.f;
                    for (int sp = 0; sp < prm.ksplit; ++sp)
                      sum += __ldcg(prm.s_part + (static_cast<size_t>(sp) * prm.max_runs + t.srun) * BT * prm.r_pad +
                                    static_cast<size_t>(n) * prm.r_pad + mr);
                    const float val = (n >= beg && n < end && mr < r_a) ? sum : 0.f;
                    __nv_bfloat16 hv = __float2bfloat16_rn(val);
                    srun[static_cast<size_t>(n) * prm.r_pad + mr] = *reinterpret_cast<uint16_t*>(&hv);
                  }
                }
              }
            }
          }
        } else if constexpr (MODE == kGateUp) {
          const int I = prm.n_feat;
          if constexpr (!SWAP) {
            for (int mt = 0; mt < C::MT; ++mt) {
              uint16_t* hrow = prm.h_out + static_cast<size_t>(row0 + mt * 128 + m) * I + f0;
              const uint32_t ta = tq + mt * C::NACC;
              for (int c0 = 0; c0 < 128; c0 += 64) {   // 64 features per TMEM wait (I % 64 == 0)
                if (f0 + c0 >= I) break;
                uint32_t g[4][16], up[4][16];
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                  tmem_ld16(ta + c0 + 16 * q4, g[q4]);          // gate features
                  tmem_ld16(ta + 128 + c0 + 16 * q4, up[q4]);   // up features
                }
                tmem_ld_wait();
                if constexpr (C::TMA_STORE) {
                  uint8_t* buf = stage_out_buffer(out_stage, q, lane, n_out);
#pragma unroll
                  for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t pk[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                      pk[j] = pack_bf16x2(silu_f(__uint_as_float(g[q4][2 * j])) * __uint_as_float(up[q4][2 * j]),
                                          silu_f(__uint_as_float(g[q4][2 * j + 1])) *
                                              __uint_as_float(up[q4][2 * j + 1]));
                    put_row_chunks(buf, lane, 2 * q4, pk);
                  }
                  store_out_chunk(&maps.out, buf, lane, f0 + c0, row0 + mt * 128 + q * 32, n_out);
                } else {
                  uint4* dst = reinterpret_cast<uint4*>(hrow + c0);
#pragma unroll
                  for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t pk[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                      pk[j] = pack_bf16x2(silu_f(__uint_as_float(g[q4][2 * j])) * __uint_as_float(up[q4][2 * j]),
                                          silu_f(__uint_as_float(g[q4][2 * j + 1])) *
                                              __uint_as_float(up[q4][2 * j + 1]));
                    dst[2 * q4] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                    dst[2 * q4 + 1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                  }
                }
              }
            }
          } else {
            const int f = f0 + m;           // feature of this thread; columns are tokens
            for (int n0 = 0; n0 < BT; n0 += 16) {
              tmem_ld16(tq + n0, v);
              tmem_ld16(tq + BT + n0, u);
              tmem_ld_wait();
              if (f < I) {
                if (prm.ksplit > 1) {
                  // K split: this split's fp32 pre-activations go to its own buffer; the
                  // SiLU pass adds the splits in order
                  float* gs = prm.g_part + (static_cast<size_t>(t.ks) * prm.part_rows + row0 + n0) * (2 * I);
#pragma unroll
                  for (int j = 0; j < 16; ++j) {
                    gs[static_cast<size_t>(j) * (2 * I) + f] = __uint_as_float(v[j]);
                    gs[static_cast<size_t>(j) * (2 * I) + I + f] = __uint_as_float(u[j]);
                  }
                } else {
#pragma unroll
                  for (int j = 0; j < 16; ++j) {
                    __nv_bfloat16 hv = __float2bfloat16_rn(silu_f(__uint_as_float(v[j])) * __uint_as_float(u[j]));
                    prm.h_out[static_cast<size_t>(row0 + n0 + j) * I + f] = *reinterpret_cast<uint16_t*>(&hv);
                  }
                }
              }
            }
          }
        } else {  // kDown: each real row's output to its own row of y (no combine here)
          const int H = prm.n_feat;
          uint16_t* y16 = static_cast<uint16_t*>(prm.y_out);
          float* y32 = static_cast<float*>(prm.y_out) + static_cast<size_t>(t.ks) * prm.part_rows * H;
          if constexpr (!SWAP) {
            if constexpr (C::TMA_STORE) {
              // 64 output features per TMA store; every row of the tile is written (a
              // padding row's output is never read).  One TMEM wait per 16 columns.
              for (int c0 = 0; c0 < 256; c0 += 64) {
                if (f0 + c0 >= H) break;
                uint8_t* buf = stage_out_buffer(out_stage, q, lane, n_out);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                  tmem_ld16(tq + c0 + 16 * q4, v);
                  tmem_ld_wait();
                  uint32_t pk[8];
#pragma unroll
                  for (int j = 0; j < 8; ++j) pk[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
                  put_row_chunks(buf, lane, 2 * q4, pk);
                }
                store_out_chunk(&maps.out, buf, lane, f0 + c0, row0 + q * 32, n_out);
              }
            } else
            for (int mt = 0; mt < C::MT; ++mt) {
              const int row = row0 + mt * 128 + m;
              const bool valid = prm.sorted_p[row] < prm.P;
              for (int c = 0; c < 256; c += 16) {
                if (f0 + c >= H) break;
                tmem_ld16(tq + mt * C::NACC + c, v);
                tmem_ld_wait();
                if (!valid) continue;
                if (prm.ksplit == 1) {
                  uint32_t pk[8];
#pragma unroll
                  for (int j = 0; j < 8; ++j) pk[j] = pack_bf16x2(__uint_as_float(v[2 * j]), __uint_as_float(v[2 * j + 1]));
                  uint4* dst = reinterpret_cast<uint4*>(y16 + static_cast<size_t>(row) * H + f0 + c);
                  dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                  dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
                } else {
                  float4* dst = reinterpret_cast<float4*>(y32 + static_cast<size_t>(row) * H + f0 + c);
#pragma unroll
                  for (int j = 0; j < 4; ++j)
                    dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                         __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
                }
              }
            }
          } else {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const int f = f0 + h * 128 + m;
              for (int n0 = 0; n0 < BT; n0 += 16) {
                tmem_ld16(tq + h * BT + n0, v);
                tmem_ld_wait();
                if (f >= H) continue;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                  const int row = row0 + n0 + j;
                  if (prm.sorted_p[row] >= prm.P) continue;
                  if (prm.ksplit == 1) {
                    __nv_bfloat16 hv = __float2bfloat16_rn(__uint_as_float(v[j]));
                    y16[static_cast<size_t>(row) * H + f] = *reinterpret_cast<uint16_t*>(&hv);
                  } else {
                    y32[static_cast<size_t>(row) * H + f] = __uint_as_float(v[j]);
                  }
                }
              }
            }
          }
        }
      }
      // release the accumulator buffer to the MMA warp and the tile slot to the producer
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (C::CTA2 && rank != 0) mbar_arrive_cluster(mapa_shared(&bars->acc_empty[ab], 0));
        else mbar_arrive(&bars->acc_empty[ab]);
        mbar_arrive(&bars->sched_empty[i & 3]);
      }
      if (!ok) break;
    }
  }

  if constexpr (C::TMA_STORE) {
    if (warp >= 2 && warp < kSchedWarp && lane == 0) bulk_wait_all();   // the epilogue's output stores have completed
  }
  __syncwarp();   // lanes of every warp reconverge before the CTA barrier
  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    // every MMA of this CTA (of a pair: of the even CTA, into both) has completed
    // before its TMEM is freed
    if (lane == 0) (void)(C::CTA2 ? mbar_wait_cluster(&bars->drain, 0) : mbar_wait(&bars->drain, 0));
    __syncwarp();
    if constexpr (C::CTA2) tmem_dealloc_pair(tmem, C::TMEM_COLS);
    else tmem_dealloc(tmem, C::TMEM_COLS);
  }
  // a pair: neither CTA leaves while the other may still arrive on its barriers or
  // have the MMA read its shared memory
  if constexpr (C::CTA2) cluster_sync();
}

template <int MODE, bool SWAP, int BT, bool BD = false, bool DEEP = false>
cudaError_t launch_gemm_t(const GemmMaps& maps, const GemmParams& prm, int64_t max_blocks, int64_t max_runs,
                          bool pdl, cudaStream_t s) {
  using C = GemmCfg<MODE, SWAP, BT, BD, DEEP>;
  auto kern = moe_gemm_kernel<MODE, SWAP, BT, BD, DEEP>;
  int64_t cap_tiles;
  // groups <= unit chunks / gch + units <= (BT / 128) * (runs + blocks) for gch >= 4
  if constexpr (C::BDIAG) cap_tiles = (BT / 128) * (max_runs + max_blocks);
  else if constexpr (MODE == kShrink) cap_tiles = max_runs * prm.ksplit * (C::HALF ? 2 : 1);
  else cap_tiles = max_blocks * prm.n_ft * prm.ksplit;
  if (cap_tiles <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;   // CTA pairs (used only by the 2-SM kernels)
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = C::CTA2 ? attr : attr + 1;
  cfg.numAttrs = (C::CTA2 ? 1 : 0) + (pdl ? 1 : 0);

  // Persistent grid: as many CTAs (CTA pairs) as fit on the device at once, no more
  // than tiles.  The attribute and the occupancy are settled on the first launch of
  // this kernel (per process: one device model), so later launches make no such calls.
  static int64_t max_ctas = 0;
  if (max_ctas == 0) {
    int dev = 0, sms = 0, occ = 0, smem_sm = 0, smem_rsv = 0;
    cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    // all of the unified L1/shared array as shared memory, so co-resident CTAs fit
    if (err == cudaSuccess)
      err = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (err == cudaSuccess) err = cudaGetDevice(&dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    if (err == cudaSuccess) err = cudaDeviceGetAttribute(&smem_rsv, cudaDevAttrReservedSharedMemoryPerBlock, dev);
    if (err != cudaSuccess) return err;
    if constexpr (C::CTA2) {
      // one pair per two SMs at most (a CTA needs all of its SM's TMEM)
      cudaLaunchConfig_t q = cfg;
      q.gridDim = dim3(static_cast<unsigned>(sms & ~1), 1, 1);
      q.numAttrs = 1;   // the cluster dimension only
      err = cudaOccupancyMaxActiveClusters(&occ, kern, &q);
      if (err != cudaSuccess) return err;
      if (occ < 1) occ = 1;
      if (occ > sms / 2) occ = sms / 2;
      max_ctas = 2 * static_cast<int64_t>(occ);
    } else {
      err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kGemmThreads, C::SMEM_BYTES);
      if (err != cudaSuccess) return err;
      // The query can answer for a smaller shared-memory carveout than the launch gets;
      // the CTAs that fit by shared memory, registers, threads and TMEM co-reside
      // (measured: two 99 KB shrink CTAs per SM run together, the query says one).
      cudaFuncAttributes fa{};
      err = cudaFuncGetAttributes(&fa, kern);
      if (err != cudaSuccess) return err;
      int fit = smem_sm / (C::SMEM_BYTES + smem_rsv);
      const int by_regs = fa.numRegs > 0 ? 65536 / (fa.numRegs * kGemmThreads) : fit;
      if (fit > by_regs) fit = by_regs;
      if (fit > 2048 / kGemmThreads) fit = 2048 / kGemmThreads;
      if (occ < fit) occ = fit;
      if (occ < 1) occ = 1;
      // co-resident CTAs share TMEM: keep their accumulators within its 512 columns
      while (occ > 1 && occ * C::TMEM_COLS > 512) --occ;
      max_ctas = static_cast<int64_t>(sms) * occ;
    }
  }
  int64_t grid = max_ctas;
  if constexpr (C::CTA2) {
    if (grid > 2 * cap_tiles) grid = 2 * cap_tiles;   // a pair per tile at most
  } else {
    if (grid > cap_tiles) grid = cap_tiles;
  }
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  return cudaLaunchKernelEx(&cfg, kern, maps, prm);
}

}  // namespace moe
