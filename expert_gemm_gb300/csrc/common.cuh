// common.cuh -- types shared by the host orchestration and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/moe_lora.h"

namespace moe {

// Which stage of the layer one grouped-GEMM launch computes.
enum GemmMode : int {
  kShrink = 0,   // S_run = X_block * A[a,e]^T       (gate_up_shrink / down_shrink)
  kGateUp = 1,   // h = silu(gate) * up, gate/up = X W_gu[e]^T + S_run B_gu[a,e] (gate_up + expand)
  kDown = 2,     // y[row] = h W_dn[e]^T + S_run B_dn[a,e]                      (down + expand)
};

constexpr int kKTile = 64;      // K elements per pipeline stage (one 128-byte swizzle row of bf16)

// K elements per pipeline stage of a GEMM launch; host tensor maps use the same value.
// Token-tiled gate_up/down may be compiled with 32 (64-byte rows, 64-byte swizzle,
// twice the stages in the same shared memory); measured on GB300 the 64-wide stages
// of the persistent kernel are faster, so 64 is the default everywhere.
#ifndef MOE_TOKEN_TILED_BK
#define MOE_TOKEN_TILED_BK 64
#endif
constexpr int gemm_bk(int mode, int block_m) {
  return (block_m >= 128 && mode != kShrink) ? MOE_TOKEN_TILED_BK : kKTile;
}
constexpr int kRankChunk = 16;  // LoRA rank elements per MMA K-step

// Parameters of one grouped-GEMM launch (passed by value, read-only on the device).
struct GemmParams {
  const int32_t* block_expert;  // [blocks]
  const int32_t* expert_begin;  // [E+1] first sorted row of each expert
  const int32_t* block_runs;    // [blocks+1]
  const int32_t* runs;          // [runs][4] {block, adapter, begin, end}
  const int32_t* totals;        // {rows, blocks, runs, dropped}
  const int32_t* sorted_p;      // [rows]
  uint16_t* h_out;              // kGateUp: h rows in sorted order [rows][I] (bf16)
  void* y_out;                  // kDown: expert outputs of the real rows in sorted order,
                                //   [rows][H] bf16 (ksplit 1) or [ksplit][part_rows][H] fp32 partials
  float* g_part;                // kGateUp with K splits: [ksplit][part_rows][2I] fp32 partial pre-activations
  int64_t part_rows;            // row stride between the K splits' partial buffers
  float* s_part;                // kShrink with K splits: [ksplit][max_runs][BT][r_pad] fp32 partials
  int32_t* s_cnt;               // kShrink with K splits: [max_runs] splits finished per run (zero at launch)
  int32_t max_runs;
  uint16_t* s_out;              // kShrink: [runs][BT][r_pad] (bf16), rows outside the run zero
  int32_t* status;              // device status word (MOE_LORA_DEV_* bits)
  uint64_t acc_wait_ns;         // limit of the single-CTA epilogue's accumulator wait (test hook;
                                //   the default limit otherwise)
  int32_t K;                    // reduction length of the base GEMM (H or I)
  int32_t n_feat;               // output features (I for kGateUp, H for kDown)
  int32_t E;
  int32_t k;
  int32_t P;                    // T*k, the padding sentinel
  int32_t r_pad;                // S row length (r_max rounded up to 16)
  int32_t* tile_ctr;            // tile counter of this launch (zero at launch; persistent CTAs take tiles)
  int32_t n_ft;                 // feature tiles per token block (kGateUp, kDown)
  int32_t ksplit;               // K splits; each split stores its own partial sums
  int32_t lora_after_pdl;       // previous kernel is the shrink: wait for it only before the LoRA K-steps
  // kShrink on token-tiled blocks: the rank-chunk groups (128-row unit, first chunk) of
  // the block-diagonal shrink tiles and their count, built by the gather launch
  const int32_t* plan_block;
  const int32_t* plan_c0;
  const int32_t* plan_count;
  int32_t shrink_gch;           // rank chunks per group of those tiles
  int32_t ranks[MOE_LORA_MAX_ADAPTERS];
};

// Tensor maps of one grouped-GEMM launch.
struct GemmMaps {
  CUtensorMap w;      // base weights (W_gu 4D / W_dn 3D / A 3D)
  CUtensorMap tok;    // token rows in sorted order (x_sorted / h_sorted) 2D
  CUtensorMap lw;     // LoRA expand weights, rank-major (B_gu 5D / B_dn 4D)
  CUtensorMap ls;     // S run tiles 3D
  CUtensorMap out;    // CTA-pair gate_up / down: output rows (h_sorted / y, bf16) 2D, box {64, 32}
  CUtensorMap w_rank[3];   // kShrink: A with boxes of 32, 48 and 64 rank rows (w: 16), so a
                           //   stage loads its adapter's ranks with one TMA
};

// Launchers (defined next to their kernels).
cudaError_t launch_route(const float* logits, int64_t T, int E, int k, int32_t* ids, float* w,
                         cudaStream_t s);

struct AlignLaunch {
  const int32_t* topk_ids;
  const int32_t* lora_ids;
  int64_t P;
  int k, E, L, BM;
  int ch_log2;                 // log2 of the chunk size
  int nchunks;
  uint32_t* chunk_keys;        // [nchunks << ch_log2]
  int32_t* counts;             // [nchunks][E*(L+1)]
  int32_t* chunk_invalid;      // [nchunks]
  int32_t* bucket_total;       // [E*(L+1)]
  int32_t* bucket_base;        // [E*(L+1)]
  int32_t* run_base;           // [E*(L+1)]
  int32_t* expert_n;           // [E]
  moe_lora_align_buf out;
};
cudaError_t launch_align(const AlignLaunch& a, cudaStream_t s);
// Route + align in one single-CTA launch; only for a.nchunks == 1 (T*k <= 4096).
// a.topk_ids is ignored: the routed ids are written to topk_ids.
cudaError_t launch_route_align_small(const AlignLaunch& a, const float* logits, float* topk_w, int32_t* topk_ids,
                                     cudaStream_t s);

// Whether the gather copies in token order (a second launch that reads each x row once).
inline bool gather_token_order(int64_t T, int H) { return T * static_cast<int64_t>(H) * 2 > (int64_t(64) << 20); }
// Gathers x rows into sorted order (in token order when gather_token_order), records
// the sorted row of every placed pair in
// pair_row [T*k], and zeroes *status and the n_ctr tile counters of the forward's
// GEMM launches.
// The group table of the block-diagonal shrink of token-tiled blocks.  A unit is 128
// rows: a 128-row block, or one half of a 256-row block.  The rank chunks of the
// adapter runs that reach a unit, in run order, are cut into groups of `gch` chunks;
// group g is (plan_block[g] = its unit b * (block_m / 128) + half, plan_c0[g] = its
// first chunk inside the unit), groups in unit order, plan_count[0] groups in all.
// block_chunks is [units] scratch.
constexpr int kShrinkGroupChunks = 16;   // the most chunks of a group (N = 256)
struct ShrinkPlanArgs {
  const int32_t* block_runs;   // [blocks+1]
  const int32_t* runs;         // [runs][4]
  int32_t* block_chunks;
  int32_t* plan_block;
  int32_t* plan_c0;
  int32_t* plan_count;
  int32_t block_m;             // 128 or 256
  int32_t gch;                 // rank chunks per group, 1 .. kShrinkGroupChunks
  int32_t ranks[MOE_LORA_MAX_ADAPTERS];
};
// plan: when non-null, one extra CTA of the launch builds the group table (it reads
// only the align outputs, so it overlaps the row copies).
cudaError_t launch_gather_rows(const uint16_t* x, const int32_t* sorted_p, const int32_t* totals, int64_t max_rows,
                               int H, int k, int P, uint16_t* x_sorted, int32_t* pair_row, int32_t* status,
                               int32_t* ctr, int n_ctr, const ShrinkPlanArgs* plan, cudaStream_t s);
// out[t] = bf16(sum_j topk_w[t,j] * y(row of pair t*k+j)) in a fixed order; y is bf16
// [rows][H] when ksplit == 1, else fp32 partials [ksplit][part_rows][H] summed in order.
cudaError_t launch_combine(const void* y, int ksplit, int64_t part_rows, const int32_t* pair_row,
                           const int32_t* sorted_p, const int32_t* totals, const float* topk_w, int64_t T, int k,
                           int H, uint16_t* out, bool pdl, cudaStream_t s);
// h = bf16(silu(g[:, :I]) * g[:, I:]) for the live sorted rows after a K-split gate_up,
// g being the sum of the ksplit partial buffers [ksplit][part_rows][2I] in split order.
cudaError_t launch_silu_rows(const float* g_part, int ksplit, int64_t part_rows, const int32_t* totals,
                             int64_t max_rows, int I, uint16_t* h, bool pdl, cudaStream_t s);
// LoRA shrink of short runs on CUDA cores (weight-streaming blocks, block_m <= 64):
// one CTA per (run, kShrinkSlice-wide K slice); fp32 slice partials added in slice
// order by the CTA that completes the run's count (s_cnt[4 * run], zero at launch).
constexpr int kShrinkSlice = 256;
struct ShrinkRowsLaunch {
  const uint16_t* xs;           // token rows in sorted order [rows][K]
  const uint16_t* A;            // [L*E][r_max][K]
  const int32_t* runs;          // [runs][4] {block, adapter, begin, end}
  const int32_t* block_expert;  // [blocks]
  const int32_t* totals;        // {rows, blocks, runs, dropped}
  float* s_part;                // [slices][max_runs][block_m][r_pad] fp32
  int32_t* s_cnt;               // [max_runs][4]
  uint16_t* s_out;              // [runs][block_m][r_pad] bf16
  int32_t K, E, r_max, r_pad, block_m, slices, max_runs;
  int32_t ranks[MOE_LORA_MAX_ADAPTERS];
};
cudaError_t launch_shrink_rows(const ShrinkRowsLaunch& a, int64_t max_runs, bool pdl, cudaStream_t s);
// pdl: launch with programmatic stream serialisation (may overlap the previous kernel).
// block_diag (kShrink, bt 128 only): the block-diagonal shrink, whose tiles are the
// group table's entries (prm.plan_*, built by the gather launch of the same forward).
// deep (kGateUp / kDown, bt 16 only): the variant with a 6-deep ring, one CTA per SM.
cudaError_t launch_gemm(int mode, int bt, const GemmMaps& maps, const GemmParams& prm, int64_t max_blocks,
                        int64_t max_runs, bool pdl, cudaStream_t s, bool block_diag = false, bool deep = false);
// K elements per pipeline stage and stage count of the compiled GEMM for (mode, bt);
// false if no kernel is compiled for it.  Host only, no device calls.
bool gemm_stage_shape(int mode, int bt, int* k_tile, int* stages, bool deep = false);

}  // namespace moe
