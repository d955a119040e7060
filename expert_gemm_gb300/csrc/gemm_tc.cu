// gemm_tc.cu -- instantiations of the tcgen05 grouped GEMM and the launch dispatch.
#include "gemm_tc.cuh"

namespace moe {

cudaError_t launch_gemm(int mode, int bt, const GemmMaps& maps, const GemmParams& prm, int64_t max_blocks,
                        int64_t max_runs, bool pdl, cudaStream_t s, bool block_diag, bool deep) {
  // the 16-token weight-streaming gate_up / down with a deeper ring
  if (deep) {
    if (bt != 16) return cudaErrorInvalidValue;
    if (mode == kGateUp) return launch_gemm_t<kGateUp, true, 16, false, true>(maps, prm, max_blocks, max_runs, pdl, s);
    if (mode == kDown) return launch_gemm_t<kDown, true, 16, false, true>(maps, prm, max_blocks, max_runs, pdl, s);
    return cudaErrorInvalidValue;
  }
  // the block-diagonal shrink of 128-row blocks: its own kernel, fed by the group table
  if (block_diag) {
    if (mode != kShrink) return cudaErrorInvalidValue;
    if (bt == 128) return launch_gemm_t<kShrink, false, 128, true>(maps, prm, max_blocks, max_runs, pdl, s);
    if (bt == 256) return launch_gemm_t<kShrink, false, 256, true>(maps, prm, max_blocks, max_runs, pdl, s);
    return cudaErrorInvalidValue;
  }
#define MOE_GEMM_CASE(BT_, SWAP_)                                                                       \
  if (bt == BT_) {                                                                                      \
    switch (mode) {                                                                                     \
      case kShrink: return launch_gemm_t<kShrink, SWAP_, BT_>(maps, prm, max_blocks, max_runs, pdl, s);     \
      case kGateUp: return launch_gemm_t<kGateUp, SWAP_, BT_>(maps, prm, max_blocks, max_runs, pdl, s);     \
      case kDown: return launch_gemm_t<kDown, SWAP_, BT_>(maps, prm, max_blocks, max_runs, pdl, s);         \
      default: return cudaErrorInvalidValue;                                                            \
    }                                                                                                   \
  }
  MOE_GEMM_CASE(16, true)
  MOE_GEMM_CASE(32, true)
  MOE_GEMM_CASE(64, true)
  MOE_GEMM_CASE(128, false)
  MOE_GEMM_CASE(256, false)
#undef MOE_GEMM_CASE
  return cudaErrorInvalidValue;
}

bool gemm_stage_shape(int mode, int bt, int* k_tile, int* stages, bool deep) {
  if (deep && bt == 16 && mode != kShrink) {
    *k_tile = GemmCfg<kGateUp, true, 16, false, true>::BK;
    *stages = GemmCfg<kGateUp, true, 16, false, true>::STAGES;
    return true;
  }
#define MOE_SHAPE_CASE(BT_, SWAP_)                                                       \
  if (bt == BT_) {                                                                       \
    switch (mode) {                                                                      \
      case kShrink: *k_tile = GemmCfg<kShrink, SWAP_, BT_>::BK; *stages = GemmCfg<kShrink, SWAP_, BT_>::STAGES; return true; \
      case kGateUp: *k_tile = GemmCfg<kGateUp, SWAP_, BT_>::BK; *stages = GemmCfg<kGateUp, SWAP_, BT_>::STAGES; return true; \
      case kDown: *k_tile = GemmCfg<kDown, SWAP_, BT_>::BK; *stages = GemmCfg<kDown, SWAP_, BT_>::STAGES; return true;       \
      default: return false;                                                             \
    }                                                                                    \
  }
  MOE_SHAPE_CASE(16, true)
  MOE_SHAPE_CASE(32, true)
  MOE_SHAPE_CASE(64, true)
  MOE_SHAPE_CASE(128, false)
  MOE_SHAPE_CASE(256, false)
#undef MOE_SHAPE_CASE
  return false;
}

}  // namespace moe
