// gemm_tc.cu -- instantiations of the tcgen05 grouped GEMM and the launch dispatch.
#include "gemm_tc.cuh"

namespace moe {

cudaError_t launch_gemm(int mode, int bt, const GemmMaps& maps, const GemmParams& prm, int64_t max_blocks,
                        int64_t max_runs, bool pdl, cudaStream_t s, bool block_diag) {
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

bool gemm_stage_shape(int mode, int bt, int* k_tile, int* stages) {
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
