// gemm_tc.cuh -- grouped expert GEMM on the 5th-generation tensor core (tcgen05 + TMEM),
// fed by TMA, for the three GEMM-shaped steps of the MoE-LoRA layer:
//
//   kShrink : S_run = X_block * A[a,e]^T           LoRA shrink of gate_up or down
//   kGateUp : g = X W_gu[e]^T (+ S_run Bt_gu[a,e]^T per adapter run), h = silu(g_gate) * g_up
//   kDown   : d = H W_dn[e]^T (+ S_run Bt_dn[a,e]^T per adapter run), out[t] += w * d
//
// The LoRA expand is not a separate kernel: every adapter run of a token block adds
// ceil(rank/16) extra K-steps to the same TMEM accumulator, with the run's S tile
// (rows outside the run are zero) as the token-side operand and Bt[a,e] as the
// weight-side operand.  SiLU gating and the weighted top-k combine happen in the
// epilogue that drains TMEM.  This is the pages' fusion of the LoRA add into the
// expand kernel (AWS ML Blog "Efficiently serve dozens of fine-tuned models with
// vLLM on Amazon SageMaker AI and Amazon Bedrock", section "Kernel optimizations")
// taken one step further: base GEMM, expand and epilogue share one accumulator.
//
// Two tile orientations (template SWAP):
//   SWAP = false (token blocks of 128 or 256 rows): MMA M = 128 tokens per accumulator
//          (one or two accumulators, MT = BT/128), N = 256 weight rows (gate_up: 128 gate
//          + 128 up rows of the same features; down: 256 features).  A 256-token block
//          uses each staged weight tile twice, which halves the L2 traffic per flop of
//          the weight side.
//   SWAP = true  (token blocks of 16/32/64 rows, few tokens per expert): MMA M = 128
//          weight rows, N = BT tokens; two accumulators (gate/up, or two feature halves).
//          Weights stream through the tensor core at full tile height however few
//          tokens an expert has.
//
// Warp roles (192 threads): warp 0 = TMA producer, warp 1 = TMEM owner + MMA issuer,
// warps 2..5 = epilogue (warp w drains TMEM lanes 32*(w%4) .. +31).
#pragma once

#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {

template <int MODE, bool SWAP, int BT>
struct GemmCfg {
  static constexpr bool kLora = MODE != kShrink;
  // weight-side rows staged per K-tile
  static constexpr int WROWS = MODE == kShrink ? (SWAP ? 128 : 64) : 256;
  static constexpr int W_BYTES = WROWS * 128;
  static constexpr int T_BYTES = BT * 128;
  static constexpr int STAGE_BYTES = W_BYTES + T_BYTES;
  static constexpr int STAGES = MODE == kShrink ? 4 : (SWAP ? (BT <= 16 ? 6 : 5) : (BT == 256 ? 3 : 4));
  // accumulators: non-swapped MT tiles of M=128 tokens x N; swapped NH tiles of 128 x BT
  static constexpr int NH = MODE == kShrink ? 1 : 2;
  static constexpr int MT = SWAP ? 1 : BT / 128;
  static constexpr int NACC = MODE == kShrink ? 64 : 256;   // columns of one non-swapped accumulator
  static constexpr int ACC_COLS = SWAP ? NH * BT : MT * NACC;
  static constexpr int TMEM_COLS =
      ACC_COLS <= 32 ? 32 : ACC_COLS <= 64 ? 64 : ACC_COLS <= 128 ? 128 : ACC_COLS <= 256 ? 256 : 512;
  static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align slack*/ + 256 /*barriers*/;
  static_assert(!SWAP || (BT == 16 || BT == 32 || BT == 64), "swapped tiles take 16/32/64 tokens");
  static_assert(SWAP || BT == 128 || BT == 256, "token-tiled blocks are 128 or 256 rows");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
  static_assert(W_BYTES % 1024 == 0 && T_BYTES % 1024 == 0, "stage regions keep 1024-byte alignment");
};

struct GemmBars {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t acc_full;
  uint32_t tmem_base;
  int32_t abort;
};

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
__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + __expf(-z)); }

template <int MODE, bool SWAP, int BT>
__global__ void __launch_bounds__(192, 1)
    moe_gemm_kernel(const __grid_constant__ GemmMaps maps, const __grid_constant__ GemmParams prm) {
  using C = GemmCfg<MODE, SWAP, BT>;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- work unit (uniform across the CTA; CTAs past the device-side count leave now).
  // The routing metadata comes from align, which finished before the previous kernel
  // started, so it may be read before waiting on that kernel.
  int b, f0 = 0, run0 = 0, nruns = 0, shrink_run = -1;
  int kb0 = 0, nk = prm.K / kKTile;
  if constexpr (MODE == kShrink) {
    shrink_run = blockIdx.x;
    if (shrink_run >= prm.totals[2]) return;
    b = prm.runs[4 * shrink_run + 0];
    // S tiles feed the next kernel's LoRA K-steps; it may launch once every shrink
    // CTA has passed this point, which is after the inputs of this kernel are ready.
    pdl_wait();
    pdl_trigger();
  } else {
    b = blockIdx.y;
    if (b >= prm.totals[1]) return;
    f0 = blockIdx.x * (MODE == kGateUp ? 128 : 256);
    if (blockIdx.z == 0) {
      run0 = prm.block_runs[b];
      nruns = prm.block_runs[b + 1] - run0;
    }
    const int nk_all = nk;
    kb0 = static_cast<int>(blockIdx.z) * nk_all / prm.ksplit;
    nk = (static_cast<int>(blockIdx.z) + 1) * nk_all / prm.ksplit - kb0;
    if (!prm.lora_after_pdl) pdl_wait();   // the previous kernel produced the token rows
    pdl_trigger();
  }
  const int e = prm.block_expert[b];
  const int row0 = b * BT;
  const int n_it = nk + nruns;
  int shrink_a = 0, shrink_nch = 0;
  if constexpr (MODE == kShrink) {
    shrink_a = prm.runs[4 * shrink_run + 1];
    shrink_nch = (prm.ranks[shrink_a] + kRankChunk - 1) / kRankChunk;
  }

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  GemmBars* bars = reinterpret_cast<GemmBars*>(smem + C::STAGES * C::STAGE_BYTES);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    mbar_init(&bars->acc_full, 1);
    bars->abort = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = bars->tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&maps.w);
      tma_prefetch_desc(&maps.tok);
      if constexpr (C::kLora) {
        tma_prefetch_desc(&maps.lw);
        tma_prefetch_desc(&maps.ls);
      }
      int issued = 0;
      for (int it = 0; it < n_it; ++it) {
        const int s = it % C::STAGES;
        const uint32_t ph = (it / C::STAGES) & 1;
        if (aborted(bars)) break;
        if (!mbar_wait(&bars->empty[s], ph ^ 1)) {
          record_timeout(bars, prm.status);
          break;
        }
        uint8_t* wdst = smem + s * C::STAGE_BYTES;
        uint8_t* tdst = wdst + C::W_BYTES;
        uint64_t* fb = &bars->full[s];
        if (it < nk) {
          const int k0 = (kb0 + it) * kKTile;
          if constexpr (MODE == kGateUp) {
            mbar_arrive_expect_tx(fb, C::W_BYTES + C::T_BYTES);
            tma_load_4d(wdst, &maps.w, fb, k0, f0, 0, e);               // gate rows f0..f0+127
            tma_load_4d(wdst + 128 * 128, &maps.w, fb, k0, f0, 1, e);   // up rows   f0..f0+127
          } else if constexpr (MODE == kDown) {
            mbar_arrive_expect_tx(fb, C::W_BYTES + C::T_BYTES);
            tma_load_3d(wdst, &maps.w, fb, k0, f0, e);
            tma_load_3d(wdst + 128 * 128, &maps.w, fb, k0, f0 + 128, e);
          } else {
            const int ae = shrink_a * prm.E + e;
            mbar_arrive_expect_tx(fb, shrink_nch * kRankChunk * 128 + C::T_BYTES);
            for (int c = 0; c < shrink_nch; ++c)
              tma_load_3d(wdst + c * kRankChunk * 128, &maps.w, fb, k0, c * kRankChunk, ae);
          }
          tma_load_2d(tdst, &maps.tok, fb, k0, row0);
        } else if constexpr (C::kLora) {
          if (it == nk && prm.lora_after_pdl) pdl_wait();   // S tiles come from the previous kernel
          const int run = run0 + (it - nk);
          const int a = prm.runs[4 * run + 1];
          const int nch = (prm.ranks[a] + kRankChunk - 1) / kRankChunk;
          const int ae = a * prm.E + e;
          mbar_arrive_expect_tx(fb, nch * (C::WROWS * 32 + BT * 32));
          for (int c = 0; c < nch; ++c) {
            uint8_t* wc = wdst + c * (C::WROWS * 32);
            if constexpr (MODE == kGateUp) {
              tma_load_4d(wc, &maps.lw, fb, c * kRankChunk, f0, 0, ae);
              tma_load_4d(wc + 128 * 32, &maps.lw, fb, c * kRankChunk, f0, 1, ae);
            } else {
              tma_load_3d(wc, &maps.lw, fb, c * kRankChunk, f0, ae);
              tma_load_3d(wc + 128 * 32, &maps.lw, fb, c * kRankChunk, f0 + 128, ae);
            }
            tma_load_3d(tdst + c * (BT * 32), &maps.ls, fb, c * kRankChunk, 0, run);
          }
        }
        issued = it + 1;
      }
      // Leave no copy in flight: wait (bounded) for the stages issued last.
      if (aborted(bars)) {
        for (int it = issued - C::STAGES < 0 ? 0 : issued - C::STAGES; it < issued; ++it)
          (void)mbar_wait(&bars->full[it % C::STAGES], (it / C::STAGES) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t acc = 0;
      for (int it = 0; it < n_it; ++it) {
        const int s = it % C::STAGES;
        const uint32_t ph = (it / C::STAGES) & 1;
        if (aborted(bars)) break;
        if (!mbar_wait(&bars->full[s], ph)) {
          record_timeout(bars, prm.status);
          break;
        }
        tc_fence_after_sync();
        const uint32_t wbase = smem_u32(smem + s * C::STAGE_BYTES);
        const uint32_t tbase = wbase + C::W_BYTES;
        if (it < nk) {
#pragma unroll
          for (int kk = 0; kk < kKTile / 16; ++kk) {
            if constexpr (!SWAP) {
              const uint32_t n_mma = MODE == kShrink ? shrink_nch * kRankChunk : 256;
              const uint64_t bd = smem_desc(wbase + kk * 32, 1024, kSw128);
#pragma unroll
              for (int mt = 0; mt < C::MT; ++mt) {
                const uint64_t ad = smem_desc(tbase + mt * 128 * 128 + kk * 32, 1024, kSw128);
                tc_mma(tmem + mt * C::NACC, ad, bd, idesc_bf16_f32(128, n_mma), acc);
              }
            } else {
              const uint64_t bd = smem_desc(tbase + kk * 32, 1024, kSw128);
#pragma unroll
              for (int h = 0; h < C::NH; ++h) {
                const uint64_t ad = smem_desc(wbase + h * 128 * 128 + kk * 32, 1024, kSw128);
                tc_mma(tmem + h * BT, ad, bd, idesc_bf16_f32(128, BT), acc);
              }
            }
            acc = 1;
          }
        } else if constexpr (C::kLora) {
          const int run = run0 + (it - nk);
          const int nch = (prm.ranks[prm.runs[4 * run + 1]] + kRankChunk - 1) / kRankChunk;
          for (int c = 0; c < nch; ++c) {
            const uint32_t wc = wbase + c * (C::WROWS * 32);
            const uint32_t tc = tbase + c * (BT * 32);
            if constexpr (!SWAP) {
              const uint64_t bd = smem_desc(wc, 256, kSw32);
#pragma unroll
              for (int mt = 0; mt < C::MT; ++mt)
                tc_mma(tmem + mt * C::NACC, smem_desc(tc + mt * 128 * 32, 256, kSw32), bd, idesc_bf16_f32(128, 256), 1);
            } else {
              const uint64_t bd = smem_desc(tc, 256, kSw32);
#pragma unroll
              for (int h = 0; h < C::NH; ++h)
                tc_mma(tmem + h * BT, smem_desc(wc + h * 128 * 32, 256, kSw32), bd, idesc_bf16_f32(128, BT), 1);
            }
          }
        }
        tc_commit(&bars->empty[s]);
      }
      tc_commit(&bars->acc_full);   // also after an abort: marks the end of all issued MMAs
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;          // TMEM lane quarter this warp may access
    const int m = q * 32 + lane;     // accumulator row (TMEM lane) of this thread
    const uint32_t tq = tmem + (static_cast<uint32_t>(q * 32) << 16);
    bool ok = mbar_wait(&bars->acc_full, 0);
    if (!ok) record_timeout(bars, prm.status);
    tc_fence_after_sync();
    ok = ok && !aborted(bars);
    if (ok) {
      uint32_t v[16], u[16];
      if constexpr (MODE == kShrink) {
        const int beg = prm.runs[4 * shrink_run + 2] - row0;
        const int end = prm.runs[4 * shrink_run + 3] - row0;
        const int r_a = prm.ranks[shrink_a];
        uint16_t* srun = prm.s_out + static_cast<size_t>(shrink_run) * BT * prm.r_pad;
        if constexpr (!SWAP) {
          // row mt*128 + m of the token block; columns are ranks
          for (int mt = 0; mt < C::MT; ++mt) {
          const int row = mt * 128 + m;
          const bool in_run = row >= beg && row < end;
          for (int c = 0; c < prm.r_pad; c += 16) {
            if (c < shrink_nch * kRankChunk) {
              tmem_ld16(tq + mt * C::NACC + c, v);
              tmem_ld_wait();
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) v[i] = 0;
            }
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int c0 = c + 2 * i;
              const float a0 = (in_run && c0 < r_a) ? __uint_as_float(v[2 * i]) : 0.f;
              const float a1 = (in_run && c0 + 1 < r_a) ? __uint_as_float(v[2 * i + 1]) : 0.f;
              pk[i] = pack_bf16x2(a0, a1);
            }
            uint4* dst = reinterpret_cast<uint4*>(srun + static_cast<size_t>(row) * prm.r_pad + c);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
          }
        } else {
          // row m is rank index m; columns are the BT tokens of the block
          for (int n0 = 0; n0 < BT; n0 += 16) {
            tmem_ld16(tq + n0, v);
            tmem_ld_wait();
            if (m < prm.r_pad) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int n = n0 + i;
                const float val = (n >= beg && n < end && m < r_a) ? __uint_as_float(v[i]) : 0.f;
                __nv_bfloat16 hv = __float2bfloat16_rn(val);
                srun[static_cast<size_t>(n) * prm.r_pad + m] = *reinterpret_cast<uint16_t*>(&hv);
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
          for (int c = 0; c < 128; c += 16) {
            if (f0 + c >= I) break;
            tmem_ld16(ta + c, v);          // gate features f0+c ..
            tmem_ld16(ta + 128 + c, u);    // up features   f0+c ..
            tmem_ld_wait();
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
              pk[i] = pack_bf16x2(silu_f(__uint_as_float(v[2 * i])) * __uint_as_float(u[2 * i]),
                                  silu_f(__uint_as_float(v[2 * i + 1])) * __uint_as_float(u[2 * i + 1]));
            uint4* dst = reinterpret_cast<uint4*>(hrow + c);
            dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
          }
          }
        } else {
          const int f = f0 + m;           // feature of this thread; columns are tokens
          for (int n0 = 0; n0 < BT; n0 += 16) {
            tmem_ld16(tq + n0, v);
            tmem_ld16(tq + BT + n0, u);
            tmem_ld_wait();
            if (f < I) {
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                __nv_bfloat16 hv = __float2bfloat16_rn(silu_f(__uint_as_float(v[i])) * __uint_as_float(u[i]));
                prm.h_out[static_cast<size_t>(row0 + n0 + i) * I + f] = *reinterpret_cast<uint16_t*>(&hv);
              }
            }
          }
        }
      } else {  // kDown
        const int H = prm.n_feat;
        if constexpr (!SWAP) {
          for (int mt = 0; mt < C::MT; ++mt) {
          const int p = prm.sorted_p[row0 + mt * 128 + m];
          const bool valid = p < prm.P;
          const float w = valid ? prm.topk_w[p] : 0.f;
          float* orow = prm.out_acc + static_cast<size_t>(valid ? p / prm.k : 0) * H + f0;
          for (int c = 0; c < 256; c += 16) {
            if (f0 + c >= H) break;
            tmem_ld16(tq + mt * C::NACC + c, v);
            tmem_ld_wait();
            if (valid) {
#pragma unroll
              for (int i = 0; i < 4; ++i)
                atomicAdd(reinterpret_cast<float4*>(orow + c + 4 * i),
                          make_float4(w * __uint_as_float(v[4 * i]), w * __uint_as_float(v[4 * i + 1]),
                                      w * __uint_as_float(v[4 * i + 2]), w * __uint_as_float(v[4 * i + 3])));
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
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int p = prm.sorted_p[row0 + n0 + i];
                if (p < prm.P && f < H)
                  atomicAdd(prm.out_acc + static_cast<size_t>(p / prm.k) * H + f, prm.topk_w[p] * __uint_as_float(v[i]));
              }
            }
          }
        }
      }
    }
    tc_fence_before_sync();
  }

  __syncwarp();   // lanes of the producer and MMA warps reconverge before the CTA barrier
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    // All MMAs were committed to acc_full; make sure they finished before freeing TMEM.
    if (lane == 0) (void)mbar_wait(&bars->acc_full, 0);
    __syncwarp();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int MODE, bool SWAP, int BT>
cudaError_t launch_gemm_t(const GemmMaps& maps, const GemmParams& prm, int64_t max_blocks, int64_t max_runs,
                          bool pdl, cudaStream_t s) {
  using C = GemmCfg<MODE, SWAP, BT>;
  auto kern = moe_gemm_kernel<MODE, SWAP, BT>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
  if (err != cudaSuccess) return err;
  dim3 grid;
  if constexpr (MODE == kShrink) {
    if (max_runs <= 0) return cudaSuccess;
    grid = dim3(static_cast<unsigned>(max_runs), 1, 1);
  } else {
    if (max_blocks <= 0) return cudaSuccess;
    const int tile = MODE == kGateUp ? 128 : 256;
    grid = dim3(static_cast<unsigned>((prm.n_feat + tile - 1) / tile), static_cast<unsigned>(max_blocks),
                static_cast<unsigned>(prm.ksplit));
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(192, 1, 1);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, maps, prm);
}

}  // namespace moe
