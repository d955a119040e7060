/*
 * moe_lora.h -- C ABI of the GB300 (sm_103a) fused Mixture-of-Experts layer with
 * per-request LoRA adapters.
 *
 * Sources (cited by page title and section):
 *   [AWS] AWS Machine Learning Blog, "Efficiently serve dozens of fine-tuned models
 *         with vLLM on Amazon SageMaker AI and Amazon Bedrock".
 *   [KO]  agentlenshq.com, "vLLM MoE 모델을 위한 Multi-LoRA 서빙".
 *   [ZH]  setupai.cc, "vLLM 多 LoRA 提升 AWS 上 MoE 模型服務".
 *
 * The layer.  Each of T tokens is routed to k of E experts and carries one adapter
 * id in [-1, L) (-1 = no adapter; adapters are swapped per request, [AWS]
 * introduction).  Each expert is a two-stage FFN that expands the hidden state to
 * an intermediate space (gate_up, H -> 2I) and compresses it back (down, I -> H)
 * ([KO] "MoE 모델을 위한 Multi-LoRA 서빙").  LoRA turns XW into XW + XAB on both
 * projections ([ZH] "增強重點摘要"), i.e. four extra ops per expert:
 * gate_up_shrink, gate_up_expand, down_shrink, down_expand ([KO] "Amazon 전용 튜닝").
 * For a pair (token t, expert e) with adapter a and rank r = ranks[a]:
 *     g = W_gu[e] x_t + B_gu[a,e][:r, :]^T (A_gu[a,e][:r, :] x_t)         (2I)
 *     h = silu(g[0:I]) * g[I:2I]                                        (I)
 *     d = W_dn[e] h   + B_dn[a,e][:r, :]^T (A_dn[a,e][:r, :] h)           (H)
 *     out_t = sum_j w_{t,j} d_{t,j}
 * where the weights w are the softmax over the E router logits, kept for the k
 * largest and renormalised; the router and the aggregation of expert outputs are
 * [AWS] "Implementing multi-LoRA inference for MoE models in vLLM".
 *
 * Conventions for every entry point:
 *   - bf16 tensors are passed as their 16-bit patterns (uint16_t).
 *   - All tensors are dense, row-major, with the shapes stated.  Device pointers
 *     must be 16-byte aligned (the kernels stream them with TMA).
 *   - `stream` is a cudaStream_t (NULL = legacy default stream).  Device work is
 *     enqueued asynchronously on it; nothing is synchronised unless stated.
 *   - Ownership: the caller allocates every buffer; the library never allocates
 *     device or pinned memory and keeps no per-call state.  Calls on different
 *     streams with different buffers may run concurrently.
 *   - Errors detectable on the host return a non-zero status before anything is
 *     enqueued; moe_lora_last_error() then describes it (per thread).
 *   - Kernels never trap.  Conditions found on the device (invalid ids, a pipeline
 *     wait that timed out) are reported in `dev_status`, to be read by the caller
 *     after synchronising.
 */
#ifndef MOE_LORA_H
#define MOE_LORA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status -- */
enum {
    MOE_LORA_OK = 0,
    MOE_LORA_EINVAL = 1,        /* null pointer, size out of range, bad rank           */
    MOE_LORA_EALIGN = 2,        /* a device pointer is not 16-byte aligned            */
    MOE_LORA_EWORKSPACE = 3,    /* workspace smaller than moe_lora_workspace_size()    */
    MOE_LORA_EUNSUPPORTED = 4,  /* shape outside the compiled kernels (see limits)     */
    MOE_LORA_ECUDA = 5,         /* a CUDA runtime call failed                          */
    MOE_LORA_EDEVICE = 6        /* the device reported an error in dev_status          */
};

/* Bits of the forward call's device status word (dropped pairs are in totals[3]). */
#define MOE_LORA_DEV_TIMEOUT 0x1   /* a bounded pipeline wait expired; outputs invalid */

/* Stages of moe_lora_forward, in launch order (see stage_events). */
#define MOE_LORA_STAGE_GATHER 0      /* x rows into sorted order               */
#define MOE_LORA_STAGE_SHRINK_GU 1   /* gate_up_shrink                         */
#define MOE_LORA_STAGE_GATE_UP 2     /* gate_up GEMM + expand + SiLU gating    */
#define MOE_LORA_STAGE_SHRINK_DN 3   /* down_shrink                            */
#define MOE_LORA_STAGE_DOWN 4        /* down GEMM + expand, one row per pair   */
#define MOE_LORA_STAGE_COMBINE 5     /* weighted top-k combine -> bf16 output  */
#define MOE_LORA_NUM_STAGES 6

/* Limits of the compiled kernels (MOE_LORA_EUNSUPPORTED beyond them). */
#define MOE_LORA_MAX_ADAPTERS 256  /* L                                    */
#define MOE_LORA_MAX_RANK 64       /* r_max                                */
#define MOE_LORA_MAX_EXPERTS 1024  /* E                                    */
#define MOE_LORA_MAX_TOPK 32       /* k                                    */

/* ---------------------------------------------------------------- shapes -- */
typedef struct moe_lora_dims {
    int64_t T;        /* tokens, >= 0                                                   */
    int32_t H;        /* hidden size, multiple of 64                                    */
    int32_t I;        /* expert intermediate size, multiple of 64                       */
    int32_t E;        /* experts, 1..MOE_LORA_MAX_EXPERTS                               */
    int32_t k;        /* experts per token, 1..min(E, MOE_LORA_MAX_TOPK)                */
    int32_t L;        /* adapters, 0..MOE_LORA_MAX_ADAPTERS                             */
    int32_t r_max;    /* storage rank: rows of A and of B; multiple of 8, <= 64         */
    int32_t block_m;  /* rows per align block: 16, 32, 64 (weight-streaming kernels)    */
                      /* or 128, 256 (token-tiled kernels); 0 = the tile table's choice */
                      /* for the dims (moe_lora_pick_block_m, moe_lora_plan_query)      */
    const int32_t *ranks; /* HOST array [L]: rank of adapter a, 1 <= ranks[a] <= r_max  */
} moe_lora_dims;

/*
 * Output of moe_lora_align: the (expert, adapter) compound-sparsity layout
 * ([AWS] "Tuning kernel configurations for Amazon SageMaker AI and Amazon
 * Bedrock": the extra LoRA-index grid dimension and the sparsity of many
 * adapters; [KO] "MoE 모델을 위한 Multi-LoRA 서빙").  All arrays are device int32,
 * caller-allocated with the capacities of moe_lora_align_capacity().
 *   Pair p = t*k + j joins expert topk_ids[p] and adapter lora_ids[t]; a pair is
 *   valid when the expert is in [0, E) and the adapter in [-1, L).  Valid pairs are
 *   sorted by (expert, adapter, p); each expert's rows are padded to a multiple of
 *   block_m with the sentinel P = T*k.
 */
typedef struct moe_lora_align_buf {
    int32_t *sorted_p;     /* [max_rows]   pair index of each row, P for padding        */
    int32_t *expert_begin; /* [E+1]        first row of each expert; [E] = rows         */
    int32_t *block_expert; /* [max_blocks] expert of each block_m-row block             */
    int32_t *block_runs;   /* [max_blocks+1] first run of each block (CSR into runs)    */
    int32_t *runs;         /* [max_runs][4] {block, adapter, begin_row, end_row}: maximal
                              stretches of one adapter >= 0 inside one block, in row order */
    int32_t *totals;       /* [4] {rows, blocks, runs, dropped pairs}                   */
} moe_lora_align_buf;

/* ----------------------------------------------------------- size queries -- */

/* Capacities of the align arrays for these dims.  Returns a status. */
int moe_lora_align_capacity(const moe_lora_dims *d, int64_t *max_rows, int64_t *max_blocks,
                            int64_t *max_runs);

/* Device scratch bytes needed by moe_lora_align and by moe_lora_forward (the two
 * use disjoint regions, so one buffer of align_bytes + forward_bytes serves both,
 * with forward's region at offset align_bytes).  Returns a status. */
int moe_lora_workspace_size(const moe_lora_dims *d, size_t *align_bytes, size_t *forward_bytes);

/* The compiled-in tile table's block_m for T*k pairs over E experts, L adapters and
 * experts of hidden size H and intermediate size I: the shape class is the pairs per
 * expert T*k/E (16, 64 weight-streaming up to 24, 95 pairs per expert; 128 token-tiled
 * up to 2047; 256, token-tiled on CTA pairs, above), and from 768 pairs per expert
 * also 256 when the adapter runs are long, i.e. T*k / (E*(L+1)) >= 20.  An expert whose
 * bf16 weights (3*H*I*2 bytes) exceed the L2 takes, up to 128 pairs per expert, the
 * smallest of 16, 32, 64, 128 that holds T*k/E pairs (each block of it streams the
 * expert from DRAM).  H or I <= 0 leaves that rule out.  The pages pick tuned tile
 * configurations per shape ([AWS] "Tuning kernel configurations for Amazon SageMaker
 * AI and Amazon Bedrock"; [KO] "Amazon 전용 튜닝").  Host only. */
int32_t moe_lora_pick_block_m(int64_t T, int32_t k, int32_t E, int32_t L, int32_t H, int32_t I);

/* What the calls will launch for these dims: the tile-table row and the per-GEMM
 * choices.  GEMM index: 0 gate_up shrink, 1 gate_up, 2 down shrink, 3 down. */
typedef struct moe_lora_plan {
    int32_t block_m;              /* token tile = align block (dims.block_m, or the table's) */
    int32_t table_row;            /* row of the compiled tile table whose constants apply    */
    int32_t weight_streaming;     /* 1: tiles of 128 weight rows x block_m tokens;
                                     0: tiles of block_m tokens x 256 weight rows (256-token
                                        tiles of gate_up/down run on a CTA pair)           */
    int32_t ksplit[4];            /* K splits per GEMM (0: not launched, L == 0 shrinks)     */
    int32_t k_tile[4];            /* K elements per pipeline stage                          */
    int32_t stages[4];            /* pipeline stages in shared memory                       */
    int32_t launches_route_align; /* kernel launches of one moe_lora_route_align           */
    int32_t launches_forward;     /* kernel launches of one moe_lora_forward               */
    int32_t shrink_on_cores;      /* 1: the LoRA shrinks run on CUDA cores, split over K in
                                     ksplit[0]/ksplit[2] slices of k_tile elements (short
                                     adapter runs); 0: tcgen05 tiles                        */
    int32_t shrink_block_diag;    /* 1: the tcgen05 shrinks of token-tiled blocks take groups
                                     of rank chunks of the adapter runs that reach a 128-row
                                     unit (a block, or a half of a 256-row block) per tile
                                     (N = their ranks side by side); 0: one run per tile    */
} moe_lora_plan;

/* Fills *out for dims d (host only: no device call).  Returns a status. */
int moe_lora_plan_query(const moe_lora_dims *d, moe_lora_plan *out);

/* ------------------------------------------------------------ the calls -- */

/*
 * Router top-k ([AWS] "Implementing multi-LoRA inference for MoE models in vLLM").
 *   logits   [T][E] fp32, device, finite values
 *   topk_ids [T][k] int32, device, out: experts in descending logit order, ties to the
 *            lower index
 *   topk_w   [T][k] fp32, device, out: exp(l_j - l_max) / sum over the chosen k
 *            (= softmax over all E renormalised over the chosen k)
 */
int moe_lora_route(const float *logits, int64_t T, int32_t E, int32_t k,
                   int32_t *topk_ids, float *topk_w, void *stream);

/*
 * Align-and-sort of the (expert, adapter) compound sparsity (layout above).
 *   topk_ids [T][k], lora_ids [T]: int32, device
 *   out:       the align arrays (bit-identical to the CPU definition)
 *   workspace: device scratch of at least align_bytes (moe_lora_workspace_size)
 * totals[3] counts the dropped (invalid) pairs.
 */
int moe_lora_align(const moe_lora_dims *d, const int32_t *topk_ids, const int32_t *lora_ids,
                   const moe_lora_align_buf *out, void *workspace, size_t workspace_bytes,
                   void *stream);

/*
 * moe_lora_route followed by moe_lora_align, with the same arguments and results
 * (topk_ids and topk_w are outputs here).  The pages route, then group the routed
 * tokens per (expert, adapter) for the fused MoE-LoRA kernels ([AWS] "Implementing
 * multi-LoRA inference for MoE models in vLLM"; [KO] "MoE 모델을 위한 Multi-LoRA
 * 서빙"); a batch of at most 4096 pairs (T*k <= 4096) is routed and aligned by one
 * single-CTA launch, larger batches take the two calls' launches.
 *   logits [T][E] fp32, lora_ids [T] int32: device, read
 *   topk_ids [T][k] int32, topk_w [T][k] fp32: device, written
 *   workspace: device scratch of at least align_bytes (moe_lora_workspace_size)
 */
int moe_lora_route_align(const moe_lora_dims *d, const float *logits, const int32_t *lora_ids,
                         int32_t *topk_ids, float *topk_w, const moe_lora_align_buf *out,
                         void *workspace, size_t workspace_bytes, void *stream);

/*
 * The fused expert computation over an aligned pair list: gate_up GEMM with its
 * LoRA shrink and expand, SiLU gating, down GEMM with its LoRA shrink and expand,
 * and the weighted top-k combine.
 *   x       [T][H]            bf16, device
 *   topk_w  [T][k]            fp32, device (the combine weights)
 *   aligned                   moe_lora_align output for the same dims
 *   W_gu    [E][2I][H]        bf16; rows [0,I) gate, rows [I,2I) up
 *   W_dn    [E][H][I]         bf16
 *   A_gu    [L][E][r_max][H]  bf16; rows >= ranks[a] must be zero
 *   B_gu    [L][E][r_max][2I] bf16, the r x 2I matrix B of XAB for gate_up (columns
 *                             [0,I) gate, [I,2I) up); rows >= ranks[a] zero
 *   A_dn    [L][E][r_max][I]  bf16; rows >= ranks[a] zero
 *   B_dn    [L][E][r_max][H]  bf16; rows >= ranks[a] zero
 *   (A and B rank-major: an adapter's rank-r slice is its first r rows, read as r
 *   contiguous rows, so a low-rank adapter in a wide bank costs only its own bytes.)
 *   out     [T][H]            bf16, device, out: fully overwritten
 *   workspace  device scratch of at least forward_bytes
 *   dev_status one int32, device: cleared by the call, then receives MOE_LORA_DEV_* bits
 *   stage_events  NULL, or MOE_LORA_NUM_STAGES + 1 cudaEvent_t recorded on `stream`
 *              before the first stage and after each stage (for timing)
 * LoRA tensors may be NULL when L == 0.
 * Deterministic: no step accumulates with atomics.  Each pair's expert output gets
 * its own row (K-split partial sums their own buffers), and the combine adds a
 * token's k rows in ascending j, so the same inputs give the same output bytes on
 * every call.
 */
int moe_lora_forward(const moe_lora_dims *d, const uint16_t *x, const float *topk_w,
                     const moe_lora_align_buf *aligned,
                     const uint16_t *W_gu, const uint16_t *W_dn,
                     const uint16_t *A_gu, const uint16_t *B_gu,
                     const uint16_t *A_dn, const uint16_t *B_dn,
                     uint16_t *out, void *workspace, size_t workspace_bytes,
                     int32_t *dev_status, void *stream, void *const *stage_events);

/*
 * The whole layer from HOST inputs to a HOST output: brings logits [T][E] fp32,
 * lora_ids [T] int32 and x [T][H] bf16 to the device, runs route, align and
 * forward on `stream`, returns out [T][H] bf16 and synchronises the stream.
 * Weights are device pointers (resident).  A host buffer of at most 4 MB that is
 * pinned and mapped at the same address on both sides (cudaHostAlloc or
 * cudaHostRegister memory under unified addressing, as on a coherent CPU-GPU link)
 * and 16-byte aligned is read or written in place by the kernels over the link
 * (x only while T*k*H*2 <= 1 MB: the gather reads a token's row once per pair);
 * any other host buffer goes through a copy on `stream` (pinned memory keeps those
 * copies asynchronous).  workspace: device scratch of at least
 * moe_lora_layer_workspace_size().  Returns MOE_LORA_EDEVICE if the device
 * reported a timeout.  *dropped (may be NULL) receives the dropped-pair count.
 */
int moe_lora_layer_workspace_size(const moe_lora_dims *d, size_t *bytes);
int moe_lora_layer_host(const moe_lora_dims *d, const float *logits_host,
                        const int32_t *lora_ids_host, const uint16_t *x_host,
                        const uint16_t *W_gu, const uint16_t *W_dn,
                        const uint16_t *A_gu, const uint16_t *B_gu,
                        const uint16_t *A_dn, const uint16_t *B_dn,
                        uint16_t *out_host, void *workspace, size_t workspace_bytes,
                        int64_t *dropped, void *stream);

/*
 * The moe_lora_layer_host sequence (inputs in, route, align, forward, output back,
 * each host buffer read or written in place or copied as moe_lora_layer_host
 * decides) captured once as a CUDA graph and replayed per step: one launch instead
 * of every copy and kernel issued from the CPU.
 * The pages capture GPU operation sequences with CUDA graphs to cut kernel-launch
 * and CPU overhead ([AWS] "Execution optimizations").
 *   create: same arguments as moe_lora_layer_host, with every host buffer pinned
 *           (cudaHostAlloc / cudaHostRegister) and status_host an extra pinned int32[8]
 *           that each run fills with {device status word, 3 unused, align totals[4]}.
 *           Runs the layer once eagerly (validation, kernel set-up), then captures it
 *           on `stream`.  *graph receives the handle.
 *   run:    launches the graph on `stream` and synchronises it; the host buffers'
 *           CURRENT contents are the step's inputs.  *dropped (may be NULL) receives
 *           the dropped-pair count; returns MOE_LORA_EDEVICE if the device reported
 *           a timeout.
 *   destroy: releases the graph.  Buffers, weights and workspace stay the caller's;
 *           none of them may move or be freed while the graph exists, and the host
 *           buffers stay pinned (not unregistered): the kernels captured at create
 *           time may read or write them in place.
 */
typedef struct moe_lora_graph moe_lora_graph;
int moe_lora_layer_graph_create(const moe_lora_dims *d, const float *logits_host,
                                const int32_t *lora_ids_host, const uint16_t *x_host,
                                const uint16_t *W_gu, const uint16_t *W_dn,
                                const uint16_t *A_gu, const uint16_t *B_gu,
                                const uint16_t *A_dn, const uint16_t *B_dn,
                                uint16_t *out_host, int32_t *status_host,
                                void *workspace, size_t workspace_bytes, void *stream,
                                moe_lora_graph **graph);
int moe_lora_layer_graph_run(moe_lora_graph *graph, void *stream, int64_t *dropped);
int moe_lora_layer_graph_destroy(moe_lora_graph *graph);

/*
 * moe_lora_align_static: moe_lora_align without a caller-supplied workspace.
 * The pages have no counterpart of this entry point.  It is for callers that cannot
 * allocate device memory when they call: a serving engine that has handed almost all
 * HBM to its own pool (weights, KV cache), so cudaMalloc has nothing left to give or
 * would fragment that pool, and latency-bound decode loops in which a cudaMalloc --
 * which may synchronise the device and takes unbounded time -- is not allowed.
 * Its scratch is one static device array of MOE_LORA_STATIC_SCRATCH_BYTES, which
 * every GPU that loads the library holds until the process exits.  Dims whose align
 * scratch (align_bytes of moe_lora_workspace_size) is larger are rejected with
 * MOE_LORA_EWORKSPACE before anything is enqueued.
 *   - The first call on a device looks up the array's device address (once per
 *     device, with that device current; again after the device's context was
 *     replaced, e.g. by cudaDeviceReset); make that first call before any stream
 *     capture.
 *   - All calls on a device share the one array: calls that overlap on the GPU
 *     (other streams, other host threads) race on it, so serialise them.
 *   - The array keeps the last call's contents; the align kernels write every
 *     scratch word before reading it, so nothing needs clearing between calls.
 * Arguments and results are those of moe_lora_align.
 */
#define MOE_LORA_STATIC_SCRATCH_BYTES (4u << 20)
int moe_lora_align_static(const moe_lora_dims *d, const int32_t *topk_ids, const int32_t *lora_ids,
                          const moe_lora_align_buf *out, void *stream);

/* ------------------------------------------------------------ diagnostics -- */

/*
 * Test hook for the failure path; the pages have no counterpart.  Every pipeline wait
 * in the GEMM kernels is bounded (2 s) and reports expiry through dev_status rather
 * than trapping.  This call sets, for the moe_lora_forward calls that follow in this
 * process, the wall-clock limit in nanoseconds of ONE of those waits: the gate_up
 * epilogue's wait for its accumulator, in the single-CTA kernels (block_m <= 128; the
 * CTA-pair kernels of 256-row blocks keep the default).  0 restores the default.  A
 * limit shorter than the accumulator takes makes that wait give up: the call sets
 * MOE_LORA_DEV_TIMEOUT in dev_status (moe_lora_layer_host and the graph run return
 * MOE_LORA_EDEVICE), the gate_up kernel winds down -- its in-flight copies and MMAs
 * drained, its TMEM freed, the MMA thread giving up its own wait after the default
 * limit -- and the call's output is invalid; the later kernels of the call still run.
 * The next call with the default limit computes normally.  Process-wide; always
 * returns MOE_LORA_OK.
 */
int moe_lora_debug_set_acc_wait_ns(uint64_t ns);

/*
 * Test hook: the tile form of the tcgen05 shrinks of token-tiled blocks (block_m 128
 * or 256) in later moe_lora_forward calls of this process.  0 (default): by shape --
 * on 128-row blocks block-diagonal tiles (several adapter runs per tile) once the
 * blocks alone fill the SMs twice, else one run per tile; on 256-row blocks one run per
 * 128-row half; 1: always block-diagonal; 2: always one run per tile.  Both forms
 * compute the same S tiles (the same fp32 sums of the same products, rounded once to
 * bf16), so the layer's output does not depend on the choice.  The forward workspace
 * size does not depend on it either.  Returns MOE_LORA_EINVAL for another mode.
 */
int moe_lora_debug_set_shrink_tiles(int32_t mode);

const char *moe_lora_status_string(int status);
const char *moe_lora_last_error(void);   /* detail of this thread's last failure */
int moe_lora_version(void);              /* MAJOR*10000 + MINOR*100 + PATCH       */

#ifdef __cplusplus
}
#endif
#endif /* MOE_LORA_H */
