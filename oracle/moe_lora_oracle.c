/*
 * moe_lora_oracle.c -- plain, slow, fp64 CPU oracle of the fused MoE layer with
 * per-request LoRA adapters.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package's smoke check and
 * the benchmark's CPU-baseline leg may load or call this library.  It shares no
 * code, header, table or helper with the CUDA path, and it never calls it.
 *
 * Sources (cited by page title and section):
 *   [AWS] AWS Machine Learning Blog, "Efficiently serve dozens of fine-tuned
 *         models with vLLM on Amazon SageMaker AI and Amazon Bedrock".
 *   [KO]  agentlenshq.com, "vLLM MoE 모델을 위한 Multi-LoRA 서빙" (Korean summary of [AWS]).
 *   [ZH]  setupai.cc, "vLLM 多 LoRA 提升 AWS 上 MoE 模型服務" (Chinese summary of [AWS]).
 *
 * What is computed (each function names the passage it follows):
 *   route   -- a router sends each token to its k most relevant experts and their
 *              outputs are aggregated ([AWS] "Implementing multi-LoRA inference for
 *              MoE models in vLLM", first paragraph).  Weights: softmax over all E
 *              logits, the k largest kept, renormalised to sum to 1.  Ties in the
 *              logit go to the lower expert index (the pages are silent on ties).
 *   align   -- the layout of the (expert, adapter) compound sparsity: the extra LoRA
 *              grid dimension and the sparsity from many adapters ([AWS] "Tuning
 *              kernel configurations for Amazon SageMaker AI and Amazon Bedrock";
 *              [KO] "MoE 모델을 위한 Multi-LoRA 서빙").  The pages give no layout; the
 *              one below is this library's definition, and the CUDA path must
 *              reproduce it bit for bit.
 *   forward -- each expert expands the hidden state (gate_up) and compresses it back
 *              (down) ([KO] "MoE 모델을 위한 Multi-LoRA 서빙"); LoRA replaces XW by
 *              XW + XAB with a frozen W ([ZH] "增強重點摘要"; [AWS] introduction), which
 *              gives the four extra ops gate_up_shrink, gate_up_expand, down_shrink,
 *              down_expand ([KO] "Amazon 전용 튜닝").  Activation SiLU(gate)*up, gate =
 *              first I rows of gate_up, up = last I rows; LoRA scale 1; adapter id -1
 *              means no adapter; the expert outputs are summed with the routing weights.
 *
 * Precision: every bf16 input is converted exactly to double, and all arithmetic,
 * intermediates (S, g, h, d) and the output stay in double.  No rounding to bf16.
 *
 * Parity pins: every function here is pinned by the CPU test suite against
 * independent results (brute-force sorts, closed forms, library matmuls,
 * hand-computed cases, merged-weight runs).  Nothing here is "parity unpinned".
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Threads of the parallel regions that later calls from this host thread start
 * (n <= 0: one per processor).  Returns the count now in force.  Timing only; the
 * results do not depend on it. */
int32_t oracle_set_threads(int32_t n)
{
    omp_set_num_threads(n > 0 ? n : omp_get_num_procs());
    return omp_get_max_threads();
}

/* bf16 bit pattern -> double (exact). */
static double bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* route                                                                     */
/* ------------------------------------------------------------------------ */

/*
 * For each token t: p_e = exp(l_e - max_e l_e) / sum_e exp(l_e - max_e l_e) for all E
 * experts; the k experts with the largest p (ties: lower index first) are chosen in
 * descending order; w_j = p_{e_j} / sum_{chosen} p.  Writes topk_ids [T][k] and
 * topk_w [T][k] (double).
 */
void oracle_route(const float *logits, int64_t T, int32_t E, int32_t k,
                  int32_t *topk_ids, double *topk_w)
{
    #pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)E);
        char *taken = (char *)malloc((size_t)E);
        #pragma omp for schedule(static)
        for (int64_t t = 0; t < T; ++t) {
            const float *l = logits + t * E;
            double mx = -INFINITY, z = 0.0;
            for (int32_t e = 0; e < E; ++e)
                if ((double)l[e] > mx) mx = (double)l[e];
            for (int32_t e = 0; e < E; ++e) {
                p[e] = exp((double)l[e] - mx);
                z += p[e];
            }
            for (int32_t e = 0; e < E; ++e) {
                p[e] /= z;
                taken[e] = 0;
            }
            double chosen_sum = 0.0;
            for (int32_t j = 0; j < k; ++j) {
                int32_t best = -1;
                for (int32_t e = 0; e < E; ++e) {
                    if (taken[e]) continue;
                    /* strict '>' keeps the lower index on ties */
                    if (best < 0 || p[e] > p[best] ||
                        (p[e] == p[best] && l[e] > l[best]))
                        best = e;
                }
                taken[best] = 1;
                topk_ids[t * k + j] = best;
                topk_w[t * k + j] = p[best];
                chosen_sum += p[best];
            }
            for (int32_t j = 0; j < k; ++j) topk_w[t * k + j] /= chosen_sum;
        }
        free(p);
        free(taken);
    }
}

/* ------------------------------------------------------------------------ */
/* align                                                                     */
/* ------------------------------------------------------------------------ */

typedef struct { int32_t e, a, p; } pair_key;

static int cmp_pair(const void *x, const void *y)
{
    const pair_key *u = (const pair_key *)x, *v = (const pair_key *)y;
    if (u->e != v->e) return u->e < v->e ? -1 : 1;
    if (u->a != v->a) return u->a < v->a ? -1 : 1;
    if (u->p != v->p) return u->p < v->p ? -1 : 1;
    return 0;
}

/*
 * Layout of the sorted, block-padded pair list.  Pair p = t*k + j joins expert
 * e_p = topk_ids[p] and adapter a_t = lora_ids[t].  A pair is valid when
 * 0 <= e_p < E and -1 <= a_t < L; invalid pairs are dropped and counted.
 *
 *   1. Valid pairs are sorted by the key (e_p, a_t, p), ascending.
 *   2. Each expert's pairs are padded to a multiple of BM rows with the sentinel
 *      P = T*k; experts without pairs get no rows.  expert_begin[e] is the first
 *      row of expert e, expert_begin[E] = num_rows.
 *   3. Blocks are the BM-row slices of the rows; block_expert[b] is their expert.
 *   4. Runs are the maximal stretches of rows inside one block that share one
 *      adapter a >= 0 (rows of adapter -1 and padding rows belong to no run), in
 *      row order: runs[i] = {block, adapter, begin_row, end_row}.  block_runs[b] is
 *      the first run of block b and block_runs[num_blocks] = num_runs.
 *
 * totals[0..3] = num_rows, num_blocks, num_runs, num_dropped.
 * Returns 0, or -1 when a capacity is too small (outputs then undefined).
 */
int oracle_align(int64_t T, int32_t E, int32_t k, int32_t L, int32_t BM,
                 const int32_t *topk_ids, const int32_t *lora_ids,
                 int32_t *sorted_p, int64_t cap_rows,
                 int32_t *expert_begin,
                 int32_t *block_expert, int32_t *block_runs, int64_t cap_blocks,
                 int32_t *runs, int64_t cap_runs,
                 int64_t *totals)
{
    const int64_t P = T * (int64_t)k;
    pair_key *keys = (pair_key *)malloc(sizeof(pair_key) * (size_t)(P > 0 ? P : 1));
    int64_t nv = 0, dropped = 0;
    for (int64_t p = 0; p < P; ++p) {
        int32_t e = topk_ids[p], a = lora_ids[p / k];
        if (e < 0 || e >= E || a < -1 || a >= L) { ++dropped; continue; }
        keys[nv].e = e; keys[nv].a = a; keys[nv].p = (int32_t)p; ++nv;
    }
    qsort(keys, (size_t)nv, sizeof(pair_key), cmp_pair);

    /* per-expert counts and padded starts */
    int64_t row = 0, idx = 0;
    for (int32_t e = 0; e < E; ++e) {
        expert_begin[e] = (int32_t)row;
        int64_t n = 0;
        while (idx + n < nv && keys[idx + n].e == e) ++n;
        int64_t padded = (n + BM - 1) / BM * BM;
        if (row + padded > cap_rows) { free(keys); return -1; }
        for (int64_t i = 0; i < padded; ++i)
            sorted_p[row + i] = i < n ? keys[idx + i].p : (int32_t)P;
        for (int64_t b = row / BM; b < (row + padded) / BM; ++b) {
            if (b >= cap_blocks) { free(keys); return -1; }
            block_expert[b] = e;
        }
        row += padded;
        idx += n;
    }
    expert_begin[E] = (int32_t)row;
    const int64_t nb = row / BM;

    /* runs: walk the rows block by block */
    int64_t nr = 0;
    for (int64_t b = 0; b < nb; ++b) {
        block_runs[b] = (int32_t)nr;
        int64_t r = b * BM, end = (b + 1) * BM;
        while (r < end) {
            int32_t p = sorted_p[r];
            if (p == (int32_t)P) { ++r; continue; }
            int32_t a = lora_ids[p / k];
            int64_t s = r;
            while (r < end && sorted_p[r] != (int32_t)P && lora_ids[sorted_p[r] / k] == a) ++r;
            if (a >= 0) {
                if (nr >= cap_runs) { free(keys); return -1; }
                runs[4 * nr + 0] = (int32_t)b;
                runs[4 * nr + 1] = a;
                runs[4 * nr + 2] = (int32_t)s;
                runs[4 * nr + 3] = (int32_t)r;
                ++nr;
            }
        }
    }
    if (nb < cap_blocks + 1) block_runs[nb] = (int32_t)nr;
    totals[0] = row;
    totals[1] = nb;
    totals[2] = nr;
    totals[3] = dropped;
    free(keys);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* forward                                                                   */
/* ------------------------------------------------------------------------ */

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* y[n] = sum_{c < rows} M[c][n] * v[c] for n < cols, M row-major bf16 with row pitch
 * `pitch` (v times the first `rows` rows of M). */
static void vecmat_bf16(const uint16_t *M, int64_t rows, int64_t cols, int64_t pitch,
                        const double *v, double *y)
{
    for (int64_t n = 0; n < cols; ++n) y[n] = 0.0;
    for (int64_t c = 0; c < rows; ++c) {
        const uint16_t *m = M + c * pitch;
        const double vc = v[c];
        for (int64_t n = 0; n < cols; ++n) y[n] += bf16_to_double(m[n]) * vc;
    }
}

/* y[n] = sum_c M[n][c] * v[c] for n < rows, M row-major bf16 with row pitch `pitch`. */
static void matvec_bf16(const uint16_t *M, int64_t rows, int64_t cols, int64_t pitch,
                        const double *v, double *y)
{
    for (int64_t n = 0; n < rows; ++n) {
        const uint16_t *m = M + n * pitch;
        double acc = 0.0;
        #pragma omp simd reduction(+ : acc)
        for (int64_t c = 0; c < cols; ++c) acc += bf16_to_double(m[c]) * v[c];
        y[n] = acc;
    }
}

/*
 * out[i][:] for token t = tokens[i] (all tokens when tokens == NULL, i = t):
 *   out_t = sum over valid pairs (t, j) of w_{t,j} * d_{t,j}, where with e = topk_ids[t][j],
 *   a = lora_ids[t], r = ranks[a]:
 *     g   = W_gu[e] x_t                                   (2I)
 *     g  += (A_gu[a][e][0:r, :] x_t) B_gu[a][e][0:r, :]   if a >= 0   (gate_up shrink, expand)
 *     h_i = silu(g_i) * g_{I+i}                           (I)
 *     d   = W_dn[e] h                                     (H)
 *     d  += (A_dn[a][e][0:r, :] h) B_dn[a][e][0:r, :]     if a >= 0   (down shrink, expand)
 * Tokens without a valid pair get out_t = 0.  *n_dropped counts invalid pairs seen.
 */
void oracle_forward(int64_t T, int32_t H, int32_t I, int32_t E, int32_t k, int32_t L,
                    int32_t r_max, const int32_t *ranks,
                    const uint16_t *x, const int32_t *topk_ids, const float *topk_w,
                    const int32_t *lora_ids,
                    const uint16_t *W_gu, const uint16_t *W_dn,
                    const uint16_t *A_gu, const uint16_t *B_gu,
                    const uint16_t *A_dn, const uint16_t *B_dn,
                    const int64_t *tokens, int64_t n_tokens,
                    double *out, int64_t *n_dropped)
{
    const int64_t n_out = tokens ? n_tokens : T;
    int64_t dropped = 0;
    #pragma omp parallel reduction(+ : dropped)
    {
        double *xt = (double *)malloc(sizeof(double) * (size_t)H);
        double *g = (double *)malloc(sizeof(double) * (size_t)(2 * I));
        double *h = (double *)malloc(sizeof(double) * (size_t)I);
        double *d = (double *)malloc(sizeof(double) * (size_t)H);
        double *s = (double *)malloc(sizeof(double) * (size_t)(r_max > 0 ? r_max : 1));
        double *u = (double *)malloc(sizeof(double) * (size_t)(2 * I > H ? 2 * I : H));
        #pragma omp for schedule(dynamic, 1)
        for (int64_t i = 0; i < n_out; ++i) {
            const int64_t t = tokens ? tokens[i] : i;
            double *o = out + i * H;
            for (int32_t c = 0; c < H; ++c) o[c] = 0.0;
            for (int32_t c = 0; c < H; ++c) xt[c] = bf16_to_double(x[t * H + c]);
            const int32_t a = lora_ids[t];
            for (int32_t j = 0; j < k; ++j) {
                const int32_t e = topk_ids[t * k + j];
                if (e < 0 || e >= E || a < -1 || a >= L) { ++dropped; continue; }
                const double w = (double)topk_w[t * k + j];

                /* gate_up projection */
                matvec_bf16(W_gu + (int64_t)e * 2 * I * H, 2 * (int64_t)I, H, H, xt, g);
                if (a >= 0) {
                    const int32_t r = ranks[a];
                    const int64_t ae = (int64_t)a * E + e;
                    /* gate_up shrink: s = A x */
                    matvec_bf16(A_gu + ae * r_max * H, r, H, H, xt, s);
                    /* gate_up expand: g += s B (B: r_max rows of 2I) */
                    vecmat_bf16(B_gu + ae * r_max * 2 * I, r, 2 * (int64_t)I, 2 * (int64_t)I, s, u);
                    for (int32_t n = 0; n < 2 * I; ++n) g[n] += u[n];
                }
                for (int32_t c = 0; c < I; ++c) h[c] = silu(g[c]) * g[I + c];

                /* down projection */
                matvec_bf16(W_dn + (int64_t)e * H * I, H, I, I, h, d);
                if (a >= 0) {
                    const int32_t r = ranks[a];
                    const int64_t ae = (int64_t)a * E + e;
                    matvec_bf16(A_dn + ae * r_max * I, r, I, I, h, s);          /* down shrink */
                    vecmat_bf16(B_dn + ae * r_max * H, r, H, H, s, u);          /* down expand */
                    for (int32_t n = 0; n < H; ++n) d[n] += u[n];
                }
                /* weighted combine over the k experts */
                for (int32_t c = 0; c < H; ++c) o[c] += w * d[c];
            }
        }
        free(xt); free(g); free(h); free(d); free(s); free(u);
    }
    if (n_dropped) *n_dropped = dropped;
}
