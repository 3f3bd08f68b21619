/*
 * moe_oracle.c -- plain, slow, obviously-correct CPU oracle of the MoE expert
 * layer (route -> permute into 128-row expert blocks -> grouped gate/up GEMM
 * with SiLU(gate)*up -> grouped down GEMM -> top-k weighted combine).
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the
 * benchmark's CPU-baseline leg may load this library.  It shares no code,
 * header, table or helper with the CUDA library it checks.
 *
 * Sources (page titles; sections as printed on each page):
 *   [P1] "通算融合算子（三）：ThunderKittens 多卡编程与可融合的 GEMM 模板", §4
 *        (grouped GEMM walk-through: rows grouped by expert, 128 rows = task
 *        block = expert alignment unit, expert-major task order).
 *   [P2] "通算融合算子（一）：为什么要把通信写进 GEMM kernel 里", §1 (the serial
 *        layer: gate/up GEMM -> SiLU -> down GEMM) and §4 (table of the four
 *        data-flow patterns: "dispatch + GEMM" reorders rows by the route,
 *        "GEMM + combine" is the top-k weighted reduction).
 *   [P3] "Lecture 11: Programming Systems for Specialized Hardware", example 4
 *        (softmax as Map(exp) -> Reduce(+) -> Zip(/)).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - softmax subtracts the row maximum before exp (an identity of the
 *     quotient; the simplified form of [P3] overflows for large logits);
 *   - top-k ranks by logit, descending, ties to the lower expert index; slot j
 *     holds the j-th pick;
 *   - weights are renormalised over the k picks in slot order;
 *   - inside an expert, rows are ordered by ascending token (stable);
 *   - padding rows of a block carry gather index -1 and are never computed;
 *   - gate and up are accumulated exactly (double), rounded once to float32,
 *     SiLU(g)*u is formed in double, rounded to float32 and then to bf16;
 *   - the down projection is accumulated in double, rounded to float32 and
 *     then to bf16;
 *   - the combine accumulates w_j * y_j in float32 in slot order, each product
 *     and each sum rounded to float32 (no fused multiply-add), and rounds the
 *     sum to bf16.
 * All roundings are round-to-nearest-even.  Build with -ffp-contract=off so
 * the compiler does not fuse the float32 multiply and add of the combine.
 *
 * Arrays: bf16 values are passed as raw uint16 bit patterns; all tensors are
 * dense row-major.  W_gate, W_up are [E][H][I]; W_down is [E][I][H].
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_ROW_BLOCK 128 /* [P1] §4: 128 rows per task block and per expert alignment */

/* ------------------------------------------------------------------ bf16 */

/* IEEE-754 binary32 -> bfloat16, round to nearest, ties to even: keep the top
 * 16 bits and add one unit when the dropped 16 bits exceed one half, or equal
 * one half and the kept part is odd.  A carry out of the mantissa increments
 * the exponent, which is the correct rounded value (up to +-inf). */
uint16_t oracle_bf16_from_f32(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu) != 0u)
        return (uint16_t)((u >> 16) | 0x0040u); /* NaN stays a (quiet) NaN */
    uint32_t kept = u >> 16;
    uint32_t dropped = u & 0xFFFFu;
    if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u)))
        kept += 1u;
    return (uint16_t)kept;
}

float oracle_f32_from_bf16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

void oracle_bf16_from_f32_array(int64_t n, const float *in, uint16_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_bf16_from_f32(in[i]);
}

int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void oracle_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* --------------------------------------------------------------- routing */

/* Route selection for every token ([P2] §4 "dispatch + GEMM" needs the route;
 * softmax per [P3] example 4):
 *   p_e = exp(l_e - max l) / sum_e exp(l_e - max l)        (double)
 *   picks: the k largest logits, ties to the lower index  (slot order)
 *   w_j = p_{id_j} / sum_{j'} p_{id_j'}                    (double -> float32)
 */
void oracle_route_select(int T, int E, int k, const float *logits,
                         int32_t *topk_ids, float *topk_w)
{
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)E);
        char *taken = (char *)malloc((size_t)E);
#pragma omp for schedule(static)
        for (int t = 0; t < T; ++t) {
            const float *l = logits + (int64_t)t * E;
            float m = l[0];
            for (int e = 1; e < E; ++e)
                if (l[e] > m)
                    m = l[e];
            double Z = 0.0;
            for (int e = 0; e < E; ++e) {
                p[e] = exp((double)l[e] - (double)m);
                Z += p[e];
            }
            for (int e = 0; e < E; ++e)
                p[e] = p[e] / Z;

            memset(taken, 0, (size_t)E);
            double S = 0.0;
            for (int j = 0; j < k; ++j) {
                int best = -1;
                for (int e = 0; e < E; ++e) {
                    if (taken[e])
                        continue;
                    if (best < 0 || l[e] > l[best]) /* strict: ties keep the lower index */
                        best = e;
                }
                taken[best] = 1;
                topk_ids[(int64_t)t * k + j] = best;
                S += p[best];
            }
            for (int j = 0; j < k; ++j)
                topk_w[(int64_t)t * k + j] = (float)(p[topk_ids[(int64_t)t * k + j]] / S);
        }
        free(p);
        free(taken);
    }
}

/* Upper bound on the number of 128-row blocks over all routings. */
int64_t oracle_max_blocks(int T, int E, int k)
{
    int64_t R = (int64_t)T * k;
    int64_t touched = R < E ? R : E;
    return (R + (ORACLE_ROW_BLOCK - 1) * touched) / ORACLE_ROW_BLOCK;
}

/* Expert-contiguous, 128-row-aligned grouping of the T*k routed rows
 * ([P1] §4: rows grouped by expert, 128 = expert alignment unit; [P2] §4:
 * rows reordered by the route):
 *   counts[e]        number of (t, j) with topk_ids[t,j] == e
 *   off_pad[e]       sum_{e' < e} ceil(counts[e'] / 128) * 128, off_pad[E] = R_pad
 *   block_expert[b]  expert owning rows [128 b, 128 b + 128)
 *   num_blocks       R_pad / 128
 *   scatter_idx[t,j] off_pad[e] + #{(t', j') : t' < t, topk_ids[t', j'] == e}
 *   gather_idx[row]  t for the row of (t, j), -1 for padding rows
 * Returns 0, or -1 when max_rows is too small. */
int oracle_route_permute(int T, int E, int k, const int32_t *topk_ids,
                         int32_t *counts, int32_t *off_pad,
                         int32_t *block_expert, int32_t *num_blocks,
                         int32_t *gather_idx, int32_t *scatter_idx,
                         int64_t max_rows)
{
    for (int e = 0; e < E; ++e)
        counts[e] = 0;
    for (int64_t i = 0; i < (int64_t)T * k; ++i)
        counts[topk_ids[i]] += 1;

    off_pad[0] = 0;
    for (int e = 0; e < E; ++e) {
        int32_t padded = (counts[e] + ORACLE_ROW_BLOCK - 1) / ORACLE_ROW_BLOCK * ORACLE_ROW_BLOCK;
        off_pad[e + 1] = off_pad[e] + padded;
    }
    if ((int64_t)off_pad[E] > max_rows)
        return -1;
    *num_blocks = off_pad[E] / ORACLE_ROW_BLOCK;

    for (int e = 0; e < E; ++e)
        for (int32_t b = off_pad[e] / ORACLE_ROW_BLOCK; b < off_pad[e + 1] / ORACLE_ROW_BLOCK; ++b)
            block_expert[b] = e;

    for (int32_t r = 0; r < off_pad[E]; ++r)
        gather_idx[r] = -1;

    int32_t *next = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (int t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            int e = topk_ids[(int64_t)t * k + j];
            int32_t row = off_pad[e] + next[e];
            next[e] += 1;
            scatter_idx[(int64_t)t * k + j] = row;
            gather_idx[row] = t;
        }
    }
    free(next);
    return 0;
}

/* ---------------------------------------------------------- expert FFN */

/* One routed row through one expert's gate/up projection ([P2] §1: gate/up
 * GEMM then SiLU):
 *   g_i = sum_h x_h Wg[h][i],  u_i = sum_h x_h Wu[h][i]   (double, ascending h)
 *   h_i = bf16(f32(silu(f32(g_i)) * f32(u_i)))            silu(g) = g / (1 + e^-g)
 * acc must hold 2*I doubles. */
void oracle_expert_up_row(int H, int I, const uint16_t *x, const uint16_t *wg,
                          const uint16_t *wu, uint16_t *h, double *acc)
{
    double *g = acc;
    double *u = acc + I;
    for (int i = 0; i < I; ++i) {
        g[i] = 0.0;
        u[i] = 0.0;
    }
    for (int hh = 0; hh < H; ++hh) {
        double xv = (double)oracle_f32_from_bf16(x[hh]);
        const uint16_t *wg_row = wg + (int64_t)hh * I;
        const uint16_t *wu_row = wu + (int64_t)hh * I;
        for (int i = 0; i < I; ++i) {
            g[i] += xv * (double)oracle_f32_from_bf16(wg_row[i]);
            u[i] += xv * (double)oracle_f32_from_bf16(wu_row[i]);
        }
    }
    for (int i = 0; i < I; ++i) {
        float gf = (float)g[i];
        float uf = (float)u[i];
        double silu = (double)gf / (1.0 + exp(-(double)gf));
        float hv = (float)(silu * (double)uf);
        h[i] = oracle_bf16_from_f32(hv);
    }
}

/* One row through one expert's down projection ([P2] §1: down GEMM):
 *   y_c = bf16(f32(sum_i h_i Wd[i][c]))   (double, ascending i)
 * acc must hold H doubles. */
void oracle_expert_down_row(int H, int I, const uint16_t *h, const uint16_t *wd,
                            uint16_t *y, double *acc)
{
    for (int c = 0; c < H; ++c)
        acc[c] = 0.0;
    for (int i = 0; i < I; ++i) {
        double hv = (double)oracle_f32_from_bf16(h[i]);
        const uint16_t *wd_row = wd + (int64_t)i * H;
        for (int c = 0; c < H; ++c)
            acc[c] += hv * (double)oracle_f32_from_bf16(wd_row[c]);
    }
    for (int c = 0; c < H; ++c)
        y[c] = oracle_bf16_from_f32((float)acc[c]);
}

/* Grouped gate/up over the permuted rows ([P1] §4: each 128-row block
 * multiplies the weights of its own expert).  Rows with gather_idx < 0 are
 * padding and are left untouched.  h is [num_blocks*128][I]. */
void oracle_grouped_up(int T, int H, int I, int E, int32_t num_blocks,
                       const int32_t *block_expert, const int32_t *gather_idx,
                       const uint16_t *X, const uint16_t *Wg, const uint16_t *Wu,
                       uint16_t *h)
{
    int64_t rows = (int64_t)num_blocks * ORACLE_ROW_BLOCK;
    (void)T;
    (void)E;
#pragma omp parallel
    {
        double *acc = (double *)malloc(sizeof(double) * 2 * (size_t)I);
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < rows; ++r) {
            int32_t t = gather_idx[r];
            if (t < 0)
                continue;
            int e = block_expert[r / ORACLE_ROW_BLOCK];
            oracle_expert_up_row(H, I, X + (int64_t)t * H, Wg + (int64_t)e * H * I,
                                 Wu + (int64_t)e * H * I, h + r * I, acc);
        }
        free(acc);
    }
}

/* Grouped down over the permuted rows; Y is [num_blocks*128][H]. */
void oracle_grouped_down(int H, int I, int E, int32_t num_blocks,
                         const int32_t *block_expert, const int32_t *gather_idx,
                         const uint16_t *h, const uint16_t *Wd, uint16_t *Y)
{
    int64_t rows = (int64_t)num_blocks * ORACLE_ROW_BLOCK;
    (void)E;
#pragma omp parallel
    {
        double *acc = (double *)malloc(sizeof(double) * (size_t)H);
#pragma omp for schedule(dynamic, 4)
        for (int64_t r = 0; r < rows; ++r) {
            if (gather_idx[r] < 0)
                continue;
            int e = block_expert[r / ORACLE_ROW_BLOCK];
            oracle_expert_down_row(H, I, h + r * I, Wd + (int64_t)e * I * H, Y + r * H, acc);
        }
        free(acc);
    }
}

/* Top-k weighted combine back to token order ([P2] §4 "GEMM + combine"):
 *   out[t][c] = bf16( sum_{j = 0..k-1} w[t][j] * Y[scatter_idx[t][j]][c] )
 * float32 accumulator in slot order, products and sums each rounded. */
void oracle_combine(int T, int H, int k, const uint16_t *Y,
                    const int32_t *scatter_idx, const float *topk_w, uint16_t *out)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; ++t) {
        for (int c = 0; c < H; ++c) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                int64_t row = scatter_idx[(int64_t)t * k + j];
                float prod = topk_w[(int64_t)t * k + j] * oracle_f32_from_bf16(Y[row * H + c]);
                acc = acc + prod;
            }
            out[(int64_t)t * H + c] = oracle_bf16_from_f32(acc);
        }
    }
}

/* The layer output of a list of tokens, computed token by token from the
 * route (same arithmetic as the grouped path, without the permutation):
 * used to check single outputs of workloads too large for the full oracle.
 * ids/w are [ntok][k] (the route of each listed token); out is [ntok][H];
 * y_out, when not NULL, receives the k expert outputs [ntok][k][H]. */
void oracle_tokens_out(int ntok, const int32_t *tokens, int H, int I, int k,
                       const int32_t *ids, const float *w, const uint16_t *X,
                       const uint16_t *Wg, const uint16_t *Wu, const uint16_t *Wd,
                       uint16_t *out, uint16_t *h_out, uint16_t *y_out)
{
    /* parallel over (token, slot) pairs, then a sequential combine */
    int64_t pairs = (int64_t)ntok * k;
    uint16_t *ys = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)pairs * H);
    uint16_t *hs = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)pairs * I);
#pragma omp parallel
    {
        double *acc = (double *)malloc(sizeof(double) * (size_t)(2 * I > H ? 2 * I : H));
#pragma omp for schedule(dynamic, 1)
        for (int64_t pj = 0; pj < pairs; ++pj) {
            int64_t n = pj / k;
            int e = ids[pj];
            int64_t t = tokens[n];
            oracle_expert_up_row(H, I, X + t * H, Wg + (int64_t)e * H * I,
                                 Wu + (int64_t)e * H * I, hs + pj * I, acc);
            oracle_expert_down_row(H, I, hs + pj * I, Wd + (int64_t)e * I * H,
                                   ys + pj * H, acc);
        }
        free(acc);
    }
    for (int64_t n = 0; n < ntok; ++n) {
        for (int c = 0; c < H; ++c) {
            float acc = 0.0f;
            for (int j = 0; j < k; ++j) {
                float prod = w[n * k + j] * oracle_f32_from_bf16(ys[(n * k + j) * H + c]);
                acc = acc + prod;
            }
            out[n * H + c] = oracle_bf16_from_f32(acc);
        }
    }
    if (y_out)
        memcpy(y_out, ys, sizeof(uint16_t) * (size_t)pairs * H);
    if (h_out)
        memcpy(h_out, hs, sizeof(uint16_t) * (size_t)pairs * I);
    free(ys);
    free(hs);
}
