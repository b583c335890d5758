/*
 * CPU oracle: router logits in single precision.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this file's library; the CUDA product path never does.
 *
 * The router is one linear layer that maps a token's hidden state to one
 * logit per expert ("Noise Top-k Gating" glossary, paragraph on the router as
 * a small trainable network; "MoE: Choosing Which MLPs to Use for Each Token",
 * section "Router: Selecting Experts and Computing Weights", Figure 2, where
 * W_r is d x N; the DeepSeekMoE layer equation, affinity u_t^T e_i). The
 * Switch explainer ("Making it work") keeps the router in higher precision than
 * the experts, so the logits are fp32 here.
 *
 * The pages fix no summation order. The top-k choice is an integer decision
 * taken on these fp32 values, so the oracle and the CUDA router take it on the
 * same values, computed in this order:
 *
 *   1. The features are cut into blocks of 8 (block b holds features 8b..8b+7).
 *      Partial sum p_l (l = 0..31) starts at 0 and takes, in increasing feature
 *      index, every feature whose block number b satisfies b mod 32 == l, each
 *      with one correctly rounded fused multiply-add: p_l = fma(x_i, w_ie, p_l).
 *   2. The 32 partials are combined by five pairwise rounds: for o = 16, 8, 4,
 *      2, 1, every p_l becomes p_l + p_(l xor o) (all l at once). The logit is
 *      p_0 after the fifth round.
 *   3. The bias (when present) is added last in fp32.
 *
 * Layout: x [T][d], w_r [d][N], b [N] (or NULL), logits [T][N], all row-major.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define LANES 32
#define BLOCK 8

void oracle_router_logits(long T, long d, long N, const float *x, const float *w_r,
                          const float *bias, float *logits)
{
    /* part[l][e]: partial l of expert e for the current token */
    float *part = (float *)malloc(sizeof(float) * LANES * (size_t)N);
    float *next = (float *)malloc(sizeof(float) * LANES * (size_t)N);
    for (long t = 0; t < T; ++t) {
        memset(part, 0, sizeof(float) * LANES * (size_t)N);
        /* step 1: feature i goes to partial (i / 8) mod 32; features of one
           partial are visited in increasing order (the e loop only lets the
           independent experts advance together) */
        for (long i = 0; i < d; ++i) {
            const long l = (i / BLOCK) % LANES;
            const float xi = x[t * d + i];
            const float *w = w_r + i * N;
            float *p = part + l * N;
            for (long e = 0; e < N; ++e)
                p[e] = fmaf(xi, w[e], p[e]);
        }
        /* step 2: five pairwise rounds */
        for (int o = LANES / 2; o >= 1; o /= 2) {
            for (int l = 0; l < LANES; ++l)
                for (long e = 0; e < N; ++e)
                    next[l * N + e] = part[l * N + e] + part[(l ^ o) * N + e];
            float *tmp = part;
            part = next;
            next = tmp;
        }
        /* step 3: bias */
        for (long e = 0; e < N; ++e)
            logits[t * N + e] = bias ? part[e] + bias[e] : part[e];
    }
    free(part);
    free(next);
}
