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
 * same values: each logit is accumulated from 0 with one correctly rounded
 * fused multiply-add per feature, in increasing feature index i, and the bias
 * (when present) is added last in fp32:
 *
 *     acc = 0;  for i in 0..d-1: acc = fma(x[t][i], w_r[i][e], acc);  acc += b[e]
 *
 * Layout: x [T][d], w_r [d][N], b [N] (or NULL), logits [T][N], all row-major.
 */
#include <math.h>
#include <stddef.h>

void oracle_router_logits(long T, long d, long N, const float *x, const float *w_r,
                          const float *bias, float *logits)
{
    for (long t = 0; t < T; ++t) {
        float *acc = logits + t * N;
        for (long e = 0; e < N; ++e)
            acc[e] = 0.0f;
        /* Loop order (i outer, e inner) keeps each logit's own additions in
           increasing i; it only lets independent logits advance together. */
        for (long i = 0; i < d; ++i) {
            const float xi = x[t * d + i];
            const float *w = w_r + i * N;
            for (long e = 0; e < N; ++e)
                acc[e] = fmaf(xi, w[e], acc[e]);
        }
        if (bias)
            for (long e = 0; e < N; ++e)
                acc[e] = acc[e] + bias[e];
    }
}
