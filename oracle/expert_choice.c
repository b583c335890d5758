/*
 * CPU oracle: Expert Choice scores in single precision.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg load this file's library; the CUDA product path never does.
 *
 * Expert Choice inverts the routing: every expert picks its top tokens ("Mixture
 * of Experts (MoE)" glossary, sparse-MoE list). The scores are the router's
 * probability distribution over experts for each token (glossary, gating-network
 * paragraph: a softmax over all experts), and expert e keeps the tokens with the
 * largest S[t][e]. That choice compares fp32 scores across tokens, so this oracle
 * and the CUDA kernel compute S with the same fp32 operations, each correctly
 * rounded, in this order:
 *
 *   m_t  = max_e L[t][e]
 *   u_te = ec_exp(L[t][e] - m_t)        (the difference rounded to fp32)
 *   Z_t  = ((u_t0 + u_t1) + u_t2) + ... (experts ascending, each sum rounded)
 *   S_te = u_te / Z_t                   (rounded to fp32)
 *
 * ec_exp is an exponential assembled from named published steps rather than a
 * library call:
 *   - the argument reduction of Cody and Waite (W. J. Cody, W. Waite, "Software
 *     Manual for the Elementary Functions", 1980): n = nearest integer (ties to
 *     even) to x * log2(e), r = x - n ln2 in two fused steps, ln2 being split into
 *     a high part of 16 significant bits (so n * ln2_hi is exact for |n| <= 256) and
 *     the remainder ln2_lo;
 *   - e^r from its Taylor series up to degree 7 (|r| <= ln2 / 2, truncation error
 *     below 6e-9 relative), evaluated by Horner's rule with fused multiply-adds;
 *   - the product with the power of two 2^n (exact scaling).
 * The constants are ln2_hi = ln2 rounded to 16 bits, ln2_lo = fp32(ln2 - ln2_hi),
 * log2(e) and 1/k! rounded to fp32, written as hexadecimal literals. Arguments
 * below -87 (where e^x approaches the smallest normal float) give 0; the scores
 * only need x <= 0.
 *
 * Layout: L [T][N] and S [T][N] row-major fp32.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static const float LOG2E = 0x1.715476p+0f;
static const float LN2_HI = 0x1.62e4p-1f;
static const float LN2_LO = 0x1.7f7d1cp-20f;
static const float C2 = 0x1.0p-1f;     /* 1/2! */
static const float C3 = 0x1.555556p-3f; /* 1/3! */
static const float C4 = 0x1.555556p-5f; /* 1/4! */
static const float C5 = 0x1.111112p-7f; /* 1/5! */
static const float C6 = 0x1.6c16c2p-10f; /* 1/6! */
static const float C7 = 0x1.a01a02p-13f; /* 1/7! */

float oracle_ec_exp(float x)
{
    if (!(x >= -87.0f)) return 0.0f;
    const float nf = nearbyintf(x * LOG2E);          /* ties to even (default mode) */
    const int n = (int)nf;
    float r = fmaf(-nf, LN2_HI, x);                  /* exact product, one rounding */
    r = fmaf(-nf, LN2_LO, r);
    float p = C7;
    p = fmaf(p, r, C6);
    p = fmaf(p, r, C5);
    p = fmaf(p, r, C4);
    p = fmaf(p, r, C3);
    p = fmaf(p, r, C2);
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    const uint32_t bits = (uint32_t)(n + 127) << 23;  /* 2^n, n in [-126, 0] here */
    float scale;
    memcpy(&scale, &bits, sizeof scale);
    return p * scale;
}

void oracle_ec_scores(long T, long N, const float *L, float *S)
{
    for (long t = 0; t < T; ++t) {
        const float *l = L + t * N;
        float *s = S + t * N;
        float m = l[0];
        for (long e = 1; e < N; ++e)
            if (l[e] > m) m = l[e];
        float z = 0.0f;
        for (long e = 0; e < N; ++e) {
            s[e] = oracle_ec_exp(l[e] - m);
            z = z + s[e];
        }
        for (long e = 0; e < N; ++e)
            s[e] = s[e] / z;
    }
}

void oracle_ec_exp_array(long n, const float *x, float *y)
{
    for (long i = 0; i < n; ++i)
        y[i] = oracle_ec_exp(x[i]);
}
