// Expert Choice routing: every expert picks its top tokens ("Mixture of Experts
// (MoE)" glossary, sparse-MoE list: Expert Choice inverts the routing).
//
// From the router logits L [T][N] (router.cu, the usual fp32 summation order):
//   k_ec_scores  one thread per token: the scores S = softmax over experts, in the
//                fixed fp32 steps below, written transposed (S_t [N][T]) so that an
//                expert's column is contiguous;
//   k_ec_select  one CTA per expert: chooses the expert's first Ce = min(C, T) tokens
//                by (score descending, token ascending) with a radix selection of the
//                score bits in shared memory, and writes them
//                in ascending token order as rows e*Ce .. e*Ce + Ce - 1 (perm_token,
//                row_gate = the score), plus the row of every (expert, token) pair
//                (-1 if not chosen) and, per token, how many experts chose it;
//   k_ec_scan / k_ec_fill  per-token row lists in expert order (tok_ptr, tok_rows);
//   k_combine_ec y_t = x_t + S(x_t) + sum of gate * y_perm over the token's rows
//                (fp32, expert order), like the token-choice combine.
// The experts in between are the grouped FFN of the token-choice path, on segments
// of Ce rows.
//
// The choice compares fp32 scores across tokens, so the scores are computed with
// the same correctly rounded fp32 operations as the CPU oracle:
//   m = max_e L[t][e];  u_e = ec_exp(L[t][e] - m);  Z = u_0 + u_1 + ... (ascending);
//   S[t][e] = u_e / Z.
// ec_exp: the argument reduction of Cody and Waite (Software Manual for the
// Elementary Functions, 1980) with ln 2 split into a 16-bit high part and its fp32
// remainder, e^r by its degree-7 Taylor series (Horner, fused multiply-adds), and an
// exact scaling by 2^n; arguments below -87 give 0.
#include <algorithm>
#include <cstdint>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr float kLog2e = 0x1.715476p+0f;
constexpr float kLn2Hi = 0x1.62e4p-1f;
constexpr float kLn2Lo = 0x1.7f7d1cp-20f;
constexpr float kC2 = 0x1.0p-1f, kC3 = 0x1.555556p-3f, kC4 = 0x1.555556p-5f;
constexpr float kC5 = 0x1.111112p-7f, kC6 = 0x1.6c16c2p-10f, kC7 = 0x1.a01a02p-13f;

__device__ __forceinline__ float ec_exp(float x) {
    if (!(x >= -87.0f)) return 0.0f;
    const float nf = rintf(__fmul_rn(x, kLog2e));  // nearest integer, ties to even
    const int n = (int)nf;
    float r = __fmaf_rn(-nf, kLn2Hi, x);
    r = __fmaf_rn(-nf, kLn2Lo, r);
    float p = kC7;
    p = __fmaf_rn(p, r, kC6);
    p = __fmaf_rn(p, r, kC5);
    p = __fmaf_rn(p, r, kC4);
    p = __fmaf_rn(p, r, kC3);
    p = __fmaf_rn(p, r, kC2);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    return __fmul_rn(p, __uint_as_float((uint32_t)(n + 127) << 23));
}

__global__ void __launch_bounds__(256) k_ec_scores(const float *__restrict__ L, int T, int N,
                                                   float *__restrict__ S_t, int32_t *__restrict__ tok_cnt) {
    pdl_enter();
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    const float *l = L + (size_t)t * N;
    float m = l[0];
    for (int e = 1; e < N; ++e)
        if (l[e] > m) m = l[e];
    float z = 0.0f;
    for (int e = 0; e < N; ++e) z = __fadd_rn(z, ec_exp(__fsub_rn(l[e], m)));
    for (int e = 0; e < N; ++e) S_t[(size_t)e * T + t] = __fdiv_rn(ec_exp(__fsub_rn(l[e], m)), z);
    tok_cnt[t] = 0;
}

// Exclusive scan of one int per thread over the block (blockDim.x a multiple of 32,
// at most 1024); *total receives the sum.
__device__ int block_scan(int v, int *sh, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) sh[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? sh[lane] : 0;
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, wi, o);
            if (lane >= o) wi += u;
        }
        if (lane < nw) sh[lane] = wi - w;
        if (lane == 31) sh[32] = wi;
    }
    __syncthreads();
    const int ex = sh[warp] + incl - v;
    *total = sh[32];
    __syncthreads();
    return ex;
}

struct SelectArgs {
    const float *S_t;  // [N][T]
    int T, N, Ce;
    int32_t *ec_row;   // [N][T]
    int32_t *tok_cnt;  // [T]
    int32_t *offsets;  // [N+1]
    int32_t *perm_token;
    float *row_gate;
};

__global__ void __launch_bounds__(1024) k_ec_select(SelectArgs a) {
    extern __shared__ __align__(16) uint8_t sm[];
    uint32_t *bits = reinterpret_cast<uint32_t *>(sm);        // [T] score bits
    uint8_t *flag = reinterpret_cast<uint8_t *>(bits + a.T);  // [T]
    __shared__ int sh[33];
    __shared__ int hist[256];
    __shared__ uint32_t s_prefix;
    __shared__ int s_need;
    const int e = blockIdx.x, tid = threadIdx.x, nt = blockDim.x;
    const int lane = tid & 31, warp = tid >> 5;
    const float *s = a.S_t + (size_t)e * a.T;
    pdl_enter();
    // Non-negative floats order like their bits (a NaN's bits above every number), so
    // the expert's first Ce tokens by (score descending, token ascending) are: every
    // token whose score bits exceed the Ce-th largest score's bits P, and of the tokens
    // at P the lowest `need`. P is found a byte at a time from the top (radix selection):
    // a histogram of the next byte over the tokens that match P's bytes so far, then the
    // byte where the count from the top reaches the number still to choose.
    for (int i = tid; i < a.T; i += nt) {
        bits[i] = __float_as_uint(s[i]);
        flag[i] = 0;
    }
    uint32_t prefix = 0;
    int need = a.Ce;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = tid; i < 256; i += nt) hist[i] = 0;
        __syncthreads();
        for (int i = tid; i < a.T; i += nt) {
            const uint32_t u = bits[i];
            if (pass == 0 || (u >> (shift + 8)) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1);
        }
        __syncthreads();
        if (warp == 0) {
            // lane l holds bytes 255 - 8l .. 248 - 8l (from the top): counts from the top
            int c[8], sum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = hist[255 - 8 * lane - j];
                sum += c[j];
            }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += u;
            }
            const int before = incl - sum;  // tokens in higher bytes than this lane's
            const unsigned hit = __ballot_sync(0xffffffffu, before < need && incl >= need);
            if (lane == __ffs(hit) - 1) {
                int cum = before, j = 0;
                while (cum + c[j] < need) cum += c[j++];
                s_prefix = (prefix << 8) | (uint32_t)(255 - 8 * lane - j);
                s_need = need - cum;
            }
        }
        __syncthreads();
        prefix = s_prefix;
        need = s_need;
    }
    // flags: above P, or at P among the lowest `need` tokens (token order)
    {
        const int per = (a.T + nt - 1) / nt;
        const int beg = min(a.T, tid * per), end = min(a.T, beg + per);
        int eq = 0;
        for (int t = beg; t < end; ++t) eq += bits[t] == prefix;
        int total_eq;
        int rank = block_scan(eq, sh, &total_eq);
        for (int t = beg; t < end; ++t) {
            const uint32_t u = bits[t];
            if (u > prefix) flag[t] = 1;
            else if (u == prefix) flag[t] = rank++ < need ? 1 : 0;
        }
    }
    __syncthreads();
    // rows of the chosen tokens in ascending token order
    const int per = (a.T + nt - 1) / nt;
    const int beg = min(a.T, tid * per), end = min(a.T, beg + per);
    int c = 0;
    for (int t = beg; t < end; ++t) c += flag[t];
    int total;
    int pos = block_scan(c, sh, &total);
    const int32_t row0 = e * a.Ce;
    for (int t = beg; t < end; ++t) {
        int32_t r = -1;
        if (flag[t]) {
            r = row0 + pos++;
            a.perm_token[r] = t;
            a.row_gate[r] = s[t];
            atomicAdd(&a.tok_cnt[t], 1);
        }
        a.ec_row[(size_t)e * a.T + t] = r;
    }
    if (tid == 0) {
        a.offsets[e] = row0;
        if (e == a.N - 1) a.offsets[a.N] = a.N * a.Ce;
    }
}

// One CTA: tok_ptr = exclusive scan of the per-token counts, in token order.
__global__ void __launch_bounds__(1024) k_ec_scan(const int32_t *__restrict__ tok_cnt, int T,
                                                  int32_t *__restrict__ tok_ptr) {
    __shared__ int sh[33];
    const int tid = threadIdx.x, nt = blockDim.x;
    const int per = (T + nt - 1) / nt;
    pdl_enter();
    const int beg = min(T, tid * per), end = min(T, beg + per);
    int c = 0;
    for (int t = beg; t < end; ++t) c += tok_cnt[t];
    int total;
    int run = block_scan(c, sh, &total);
    for (int t = beg; t < end; ++t) {
        tok_ptr[t] = run;
        run += tok_cnt[t];
    }
    if (tid == 0) tok_ptr[T] = total;
}

// One thread per token: its rows in expert order.
__global__ void __launch_bounds__(256) k_ec_fill(const int32_t *__restrict__ ec_row, const int32_t *__restrict__ tok_ptr,
                                                 int T, int N, int32_t *__restrict__ tok_rows) {
    pdl_enter();
    const int t = blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    int p = tok_ptr[t];
    for (int e = 0; e < N; ++e) {
        const int32_t r = ec_row[(size_t)e * T + t];
        if (r >= 0) tok_rows[p++] = r;
    }
}

template <typename T, bool SHARED>
__global__ void __launch_bounds__(256) k_combine_ec(const T *__restrict__ x, const T *__restrict__ y_perm,
                                                    const T *__restrict__ s_out, const int32_t *__restrict__ tok_ptr,
                                                    const int32_t *__restrict__ tok_rows,
                                                    const float *__restrict__ row_gate, int Ttok, int d, int64_t rmax,
                                                    T *__restrict__ y, uint32_t *err) {
    constexpr int V = Vec16<T>::n;
    const int vpr = d / V;
    const int64_t total = (int64_t)Ttok * vpr;
    pdl_enter();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / vpr);
        const int v = (int)(i - (int64_t)t * vpr);
        float acc[V];
#pragma unroll
        for (int q = 0; q < V; ++q) acc[q] = 0.0f;
        const int p1 = tok_ptr[t + 1];
        for (int p = tok_ptr[t]; p < p1; ++p) {
            const int r = tok_rows[p];
            if (r < 0 || r >= rmax) {
                if (v == 0) record_error(err, kErrFault);
                continue;
            }
            const float g = row_gate[r];
            float yv[V];
            Vec16<T>::load(y_perm + (size_t)r * d + (size_t)v * V, yv);
#pragma unroll
            for (int q = 0; q < V; ++q) acc[q] = __fmaf_rn(g, yv[q], acc[q]);
        }
        if constexpr (SHARED) {
            float sv[V];
            Vec16<T>::load(s_out + (size_t)t * d + (size_t)v * V, sv);
#pragma unroll
            for (int q = 0; q < V; ++q) acc[q] = __fadd_rn(acc[q], sv[q]);
        }
        float xv[V];
        Vec16<T>::load(x + (size_t)t * d + (size_t)v * V, xv);
#pragma unroll
        for (int q = 0; q < V; ++q) acc[q] = __fadd_rn(acc[q], xv[q]);
        Vec16<T>::store(y + (size_t)t * d + (size_t)v * V, acc);
    }
}

template <typename T>
cudaError_t combine_ec_typed(const moe_config &c, const void *x, const void *y_perm, const void *s_out,
                             const int32_t *tok_ptr, const int32_t *tok_rows, const float *row_gate, void *y,
                             uint32_t *err, cudaStream_t s) {
    const int64_t work = (int64_t)c.T * (c.d / Vec16<T>::n);
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>((work + 255) / 256, (int64_t)device_sm_count() * 8));
    const int64_t rmax = max_rows(c);
    const T *sp = static_cast<const T *>(s_out);
    return s_out ? launch_pdl(k_combine_ec<T, true>, dim3(grid), dim3(256), 0, s, static_cast<const T *>(x),
                              static_cast<const T *>(y_perm), sp, tok_ptr, tok_rows, row_gate, c.T, c.d, rmax,
                              static_cast<T *>(y), err)
                 : launch_pdl(k_combine_ec<T, false>, dim3(grid), dim3(256), 0, s, static_cast<const T *>(x),
                              static_cast<const T *>(y_perm), sp, tok_ptr, tok_rows, row_gate, c.T, c.d, rmax,
                              static_cast<T *>(y), err);
}

}  // namespace

cudaError_t launch_expert_choice(const moe_config &c, const float *logits, int32_t *expert_offsets,
                                 int32_t *perm_token, float *row_gate, int32_t *tok_ptr, int32_t *tok_rows,
                                 uint8_t *ws, cudaStream_t s) {
    const WsLayout L = ws_layout(c);
    float *S_t = reinterpret_cast<float *>(ws + L.ec_scores);
    int32_t *ec_row = reinterpret_cast<int32_t *>(ws + L.ec_row);
    int32_t *tok_cnt = reinterpret_cast<int32_t *>(ws + L.ec_tok_cnt);
    cudaError_t e = launch_pdl(k_ec_scores, dim3((c.T + 255) / 256), dim3(256), 0, s, logits, c.T, c.N, S_t, tok_cnt);
    if (e != cudaSuccess) return e;
    const int Ce = (int)(max_rows(c) / c.N);
    const size_t smem = (size_t)c.T * 5;  // score bits and flags
    static bool attr_done = false;
    if (!attr_done) {
        e = cudaFuncSetAttribute(k_ec_select, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)((size_t)kMaxExpertChoiceTokens * 5));
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    SelectArgs sa{S_t, c.T, c.N, Ce, ec_row, tok_cnt, expert_offsets, perm_token, row_gate};
    if ((e = launch_pdl(k_ec_select, dim3(c.N), dim3(1024), smem, s, sa)) != cudaSuccess) return e;
    if ((e = launch_pdl(k_ec_scan, dim3(1), dim3(1024), 0, s, tok_cnt, c.T, tok_ptr)) != cudaSuccess) return e;
    return launch_pdl(k_ec_fill, dim3((c.T + 255) / 256), dim3(256), 0, s, ec_row, tok_ptr, c.T, c.N, tok_rows);
}

cudaError_t launch_combine_ec(const moe_config &c, const void *x, const void *y_perm, const void *s_out,
                              const int32_t *tok_ptr, const int32_t *tok_rows, const float *row_gate, void *y,
                              uint32_t *err, cudaStream_t s) {
    if (c.dtype == MOE_BF16)
        return combine_ec_typed<__nv_bfloat16>(c, x, y_perm, s_out, tok_ptr, tok_rows, row_gate, y, err, s);
    return combine_ec_typed<float>(c, x, y_perm, s_out, tok_ptr, tok_rows, row_gate, y, err, s);
}

}  // namespace moe
