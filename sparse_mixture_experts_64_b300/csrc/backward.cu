// Backward of the layer (token choice): the gradients of sum(dy ⊙ y) + aux_coef *
// aux[0] + z_coef * z with the routing held fixed (selections and capacity are
// piecewise constant). The chain rule runs back through the combine ("From Router
// to Combine": y_t = x_t + S(x_t) + sum_j g_tj O_r), the experts (O = H W_outᵀ,
// H = SiLU(X W_aᵀ) ⊙ X W_bᵀ or max(0, X W_aᵀ)) and the router (the gates are a
// softmax of the fp32 logits; the aux loss N sum_e f_e P_e with f held fixed; the
// z-loss mean_t lse_t²).
//
// This file holds the kernels that are not GEMMs and the orchestration; the row
// GEMMs run on ffn_tc.cu's kernels, the weight gradients on ffn_bwd.cu's, the two
// router contractions (T x d x N) on the weight-gradient kernel as plain products of
// bf16-split operands (an fp32 value v = hi + lo + r with hi = bf16(v), lo = bf16(v - hi),
// |r| <= 2^-16 |v|; bf16 products are exact in the fp32 accumulator):
//   k_bwd_slots   per kept slot: dO_r = g dy_t (bf16) and dg = <dy_t, O_r> (fp32)
//   k_act_bwd     dA = dH ⊙ B ⊙ SiLU'(A), dB = dH ⊙ SiLU(A) (ReLU: dA = dH ⊙ [A > 0])
//   k_count_routed, k_router_bwd  dL per token from dg, aux and z (warp per token)
//   k_split3, k_split_t  the split operands of dx_router = dL W_rᵀ (the hi·hi, hi·lo and
//                 lo·hi terms, concatenated along K) and of dW_rᵀ = dLᵀ x (hi and lo
//                 stacked along M, x exact in bf16), k_sum_hi_lo_t  dW_r from the two halves
//   k_bwd_dx      dx = dy + sum_j dX_r + dX_shared + dx_router
#include <algorithm>
#include <cmath>
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One warp per slot (t, j): the slot's row of dO and its gate gradient.
__global__ void __launch_bounds__(256) k_bwd_slots(const __nv_bfloat16 *__restrict__ dy,
                                                   const __nv_bfloat16 *__restrict__ y_perm,
                                                   const int32_t *__restrict__ slot_row,
                                                   const float *__restrict__ gate, int T, int k, int d,
                                                   int64_t rmax, __nv_bfloat16 *__restrict__ dO,
                                                   float *__restrict__ dgate, uint32_t *err) {
    const int lane = threadIdx.x & 31;
    const int64_t slot = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (slot >= (int64_t)T * k) return;
    const int t = (int)(slot / k);
    const int r = slot_row[slot];
    if (r < 0 || r >= rmax) {
        if (r >= rmax && lane == 0) record_error(err, kErrFault);
        if (lane == 0) dgate[slot] = 0.0f;
        return;
    }
    const float g = gate[slot];
    const __nv_bfloat16 *dyr = dy + (size_t)t * d;
    const __nv_bfloat16 *orow = y_perm + (size_t)r * d;
    __nv_bfloat16 *dor = dO + (size_t)r * d;
    float dot = 0.0f;
    for (int f = lane * 8; f < d; f += 256) {
        float a[8], o[8], out[8];
        Vec16<__nv_bfloat16>::load(dyr + f, a);
        Vec16<__nv_bfloat16>::load(orow + f, o);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            dot = __fmaf_rn(a[q], o[q], dot);
            out[q] = g * a[q];
        }
        Vec16<__nv_bfloat16>::store(dor + f, out);
    }
    dot = warp_sum(dot);
    if (lane == 0) dgate[slot] = dot;
}

// Activation backward over rows: AB [rows][2h] = [A | B] pre-activations (gated) or
// A [rows][h] (ReLU); dH [rows][h]; writes dAB [rows][2h] = [dA | dB] or dA [rows][h].
template <bool GATED>
__global__ void __launch_bounds__(256) k_act_bwd(const __nv_bfloat16 *__restrict__ AB,
                                                 const __nv_bfloat16 *__restrict__ dH, int64_t rows, int h,
                                                 __nv_bfloat16 *__restrict__ dAB) {
    const int vpr = h / 8;
    const int64_t total = rows * vpr;
    const int W = GATED ? 2 * h : h;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / vpr;
        const int c = (int)(i - r * vpr) * 8;
        float a[8], dh[8], da[8];
        Vec16<__nv_bfloat16>::load(AB + r * W + c, a);
        Vec16<__nv_bfloat16>::load(dH + r * h + c, dh);
        if constexpr (GATED) {
            float b[8], db[8];
            Vec16<__nv_bfloat16>::load(AB + r * W + h + c, b);
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const float sig = 1.0f / (1.0f + __expf(-a[q]));
                const float silu = a[q] * sig;
                const float dsilu = sig * (1.0f + a[q] * (1.0f - sig));
                da[q] = dh[q] * b[q] * dsilu;
                db[q] = dh[q] * silu;
            }
            Vec16<__nv_bfloat16>::store(dAB + r * W + h + c, db);
        } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) da[q] = a[q] > 0.0f ? dh[q] : 0.0f;
        }
        Vec16<__nv_bfloat16>::store(dAB + r * W + c, da);
    }
}

__global__ void __launch_bounds__(256) k_count_routed(const int32_t *__restrict__ idx, int64_t n, int N,
                                                      int32_t *__restrict__ routed) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
        const int e = idx[i];
        if (e >= 0 && e < N) atomicAdd(&routed[e], 1);
    }
}

struct RouterBwdArgs {
    const float *logits;     // [T][N]
    const int32_t *idx;      // [T][k]
    const float *gate;       // [T][k]
    const float *dgate;      // [T][k]
    const int32_t *routed;   // [N] selections before capacity
    int T, N, k, gating;
    float aux_coef, z_coef;
    float *dL;               // [T][N]
};

// One warp per token; lane l holds experts l, l + 32, ... (N <= 256).
__global__ void __launch_bounds__(256) k_router_bwd(RouterBwdArgs a) {
    constexpr int Q = 8;
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= a.T) return;
    const int N = a.N, k = a.k;
    const float *l = a.logits + (size_t)t * N;
    float v[Q], p[Q];
    float m = -INFINITY;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const int e = lane + 32 * q;
        v[q] = e < N ? l[e] : -INFINITY;
        m = fmaxf(m, v[q]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float z = 0.0f;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        p[q] = lane + 32 * q < N ? expf(v[q] - m) : 0.0f;
        z += p[q];
    }
    z = warp_sum(z);
#pragma unroll
    for (int q = 0; q < Q; ++q) p[q] /= z;
    const float lse = m + logf(z);
    // dp: gradient with respect to the softmax p (softmax-then-top-k gates, aux)
    float dp[Q], dl[Q];
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const int e = lane + 32 * q;
        dp[q] = 0.0f;
        dl[q] = 0.0f;
        if (e < N && a.aux_coef != 0.0f)
            dp[q] = a.aux_coef * (float)N * ((float)a.routed[e] / ((float)a.T * (float)k)) / (float)a.T;
    }
    if (a.gating == MOE_SOFTMAX_THEN_TOPK) {
        for (int j = 0; j < k; ++j) {
            const int e = a.idx[(size_t)t * k + j];
            const float g = a.dgate[(size_t)t * k + j];
#pragma unroll
            for (int q = 0; q < Q; ++q)
                if (lane + 32 * q == e) dp[q] += g;
        }
    } else {
        // top-k then softmax: dL_sel = g (dg - sum_j g_j dg_j) on the selected experts
        float s = 0.0f;
        for (int j = 0; j < k; ++j) s += a.gate[(size_t)t * k + j] * a.dgate[(size_t)t * k + j];
        for (int j = 0; j < k; ++j) {
            const int e = a.idx[(size_t)t * k + j];
            const float g = a.gate[(size_t)t * k + j];
            const float add = g * (a.dgate[(size_t)t * k + j] - s);
#pragma unroll
            for (int q = 0; q < Q; ++q)
                if (lane + 32 * q == e) dl[q] += add;
        }
    }
    float pd = 0.0f;
#pragma unroll
    for (int q = 0; q < Q; ++q) pd += p[q] * dp[q];
    pd = warp_sum(pd);
    const float zc = a.z_coef != 0.0f ? a.z_coef * 2.0f * lse / (float)a.T : 0.0f;
#pragma unroll
    for (int q = 0; q < Q; ++q) {
        const int e = lane + 32 * q;
        if (e < N) a.dL[(size_t)t * N + e] = dl[q] + p[q] * (dp[q] - pd) + zc * p[q];
    }
}

__device__ __forceinline__ __nv_bfloat16 split_part(float v, int part) {
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    return part == 0 ? hi : __float2bfloat16_rn(v - __bfloat162float(hi));  // v - hi is exact
}

// src fp32 [rows][n] -> dst bf16 [rows][kp]: column q * n + j (q < 3) holds part p_q of
// src[r][j] (0: hi, 1: lo), columns from 3n to kp are zero.
__global__ void __launch_bounds__(256) k_split3(const float *__restrict__ src, int rows, int n, int kp, int p0,
                                                int p1, int p2, __nv_bfloat16 *__restrict__ dst) {
    const int64_t total = (int64_t)rows * kp;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int r = (int)(i / kp), j = (int)(i - (int64_t)r * kp);
        const int q = j / n;
        __nv_bfloat16 v = __float2bfloat16_rn(0.0f);
        if (q < 3) v = split_part(src[(size_t)r * n + (j - q * n)], q == 0 ? p0 : q == 1 ? p1 : p2);
        dst[i] = v;
    }
}

// dL fp32 [T][N] -> dst bf16 [2N][Tp]: row e = hi(dL[:, e]), row N + e = lo(dL[:, e]),
// zero from column T on. 32 x 32 tiles through shared memory.
__global__ void __launch_bounds__(256) k_split_t(const float *__restrict__ dL, int T, int N, int Tp,
                                                 __nv_bfloat16 *__restrict__ dst) {
    __shared__ float tile[32][33];
    const int t0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int i = ty; i < 32; i += 8) {
        const int t = t0 + i, e = e0 + tx;
        tile[i][tx] = (t < T && e < N) ? dL[(size_t)t * N + e] : 0.0f;
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
        const int e = e0 + i, t = t0 + tx;
        if (e < N && t < Tp) {
            const float v = tile[tx][i];
            dst[(size_t)e * Tp + t] = split_part(v, 0);
            dst[(size_t)(N + e) * Tp + t] = split_part(v, 1);
        }
    }
}

// dw_r [d][N] = C[e][i] + C[N + e][i] from C fp32 [2N][d] (the hi and lo halves).
__global__ void __launch_bounds__(256) k_sum_hi_lo_t(const float *__restrict__ C, int N, int d,
                                                     float *__restrict__ dw_r) {
    __shared__ float tile[32][33];
    const int i0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int j = ty; j < 32; j += 8) {
        const int e = e0 + j, i = i0 + tx;
        tile[j][tx] = (e < N && i < d) ? C[(size_t)e * d + i] + C[(size_t)(N + e) * d + i] : 0.0f;
    }
    __syncthreads();
    for (int j = ty; j < 32; j += 8) {
        const int i = i0 + j, e = e0 + tx;
        if (i < d && e < N) dw_r[(size_t)i * N + e] = tile[tx][j];
    }
}

// dx = dy + sum_j dX[slot_row] + dX_sh + dx_router, per 8 features of a token.
__global__ void __launch_bounds__(256) k_bwd_dx(const __nv_bfloat16 *__restrict__ dy,
                                                const __nv_bfloat16 *__restrict__ dX,
                                                const int32_t *__restrict__ slot_row,
                                                const __nv_bfloat16 *__restrict__ dX_sh,
                                                const float *__restrict__ dxr, int T, int k, int d, int64_t rmax,
                                                __nv_bfloat16 *__restrict__ dx, uint32_t *err) {
    const int vpr = d / 8;
    const int64_t total = (int64_t)T * vpr;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / vpr);
        const int f = (int)(i - (int64_t)t * vpr) * 8;
        float acc[8], v[8];
        Vec16<__nv_bfloat16>::load(dy + (size_t)t * d + f, acc);
        for (int j = 0; j < k; ++j) {
            const int r = slot_row[(size_t)t * k + j];
            if (r < 0) continue;
            if (r >= rmax) {
                if (f == 0) record_error(err, kErrFault);
                continue;
            }
            Vec16<__nv_bfloat16>::load(dX + (size_t)r * d + f, v);
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] += v[q];
        }
        if (dX_sh) {
            Vec16<__nv_bfloat16>::load(dX_sh + (size_t)t * d + f, v);
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] += v[q];
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] += dxr[(size_t)t * d + f + q];
        Vec16<__nv_bfloat16>::store(dx + (size_t)t * d + f, acc);
    }
}

__global__ void k_col_sum(const float *__restrict__ a, int rows, int cols, float *__restrict__ out) {
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= cols) return;
    float s = 0.0f;
    for (int r = 0; r < rows; ++r) s += a[(size_t)r * cols + c];
    out[c] = s;
}

int grid_of(int64_t work, int threads) {
    const int64_t b = (work + threads - 1) / threads;
    return (int)std::max<int64_t>(1, std::min<int64_t>(b, (int64_t)device_sm_count() * 8));
}

}  // namespace

BwdLayout bwd_layout(const moe_config &c) {
    BwdLayout L;
    const size_t R = (size_t)max_rows(c), T = c.T, d = c.d, h = c.h, hs = c.h_shared, N = c.N;
    const size_t W = c.act == MOE_ACT_SILU_GATED ? 2 * h : h;  // [A | B] or A
    const size_t Tp = (T + 63) / 64 * 64;
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = (o + std::max<size_t>(bytes, 1) + 255) & ~(size_t)255;
        return at;
    };
    L.dO = take(R * d * 2);
    L.dgate = take(T * c.k * 4);
    const bool kept_pre = saves_preact(c);  // then the forward's workspace holds the pre-activations
    L.AB = take(kept_pre ? 0 : R * W * 2);
    L.dH = take(R * h * 2);
    L.dAB = take(R * W * 2);
    L.dX = take(R * d * 2);
    L.AB_sh = take(hs && !kept_pre ? T * 2 * hs * 2 : 0);
    L.dH_sh = take(hs ? T * hs * 2 : 0);
    L.dAB_sh = take(hs ? T * 2 * hs * 2 : 0);
    L.dX_sh = take(hs ? T * d * 2 : 0);
    L.logits = take(N > 32 ? 0 : T * N * 4);  // N > 32: the forward's logits in its workspace serve
    L.routed = take(N * 4);
    L.dL = take(T * N * 4);
    L.dxr = take(T * d * 4);
    const size_t Kr = (3 * N + 63) / 64 * 64;
    L.rA = take(T * Kr * 2);
    L.rB = take(d * Kr * 2);
    L.dLt = take(2 * N * Tp * 2);
    L.wrC = take(2 * N * d * 4);
    L.total = o;
    return L;
}

cudaError_t launch_bwd_slots(const moe_config &c, const void *dy, const void *y_perm, const int32_t *slot_row,
                             const float *gate, void *dO, float *dgate, uint32_t *err, cudaStream_t s) {
    const int64_t slots = (int64_t)c.T * c.k;
    k_bwd_slots<<<(unsigned)((slots + 7) / 8), 256, 0, s>>>(
        static_cast<const __nv_bfloat16 *>(dy), static_cast<const __nv_bfloat16 *>(y_perm), slot_row, gate, c.T, c.k,
        c.d, max_rows(c), static_cast<__nv_bfloat16 *>(dO), dgate, err);
    return cudaGetLastError();
}

cudaError_t launch_act_bwd(bool gated, const void *AB, const void *dH, int64_t rows, int h, void *dAB,
                           cudaStream_t s) {
    const int grid = grid_of(rows * (h / 8), 256);
    if (gated)
        k_act_bwd<true><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(AB),
                                             static_cast<const __nv_bfloat16 *>(dH), rows, h,
                                             static_cast<__nv_bfloat16 *>(dAB));
    else
        k_act_bwd<false><<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(AB),
                                              static_cast<const __nv_bfloat16 *>(dH), rows, h,
                                              static_cast<__nv_bfloat16 *>(dAB));
    return cudaGetLastError();
}

cudaError_t launch_router_bwd(const moe_config &c, const void *x, const float *w_r, const float *logits,
                              const int32_t *topk_idx, const float *topk_gate, const BwdLayout &L, uint8_t *bw,
                              float aux_coef, float z_coef, float *dw_r, float *db_r, uint32_t *err, bool allow_pair,
                              cudaStream_t s) {
    int32_t *routed = reinterpret_cast<int32_t *>(bw + L.routed);
    float *dL = reinterpret_cast<float *>(bw + L.dL);
    float *dxr = reinterpret_cast<float *>(bw + L.dxr);
    cudaError_t e = cudaMemsetAsync(routed, 0, (size_t)c.N * 4, s);
    if (e != cudaSuccess) return e;
    k_count_routed<<<grid_of((int64_t)c.T * c.k, 256), 256, 0, s>>>(topk_idx, (int64_t)c.T * c.k, c.N, routed);
    RouterBwdArgs ra{logits, topk_idx, topk_gate, reinterpret_cast<const float *>(bw + L.dgate), routed, c.T, c.N,
                     c.k, c.gating, aux_coef, z_coef, dL};
    k_router_bwd<<<(c.T + 7) / 8, 256, 0, s>>>(ra);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int Kr = (3 * c.N + 63) / 64 * 64, Tp = (c.T + 63) / 64 * 64;
    __nv_bfloat16 *rA = reinterpret_cast<__nv_bfloat16 *>(bw + L.rA), *rB = reinterpret_cast<__nv_bfloat16 *>(bw + L.rB);
    __nv_bfloat16 *dLt = reinterpret_cast<__nv_bfloat16 *>(bw + L.dLt);
    // dx_router [T][d] = [dL_hi | dL_hi | dL_lo] · [W_hi | W_lo | W_hi]ᵀ  (W_r is [d][N]: K-major)
    k_split3<<<grid_of((int64_t)c.T * Kr, 256), 256, 0, s>>>(dL, c.T, c.N, Kr, 0, 0, 1, rA);
    k_split3<<<grid_of((int64_t)c.d * Kr, 256), 256, 0, s>>>(w_r, c.d, c.N, Kr, 0, 1, 0, rB);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const WgOperand none{nullptr, 0, 0, false};
    e = launch_wgrad(nullptr, 0, 0, none, none, c.T, c.d, nullptr, WgOperand{rA, Kr, 0, false},
                     WgOperand{rB, Kr, 0, false}, Kr, dxr, err, s, allow_pair, true);
    if (e != cudaSuccess) return e;
    // dW_rᵀ halves [2N][d] = [dL_hiᵀ ; dL_loᵀ] · x over the tokens (x exact in bf16, read
    // in its own layout [T][d] as the MN-major operand; tokens past T read as zero)
    k_split_t<<<dim3(Tp / 32, (c.N + 31) / 32), 256, 0, s>>>(dL, c.T, c.N, Tp, dLt);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    float *wrC = reinterpret_cast<float *>(bw + L.wrC);
    e = launch_wgrad(nullptr, 0, 0, none, none, 2 * c.N, c.d, nullptr, WgOperand{dLt, Tp, 0, false},
                     WgOperand{x, c.d, c.T, true}, Tp, wrC, err, s, allow_pair, true);
    if (e != cudaSuccess) return e;
    k_sum_hi_lo_t<<<dim3((c.d + 31) / 32, (c.N + 31) / 32), 256, 0, s>>>(wrC, c.N, c.d, dw_r);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (db_r) {
        k_col_sum<<<(c.N + 255) / 256, 256, 0, s>>>(dL, c.T, c.N, db_r);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_bwd_dx(const moe_config &c, const void *dy, const void *dX, const int32_t *slot_row,
                          const void *dX_sh, const float *dxr, void *dx, uint32_t *err, cudaStream_t s) {
    k_bwd_dx<<<grid_of((int64_t)c.T * (c.d / 8), 256), 256, 0, s>>>(
        static_cast<const __nv_bfloat16 *>(dy), static_cast<const __nv_bfloat16 *>(dX), slot_row,
        static_cast<const __nv_bfloat16 *>(dX_sh), dxr, c.T, c.k, c.d, max_rows(c), static_cast<__nv_bfloat16 *>(dx),
        err);
    return cudaGetLastError();
}

}  // namespace moe
