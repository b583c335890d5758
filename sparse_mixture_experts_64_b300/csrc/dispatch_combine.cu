// Dispatch (row gather into expert order) and combine (gate-weighted sum back to
// token order, plus shared expert and residual).
//
// "MoE: Choosing Which MLPs to Use for Each Token", section "From Router to
// Combine" (Figure 3): dispatch sends each token's own vector to the experts that
// chose it; combine gathers each token's expert outputs and sums them with the
// router weights. Section "Shared Expert" (Figure 4): y = S(x) + R(x). DeepSeekMoE
// layer equation: the residual u_t is added. "Mixture of Experts (MoE)" glossary:
// a dropped (over-capacity) slot leaves only the residual path.
//
// Both kernels move 16-byte vectors; consecutive threads take consecutive
// vectors of one row, so every warp reads and writes whole 512-byte spans.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

template <typename T>
__global__ void __launch_bounds__(256) k_dispatch(const T *__restrict__ x, const int32_t *__restrict__ perm,
                                                  const int32_t *__restrict__ offsets, int N, int Ttok,
                                                  int d, int64_t rmax, T *__restrict__ x_perm,
                                                  uint32_t *err) {
    constexpr int V = Vec16<T>::n;
    const int vpr = d / V;  // vectors per row
    pdl_enter();
    int64_t R = offsets[N];
    if (R < 0 || R > rmax) {
        if (blockIdx.x == 0 && threadIdx.x == 0) record_error(err, kErrFault);
        R = R < 0 ? 0 : rmax;
    }
    const int64_t total = R * vpr;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = i / vpr;
        const int v = (int)(i - r * vpr);
        const int t = perm[r];
        if (t < 0 || t >= Ttok) {
            if (v == 0) record_error(err, kErrFault);
            continue;
        }
        const uint4 q = *reinterpret_cast<const uint4 *>(x + (size_t)t * d + (size_t)v * V);
        *reinterpret_cast<uint4 *>(x_perm + (size_t)r * d + (size_t)v * V) = q;
    }
}

// The same rows written in token order: each token's vector is read once and stored
// at the rows of its kept slots (slot_row[t][j], -1 = dropped). The expert-order
// gather above reads a token k times at distant moments, so once the activations
// outgrow L2 it reads them k times from HBM (DeepSeek-shaped layer: 0.70 GB for a
// 117 MB x); this order reads them once.
template <typename T>
__global__ void __launch_bounds__(256) k_dispatch_tokens(const T *__restrict__ x, const int32_t *__restrict__ slot_row,
                                                         int Ttok, int k, int d, int64_t rmax, T *__restrict__ x_perm,
                                                         uint32_t *err) {
    constexpr int V = Vec16<T>::n;
    const int vpr = d / V;
    const int64_t total = (int64_t)Ttok * vpr;
    pdl_enter();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int t = (int)(i / vpr);
        const int v = (int)(i - (int64_t)t * vpr);
        const uint4 q = *reinterpret_cast<const uint4 *>(x + (size_t)t * d + (size_t)v * V);
        for (int j = 0; j < k; ++j) {
            const int r = slot_row[(size_t)t * k + j];
            if (r < 0) continue;
            if (r >= rmax) {
                if (v == 0) record_error(err, kErrFault);
                continue;
            }
            *reinterpret_cast<uint4 *>(x_perm + (size_t)r * d + (size_t)v * V) = q;
        }
    }
}

// y[t] = x[t] + S[t] + sum_j g[t][j] * y_perm[slot_row[t][j]]; the expert terms
// are accumulated in fp32 in slot order, then S is added, then x.
template <typename T, bool SHARED>
__global__ void __launch_bounds__(256) k_combine(const T *__restrict__ x, const T *__restrict__ y_perm,
                                                 const T *__restrict__ s_out,
                                                 const int32_t *__restrict__ slot_row,
                                                 const float *__restrict__ gate, int Ttok, int d, int k,
                                                 int64_t rmax, T *__restrict__ y, uint32_t *err) {
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
        for (int j = 0; j < k; ++j) {
            const int r = slot_row[(size_t)t * k + j];
            if (r < 0) continue;
            if (r >= rmax) {
                if (v == 0) record_error(err, kErrFault);
                continue;
            }
            const float g = gate[(size_t)t * k + j];
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

int grid_for(int64_t work, int threads) {
    const int64_t blocks = (work + threads - 1) / threads;
    const int64_t cap = (int64_t)device_sm_count() * 8;
    return (int)std::max<int64_t>(1, std::min(blocks, cap));
}

}  // namespace

cudaError_t launch_dispatch(const moe_config &c, const void *x, const int32_t *perm_token,
                            const int32_t *offsets, void *x_perm, uint32_t *err, cudaStream_t s) {
    const int64_t rmax = max_rows(c);
    if (c.dtype == MOE_BF16)
        return launch_pdl(k_dispatch<__nv_bfloat16>, dim3(grid_for(rmax * (c.d / 8), 256)), dim3(256), 0, s,
                          static_cast<const __nv_bfloat16 *>(x), perm_token, offsets, c.N, c.T, c.d, rmax,
                          static_cast<__nv_bfloat16 *>(x_perm), err);
    return launch_pdl(k_dispatch<float>, dim3(grid_for(rmax * (c.d / 4), 256)), dim3(256), 0, s,
                      static_cast<const float *>(x), perm_token, offsets, c.N, c.T, c.d, rmax,
                      static_cast<float *>(x_perm), err);
}

cudaError_t launch_dispatch_tokens(const moe_config &c, const void *x, const int32_t *slot_row, void *x_perm,
                                   uint32_t *err, cudaStream_t s) {
    const int64_t rmax = max_rows(c);
    if (c.dtype == MOE_BF16)
        return launch_pdl(k_dispatch_tokens<__nv_bfloat16>, dim3(grid_for((int64_t)c.T * (c.d / 8), 256)), dim3(256),
                          0, s, static_cast<const __nv_bfloat16 *>(x), slot_row, c.T, c.k, c.d, rmax,
                          static_cast<__nv_bfloat16 *>(x_perm), err);
    return launch_pdl(k_dispatch_tokens<float>, dim3(grid_for((int64_t)c.T * (c.d / 4), 256)), dim3(256), 0, s,
                      static_cast<const float *>(x), slot_row, c.T, c.k, c.d, rmax, static_cast<float *>(x_perm),
                      err);
}

template <typename T>
static cudaError_t combine_typed(const moe_config &c, const void *x, const void *y_perm, const void *s_out,
                                 const int32_t *slot_row, const float *gate, void *y, uint32_t *err, cudaStream_t s) {
    const dim3 grid(grid_for((int64_t)c.T * (c.d / Vec16<T>::n), 256));
    const T *sp = static_cast<const T *>(s_out);
    return s_out ? launch_pdl(k_combine<T, true>, grid, dim3(256), 0, s, static_cast<const T *>(x),
                              static_cast<const T *>(y_perm), sp, slot_row, gate, c.T, c.d, c.k, max_rows(c),
                              static_cast<T *>(y), err)
                 : launch_pdl(k_combine<T, false>, grid, dim3(256), 0, s, static_cast<const T *>(x),
                              static_cast<const T *>(y_perm), sp, slot_row, gate, c.T, c.d, c.k, max_rows(c),
                              static_cast<T *>(y), err);
}

cudaError_t launch_combine(const moe_config &c, const void *x, const void *y_perm, const void *s_out,
                           const int32_t *slot_row, const float *gate, void *y, uint32_t *err,
                           cudaStream_t s) {
    if (c.dtype == MOE_BF16) return combine_typed<__nv_bfloat16>(c, x, y_perm, s_out, slot_row, gate, y, err, s);
    return combine_typed<float>(c, x, y_perm, s_out, slot_row, gate, y, err, s);
}

}  // namespace moe
