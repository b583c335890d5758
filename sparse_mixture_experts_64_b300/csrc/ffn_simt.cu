// Grouped expert FFN on CUDA cores (fp32 FMA). This is the path for fp32 layers,
// whose tolerance TF32 tensor cores cannot meet, and a cross-check path for bf16
// (MOE_DEBUG_FORCE_SIMT_FFN).
//
// Each expert is an independent feed-forward network applied row by row to the
// tokens dispatched to it ("Mixture of Experts (MoE)" glossary; "MoE: Choosing
// Which MLPs to Use for Each Token", sections "Dense MLP and MoE" and "From Router
// to Combine"): gated  W_down (SiLU(W_gate x) * (W_up x)),  or  W2 max(0, W1 x).
//
// One launch per product (hidden, then output). A CTA owns a 64x64 output tile of
// one segment; blockIdx.y enumerates the m-tiles of all segments in order (routed
// experts from the device-side offsets, then the shared expert), so row counts
// never travel to the host. Every output is one fp32 FMA chain in increasing k.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16;

enum { MODE_GATED = 0, MODE_RELU = 1, MODE_PLAIN = 2 };

template <typename T> struct SimtProblem {
    const int32_t *offsets;
    int n_seg, sh_rows;
    int64_t a_rows;          // rows of the routed buffers; offsets are clamped to it
    const T *a, *a_sh;       // A [rows][K]
    int K, K_sh;
    const T *b0, *b1;        // routed weights [n_seg][n_out][K]
    const T *b0_sh, *b1_sh;  // shared weights [n_out_sh][K_sh]
    T *c, *c_sh;             // outputs [rows][n_out]
    int n_out, n_out_sh;
};

template <typename T> __device__ __forceinline__ void load4(const T *p, float *v);
template <> __device__ __forceinline__ void load4<float>(const float *p, float *v) {
    float4 q = *reinterpret_cast<const float4 *>(p);
    v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
}
template <> __device__ __forceinline__ void load4<__nv_bfloat16>(const __nv_bfloat16 *p, float *v) {
    uint2 q = *reinterpret_cast<const uint2 *>(p);
    v[0] = __uint_as_float(q.x << 16); v[1] = __uint_as_float(q.x & 0xffff0000u);
    v[2] = __uint_as_float(q.y << 16); v[3] = __uint_as_float(q.y & 0xffff0000u);
}

template <typename T, int MODE>
__global__ void __launch_bounds__(256) k_ffn_simt(SimtProblem<T> p) {
    constexpr bool TWO = MODE == MODE_GATED;
    __shared__ __align__(16) float As[BK][BM];
    __shared__ __align__(16) float Bs[TWO ? 2 : 1][BK][BN];

    pdl_enter();
    // ---- locate this CTA's segment and m-tile ----
    int y = blockIdx.y, seg = -1;
    int row0 = 0, rows = 0;
    for (int e = 0; e < p.n_seg; ++e) {
        const int ar = (int)p.a_rows;
        const int r0 = min(max(p.offsets[e], 0), ar);
        const int r1 = min(max(p.offsets[e + 1], r0), ar);
        const int mt = (r1 - r0 + BM - 1) / BM;
        if (y < mt) {
            seg = e;
            row0 = r0 + y * BM;
            rows = min(BM, r1 - row0);
            break;
        }
        y -= mt;
    }
    const T *A, *B0, *B1 = nullptr;
    T *C;
    int K, n_out;
    if (seg >= 0) {
        A = p.a; K = p.K; n_out = p.n_out; C = p.c;
        B0 = p.b0 + (size_t)seg * n_out * K;
        if (TWO) B1 = p.b1 + (size_t)seg * n_out * K;
    } else {
        const int mt = (p.sh_rows + BM - 1) / BM;
        if (y >= mt) return;
        row0 = y * BM;
        rows = min(BM, p.sh_rows - row0);
        A = p.a_sh; K = p.K_sh; n_out = p.n_out_sh; C = p.c_sh;
        B0 = p.b0_sh;
        if (TWO) B1 = p.b1_sh;
    }
    const int n0 = blockIdx.x * BN;
    if (n0 >= n_out) return;

    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    const int lr = tid / 4, lk = (tid % 4) * 4;  // loader: row/col and 4 consecutive k
    float acc0[4][4], acc1[4][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc0[i][j] = acc1[i][j] = 0.0f;

    for (int k0 = 0; k0 < K; k0 += BK) {
        float v[4];
        const int kk = k0 + lk;
        // A tile (rows lr of the segment), zero outside
        if (lr < rows && kk < K) load4<T>(A + (size_t)(row0 + lr) * K + kk, v);
        else v[0] = v[1] = v[2] = v[3] = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) As[lk + i][lr] = v[i];
        const int n = n0 + lr;
        if (n < n_out && kk < K) load4<T>(B0 + (size_t)n * K + kk, v);
        else v[0] = v[1] = v[2] = v[3] = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) Bs[0][lk + i][lr] = v[i];
        if constexpr (TWO) {
            if (n < n_out && kk < K) load4<T>(B1 + (size_t)n * K + kk, v);
            else v[0] = v[1] = v[2] = v[3] = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i) Bs[TWO ? 1 : 0][lk + i][lr] = v[i];
        }
        __syncthreads();
        const int kc = min(BK, K - k0);
        for (int q = 0; q < kc; ++q) {
            float a[4], b[4];
            load4<float>(&As[q][ty * 4], a);
            load4<float>(&Bs[0][q][tx * 4], b);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc0[i][j] = __fmaf_rn(a[i], b[j], acc0[i][j]);
            if constexpr (TWO) {
                load4<float>(&Bs[TWO ? 1 : 0][q][tx * 4], b);
#pragma unroll
                for (int i = 0; i < 4; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) acc1[i][j] = __fmaf_rn(a[i], b[j], acc1[i][j]);
            }
        }
        __syncthreads();
    }

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = ty * 4 + i;
        if (r >= rows) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int n = n0 + tx * 4 + j;
            if (n >= n_out) continue;
            float o = acc0[i][j];
            if constexpr (MODE == MODE_GATED) o = silu_f32(o) * acc1[i][j];
            if constexpr (MODE == MODE_RELU) o = fmaxf(o, 0.0f);
            C[(size_t)(row0 + r) * n_out + n] = from_f32<T>(o);
        }
    }
}

template <typename T>
cudaError_t run(const moe_config &c, const FfnGroup &g, cudaStream_t s) {
    const int64_t mslots = (g.a_rows + BM - 1) / BM + g.n_seg + (g.sh_rows + BM - 1) / BM;
    if (mslots > 65535) return cudaErrorInvalidConfiguration;
    // product 1: hidden = act(A W_aᵀ) [* (A W_bᵀ)]
    SimtProblem<T> p1{g.offsets, g.n_seg, g.sh_rows, g.a_rows,
                      static_cast<const T *>(g.a), static_cast<const T *>(g.sh_a), c.d, c.d,
                      static_cast<const T *>(g.w_a), static_cast<const T *>(g.w_b),
                      static_cast<const T *>(g.sh_w_gate), static_cast<const T *>(g.sh_w_up),
                      static_cast<T *>(g.hid), static_cast<T *>(g.sh_hid), g.h, g.h_sh};
    const int nmax1 = std::max(g.n_seg ? g.h : 0, g.sh_rows ? g.h_sh : 0);
    dim3 grid1((nmax1 + BN - 1) / BN, (unsigned)mslots);
    cudaError_t e;
    if (g.act == MOE_ACT_RELU && g.sh_rows == 0) {
        e = launch_pdl(k_ffn_simt<T, MODE_RELU>, grid1, dim3(256), 0, s, p1);
    } else if (g.act == MOE_ACT_RELU) {
        // routed ReLU experts and a gated shared expert: two launches
        SimtProblem<T> pr = p1;
        pr.sh_rows = 0;
        e = launch_pdl(k_ffn_simt<T, MODE_RELU>, grid1, dim3(256), 0, s, pr);
        SimtProblem<T> ps = p1;
        ps.n_seg = 0;
        if (e == cudaSuccess)
            e = launch_pdl(k_ffn_simt<T, MODE_GATED>, dim3(grid1.x, (g.sh_rows + BM - 1) / BM), dim3(256), 0, s, ps);
    } else {
        e = launch_pdl(k_ffn_simt<T, MODE_GATED>, grid1, dim3(256), 0, s, p1);
    }
    if (e != cudaSuccess) return e;
    if (g.mid_event && (e = cudaEventRecordWithFlags(g.mid_event, s, g.event_flags)) != cudaSuccess) return e;
    // product 2: out = hidden W_outᵀ
    SimtProblem<T> p2{g.offsets, g.n_seg, g.sh_rows, g.a_rows,
                      static_cast<const T *>(g.hid), static_cast<const T *>(g.sh_hid), g.h, g.h_sh,
                      static_cast<const T *>(g.w_out), nullptr,
                      static_cast<const T *>(g.sh_w_down), nullptr,
                      static_cast<T *>(g.out), static_cast<T *>(g.sh_out), c.d, c.d};
    dim3 grid2((c.d + BN - 1) / BN, (unsigned)mslots);
    return launch_pdl(k_ffn_simt<T, MODE_PLAIN>, grid2, dim3(256), 0, s, p2);
}

}  // namespace

cudaError_t launch_ffn_simt(const moe_config &c, const FfnGroup &g, uint32_t *, cudaStream_t s) {
    if (c.dtype == MOE_BF16) return run<__nv_bfloat16>(c, g, s);
    return run<float>(c, g, s);
}

}  // namespace moe
