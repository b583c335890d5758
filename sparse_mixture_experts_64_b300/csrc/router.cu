// Router: fp32 logits, softmax / top-k gating, per-expert counts, capacity and
// dispatch order.
//
// "Noise Top-k Gating" glossary (the router is one linear layer producing one
// logit per expert); "MoE: Choosing Which MLPs to Use for Each Token", section
// "Router: Selecting Experts and Computing Weights" (Figure 2: W_r is d x N,
// top-2 of the scores, softmax over the selected two); the DeepSeekMoE layer
// equation (softmax over all N affinities, then Topk, gates not renormalised);
// "Mixture of Experts (MoE)" glossary (capacity = tokens / experts * factor, the
// overflow keeps only the residual; auxiliary load-balancing loss); "Switch
// Transformers ... explained", section "Making it work" (router in higher
// precision, capacity with overflow skipping the layer).
//
// Three kernels, no atomics, deterministic:
//   k_router       one CTA per tile of 8*warps tokens: logits (fp32 FMA chain over
//                  d in increasing order), top-k, gates, full softmax; writes per
//                  tile, per expert: routed counts per slot and the sum of p.
//   k_expert_scan  one CTA per expert: priority-order prefix of the tile counts
//                  (slot-major, token order), capacity clamp, kept-per-tile prefix,
//                  routed/kept totals, mean routing probability P_e.
//   k_assign       one CTA per tile: expert offsets, keep/drop per slot, row of
//                  each kept slot (expert ascending, token ascending), perm_token;
//                  CTA 0 also writes expert_offsets and the aux losses.
#include <algorithm>
#include <climits>
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace moe {

int router_warps(const moe_config &c) {
    if (c.N > 32) {
        const int warp_tiles = (c.T + 7) / 8;
        const int w = (warp_tiles + kSmCountForTiling - 1) / kSmCountForTiling;
        return std::min(8, std::max(1, w));
    }
    return 2;
}

namespace {

constexpr int KC = 32;  // features staged per chunk

struct RouterArgs {
    int T, d, N, k, gating, tiles, has_bias;
    int32_t *topk_idx;
    float *topk_gate;
    int32_t *cnt;   // [N][k][tiles]
    float *psum;    // [N][tiles]
};

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
    uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
    uint32_t s = static_cast<uint32_t>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int n> __device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(n) : "memory");
}

template <int n> __device__ __forceinline__ void lds(const float *p, float *v) {
    if constexpr (n % 4 == 0) {
#pragma unroll
        for (int i = 0; i < n; i += 4) {
            float4 q = *reinterpret_cast<const float4 *>(p + i);
            v[i] = q.x; v[i + 1] = q.y; v[i + 2] = q.z; v[i + 3] = q.w;
        }
    } else if constexpr (n == 2) {
        float2 q = *reinterpret_cast<const float2 *>(p);
        v[0] = q.x; v[1] = q.y;
    } else {
#pragma unroll
        for (int i = 0; i < n; ++i) v[i] = p[i];
    }
}

__device__ __forceinline__ float warp_sum_bcast(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return __shfl_sync(0xffffffffu, v, 0);
}

// Thread tile: TPT tokens x EPT experts; a warp is (32/LE) token groups x LE
// expert groups = 8 tokens x LE*EPT experts; warps stack along tokens.
template <typename XT, int LE, int EPT, int TPT, bool NALIGN4>
__global__ void __launch_bounds__(256) k_router(const XT *__restrict__ x, const float *__restrict__ w_r,
                                                const float *__restrict__ b_r, RouterArgs a) {
    constexpr int NP = LE * EPT;
    constexpr int QMAX = (NP + 31) / 32;
    constexpr int VX = 16 / sizeof(XT);         // x elements per 16-byte load
    constexpr int XPAIRS = (KC / VX) * 8 / 32;  // (token, 16B) pairs per thread
    static_assert((32 / LE) * TPT == 8, "a warp covers 8 tokens");
    extern __shared__ __align__(16) float smem[];

    const int nthreads = blockDim.x;
    const int nwarps = nthreads / 32;
    const int TT = nwarps * 8;
    const int N = a.N, d = a.d, T = a.T;
    const int wbuf = KC * N + NP;  // W chunk [KC][N] + padding read by lanes with e >= N
    float *Ws = smem;
    float *Xs = smem + 2 * wbuf;   // [2][KC][TT], transposed, fp32
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int le = lane % LE, lt = lane / LE;
    const int t0 = blockIdx.x * TT;
    const int tok_base = warp * 8 + lt * TPT;
    const int e_base = le * EPT;

    float acc[TPT][EPT];
#pragma unroll
    for (int i = 0; i < TPT; ++i)
#pragma unroll
        for (int j = 0; j < EPT; ++j) acc[i][j] = 0.0f;

    const int nchunks = (d + KC - 1) / KC;
    float xr[XPAIRS][VX];

    auto load_x = [&](int c) {
#pragma unroll
        for (int p = 0; p < XPAIRS; ++p) {
            const int pi = tid + p * nthreads;
            const int tok = pi / (KC / VX), kq = pi % (KC / VX);
            const int t = t0 + tok, kf = c * KC + kq * VX;
            if (t < T && kf < d) {
                Vec16<XT>::load(x + (size_t)t * d + kf, xr[p]);
            } else {
#pragma unroll
                for (int i = 0; i < VX; ++i) xr[p][i] = 0.0f;
            }
        }
    };
    auto store_x = [&](int buf) {
        float *xb = Xs + buf * KC * TT;
#pragma unroll
        for (int p = 0; p < XPAIRS; ++p) {
            const int pi = tid + p * nthreads;
            const int tok = pi / (KC / VX), kq = pi % (KC / VX);
#pragma unroll
            for (int i = 0; i < VX; ++i) xb[(kq * VX + i) * TT + tok] = xr[p][i];
        }
    };
    auto issue_w = [&](int c, int buf) {
        const int k0 = c * KC;
        const int kc = min(KC, d - k0);
        const float *src = w_r + (size_t)k0 * N;
        float *dst = Ws + buf * wbuf;
        if constexpr (NALIGN4) {
            const int nvec = kc * N / 4;
            for (int v = tid; v < nvec; v += nthreads) cp_async16(dst + 4 * v, src + 4 * v);
        } else {
            const int n = kc * N;
            for (int v = tid; v < n; v += nthreads) cp_async4(dst + v, src + v);
        }
        cp_async_commit();
    };

    load_x(0);
    issue_w(0, 0);
    for (int c = 0; c < nchunks; ++c) {
        const int buf = c & 1;
        store_x(buf);
        if (c + 1 < nchunks) {
            issue_w(c + 1, buf ^ 1);
            load_x(c + 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const float *wb = Ws + buf * wbuf + e_base;
        const float *xb = Xs + buf * KC * TT + tok_base;
        const int kc = min(KC, d - c * KC);
#pragma unroll 8
        for (int kk = 0; kk < kc; ++kk) {
            float xv[TPT], wv[EPT];
            lds<TPT>(xb + kk * TT, xv);
            if constexpr (NALIGN4) {
                lds<EPT>(wb + kk * N, wv);
            } else {
#pragma unroll
                for (int j = 0; j < EPT; ++j) wv[j] = wb[kk * N + j];
            }
#pragma unroll
            for (int i = 0; i < TPT; ++i)
#pragma unroll
                for (int j = 0; j < EPT; ++j) acc[i][j] = __fmaf_rn(xv[i], wv[j], acc[i][j]);
        }
        __syncthreads();
    }

    // ---- logits to shared memory: Ls[TT][N]; Is[TT][8] behind it ----
    float *Ls = smem;
    int *Is = reinterpret_cast<int *>(smem + TT * N);
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
        const int e = e_base + j;
        if (e < N) {
            const float bj = a.has_bias ? b_r[e] : 0.0f;
#pragma unroll
            for (int i = 0; i < TPT; ++i) {
                float v = acc[i][j];
                if (a.has_bias) v = __fadd_rn(v, bj);
                Ls[(tok_base + i) * N + e] = v;
            }
        }
    }
    __syncthreads();

    // ---- gating: one warp per token ----
    const int k = a.k;
    for (int tok = warp; tok < TT; tok += nwarps) {
        const int t = t0 + tok;
        if (t >= T) {
            for (int e = lane; e < N; e += 32) Ls[tok * N + e] = 0.0f;
            if (lane < 8) Is[tok * 8 + lane] = -1;
            continue;
        }
        float v[QMAX];
#pragma unroll
        for (int q = 0; q < QMAX; ++q) {
            const int e = lane + 32 * q;
            v[q] = e < N ? Ls[tok * N + e] : -INFINITY;
        }
        unsigned taken = 0;
        float my_v = 0.0f, vmax = 0.0f;
        int my_e = 0;
        for (int s = 0; s < k; ++s) {
            float bv = -INFINITY;
            int bi = INT_MAX;
#pragma unroll
            for (int q = 0; q < QMAX; ++q) {
                const int e = lane + 32 * q;
                if (e < N && !((taken >> q) & 1u) && (v[q] > bv || (v[q] == bv && e < bi))) {
                    bv = v[q];
                    bi = e;
                }
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ov > bv || (ov == bv && oi < bi)) {
                    bv = ov;
                    bi = oi;
                }
            }
            if (s == 0) vmax = bv;
            if (lane == s) {
                my_v = bv;
                my_e = bi;
            }
            if (bi != INT_MAX && (bi & 31) == lane) taken |= 1u << (bi >> 5);
        }
        float part = 0.0f;
#pragma unroll
        for (int q = 0; q < QMAX; ++q) {
            const int e = lane + 32 * q;
            if (e < N) part += expf(v[q] - vmax);
        }
        const float sum = warp_sum_bcast(part);
#pragma unroll
        for (int q = 0; q < QMAX; ++q) {
            const int e = lane + 32 * q;
            if (e < N) Ls[tok * N + e] = expf(v[q] - vmax) / sum;
        }
        const float ex = lane < k ? expf(my_v - vmax) : 0.0f;
        float g;
        if (a.gating == MOE_SOFTMAX_THEN_TOPK) {
            g = ex / sum;
        } else {
            const float den = warp_sum_bcast(ex);
            g = ex / den;
        }
        if (lane < k) {
            a.topk_idx[(size_t)t * k + lane] = my_e;
            a.topk_gate[(size_t)t * k + lane] = g;
        }
        if (lane < 8) Is[tok * 8 + lane] = lane < k ? my_e : -1;
    }
    __syncthreads();

    // ---- per-expert statistics of this tile ----
    for (int e = tid; e < N; e += nthreads) {
        float ps = 0.0f;
        int cj[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        for (int tok = 0; tok < TT; ++tok) {
            ps += Ls[tok * N + e];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                if (j < k && Is[tok * 8 + j] == e) ++cj[j];
        }
        a.psum[(size_t)e * a.tiles + blockIdx.x] = ps;
#pragma unroll
        for (int j = 0; j < 8; ++j)
            if (j < k) a.cnt[((size_t)e * k + j) * a.tiles + blockIdx.x] = cj[j];
    }
}

// Block-wide exclusive scan of one int per thread; returns the exclusive prefix
// and writes the block total to *total. blockDim.x must be a multiple of 32.
__device__ int block_exclusive_scan(int v, int *sh /* >= 33 ints */, int *total) {
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
    const int res = sh[warp] + incl - v;
    *total = sh[32];
    __syncthreads();
    return res;
}

// Fixed-shape block sum (same association order on every run).
__device__ float block_sum(float v, float *sh /* >= 32 floats */) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) sh[warp] = v;
    __syncthreads();
    float r = 0.0f;
    if (warp == 0) {
        r = lane < nw ? sh[lane] : 0.0f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
        if (lane == 0) sh[0] = r;
    }
    __syncthreads();
    r = sh[0];
    __syncthreads();
    return r;
}

struct ScanArgs {
    int T, N, k, tiles, cap;  // cap 0: no limit
    const int32_t *cnt;       // [N][k][tiles]
    int32_t *pre;             // [N][k][tiles]
    int32_t *kpre;            // [N][tiles]
    const float *psum;        // [N][tiles]
    float *pmean;             // [N]
    int32_t *routed, *kept;   // [N]
};

__global__ void __launch_bounds__(256) k_expert_scan(ScanArgs a) {
    __shared__ int shi[33];
    __shared__ float shf[32];
    const int e = blockIdx.x, tid = threadIdx.x, nt = blockDim.x;
    const int n = a.k * a.tiles;
    const int32_t *ce = a.cnt + (size_t)e * n;
    int32_t *pe = a.pre + (size_t)e * n;
    const int C = a.cap > 0 ? a.cap : INT_MAX;

    // 1) exclusive prefix over (slot j, tile) = priority order
    const int per = (n + nt - 1) / nt;
    const int beg = min(n, tid * per), end = min(n, beg + per);
    int s = 0;
    for (int i = beg; i < end; ++i) s += ce[i];
    int total;
    int run = block_exclusive_scan(s, shi, &total);
    for (int i = beg; i < end; ++i) {
        pe[i] = run;
        run += ce[i];
    }
    __syncthreads();

    // 2) kept slots per tile, exclusive prefix over tiles
    const int per2 = (a.tiles + nt - 1) / nt;
    const int b2 = min(a.tiles, tid * per2), e2 = min(a.tiles, b2 + per2);
    int ks = 0;
    for (int tl = b2; tl < e2; ++tl)
        for (int j = 0; j < a.k; ++j) {
            const int i = j * a.tiles + tl;
            ks += min(max(C - pe[i], 0), ce[i]);
        }
    int ktot;
    int krun = block_exclusive_scan(ks, shi, &ktot);
    for (int tl = b2; tl < e2; ++tl) {
        a.kpre[(size_t)e * a.tiles + tl] = krun;
        for (int j = 0; j < a.k; ++j) {
            const int i = j * a.tiles + tl;
            krun += min(max(C - pe[i], 0), ce[i]);
        }
    }

    // 3) mean routing probability
    float ps = 0.0f;
    for (int tl = b2; tl < e2; ++tl) ps += a.psum[(size_t)e * a.tiles + tl];
    const float psum = block_sum(ps, shf);
    if (tid == 0) {
        a.routed[e] = total;
        a.kept[e] = ktot;
        a.pmean[e] = psum / (float)a.T;
    }
}

struct AssignArgs {
    int T, N, k, tiles, TT, cap;
    int64_t rmax;
    const int32_t *topk_idx;
    const int32_t *pre, *kpre;
    const int32_t *routed, *kept;
    const float *pmean;
    int32_t *offsets_out;  // may be null (then only the local copy is used)
    int32_t *slot_row, *perm_token;
    float *aux;            // may be null
    uint32_t *err;
};

__global__ void __launch_bounds__(256) k_assign(AssignArgs a) {
    extern __shared__ int sm[];
    int *offs = sm;                       // [N+1]
    int *Is = offs + a.N + 1;             // [TT][8]
    int *Ks = Is + a.TT * 8;              // [TT][8]
    __shared__ int shi[33];
    __shared__ float shf[32];
    const int tid = threadIdx.x, nt = blockDim.x, N = a.N, k = a.k;
    const int tile = blockIdx.x, t0 = tile * a.TT;
    const int C = a.cap > 0 ? a.cap : INT_MAX;

    // expert offsets (every CTA computes them; N <= 256 <= blockDim)
    {
        const int v = tid < N ? a.kept[tid] : 0;
        int total;
        const int ex = block_exclusive_scan(v, shi, &total);
        if (tid < N) offs[tid] = ex;
        if (tid == 0) offs[N] = total;
        __syncthreads();
        if (tile == 0 && a.offsets_out)
            for (int e = tid; e <= N; e += nt) a.offsets_out[e] = offs[e];
    }
    if (tile == 0 && a.aux) {
        const float invN = 1.0f / (float)N;
        float f0 = 0.0f, f1 = 0.0f;
        if (tid < N) {
            const float pm = a.pmean[tid];
            f0 = ((float)a.routed[tid] / (float)((int64_t)a.T * k)) * pm;
            f1 = (pm - invN) * (pm - invN);
        }
        const float s0 = block_sum(f0, shf);
        const float s1 = block_sum(f1, shf);
        if (tid == 0) {
            a.aux[0] = (float)N * s0;
            a.aux[1] = s1 * invN;
        }
    }

    for (int s = tid; s < a.TT * 8; s += nt) {
        const int tok = s >> 3, j = s & 7;
        const int t = t0 + tok;
        Is[s] = (t < a.T && j < k) ? a.topk_idx[(size_t)t * k + j] : -1;
        Ks[s] = 0;
    }
    __syncthreads();

    for (int s = tid; s < a.TT * k; s += nt) {
        const int tok = s / k, j = s % k, t = t0 + tok;
        if (t >= a.T) continue;
        const int e = Is[tok * 8 + j];
        if (e < 0 || e >= N) {
            record_error(a.err, kErrFault);
            continue;
        }
        int local = 0;
        for (int u = 0; u < tok; ++u) local += (Is[u * 8 + j] == e);
        const int r = a.pre[((size_t)e * k + j) * a.tiles + tile] + local;
        Ks[tok * 8 + j] = r < C;
    }
    __syncthreads();

    for (int s = tid; s < a.TT * k; s += nt) {
        const int tok = s / k, j = s % k, t = t0 + tok;
        if (t >= a.T) continue;
        const int e = Is[tok * 8 + j];
        int row = -1;
        if (e >= 0 && e < N && Ks[tok * 8 + j]) {
            int pos = a.kpre[(size_t)e * a.tiles + tile];
            for (int u = 0; u < tok; ++u)
                for (int jj = 0; jj < k; ++jj) pos += (Is[u * 8 + jj] == e && Ks[u * 8 + jj]);
            row = offs[e] + pos;
            if (row < 0 || row >= a.rmax) {
                record_error(a.err, kErrFault);
                row = -1;
            } else {
                a.perm_token[row] = t;
            }
        }
        a.slot_row[(size_t)t * k + j] = row;
    }
}

template <typename XT, int LE, int EPT, int TPT, bool A4>
cudaError_t launch_router_t(const moe_config &c, const XT *x, const float *w_r, const float *b_r,
                            RouterArgs ra, int warps, cudaStream_t s) {
    constexpr int NP = LE * EPT;
    const int TT = warps * 8;
    const size_t wbuf = (size_t)KC * c.N + NP;
    const size_t stage = 2 * wbuf + 2 * (size_t)KC * TT;
    const size_t gate = (size_t)TT * c.N + (size_t)TT * 8;
    const size_t bytes = std::max(stage, gate) * sizeof(float);
    auto kern = k_router<XT, LE, EPT, TPT, A4>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    kern<<<ra.tiles, warps * 32, bytes, s>>>(x, w_r, b_r, ra);
    return cudaGetLastError();
}

template <typename XT, int LE, int EPT, int TPT>
cudaError_t launch_router_a(const moe_config &c, const XT *x, const float *w_r, const float *b_r,
                            RouterArgs ra, int warps, cudaStream_t s) {
    if (c.N % 4 == 0) return launch_router_t<XT, LE, EPT, TPT, true>(c, x, w_r, b_r, ra, warps, s);
    return launch_router_t<XT, LE, EPT, TPT, false>(c, x, w_r, b_r, ra, warps, s);
}

template <typename XT>
cudaError_t launch_router_x(const moe_config &c, const XT *x, const float *w_r, const float *b_r,
                            RouterArgs ra, int warps, cudaStream_t s) {
    if (c.N <= 4) return launch_router_a<XT, 4, 1, 1>(c, x, w_r, b_r, ra, warps, s);
    if (c.N <= 8) return launch_router_a<XT, 4, 2, 1>(c, x, w_r, b_r, ra, warps, s);
    if (c.N <= 16) return launch_router_a<XT, 8, 2, 2>(c, x, w_r, b_r, ra, warps, s);
    if (c.N <= 32) return launch_router_a<XT, 16, 2, 4>(c, x, w_r, b_r, ra, warps, s);
    if (c.N <= 64) return launch_router_a<XT, 32, 2, 8>(c, x, w_r, b_r, ra, warps, s);
    if (c.N <= 128) return launch_router_a<XT, 32, 4, 8>(c, x, w_r, b_r, ra, warps, s);
    return launch_router_a<XT, 32, 8, 8>(c, x, w_r, b_r, ra, warps, s);
}

}  // namespace

cudaError_t launch_router(const moe_config &c, const void *x, const float *w_r, const float *b_r,
                          const RouterOut &o, uint8_t *ws, cudaStream_t s) {
    const WsLayout L = ws_layout(c);
    const int warps = router_warps(c);
    const int tiles = router_tiles(c);
    uint32_t *err = reinterpret_cast<uint32_t *>(ws + L.err);
    int32_t *cnt = reinterpret_cast<int32_t *>(ws + L.cnt);
    int32_t *pre = reinterpret_cast<int32_t *>(ws + L.pre);
    int32_t *kpre = reinterpret_cast<int32_t *>(ws + L.kpre);
    float *psum = reinterpret_cast<float *>(ws + L.psum);
    float *pmean = reinterpret_cast<float *>(ws + L.pmean);
    int32_t *routed = o.counts_routed ? o.counts_routed : reinterpret_cast<int32_t *>(ws + L.routed);
    int32_t *kept = o.counts_kept ? o.counts_kept : reinterpret_cast<int32_t *>(ws + L.kept);

    RouterArgs ra{c.T, c.d, c.N, c.k, c.gating, tiles, c.has_router_bias ? 1 : 0,
                  o.topk_idx, o.topk_gate, cnt, psum};
    cudaError_t e;
    if (c.dtype == MOE_BF16)
        e = launch_router_x<__nv_bfloat16>(c, static_cast<const __nv_bfloat16 *>(x), w_r, b_r, ra, warps, s);
    else
        e = launch_router_x<float>(c, static_cast<const float *>(x), w_r, b_r, ra, warps, s);
    if (e != cudaSuccess) return e;

    const int cap = capacity_of(c);
    ScanArgs sa{c.T, c.N, c.k, tiles, cap, cnt, pre, kpre, psum, pmean, routed, kept};
    k_expert_scan<<<c.N, 256, 0, s>>>(sa);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;

    const int TT = router_tile_tokens(c);
    AssignArgs aa{c.T, c.N, c.k, tiles, TT, cap, max_rows(c), o.topk_idx, pre, kpre, routed, kept,
                  pmean, o.expert_offsets, o.slot_row, o.perm_token, o.aux, err};
    const size_t sbytes = (size_t)(c.N + 1 + 2 * TT * 8) * sizeof(int);
    k_assign<<<tiles, 256, sbytes, s>>>(aa);
    return cudaGetLastError();
}

}  // namespace moe
