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
#include "tc_ptx.cuh"

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

struct RouterArgs {
    int T, d, N, k, gating, tiles, has_bias;
    int32_t *topk_idx;
    float *topk_gate;
    int32_t *cnt;   // [N][k][tiles]
    float *psum;    // [N][tiles]
    uint32_t *err;  // device error word (bounded waits)
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

// Expert of accumulator j of a thread in expert group le. With EPT >= 4 the
// experts come in runs of 4 interleaved across the LE groups, so one 128-bit
// shared load per run covers LE*16 contiguous bytes (no bank conflicts).
template <int LE, int EPT>
__device__ __forceinline__ int expert_of(int le, int j) {
    if constexpr (EPT >= 4) return (j / 4) * (LE * 4) + le * 4 + (j % 4);
    else return le * EPT + j;
}

template <int LE, int EPT, bool VEC>
__device__ __forceinline__ void load_w(const float *row, int le, float *wv) {
    if constexpr (VEC && EPT >= 4) {
#pragma unroll
        for (int g = 0; g < EPT / 4; ++g) lds<4>(row + g * LE * 4 + le * 4, wv + 4 * g);
    } else if constexpr (VEC) {
        lds<EPT>(row + le * EPT, wv);
    } else {
#pragma unroll
        for (int j = 0; j < EPT; ++j) wv[j] = row[expert_of<LE, EPT>(le, j)];
    }
}

// Logits -> gating -> per-tile statistics, shared by both router kernels.
// acc holds this thread's logits (TPT tokens x EPT experts, expert_of mapping);
// smem must hold TT*N + TT*8 words and be free (all staging consumed).
template <int LE, int EPT, int TPT>
__device__ __forceinline__ void router_tail(float (&acc)[TPT][EPT], float *smem, const float *__restrict__ b_r,
                                            const RouterArgs &a, int TT, int tok_base, int le) {
    constexpr int NP = LE * EPT;
    constexpr int QMAX = (NP + 31) / 32;
    const int N = a.N, T = a.T;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthreads = blockDim.x, nwarps = nthreads / 32;
    const int t0 = blockIdx.x * TT;
    // ---- logits to shared memory: Ls[TT][N]; Is[TT][8] behind it ----
    float *Ls = smem;
    int *Is = reinterpret_cast<int *>(smem + TT * N);
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
        const int e = expert_of<LE, EPT>(le, j);
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

// Gating tail for few experts (N <= 32): one thread per token (no shuffles),
// then per-tile statistics. Same rules as router_tail: top-k by logit, lower
// index first on ties, softmax over all N in fp32, gates per convention.
template <int LE, int EPT, int TPT>
__device__ __forceinline__ void router_tail_small(float (&acc)[TPT][EPT], float *smem,
                                                  const float *__restrict__ b_r, const RouterArgs &a, int TT,
                                                  int tok_base, int le) {
    const int N = a.N, T = a.T, k = a.k;
    const int tid = threadIdx.x, nthreads = blockDim.x;
    const int t0 = blockIdx.x * TT;
    float *Ls = smem;                                   // [TT][N] logits, then p
    int *Is = reinterpret_cast<int *>(smem + TT * N);   // [TT][8]
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
        const int e = expert_of<LE, EPT>(le, j);
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
    constexpr int NP = LE * EPT;  // <= 32: one token's logits fit in registers
    for (int tok = tid; tok < TT; tok += nthreads) {
        float *L = Ls + tok * N;
        const int t = t0 + tok;
        if (t >= T) {
            for (int e = 0; e < N; ++e) L[e] = 0.0f;
            for (int j = 0; j < 8; ++j) Is[tok * 8 + j] = -1;
            continue;
        }
        float Lr[NP];
#pragma unroll
        for (int e = 0; e < NP; ++e) Lr[e] = e < N ? L[e] : 0.0f;
        uint32_t taken = 0;
        float vmax = 0.0f, den = 0.0f;
        for (int s = 0; s < k; ++s) {
            float bv = -INFINITY;
            int bi = -1;
#pragma unroll
            for (int e = 0; e < NP; ++e)  // ascending e, strict '>': lowest index wins ties
                if (e < N && !((taken >> e) & 1u) && (bi < 0 || Lr[e] > bv)) {
                    bv = Lr[e];
                    bi = e;
                }
            taken |= 1u << bi;
            if (s == 0) vmax = bv;
            Is[tok * 8 + s] = bi;
        }
        float sum = 0.0f;
#pragma unroll
        for (int e = 0; e < NP; ++e) {
            Lr[e] = e < N ? expf(Lr[e] - vmax) : 0.0f;
            sum += Lr[e];
        }
        // exp of a selected expert's logit, picked without dynamic register indexing
        auto pick = [&](int e) {
            float v = 0.0f;
#pragma unroll
            for (int q = 0; q < NP; ++q) v = q == e ? Lr[q] : v;
            return v;
        };
        if (a.gating != MOE_SOFTMAX_THEN_TOPK)
            for (int s = 0; s < k; ++s) den += pick(Is[tok * 8 + s]);
        for (int s = 0; s < k; ++s) {
            const int e = Is[tok * 8 + s];
            const float ex = pick(e);
            a.topk_idx[(size_t)t * k + s] = e;
            a.topk_gate[(size_t)t * k + s] = a.gating == MOE_SOFTMAX_THEN_TOPK ? ex / sum : ex / den;
        }
        for (int s = k; s < 8; ++s) Is[tok * 8 + s] = -1;
#pragma unroll
        for (int e = 0; e < NP; ++e)
            if (e < N) L[e] = Lr[e] / sum;
    }
    __syncthreads();
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

// Shared-memory plan of the logits loop: a ring of STAGES chunks, each holding
// KC features of the router weight ([KC][N] fp32) and of the tile's token rows
// ([TT][KC] input type, rows padded by 16 bytes), filled by cp.async; plus one
// fp32 transposed copy of the current chunk's token values ([KC][TT]).
template <typename XT, int KC>
struct RouterSmem {
    static constexpr int STAGES = 4;
    static constexpr int XROW = KC * (int)sizeof(XT) + 16;  // bytes per staged token row
    static __host__ __device__ size_t w_bytes(int N) { return (size_t)KC * N * 4; }
    static __host__ __device__ size_t x_bytes(int TT) { return (size_t)TT * XROW; }
    static __host__ __device__ size_t stage_bytes(int N, int TT) { return w_bytes(N) + x_bytes(TT); }
    static __host__ __device__ size_t xf_offset(int N, int TT) { return STAGES * stage_bytes(N, TT); }
    // + NP floats of padding: lanes whose experts are >= N read (and discard) past the last row
    static __host__ __device__ size_t loop_bytes(int N, int TT, int NP) {
        return xf_offset(N, TT) + (size_t)KC * TT * 4 + (size_t)NP * 4;
    }
};

// Thread tile: TPT tokens x EPT experts; a warp is (32/LE) token groups x LE
// expert groups = 8 tokens x LE*EPT experts; warps stack along tokens.
template <typename XT, int LE, int EPT, int TPT, int KC, bool NALIGN4>
__global__ void __launch_bounds__(256) k_router(const XT *__restrict__ x, const float *__restrict__ w_r,
                                                const float *__restrict__ b_r, RouterArgs a) {
    using SM = RouterSmem<XT, KC>;
    constexpr int STAGES = SM::STAGES;
    constexpr int NP = LE * EPT;
    constexpr int VX = 16 / sizeof(XT);  // input elements per 16 bytes
    static_assert((32 / LE) * TPT == 8, "a warp covers 8 tokens");
    static_assert(KC % 8 == 0, "chunks hold whole 16-byte pieces");
    extern __shared__ __align__(16) float smem[];
    uint8_t *sbytes = reinterpret_cast<uint8_t *>(smem);

    const int nthreads = blockDim.x;
    const int nwarps = nthreads / 32;
    const int TT = nwarps * 8;
    const int N = a.N, d = a.d, T = a.T;
    const size_t stage_b = SM::stage_bytes(N, TT);
    const size_t wb_b = SM::w_bytes(N);
    float *Xf = reinterpret_cast<float *>(sbytes + SM::xf_offset(N, TT));  // [KC][TT]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int le = lane % LE, lt = lane / LE;
    const int t0 = blockIdx.x * TT;
    const int tok_base = warp * 8 + lt * TPT;

    float acc[TPT][EPT];
#pragma unroll
    for (int i = 0; i < TPT; ++i)
#pragma unroll
        for (int j = 0; j < EPT; ++j) acc[i][j] = 0.0f;

    const int nchunks = (d + KC - 1) / KC;

    // Copy chunk c into ring slot c % STAGES (one commit group per call, even if empty).
    auto issue = [&](int c) {
        if (c < nchunks) {
            const int k0 = c * KC;
            const int kc = min(KC, d - k0);
            uint8_t *slot = sbytes + (size_t)(c % STAGES) * stage_b;
            float *wdst = reinterpret_cast<float *>(slot);
            const float *wsrc = w_r + (size_t)k0 * N;
            if constexpr (NALIGN4) {
                const int nvec = kc * N / 4;
                for (int v = tid; v < nvec; v += nthreads) cp_async16(wdst + 4 * v, wsrc + 4 * v);
            } else {
                const int n = kc * N;
                for (int v = tid; v < n; v += nthreads) cp_async4(wdst + v, wsrc + v);
            }
            uint8_t *xdst = slot + wb_b;
            const int pieces = kc / VX;  // 16-byte pieces per token row in this chunk
            for (int v = tid; v < TT * pieces; v += nthreads) {
                const int tok = v / pieces, q = v % pieces;
                const int t = t0 + tok;
                if (t < T) cp_async16(xdst + (size_t)tok * SM::XROW + q * 16, x + (size_t)t * d + k0 + q * VX);
            }
        }
        cp_async_commit();
    };

#pragma unroll
    for (int c = 0; c < STAGES - 1; ++c) issue(c);

    for (int c = 0; c < nchunks; ++c) {
        cp_async_wait<STAGES - 2>();  // this thread's copies of chunk c have landed
        __syncthreads();              // ... everyone's; and chunk c-1 is fully consumed
        issue(c + STAGES - 1);        // into the slot chunk c-1 used
        const uint8_t *slot = sbytes + (size_t)(c % STAGES) * stage_b;
        const int kc = min(KC, d - c * KC);
        // token values of this chunk -> fp32, transposed to [KC][TT]
        {
            const uint8_t *xs = slot + wb_b;
            const int pieces = kc / VX;
            for (int v = tid; v < TT * pieces; v += nthreads) {
                const int q = v / TT, tok = v % TT;
                float f[VX];
                if (t0 + tok < T) {
                    Vec16<XT>::load(reinterpret_cast<const XT *>(xs + (size_t)tok * SM::XROW + q * 16), f);
                } else {
#pragma unroll
                    for (int i = 0; i < VX; ++i) f[i] = 0.0f;
                }
#pragma unroll
                for (int i = 0; i < VX; ++i) Xf[(q * VX + i) * TT + tok] = f[i];
            }
        }
        __syncthreads();
        const float *wb = reinterpret_cast<const float *>(slot);
        const float *xb = Xf + tok_base;
        if constexpr (TPT * EPT <= 8) {
            // Few accumulators: the FMA chains are the critical path, so load the
            // operands of the next 8 features while the current 8 are consumed.
            float xa[8][TPT], wa[8][EPT], xn[8][TPT], wn[8][EPT];
            auto load8 = [&](int k0, float (*xv)[TPT], float (*wv)[EPT]) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    lds<TPT>(xb + (k0 + q) * TT, xv[q]);
                    load_w<LE, EPT, NALIGN4>(wb + (k0 + q) * N, le, wv[q]);
                }
            };
            auto fma8 = [&](float (*xv)[TPT], float (*wv)[EPT]) {
#pragma unroll
                for (int q = 0; q < 8; ++q)
#pragma unroll
                    for (int i = 0; i < TPT; ++i)
#pragma unroll
                        for (int j = 0; j < EPT; ++j) acc[i][j] = __fmaf_rn(xv[q][i], wv[q][j], acc[i][j]);
            };
            load8(0, xa, wa);
            for (int k8 = 0; k8 < kc; k8 += 16) {
                if (k8 + 8 < kc) load8(k8 + 8, xn, wn);
                fma8(xa, wa);
                if (k8 + 8 < kc) {
                    if (k8 + 16 < kc) load8(k8 + 16, xa, wa);
                    fma8(xn, wn);
                }
            }
        } else {
#pragma unroll 4
            for (int kk = 0; kk < kc; ++kk) {
                float xv[TPT], wv[EPT];
                lds<TPT>(xb + kk * TT, xv);
                load_w<LE, EPT, NALIGN4>(wb + kk * N, le, wv);
#pragma unroll
                for (int i = 0; i < TPT; ++i)
#pragma unroll
                    for (int j = 0; j < EPT; ++j) acc[i][j] = __fmaf_rn(xv[i], wv[j], acc[i][j]);
            }
        }
    }
    cp_async_wait<0>();
    __syncthreads();

    router_tail<LE, EPT, TPT>(acc, smem, b_r, a, TT, tok_base, le);
}

// Router for few experts (LE*EPT <= 32). Here every logit's FMA chain over d is
// the critical path, so the loop is shaped for latency: the tile shape is fixed
// at compile time (NW warps, 8*NW tokens), the weight chunk is staged with row
// stride NP so every shared load uses an immediate offset, the token rows stay in
// their input type and are converted in registers (8 features per 128-bit load),
// and one barrier per chunk recycles the ring slot used two chunks earlier.
template <typename XT, int LE, int EPT, int NW, int KC, bool BULK>
__global__ void __launch_bounds__(NW * 32) k_router_small(const XT *__restrict__ x, const float *__restrict__ w_r,
                                                         const float *__restrict__ b_r, RouterArgs a) {
    constexpr int NP = LE * EPT;
    constexpr int TT = NW * 8;
    constexpr int TPT = 8 * LE / 32;
    constexpr int STAGES = 4;
    constexpr int ES = (int)sizeof(XT);
    constexpr int VX = 16 / ES;
    constexpr int XROW = KC * ES + 16;                       // bytes per staged token row
    constexpr int W_BYTES = KC * NP * 4;
    constexpr int STAGE = W_BYTES + TT * XROW;
    static_assert(NP <= 32 && (32 / LE) * TPT == 8, "small-N tile");
    static_assert(KC % 8 == 0 && (W_BYTES % 16) == 0, "16-byte pieces");
    static_assert(TT <= 31, "one token row per lane of warp 0");
    extern __shared__ __align__(16) float smem[];
    __shared__ uint64_t full[STAGES];
    __shared__ int abort_flag;
    uint8_t *sb = reinterpret_cast<uint8_t *>(smem);

    const int N = a.N, d = a.d, T = a.T;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int le = lane % LE, lt = lane / LE;
    const int t0 = blockIdx.x * TT;
    const int tok_base = warp * 8 + lt * TPT;
    const int nchunks = (d + KC - 1) / KC;
    const int ntok = min(TT, T - t0);

    float acc[TPT][EPT];
#pragma unroll
    for (int i = 0; i < TPT; ++i)
#pragma unroll
        for (int j = 0; j < EPT; ++j) acc[i][j] = 0.0f;

    if (tid == 0) {
        abort_flag = 0;
        if constexpr (BULK) {
            for (int i = 0; i < STAGES; ++i) tc::mbar_init(&full[i], 1);
            tc::fence_mbar_init();
        }
    }
    __syncthreads();

    // Stage chunk c into ring slot c % STAGES. BULK: one thread issues one bulk
    // copy for the weight rows (contiguous, N == NP) and one per token row, all
    // completing on the slot's mbarrier. Otherwise every thread issues cp.async.
    auto issue = [&](int c) {
        if constexpr (BULK) {
            // warp 0: lane 0 arms the barrier, then lane 0 copies the weight rows
            // and lanes 1..ntok one token row each (TT <= 31)
            if (warp == 0 && c < nchunks) {
                const int k0 = c * KC, kc = min(KC, d - k0);
                uint8_t *slot = sb + (c % STAGES) * STAGE;
                const uint32_t wbytes = (uint32_t)(kc * N * 4), xbytes = (uint32_t)(kc * ES);
                uint64_t *bar = &full[c % STAGES];
                if (lane == 0) tc::mbar_arrive_expect_tx(bar, wbytes + xbytes * (uint32_t)ntok);
                __syncwarp();
                if (lane == 0) tc::bulk_copy_g2s(slot, w_r + (size_t)k0 * N, wbytes, bar);
                else if (lane <= ntok)
                    tc::bulk_copy_g2s(slot + W_BYTES + (lane - 1) * XROW, x + (size_t)(t0 + lane - 1) * d + k0,
                                      xbytes, bar);
            }
        } else {
            if (c < nchunks) {
                const int k0 = c * KC, kc = min(KC, d - k0);
                uint8_t *slot = sb + (c % STAGES) * STAGE;
                float *wdst = reinterpret_cast<float *>(slot);
                const float *wsrc = w_r + (size_t)k0 * N;
                for (int v = tid; v < kc * N; v += NW * 32) {
                    const int r = v / N, e = v - r * N;
                    cp_async4(wdst + r * NP + e, wsrc + v);
                }
                uint8_t *xdst = slot + W_BYTES;
                const int pieces = kc / VX;
                for (int v = tid; v < ntok * pieces; v += NW * 32) {
                    const int tok = v / pieces, q = v - tok * pieces;
                    cp_async16(xdst + tok * XROW + q * 16, x + (size_t)(t0 + tok) * d + k0 + q * VX);
                }
            }
            cp_async_commit();
        }
    };
    // Wait until chunk c has landed; false if the wait ran out (error recorded).
    auto wait_chunk = [&](int c) -> bool {
        if constexpr (BULK) {
            uint64_t *bar = &full[c % STAGES];
            const uint32_t par = (uint32_t)((c / STAGES) & 1);
            if (!tc::mbar_try_wait(bar, par)) {
                const uint64_t ts = tc::globaltimer_ns();
                while (!tc::mbar_try_wait(bar, par)) {
                    if (*(volatile int *)&abort_flag) return false;
                    if (tc::globaltimer_ns() - ts > 1000000000ull) {
                        *(volatile int *)&abort_flag = 1;
                        record_error(a.err, kErrTimeout);
                        return false;
                    }
                }
            }
            return true;
        } else {
            cp_async_wait<STAGES - 2>();
            return true;
        }
    };

    auto load_x8 = [&](const uint8_t *xs, int k8, float (*xv)[TPT]) {
#pragma unroll
        for (int i = 0; i < TPT; ++i) {
            float f[8];
            const XT *p = reinterpret_cast<const XT *>(xs + (tok_base + i) * XROW) + k8;
            Vec16<XT>::load(p, f);
            if constexpr (VX == 4) Vec16<XT>::load(p + 4, f + 4);
#pragma unroll
            for (int q = 0; q < 8; ++q) xv[q][i] = f[q];
        }
    };
    auto step8 = [&](const float *ws, const uint8_t *xs, int k8) {
        float xv[8][TPT], wv[8][EPT];
        load_x8(xs, k8, xv);
#pragma unroll
        for (int q = 0; q < 8; ++q) lds<EPT>(ws + (k8 + q) * NP + le * EPT, wv[q]);
#pragma unroll
        for (int q = 0; q < 8; ++q)
#pragma unroll
            for (int i = 0; i < TPT; ++i)
#pragma unroll
                for (int j = 0; j < EPT; ++j) acc[i][j] = __fmaf_rn(xv[q][i], wv[q][j], acc[i][j]);
    };

#pragma unroll
    for (int c = 0; c < STAGES - 1; ++c) issue(c);
    int issued = STAGES - 1;
    bool ok = true;
    for (int c = 0; c < nchunks; ++c) {
        ok = wait_chunk(c);
        __syncthreads();
        if (!ok || *(volatile int *)&abort_flag) {
            ok = false;
            break;
        }
        issue(c + STAGES - 1);
        ++issued;
        const uint8_t *slot = sb + (c % STAGES) * STAGE;
        const float *ws = reinterpret_cast<const float *>(slot);
        const uint8_t *xs = slot + W_BYTES;
        const int kc = min(KC, d - c * KC);
        if (kc == KC) {
#pragma unroll
            for (int k8 = 0; k8 < KC; k8 += 8) step8(ws, xs, k8);
        } else {
            for (int k8 = 0; k8 < kc; k8 += 8) step8(ws, xs, k8);
        }
    }
    if constexpr (BULK) {
        // every copy issued lands before shared memory is reused or the CTA exits
        if (tid == 0)
            for (int c = max(0, issued - STAGES); c < min(issued, nchunks); ++c) {
                const uint64_t ts = tc::globaltimer_ns();
                while (!tc::mbar_try_wait(&full[c % STAGES], (uint32_t)((c / STAGES) & 1)))
                    if (tc::globaltimer_ns() - ts > 1000000000ull) break;
            }
    } else {
        cp_async_wait<0>();
    }
    __syncthreads();
    if (!ok) return;
    router_tail_small<LE, EPT, TPT>(acc, smem, b_r, a, TT, tok_base, le);
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

template <typename XT, int LE, int EPT, int TPT, int KC, bool A4>
cudaError_t launch_router_t(const moe_config &c, const XT *x, const float *w_r, const float *b_r,
                            RouterArgs ra, int warps, cudaStream_t s) {
    constexpr int NP = LE * EPT;
    const int TT = warps * 8;
    const size_t loop = RouterSmem<XT, KC>::loop_bytes(c.N, TT, NP);
    const size_t gate = ((size_t)TT * c.N + (size_t)TT * 8) * sizeof(float);
    const size_t bytes = std::max(loop, gate);
    auto kern = k_router<XT, LE, EPT, TPT, KC, A4>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    kern<<<ra.tiles, warps * 32, bytes, s>>>(x, w_r, b_r, ra);
    return cudaGetLastError();
}

// Many experts: chunks of 32 features so that four stages of [KC][N] weights fit.
template <typename XT, int LE, int EPT, int TPT>
cudaError_t launch_router_a(const moe_config &c, const XT *x, const float *w_r, const float *b_r,
                            RouterArgs ra, int warps, cudaStream_t s) {
    constexpr int KC = 32;
    if (c.N % 4 == 0) return launch_router_t<XT, LE, EPT, TPT, KC, true>(c, x, w_r, b_r, ra, warps, s);
    return launch_router_t<XT, LE, EPT, TPT, KC, false>(c, x, w_r, b_r, ra, warps, s);
}

// Few experts: 2 warps (16 tokens) per CTA, chunks of 256 features; bulk copies
// when the weight chunk is one contiguous block of whole 16-byte pieces.
template <typename XT, int LE, int EPT>
cudaError_t launch_router_small(const moe_config &c, const XT *x, const float *w_r, const float *b_r,
                                RouterArgs ra, cudaStream_t s) {
    constexpr int NW = 2, KC = 256, TT = NW * 8;
    constexpr size_t stage = (size_t)KC * LE * EPT * 4 + (size_t)TT * (KC * sizeof(XT) + 16);
    const size_t gate = ((size_t)TT * c.N + (size_t)TT * 8) * sizeof(float);
    const size_t bytes = std::max(4 * stage, gate);
    const bool bulk = c.N == LE * EPT && c.N % 4 == 0;
    auto kern = bulk ? k_router_small<XT, LE, EPT, NW, KC, true> : k_router_small<XT, LE, EPT, NW, KC, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    kern<<<ra.tiles, NW * 32, bytes, s>>>(x, w_r, b_r, ra);
    return cudaGetLastError();
}

template <typename XT>
cudaError_t launch_router_x(const moe_config &c, const XT *x, const float *w_r, const float *b_r,
                            RouterArgs ra, int warps, cudaStream_t s) {
    if (c.N <= 4) return launch_router_small<XT, 4, 1>(c, x, w_r, b_r, ra, s);
    if (c.N <= 8) return launch_router_small<XT, 4, 2>(c, x, w_r, b_r, ra, s);
    if (c.N <= 16) return launch_router_small<XT, 8, 2>(c, x, w_r, b_r, ra, s);
    if (c.N <= 32) return launch_router_small<XT, 16, 2>(c, x, w_r, b_r, ra, s);
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
                  o.topk_idx, o.topk_gate, cnt, psum, err};
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
