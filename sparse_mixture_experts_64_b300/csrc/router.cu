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
// Logit summation order (the pages fix none; routing must be bit-exact, so one
// order is specified): features in blocks of 8; lane l of a warp accumulates
// blocks l, l+32, l+64, ... with one fp32 fma per feature in increasing order,
// starting from 0; the 32 lane partials are combined by five xor-butterfly
// rounds v = v + shfl_xor(v, o), o = 16, 8, 4, 2, 1, and lane 0's value is the
// logit; the bias is added last. Every kernel below keeps exactly this order.
//
// Kernels (no atomics, deterministic):
//   k_router_small   N <= 32: one CTA per tile of tokens; each lane holds every
//                    expert's partial for its tokens; gating fused (one thread per
//                    token). Per-tile routed counts per slot and sums of p.
//   k_transpose_wr   N > 32: router weight [d][N] -> [N][d] (workspace), so that a
//                    lane's 8 features of one expert are contiguous.
//   k_logits_large   N > 32: 16 tokens x 32 experts per CTA -> logits [T][N].
//   k_gate           N > 32: one warp per token: top-k, softmax, gates; per-tile stats.
//   k_expert_scan    one CTA per expert: priority-order prefix of the tile counts
//                    (slot-major, token order), capacity clamp, kept-per-tile
//                    prefix, routed/kept totals, mean routing probability P_e.
//   k_assign         one CTA per tile: keep/drop per slot, row of each kept slot
//                    (expert ascending, token ascending), perm_token; CTA 0 also
//                    writes expert_offsets and the aux losses.
#include <algorithm>
#include <climits>
#include <cmath>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace moe {

// Experts per lane register row of the small kernel: 4, 8, 16 or 32.
static int router_np(int N) { return N <= 4 ? 4 : N <= 8 ? 8 : N <= 16 ? 16 : 32; }

int router_tile_tokens(const moe_config &c) {
    if (c.N > 32) return 64;           // k_gate: 8 warps x 8 tokens
    return 4 * (32 / router_np(c.N));  // k_router_small: 4 warps x (32 / NP) tokens
}

namespace {

constexpr uint64_t kWaitNs = 1000000000ull;  // bound of every mbarrier wait (1 s)

struct RouterArgs {
    int T, d, N, k, gating, tiles, has_bias;
    int32_t *topk_idx;
    float *topk_gate;
    int32_t *cnt;   // [N][k][tiles]
    float *psum;    // [N][tiles]
    uint32_t *err;  // device error word
};

// 8 consecutive features of one token as fp32 (16 bytes of bf16, 32 of fp32).
template <typename XT>
__device__ __forceinline__ void load8(const uint8_t *p, float *f) {
    Vec16<XT>::load(reinterpret_cast<const XT *>(p), f);
    if constexpr (sizeof(XT) == 4) Vec16<XT>::load(reinterpret_cast<const XT *>(p) + 4, f + 4);
}

template <int n> __device__ __forceinline__ void lds(const float *p, float *v) {
#pragma unroll
    for (int i = 0; i < n; i += 4) {
        const float4 q = *reinterpret_cast<const float4 *>(p + i);
        v[i] = q.x; v[i + 1] = q.y; v[i + 2] = q.z; v[i + 3] = q.w;
    }
}

// v <- v + shfl_xor(v, o) for o = 16 .. 1; lane 0 then holds the specified sum.
__device__ __forceinline__ float butterfly32(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Bounded wait for phase `par` of `bar`; on expiry sets *abort_flag and records
// MOE_ERR_TIMEOUT. Returns false if the wait ran out or another thread aborted.
__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t par, int *abort_flag, uint32_t *err) {
    if (tc::mbar_try_wait(bar, par)) return true;
    const uint64_t t0 = tc::globaltimer_ns();
    while (!tc::mbar_try_wait(bar, par)) {
        if (*(volatile int *)abort_flag) return false;
        if (tc::globaltimer_ns() - t0 > kWaitNs) {
            *(volatile int *)abort_flag = 1;
            record_error(err, kErrTimeout);
            return false;
        }
    }
    return true;
}

// Stride (in floats) of one staged block of 8 router-weight rows [8][N] in the
// small kernel: room for reads up to column NP-1 and == 4 (mod 32) words, so the
// 32 lanes reading 32 different blocks spread over the banks.
__host__ __device__ inline int wblock_stride(int N, int NP) {
    int s = 8 * N + (NP > N ? NP - N : 0);
    s = (s + 3) & ~3;
    s += ((4 - (s & 31)) + 32) & 31;
    return s;
}

// ------------------------------------------------------------------ gating

// Per-tile statistics from p (Ls) and the selections (Is): per expert, the sum of
// p over the tile's tokens and the number of tokens choosing it in each slot.
__device__ __forceinline__ void tile_stats(const float *Ls, const int *Is, const RouterArgs &a, int TT) {
    const int N = a.N, k = a.k;
    for (int e = threadIdx.x; e < N; e += blockDim.x) {
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

// Gating for N <= NP <= 32 experts, one thread per token. Ls [TT][N] holds the
// logits on entry and p on exit; Is [TT][8] receives the selections.
template <int NP>
__device__ __forceinline__ void gate_tokens_thread(float *Ls, int *Is, const RouterArgs &a, int TT) {
    const int N = a.N, T = a.T, k = a.k;
    const int t0 = blockIdx.x * TT;
    for (int tok = threadIdx.x; tok < TT; tok += blockDim.x) {
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
        auto pick = [&](int e) {  // Lr[e] without dynamic register indexing
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
}

__device__ __forceinline__ float warp_sum_bcast(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return __shfl_sync(0xffffffffu, v, 0);
}

// Gating for any N <= 256, one warp per token (lane holds experts lane + 32q).
__device__ __forceinline__ void gate_tokens_warp(float *Ls, int *Is, const RouterArgs &a, int TT) {
    constexpr int QMAX = 8;
    const int N = a.N, T = a.T, k = a.k;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
    const int t0 = blockIdx.x * TT;
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
}

// ------------------------------------------------------------------ N <= 32

// One CTA = 4 warps; warp w owns TO = 32/NP tokens and all NP experts; lane l
// owns partial l. Chunks of 256 features (one 8-feature block per lane) are
// staged by bulk copies issued from warp 0 (lane j copies weight block j and
// token row j) into a 6-slot ring, each slot completing on its own mbarrier.
template <typename XT, int NP, bool VEC>
__global__ void __launch_bounds__(128) k_router_small(const XT *__restrict__ x, const float *__restrict__ w_r,
                                                     const float *__restrict__ b_r, RouterArgs a) {
    constexpr int NW = 4, TO = 32 / NP, TT = NW * TO;
    constexpr int KC = 256, NBLK = KC / 8;
    constexpr int STAGES = 6;
    constexpr int ES = (int)sizeof(XT);
    constexpr int XROW = KC * ES + 16;
    static_assert(TT <= 32, "one token row per lane of warp 0");
    extern __shared__ __align__(16) float smem[];
    __shared__ uint64_t full[STAGES];
    __shared__ int abort_flag;
    uint8_t *sb = reinterpret_cast<uint8_t *>(smem);

    const int N = a.N, d = a.d, T = a.T;
    const int BST = wblock_stride(N, NP);
    const int W_BYTES = NBLK * BST * 4;
    const int STAGE = W_BYTES + TT * XROW;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = blockIdx.x * TT;
    const int ntok = min(TT, T - t0);
    const int nblocks = d / 8;
    const int nchunks = (nblocks + NBLK - 1) / NBLK;

    if (tid == 0) {
        abort_flag = 0;
        for (int i = 0; i < STAGES; ++i) tc::mbar_init(&full[i], 1);
        tc::fence_mbar_init();
    }
    __syncthreads();

    auto issue = [&](int c) {
        if (warp != 0 || c >= nchunks) return;
        const int b0 = c * NBLK, nb = min(NBLK, nblocks - b0);
        uint8_t *slot = sb + (size_t)(c % STAGES) * STAGE;
        uint64_t *bar = &full[c % STAGES];
        const uint32_t wb = (uint32_t)(8 * N * 4), xb = (uint32_t)(nb * 8 * ES);
        if (lane == 0) tc::mbar_arrive_expect_tx(bar, (uint32_t)nb * wb + (uint32_t)ntok * xb);
        __syncwarp();
        if (lane < nb) tc::bulk_copy_g2s(slot + lane * BST * 4, w_r + (size_t)(b0 + lane) * 8 * N, wb, bar);
        if (lane < ntok)
            tc::bulk_copy_g2s(slot + W_BYTES + lane * XROW, x + (size_t)(t0 + lane) * d + (size_t)b0 * 8, xb, bar);
    };

    float acc[TO][NP];
#pragma unroll
    for (int i = 0; i < TO; ++i)
#pragma unroll
        for (int e = 0; e < NP; ++e) acc[i][e] = 0.0f;

#pragma unroll
    for (int c = 0; c < STAGES - 1; ++c) issue(c);
    bool ok = true;
    int issued = min(STAGES - 1, nchunks);
    for (int c = 0; c < nchunks; ++c) {
        const bool mine = wait_phase(&full[c % STAGES], (uint32_t)((c / STAGES) & 1), &abort_flag, a.err);
        __syncthreads();
        if (!mine || *(volatile int *)&abort_flag) {
            ok = false;
            break;
        }
        issue(c + STAGES - 1);
        if (c + STAGES - 1 < nchunks) ++issued;
        const uint8_t *slot = sb + (size_t)(c % STAGES) * STAGE;
        if (c * NBLK + lane < nblocks) {
            const float *wbk = reinterpret_cast<const float *>(slot) + lane * BST;
            float xf[TO][8];
#pragma unroll
            for (int i = 0; i < TO; ++i) load8<XT>(slot + W_BYTES + (warp * TO + i) * XROW + lane * 8 * ES, xf[i]);
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                float wv[NP];
                if constexpr (VEC) {
                    lds<NP>(wbk + r * N, wv);
                } else {
#pragma unroll
                    for (int e = 0; e < NP; ++e) wv[e] = wbk[r * N + e];
                }
#pragma unroll
                for (int i = 0; i < TO; ++i)
#pragma unroll
                    for (int e = 0; e < NP; ++e) acc[i][e] = __fmaf_rn(xf[i][r], wv[e], acc[i][e]);
            }
        }
    }
    // every copy issued has landed before shared memory is reused or the CTA exits
    if (tid == 0)
        for (int c = max(0, issued - STAGES); c < issued; ++c) {
            const uint64_t ts = tc::globaltimer_ns();
            while (!tc::mbar_try_wait(&full[c % STAGES], (uint32_t)((c / STAGES) & 1)))
                if (tc::globaltimer_ns() - ts > kWaitNs) break;
        }
    __syncthreads();
    if (!ok) return;

    float *Ls = smem;                                    // [TT][N]
    int *Is = reinterpret_cast<int *>(smem + TT * N);    // [TT][8]
#pragma unroll
    for (int i = 0; i < TO; ++i)
#pragma unroll
        for (int e = 0; e < NP; ++e) {
            const float v = butterfly32(acc[i][e]);
            if (lane == 0 && e < N) Ls[(warp * TO + i) * N + e] = a.has_bias ? __fadd_rn(v, b_r[e]) : v;
        }
    __syncthreads();
    gate_tokens_thread<NP>(Ls, Is, a, TT);
    __syncthreads();
    tile_stats(Ls, Is, a, TT);
}

// ------------------------------------------------------------------ N > 32

__global__ void __launch_bounds__(256) k_transpose_wr(const float *__restrict__ w_r, float *__restrict__ w_t,
                                                      int d, int N) {
    __shared__ float tile[32][33];
    const int i0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    for (int r = ty; r < 32; r += 8)
        if (i0 + r < d && e0 + tx < N) tile[r][tx] = w_r[(size_t)(i0 + r) * N + e0 + tx];
    __syncthreads();
    for (int r = ty; r < 32; r += 8)
        if (e0 + r < N && i0 + tx < d) w_t[(size_t)(e0 + r) * d + i0 + tx] = tile[tx][r];
}

struct LogitsArgs {
    int T, d, N, has_bias;
    float *logits;  // [T][N]
    uint32_t *err;
};

// One CTA = 16 warps = 4 token groups x 4 expert groups; warp tile 4 tokens x 8
// experts, lane l = partial l. Tile 16 tokens x 32 experts; chunks of 256 features:
// token rows and transposed weight rows ([expert][feature], so a lane's 8 features
// of one expert are one 32-byte run) by bulk copies into a 4-slot ring.
template <typename XT>
__global__ void __launch_bounds__(512, 1) k_logits_large(const XT *__restrict__ x, const float *__restrict__ w_t,
                                                        const float *__restrict__ b_r, LogitsArgs a) {
    constexpr int TOK = 16, EXP = 32, TO = 4, EO = 8;
    constexpr int KC = 256, NBLK = KC / 8, STAGES = 4;
    constexpr int ES = (int)sizeof(XT);
    constexpr int XROW = KC * ES + 16;
    constexpr int WROW = KC * 4 + 16;
    constexpr int X_BYTES = TOK * XROW;
    constexpr int STAGE = X_BYTES + EXP * WROW;
    extern __shared__ __align__(16) float smem[];
    __shared__ uint64_t full[STAGES];
    __shared__ int abort_flag;
    uint8_t *sb = reinterpret_cast<uint8_t *>(smem);

    const int T = a.T, d = a.d, N = a.N;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tg = warp >> 2, eg = warp & 3;
    const int t0 = blockIdx.x * TOK, e0 = blockIdx.y * EXP;
    const int ntok = min(TOK, T - t0), nexp = min(EXP, N - e0);
    const int nblocks = d / 8;
    const int nchunks = (nblocks + NBLK - 1) / NBLK;

    if (tid == 0) {
        abort_flag = 0;
        for (int i = 0; i < STAGES; ++i) tc::mbar_init(&full[i], 1);
        tc::fence_mbar_init();
    }
    __syncthreads();

    auto issue = [&](int c) {
        if (warp != 0 || c >= nchunks) return;
        const int b0 = c * NBLK, nb = min(NBLK, nblocks - b0);
        uint8_t *slot = sb + (size_t)(c % STAGES) * STAGE;
        uint64_t *bar = &full[c % STAGES];
        const uint32_t xb = (uint32_t)(nb * 8 * ES), wb = (uint32_t)(nb * 8 * 4);
        if (lane == 0) tc::mbar_arrive_expect_tx(bar, (uint32_t)ntok * xb + (uint32_t)nexp * wb);
        __syncwarp();
        if (lane < ntok)
            tc::bulk_copy_g2s(slot + lane * XROW, x + (size_t)(t0 + lane) * d + (size_t)b0 * 8, xb, bar);
        if (lane < nexp)
            tc::bulk_copy_g2s(slot + X_BYTES + lane * WROW, w_t + (size_t)(e0 + lane) * d + (size_t)b0 * 8, wb, bar);
    };

    float acc[TO][EO];
#pragma unroll
    for (int i = 0; i < TO; ++i)
#pragma unroll
        for (int j = 0; j < EO; ++j) acc[i][j] = 0.0f;

#pragma unroll
    for (int c = 0; c < STAGES - 1; ++c) issue(c);
    bool ok = true;
    int issued = min(STAGES - 1, nchunks);
    for (int c = 0; c < nchunks; ++c) {
        const bool mine = wait_phase(&full[c % STAGES], (uint32_t)((c / STAGES) & 1), &abort_flag, a.err);
        __syncthreads();
        if (!mine || *(volatile int *)&abort_flag) {
            ok = false;
            break;
        }
        issue(c + STAGES - 1);
        if (c + STAGES - 1 < nchunks) ++issued;
        const uint8_t *slot = sb + (size_t)(c % STAGES) * STAGE;
        if (c * NBLK + lane < nblocks) {
            float xf[TO][8];
#pragma unroll
            for (int i = 0; i < TO; ++i) load8<XT>(slot + (tg * TO + i) * XROW + lane * 8 * ES, xf[i]);
            const float *wl = reinterpret_cast<const float *>(slot + X_BYTES) + lane * 8;
#pragma unroll
            for (int jp = 0; jp < EO; jp += 2) {
                float w0[8], w1[8];
                lds<8>(wl + (eg * EO + jp) * (WROW / 4), w0);
                lds<8>(wl + (eg * EO + jp + 1) * (WROW / 4), w1);
#pragma unroll
                for (int r = 0; r < 8; ++r)
#pragma unroll
                    for (int i = 0; i < TO; ++i) {
                        acc[i][jp] = __fmaf_rn(xf[i][r], w0[r], acc[i][jp]);
                        acc[i][jp + 1] = __fmaf_rn(xf[i][r], w1[r], acc[i][jp + 1]);
                    }
            }
        }
    }
    if (tid == 0)
        for (int c = max(0, issued - STAGES); c < issued; ++c) {
            const uint64_t ts = tc::globaltimer_ns();
            while (!tc::mbar_try_wait(&full[c % STAGES], (uint32_t)((c / STAGES) & 1)))
                if (tc::globaltimer_ns() - ts > kWaitNs) break;
        }
    __syncthreads();
    if (!ok) return;
#pragma unroll
    for (int i = 0; i < TO; ++i)
#pragma unroll
        for (int j = 0; j < EO; ++j) {
            const float v = butterfly32(acc[i][j]);
            const int t = t0 + tg * TO + i, e = e0 + eg * EO + j;
            if (lane == 0 && t < T && e < N) a.logits[(size_t)t * N + e] = a.has_bias ? __fadd_rn(v, b_r[e]) : v;
        }
}

// One CTA = 8 warps, 64 tokens: logits tile -> shared memory -> gating -> stats.
__global__ void __launch_bounds__(256) k_gate(const float *__restrict__ logits, RouterArgs a) {
    constexpr int TT = 64;
    extern __shared__ __align__(16) float smem[];
    float *Ls = smem;                                    // [TT][N]
    int *Is = reinterpret_cast<int *>(smem + TT * a.N);  // [TT][8]
    const int t0 = blockIdx.x * TT;
    const int nrows = min(TT, a.T - t0);
    for (int i = threadIdx.x; i < nrows * a.N; i += blockDim.x) Ls[i] = logits[(size_t)t0 * a.N + i];
    __syncthreads();
    gate_tokens_warp(Ls, Is, a, TT);
    __syncthreads();
    tile_stats(Ls, Is, a, TT);
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

template <typename XT, int NP>
cudaError_t launch_small(const moe_config &c, const XT *x, const float *w_r, const float *b_r, RouterArgs ra,
                         cudaStream_t s) {
    constexpr int TT = 4 * (32 / NP);
    const size_t stage = (size_t)32 * wblock_stride(c.N, NP) * 4 + (size_t)TT * (256 * sizeof(XT) + 16);
    const size_t gate = ((size_t)TT * c.N + (size_t)TT * 8) * sizeof(float);
    const size_t bytes = std::max(6 * stage, gate);
    auto kern = c.N % 4 == 0 ? k_router_small<XT, NP, true> : k_router_small<XT, NP, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    kern<<<ra.tiles, 128, bytes, s>>>(x, w_r, b_r, ra);
    return cudaGetLastError();
}

template <typename XT>
cudaError_t launch_large(const moe_config &c, const XT *x, const float *w_r, const float *b_r, RouterArgs ra,
                         float *logits, float *w_t, cudaStream_t s) {
    k_transpose_wr<<<dim3((c.d + 31) / 32, (c.N + 31) / 32), 256, 0, s>>>(w_r, w_t, c.d, c.N);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    LogitsArgs la{c.T, c.d, c.N, ra.has_bias, logits, ra.err};
    const size_t lbytes = 4 * (size_t)(16 * (256 * sizeof(XT) + 16) + 32 * (256 * 4 + 16));
    e = cudaFuncSetAttribute(k_logits_large<XT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lbytes);
    if (e != cudaSuccess) return e;
    k_logits_large<XT><<<dim3((c.T + 15) / 16, (c.N + 31) / 32), 512, lbytes, s>>>(x, w_t, b_r, la);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const size_t gbytes = ((size_t)64 * c.N + 64 * 8) * sizeof(float);
    e = cudaFuncSetAttribute(k_gate, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gbytes);
    if (e != cudaSuccess) return e;
    k_gate<<<ra.tiles, 256, gbytes, s>>>(logits, ra);
    return cudaGetLastError();
}

template <typename XT>
cudaError_t launch_logits_gate(const moe_config &c, const XT *x, const float *w_r, const float *b_r, RouterArgs ra,
                               float *logits, float *w_t, cudaStream_t s) {
    if (c.N <= 4) return launch_small<XT, 4>(c, x, w_r, b_r, ra, s);
    if (c.N <= 8) return launch_small<XT, 8>(c, x, w_r, b_r, ra, s);
    if (c.N <= 16) return launch_small<XT, 16>(c, x, w_r, b_r, ra, s);
    if (c.N <= 32) return launch_small<XT, 32>(c, x, w_r, b_r, ra, s);
    return launch_large<XT>(c, x, w_r, b_r, ra, logits, w_t, s);
}

}  // namespace

cudaError_t launch_router(const moe_config &c, const void *x, const float *w_r, const float *b_r,
                          const RouterOut &o, uint8_t *ws, cudaStream_t s) {
    const WsLayout L = ws_layout(c);
    const int tiles = router_tiles(c);
    uint32_t *err = reinterpret_cast<uint32_t *>(ws + L.err);
    int32_t *cnt = reinterpret_cast<int32_t *>(ws + L.cnt);
    int32_t *pre = reinterpret_cast<int32_t *>(ws + L.pre);
    int32_t *kpre = reinterpret_cast<int32_t *>(ws + L.kpre);
    float *psum = reinterpret_cast<float *>(ws + L.psum);
    float *pmean = reinterpret_cast<float *>(ws + L.pmean);
    float *logits = reinterpret_cast<float *>(ws + L.logits);
    float *w_t = reinterpret_cast<float *>(ws + L.w_t);
    int32_t *routed = o.counts_routed ? o.counts_routed : reinterpret_cast<int32_t *>(ws + L.routed);
    int32_t *kept = o.counts_kept ? o.counts_kept : reinterpret_cast<int32_t *>(ws + L.kept);

    RouterArgs ra{c.T, c.d, c.N, c.k, c.gating, tiles, c.has_router_bias ? 1 : 0,
                  o.topk_idx, o.topk_gate, cnt, psum, err};
    cudaError_t e;
    if (c.dtype == MOE_BF16)
        e = launch_logits_gate<__nv_bfloat16>(c, static_cast<const __nv_bfloat16 *>(x), w_r, b_r, ra, logits, w_t, s);
    else
        e = launch_logits_gate<float>(c, static_cast<const float *>(x), w_r, b_r, ra, logits, w_t, s);
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
