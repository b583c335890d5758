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
//   k_transpose_wr   router weight [d][N] -> chunk-major copy in the workspace, per
//                    expert (k_router_small) or per expert pair (k_logits_large),
//                    so that a lane's features of a block load as 16-byte runs.
//   k_logits_large   N > 32: 48 (bf16) or 32 (fp32) tokens x 16 experts per CTA -> logits [T][N]; one
//                    packed fp32x2 fma updates two experts' partials (each half
//                    rounds exactly like a scalar fma, so the order above holds).
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
    if (c.N > 32) return 64;           // k_gate: 32 warps x 2 tokens
    return 4 * (32 / router_np(c.N));  // k_router_small: 4 warps x (32 / NP) tokens
}

namespace {

constexpr uint64_t kWaitNs = 1000000000ull;  // bound of every mbarrier wait (1 s)
// Bound of the waits of k_router_small under MOE_DEBUG_ROUTER_STALL (1 ms): its producer
// then issues no copy, so the consumers' first wait runs out with nothing in flight.
constexpr uint64_t kStallWaitNs = 1000000ull;

struct RouterArgs {
    int T, d, N, k, gating, tiles, has_bias;
    int32_t *topk_idx;
    float *topk_gate;
    int32_t *cnt;   // [N][k][tiles]
    float *psum;    // [N][tiles]
    uint32_t *err;  // device error word
    // training-time router: noise draws [T][N] (null: none) and their weight; per-tile
    // sums of the z-loss terms (null: no z-loss)
    const float *noise = nullptr;
    float noise_w = 0.0f;
    float *zpart = nullptr;
    int stall = 0;  // MOE_DEBUG_ROUTER_STALL (k_router_small only)
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
__device__ __forceinline__ bool wait_phase(uint64_t *bar, uint32_t par, int *abort_flag, uint32_t *err,
                                           uint64_t limit_ns = kWaitNs) {
    if (tc::mbar_try_wait(bar, par)) return true;
    const uint64_t t0 = tc::globaltimer_ns();
    while (!tc::mbar_try_wait(bar, par)) {
        if (*(volatile int *)abort_flag) return false;
        if (tc::globaltimer_ns() - t0 > limit_ns) {
            *(volatile int *)abort_flag = 1;
            record_error(err, kErrTimeout);
            return false;
        }
    }
    return true;
}

// ------------------------------------------------------------------ gating

// Selection key of a logit: the fp32 order as a signed integer, with -0 equal to +0,
// a NaN below every number (-inf included), and taken or absent experts below that.
// For numeric logits the larger key is the larger logit, so selecting the largest key,
// lower expert index first on equal keys, is selection by logit; a NaN logit (a NaN in
// the token or the router weight) is chosen only when no numeric logit is left, and
// every token still gets k distinct experts.
constexpr int kKeyNaN = INT_MIN + 1;
constexpr int kKeyNone = INT_MIN;
__device__ __forceinline__ int sel_key(float v) {
    if (v != v) return kKeyNaN;
    const int b = __float_as_int(__fadd_rn(v, 0.0f));  // -0 + 0 = +0
    return b >= 0 ? b : b ^ 0x7fffffff;
}
// The logit of a numeric key (+0 for a zero logit), NaN for kKeyNaN.
__device__ __forceinline__ float key_value(int key) {
    if (key == kKeyNaN) return __int_as_float(0x7fc00000);
    return __int_as_float(key >= 0 ? key : key ^ 0x7fffffff);
}

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
        int key[NP];
#pragma unroll
        for (int e = 0; e < NP; ++e) {
            Lr[e] = e < N ? L[e] : 0.0f;
            key[e] = e < N ? sel_key(Lr[e]) : kKeyNone;
        }
        float vmax = 0.0f, den = 0.0f;
        for (int s = 0; s < k; ++s) {
            // an untaken expert of this token has a key above kKeyNone (k <= N)
            int bk = kKeyNone, bi = 0;
#pragma unroll
            for (int e = 0; e < NP; ++e)  // ascending e, strict '>': lowest index wins ties
                if (key[e] > bk) {
                    bk = key[e];
                    bi = e;
                }
#pragma unroll
            for (int e = 0; e < NP; ++e) key[e] = e == bi ? kKeyNone : key[e];
            if (s == 0) vmax = key_value(bk);
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
        // Candidates still open: the selection keys of v, taken and absent experts at
        // kKeyNone. An untaken expert's key is above kKeyNone (k <= N), so the winner
        // is always a real expert; a lane's experts rise with q, so keeping the first
        // of equal keys picks the lower index inside the lane, and the butterfly
        // breaks ties between lanes by index.
        int open[QMAX];
#pragma unroll
        for (int q = 0; q < QMAX; ++q) open[q] = lane + 32 * q < N ? sel_key(v[q]) : kKeyNone;
        float my_v = 0.0f, vmax = 0.0f;
        int my_e = 0;
        for (int s = 0; s < k; ++s) {
            int bk = open[0];
            int bq = 0;
#pragma unroll
            for (int q = 1; q < QMAX; ++q)
                if (open[q] > bk) {
                    bk = open[q];
                    bq = q;
                }
            int bi = bk == kKeyNone ? INT_MAX : lane + 32 * bq;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const int ok = __shfl_xor_sync(0xffffffffu, bk, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (ok > bk || (ok == bk && oi < bi)) {
                    bk = ok;
                    bi = oi;
                }
            }
            const float bv = key_value(bk);
            if (s == 0) vmax = bv;
            if (lane == s) {
                my_v = bv;
                my_e = bi;
            }
            const int tq = (bi & 31) == lane ? (bi >> 5) : -1;  // taken here
#pragma unroll
            for (int q = 0; q < QMAX; ++q) open[q] = q == tq ? kKeyNone : open[q];
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

__device__ __forceinline__ float warp_max_bcast(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return __shfl_sync(0xffffffffu, v, 0);
}

// Training-time step between the logits and the gating ("Noise Top-k Gating":
// noise is added to the raw logits before the top-k choice), one warp per token of
// the tile; called by every thread of the CTA when a.noise or a.zpart is set.
//   z-loss: the token's (log sum_e exp L)^2 on the noiseless logits; the tile's sum,
//           in token order, goes to zpart[tile];
//   noise:  L <- fl(L + fl(w * n)), the product and the sum each rounded to fp32.
constexpr int kMaxTileTokens = 64;
__device__ void train_step(float *Ls, const RouterArgs &a, int TT) {
    __shared__ float zs[kMaxTileTokens];
    const int N = a.N, lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    const int t0 = blockIdx.x * TT;
    const int nrows = min(TT, a.T - t0);
    for (int tok = warp; tok < nrows; tok += nw) {
        float *L = Ls + tok * N;
        if (a.zpart) {
            float m = -INFINITY;
            for (int e = lane; e < N; e += 32) m = fmaxf(m, L[e]);
            m = warp_max_bcast(m);
            float part = 0.0f;
            for (int e = lane; e < N; e += 32) part += expf(L[e] - m);
            const float lse = m + logf(warp_sum_bcast(part));
            if (lane == 0) zs[tok] = lse * lse;
        }
        if (a.noise) {
            const float *n = a.noise + (size_t)(t0 + tok) * N;
            for (int e = lane; e < N; e += 32) L[e] = __fadd_rn(L[e], __fmul_rn(a.noise_w, n[e]));
        }
    }
    __syncthreads();
    if (a.zpart && threadIdx.x == 0) {
        float sum = 0.0f;
        for (int tok = 0; tok < nrows; ++tok) sum += zs[tok];
        a.zpart[blockIdx.x] = sum;
    }
}

// ------------------------------------------------------------------ pipeline

// Ring of STAGES staging slots between one producer warp (bulk copies) and NC
// consumer warps. full[s]: the copies of the chunk in slot s have landed (one
// arrival + transaction bytes); empty[s]: all NC consumer warps are done with it.
template <int STAGES>
struct Ring {
    uint64_t full[STAGES], empty[STAGES];
    int abort_flag;

    __device__ void init(int nc) {
        abort_flag = 0;
        for (int i = 0; i < STAGES; ++i) {
            tc::mbar_init(&full[i], 1);
            tc::mbar_init(&empty[i], (uint32_t)nc);
        }
        tc::fence_mbar_init();
    }
    __device__ bool aborted() { return *(volatile int *)&abort_flag != 0; }
    // producer: wait until slot c % STAGES may be refilled with chunk c
    __device__ bool acquire(int c, uint32_t *err) {
        if (c < STAGES) return !aborted();
        return wait_phase(&empty[c % STAGES], (uint32_t)((c / STAGES - 1) & 1), &abort_flag, err);
    }
    // consumer: wait until chunk c has landed
    __device__ bool ready(int c, uint32_t *err, uint64_t limit_ns = kWaitNs) {
        return wait_phase(&full[c % STAGES], (uint32_t)((c / STAGES) & 1), &abort_flag, err, limit_ns);
    }
    // consumer warp: done reading chunk c
    __device__ void release(int c) {
        __syncwarp();
        if ((threadIdx.x & 31) == 0) tc::mbar_arrive(&empty[c % STAGES]);
    }
    // producer lane 0: every chunk issued lands before the CTA moves on
    __device__ void drain(int issued) {
        for (int c = max(0, issued - STAGES); c < issued; ++c) {
            const uint64_t ts = tc::globaltimer_ns();
            while (!tc::mbar_try_wait(&full[c % STAGES], (uint32_t)((c / STAGES) & 1)))
                if (tc::globaltimer_ns() - ts > kWaitNs) break;
        }
    }
};

// ------------------------------------------------------------------ weight layout

// The router weight is re-laid out once per call (k_transpose_wr) as
// [chunk of 256 features][expert][256 positions]: one chunk of every expert is
// one contiguous run (a single bulk copy), and inside an expert's 256 positions
// features 0-3 of every 8-feature block come first (block after block), then
// features 4-7, so lane l's two 16-byte halves of block l sit at 16*l and
// 16*(nb + l) bytes (nb = blocks in the chunk): every half-load of a warp reads
// one contiguous 512-byte run.
__device__ __forceinline__ size_t wt_index(int i, int e, int d, int N) {
    const int c = i >> 8, p = i & 255;
    const int nb = min(32, (d - (c << 8)) >> 3);
    const int l = p >> 3, r = p & 7;
    return ((size_t)c * N + e) * 256 + (r >> 2) * (nb * 4) + l * 4 + (r & 3);
}

// Expert-pair layout of k_logits_large, whose lanes update two experts with one
// packed fp32x2 FMA: [chunk of 256 features][expert pair][512 positions] over
// N rounded up to even (the extra expert of an odd N holds zeros). Inside a pair,
// quarter q (features 2q and 2q+1 of every 8-feature block) comes block after
// block, and each block's 16 bytes of the quarter hold (f = 2q: expert 2p, 2p+1;
// f = 2q+1: expert 2p, 2p+1), so lane l's quarter-q load sits at 16*(q*nb + l)
// bytes and one 16-byte load gives the two experts' weights of two features as
// float pairs; every quarter-load of a warp reads one contiguous 512-byte run.
__device__ __forceinline__ size_t wt_index_paired(int i, int e, int d, int n_even) {
    const int c = i >> 8, p = i & 255;
    const int nb = min(32, (d - (c << 8)) >> 3);
    const int l = p >> 3, r = p & 7;
    return ((size_t)c * n_even + (e & ~1)) * 256 + (r >> 1) * (nb * 4) + l * 4 + (r & 1) * 2 + (e & 1);
}

// Grid: (ceil(d/32), ceil(N'/32)) with N' = N (per-expert layout) or N rounded up
// to even (pair layout, whose extra expert is written as zeros).
template <bool PAIRED>
__global__ void __launch_bounds__(256) k_transpose_wr(const float *__restrict__ w_r, float *__restrict__ w_t,
                                                      int d, int N) {
    __shared__ float tile[32][33];
    const int i0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int n_out = PAIRED ? (N + 1) & ~1 : N;
    pdl_enter();
    for (int r = ty; r < 32; r += 8)
        if (i0 + r < d && e0 + tx < N) tile[r][tx] = w_r[(size_t)(i0 + r) * N + e0 + tx];
    __syncthreads();
    for (int r = ty; r < 32; r += 8) {
        const int e = e0 + r, i = i0 + tx;
        if (e >= n_out || i >= d) continue;
        const float v = e < N ? tile[tx][r] : 0.0f;
        if constexpr (PAIRED)
            w_t[wt_index_paired(i, e, d, n_out)] = v;
        else
            w_t[wt_index(i, e, d, N)] = v;
    }
}

// 8 weights of expert row `row` (256 floats of one chunk) for lane's block.
__device__ __forceinline__ void load_w8(const float *row, int lane, int nb, float *w) {
    lds<4>(row + lane * 4, w);
    lds<4>(row + nb * 4 + lane * 4, w + 4);
}

// ------------------------------------------------------------------ N <= 32

// One CTA = 4 consumer warps + 1 producer warp. Consumer warp w owns TO = 32/NP
// tokens and all NP experts; lane l owns partial l. Per chunk of 256 features the
// producer issues one 2D TMA copy of the token tile ([TT][256]) and one bulk copy
// of the weight chunk ([N][256]) into a 6-slot ring.
template <typename XT, int NP>
__global__ void __launch_bounds__(160) k_router_small(const __grid_constant__ CUtensorMap tmx,
                                                     const float *__restrict__ w_t, const float *__restrict__ b_r,
                                                     RouterArgs a) {
    constexpr int NW = 4, TO = 32 / NP, TT = NW * TO;
    constexpr int KC = 256, NBLK = KC / 8;
    constexpr int STAGES = 6;
    constexpr int ES = (int)sizeof(XT);
    constexpr int X_BYTES = TT * KC * ES;
    constexpr int STAGE = (X_BYTES + NP * KC * 4 + 1023) & ~1023;
    extern __shared__ __align__(1024) uint8_t router_smem[];
    __shared__ Ring<STAGES> ring;
    uint8_t *sb = router_smem + ((1024 - (tc::smem_u32(router_smem) & 1023)) & 1023);

    const int N = a.N, d = a.d;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t0 = blockIdx.x * TT;
    const int nblocks = d / 8;
    const int nchunks = (nblocks + NBLK - 1) / NBLK;

    if (tid == 0) ring.init(NW);
    __syncthreads();
    pdl_enter();

    float acc[TO][NP];
#pragma unroll
    for (int i = 0; i < TO; ++i)
#pragma unroll
        for (int e = 0; e < NP; ++e) acc[i][e] = 0.0f;

    // MOE_DEBUG_ROUTER_STALL: the producer issues nothing and the consumers' first wait
    // gives up after kStallWaitNs (records MOE_ERR_TIMEOUT; no copy is in flight)
    const uint64_t wait_ns = a.stall ? kStallWaitNs : kWaitNs;
    if (warp == NW) {
        // ---- producer (lane 0)
        if (lane == 0 && !a.stall) {
            int issued = 0;
            for (int c = 0; c < nchunks; ++c) {
                if (!ring.acquire(c, a.err)) break;
                uint8_t *slot = sb + (size_t)(c % STAGES) * STAGE;
                uint64_t *bar = &ring.full[c % STAGES];
                const uint32_t wbytes = (uint32_t)(N * KC * 4);
                tc::mbar_arrive_expect_tx(bar, (uint32_t)X_BYTES + wbytes);
                tc::tma_load_2d(slot, &tmx, c * KC, t0, bar);
                tc::bulk_copy_g2s(slot + X_BYTES, w_t + (size_t)c * N * KC, wbytes, bar);
                issued = c + 1;
            }
            ring.drain(issued);
        }
    } else {
        // ---- consumers
        for (int c = 0; c < nchunks; ++c) {
            if (!ring.ready(c, a.err, wait_ns)) break;
            const uint8_t *slot = sb + (size_t)(c % STAGES) * STAGE;
            const int nb = min(NBLK, nblocks - c * NBLK);
            if (lane < nb) {
                const float *wl = reinterpret_cast<const float *>(slot + X_BYTES);
                float xf[TO][8];
#pragma unroll
                for (int i = 0; i < TO; ++i) load8<XT>(slot + ((warp * TO + i) * KC + lane * 8) * ES, xf[i]);
#pragma unroll
                for (int e = 0; e < NP; ++e) {
                    float w[8];
                    load_w8(wl + e * KC, lane, nb, w);
#pragma unroll
                    for (int r = 0; r < 8; ++r)
#pragma unroll
                        for (int i = 0; i < TO; ++i) acc[i][e] = __fmaf_rn(xf[i][r], w[r], acc[i][e]);
                }
            }
            ring.release(c);
        }
    }
    __syncthreads();
    if (ring.aborted()) return;

    float *Ls = reinterpret_cast<float *>(sb);            // [TT][N]
    int *Is = reinterpret_cast<int *>(Ls + TT * N);       // [TT][8]
    if (warp < NW) {
#pragma unroll
        for (int i = 0; i < TO; ++i)
#pragma unroll
            for (int e = 0; e < NP; ++e) {
                const float v = butterfly32(acc[i][e]);
                if (lane == 0 && e < N) Ls[(warp * TO + i) * N + e] = a.has_bias ? __fadd_rn(v, b_r[e]) : v;
            }
    }
    __syncthreads();
    if (a.noise || a.zpart) train_step(Ls, a, TT);
    gate_tokens_thread<NP>(Ls, Is, a, TT);
    __syncthreads();
    tile_stats(Ls, Is, a, TT);
}

// ------------------------------------------------------------------ N > 32

struct LogitsArgs {
    int T, d, N, has_bias;
    float *logits;  // [T][N]
    uint32_t *err;
};

// One CTA = TG x EG consumer warps (warp tile TO tokens x EO experts, lane l =
// partial l) + 1 producer warp. Tile TG*TO tokens x EG*EO experts; per chunk of 256
// features one 2D TMA copy of the token tile and one bulk copy of the tile's expert
// weight rows, into a STAGES-slot ring. Per feature a lane loads TO x values and EO
// weights from shared memory for TO*EO FMAs.
// 8 consecutive features of one token, kept as loaded; dup(r) gives feature r
// as the float pair (x, x) for a packed FMA against two experts' weights.
template <typename XT> struct XRow8;
template <> struct XRow8<__nv_bfloat16> {
    uint32_t w[4];
    __device__ __forceinline__ void load(const uint8_t *p) {
        const uint4 q = *reinterpret_cast<const uint4 *>(p);
        w[0] = q.x; w[1] = q.y; w[2] = q.z; w[3] = q.w;
    }
    __device__ __forceinline__ float2 dup(int r) const {
        const float v = __uint_as_float((r & 1) ? (w[r >> 1] & 0xffff0000u) : (w[r >> 1] << 16));
        return make_float2(v, v);
    }
};
template <> struct XRow8<float> {
    float f[8];
    __device__ __forceinline__ void load(const uint8_t *p) { lds<8>(reinterpret_cast<const float *>(p), f); }
    __device__ __forceinline__ float2 dup(int r) const { return make_float2(f[r], f[r]); }
};

template <typename XT, int TO, int EO, int TG, int EG>
__global__ void __launch_bounds__((TG * EG + 1) * 32, 1) k_logits_large(const __grid_constant__ CUtensorMap tmx,
                                                                     const float *__restrict__ w_t,
                                                                     const float *__restrict__ b_r, LogitsArgs a) {
    constexpr int NC = TG * EG, TOK = TG * TO, EXP = EG * EO;
    constexpr int KC = 256, NBLK = KC / 8, STAGES = 4;
    constexpr int ES = (int)sizeof(XT);
    constexpr int X_BYTES = TOK * KC * ES;
    constexpr int STAGE = (X_BYTES + EXP * KC * 4 + 1023) & ~1023;
    static_assert(EO % 2 == 0, "experts are taken in pairs");
    extern __shared__ __align__(1024) uint8_t router_smem[];
    __shared__ Ring<STAGES> ring;
    uint8_t *sb = router_smem + ((1024 - (tc::smem_u32(router_smem) & 1023)) & 1023);

    const int T = a.T, d = a.d, N = a.N, n_even = (N + 1) & ~1;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int tg = warp / EG, eg = warp % EG;
    const int e0 = blockIdx.x * EXP, t0 = blockIdx.y * TOK;   // experts fastest: CTAs sharing a token tile run together
    const int nexp = min(EXP, n_even - e0);                    // even: whole pairs
    const int nblocks = d / 8;
    const int nchunks = (nblocks + NBLK - 1) / NBLK;

    if (tid == 0) ring.init(NC);
    __syncthreads();
    pdl_enter();

    // acc[i][p] = partials of token i for experts 2p and 2p+1 of the warp's EO
    float2 acc[TO][EO / 2];
#pragma unroll
    for (int i = 0; i < TO; ++i)
#pragma unroll
        for (int p = 0; p < EO / 2; ++p) acc[i][p] = make_float2(0.0f, 0.0f);

    if (warp == NC) {
        if (lane == 0) {
            int issued = 0;
            for (int c = 0; c < nchunks; ++c) {
                if (!ring.acquire(c, a.err)) break;
                uint8_t *slot = sb + (size_t)(c % STAGES) * STAGE;
                uint64_t *bar = &ring.full[c % STAGES];
                const uint32_t wbytes = (uint32_t)(nexp * KC * 4);
                tc::mbar_arrive_expect_tx(bar, (uint32_t)X_BYTES + wbytes);
                tc::tma_load_2d(slot, &tmx, c * KC, t0, bar);
                tc::bulk_copy_g2s(slot + X_BYTES, w_t + ((size_t)c * n_even + e0) * KC, wbytes, bar);
                issued = c + 1;
            }
            ring.drain(issued);
        }
    } else {
        for (int c = 0; c < nchunks; ++c) {
            if (!ring.ready(c, a.err)) break;
            const uint8_t *slot = sb + (size_t)(c % STAGES) * STAGE;
            const int nb = min(NBLK, nblocks - c * NBLK);
            if (lane < nb) {
                XRow8<XT> xr[TO];
#pragma unroll
                for (int i = 0; i < TO; ++i) xr[i].load(slot + ((tg * TO + i) * KC + lane * 8) * ES);
                // pair p of the warp's experts: 2 * KC floats per chunk
                const float *wl = reinterpret_cast<const float *>(slot + X_BYTES) + (eg * EO) * KC + lane * 4;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float2 wp[EO / 2][2];
#pragma unroll
                    for (int p = 0; p < EO / 2; ++p) {
                        const float4 v = *reinterpret_cast<const float4 *>(wl + p * 2 * KC + q * nb * 4);
                        wp[p][0] = make_float2(v.x, v.y);
                        wp[p][1] = make_float2(v.z, v.w);
                    }
                    // features 2q, 2q+1 of the block, in increasing order for every partial
#pragma unroll
                    for (int f = 0; f < 2; ++f)
#pragma unroll
                        for (int i = 0; i < TO; ++i) {
                            const float2 xv = xr[i].dup(2 * q + f);
#pragma unroll
                            for (int p = 0; p < EO / 2; ++p) acc[i][p] = __ffma2_rn(xv, wp[p][f], acc[i][p]);
                        }
                }
            }
            ring.release(c);
        }
    }
    __syncthreads();
    if (ring.aborted() || warp == NC) return;
#pragma unroll
    for (int i = 0; i < TO; ++i)
#pragma unroll
        for (int j = 0; j < EO; ++j) {
            const float v = butterfly32((j & 1) ? acc[i][j >> 1].y : acc[i][j >> 1].x);
            const int t = t0 + tg * TO + i, e = e0 + eg * EO + j;
            if (lane == 0 && t < T && e < N) a.logits[(size_t)t * N + e] = a.has_bias ? __fadd_rn(v, b_r[e]) : v;
        }
}

// One CTA = 32 warps, 64 tokens: logits tile -> shared memory -> gating -> stats.
// The tile is one contiguous run of logits; it is loaded as 16-byte vectors with
// every load of a thread in flight before the first store (one round trip to L2,
// where the logits kernel left them), then each warp gates 2 tokens.
constexpr int kGateThreads = 1024;
__global__ void __launch_bounds__(kGateThreads) k_gate(const float *__restrict__ logits, RouterArgs a) {
    constexpr int TT = 64, U = 8;
    extern __shared__ __align__(16) float smem[];
    float *Ls = smem;                                    // [TT][N]
    int *Is = reinterpret_cast<int *>(smem + TT * a.N);  // [TT][8]
    const int t0 = blockIdx.x * TT;
    const int nrows = min(TT, a.T - t0);
    pdl_enter();
    const float *src = logits + (size_t)t0 * a.N;
    const int n = nrows * a.N;
    int done = 0;
    if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
        const int n4 = n >> 2;
        const float4 *src4 = reinterpret_cast<const float4 *>(src);
        float4 *dst4 = reinterpret_cast<float4 *>(Ls);
        for (int base = 0; base < n4; base += U * kGateThreads) {
            float4 r[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = base + u * kGateThreads + (int)threadIdx.x;
                if (i < n4) r[u] = src4[i];
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int i = base + u * kGateThreads + (int)threadIdx.x;
                if (i < n4) dst4[i] = r[u];
            }
        }
        done = n4 << 2;
    }
    for (int i = done + (int)threadIdx.x; i < n; i += kGateThreads) Ls[i] = src[i];
    __syncthreads();
    if (a.noise || a.zpart) {
        train_step(Ls, a, TT);
        __syncthreads();
    }
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
    // token-sharded router: slot_base [N][k] = global priority of this shard's first
    // selection of (expert, slot) (null: this batch is the whole batch); stats_only:
    // write slot_counts [N][k] and prob_sums [N] and stop before the capacity step
    const int32_t *slot_base = nullptr;
    int stats_only = 0;
    int32_t *slot_counts = nullptr;
    float *prob_sums = nullptr;
};

__global__ void __launch_bounds__(256) k_expert_scan(ScanArgs a) {
    __shared__ int shi[33];
    __shared__ float shf[32];
    const int e = blockIdx.x, tid = threadIdx.x, nt = blockDim.x;
    const int n = a.k * a.tiles;
    pdl_enter();
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

    // per-slot totals (the prefix at each slot's first tile) and, for a shard, the
    // move from this batch's priorities to the global ones
    __shared__ int slot_first[9];
    if (tid < a.k) slot_first[tid] = pe[tid * a.tiles];
    if (tid == 0) slot_first[a.k] = total;
    __syncthreads();
    if (a.slot_counts && tid < a.k) a.slot_counts[(size_t)e * a.k + tid] = slot_first[tid + 1] - slot_first[tid];
    if (a.stats_only) {
        float ps = 0.0f;
        for (int tl = tid; tl < a.tiles; tl += nt) ps += a.psum[(size_t)e * a.tiles + tl];
        const float psum = block_sum(ps, shf);
        if (tid == 0) {
            a.routed[e] = total;
            if (a.prob_sums) a.prob_sums[e] = psum;
        }
        return;
    }
    if (a.slot_base) {
        for (int i = beg; i < end; ++i) {
            const int j = i / a.tiles;
            pe[i] += a.slot_base[(size_t)e * a.k + j] - slot_first[j];
        }
        __syncthreads();
    }

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
    const float *zpart = nullptr;  // [tiles] z-loss tile sums (with z_out)
    float *z_out = nullptr;        // [1] may be null
    // token-sharded router: aux from the global statistics of all shards
    const int32_t *g_routed = nullptr;  // [N] selections per expert, all shards
    const float *g_psum = nullptr;      // [N] sum over all tokens of softmax
    float g_T = 0.0f;                   // tokens of all shards
    // Small problems (at most kFusedScanTiles tiles and kFusedScanMax counts): k_expert_scan is not launched and
    // every CTA derives what it needs of it from the tile counts itself; CTA 0 writes
    // routed, kept and the mean probabilities.
    int fused_scan = 0;
    const int32_t *cnt = nullptr;  // [N][k][tiles]
    const float *psum = nullptr;   // [N][tiles]
    int32_t *routed_out = nullptr, *kept_out = nullptr;
};
constexpr int kFusedScanMax = 4096, kFusedScanTiles = 32;

// One warp: expert e's priority-order prefix over its (slot, tile) counts (what
// k_expert_scan computes), reduced to what tile `tile` needs: pre for each slot of the
// tile, kept slots of earlier tiles, and the totals.
__device__ void scan_expert_warp(const AssignArgs &a, const int *cnt_s, int e, int tile, int C, int *pre_t,
                                 int *kpre_t, int *routed_e, int *kept_e, float *pmean_e) {
    const int lane = threadIdx.x & 31, n = a.k * a.tiles;
    const int *ce = cnt_s + (size_t)e * n;
    int run = 0, kb = 0, kt = 0;
    for (int i0 = 0; i0 < n; i0 += 32) {
        const int i = i0 + lane;
        const int v = i < n ? ce[i] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        const int ex = run + incl - v;
        if (i < n) {
            const int j = i / a.tiles, tl = i - j * a.tiles;
            const int kv = min(max(C - ex, 0), v);
            if (tl == tile) pre_t[j] = ex;
            if (tl < tile) kb += kv;
            kt += kv;
        }
        run += __shfl_sync(0xffffffffu, incl, 31);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        kb += __shfl_xor_sync(0xffffffffu, kb, o);
        kt += __shfl_xor_sync(0xffffffffu, kt, o);
    }
    if (lane == 0) {
        *kpre_t = kb;
        *routed_e = run;
        *kept_e = kt;
    }
    if (pmean_e) {  // mean routing probability: lane-strided tile sums, then a fixed butterfly
        float ps = 0.0f;
        for (int tl = lane; tl < a.tiles; tl += 32) ps += a.psum[(size_t)e * a.tiles + tl];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        if (lane == 0) *pmean_e = ps / (float)a.T;
    }
}

__global__ void __launch_bounds__(256) k_assign(AssignArgs a) {
    extern __shared__ int sm[];
    int *offs = sm;                       // [N+1]
    int *Is = offs + a.N + 1;             // [TT][8] expert of each slot (-1 none, -2 invalid)
    int *Ks = Is + a.TT * 8;              // [TT][8] kept
    int *Cs = Ks + a.TT * 8;              // [9][N] running counts: per slot, then kept per expert
    int *Fp = Cs + 9 * a.N;               // fused scan: [N][8] pre of this tile, [N] kpre, routed, kept, pmean
    __shared__ int shi[33];
    __shared__ float shf[32];
    const int tid = threadIdx.x, nt = blockDim.x, N = a.N, k = a.k;
    const int tile = blockIdx.x, t0 = tile * a.TT;
    const int C = a.cap > 0 ? a.cap : INT_MAX;
    pdl_enter();

    const int32_t *kept_of = a.kept;
    const int32_t *routed_of = a.routed;
    if (a.fused_scan) {
        float *pm = reinterpret_cast<float *>(Fp + 11 * N);
        int *cnt_s = Fp + 12 * N;  // the tile counts, loaded once with every load in flight
        const int ncnt = N * k * a.tiles;
        for (int i = tid; i < ncnt; i += nt) cnt_s[i] = a.cnt[i];
        __syncthreads();
        for (int e = tid >> 5; e < N; e += nt >> 5)
            scan_expert_warp(a, cnt_s, e, tile, C, Fp + e * 8, Fp + 8 * N + e, Fp + 9 * N + e, Fp + 10 * N + e,
                             tile == 0 ? pm + e : nullptr);
        __syncthreads();
        kept_of = Fp + 10 * N;
        routed_of = Fp + 9 * N;
        if (tile == 0)
            for (int e = tid; e < N; e += nt) {
                if (a.routed_out) a.routed_out[e] = routed_of[e];
                if (a.kept_out) a.kept_out[e] = kept_of[e];
            }
    }
    auto pre_of = [&](int e, int j) {
        return a.fused_scan ? Fp[e * 8 + j] : a.pre[((size_t)e * k + j) * a.tiles + tile];
    };
    auto kpre_of = [&](int e) { return a.fused_scan ? Fp[8 * N + e] : a.kpre[(size_t)e * a.tiles + tile]; };

    // expert offsets (every CTA computes them; N <= 256 <= blockDim)
    {
        const int v = tid < N ? kept_of[tid] : 0;
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
            const bool global = a.g_routed != nullptr;
            const float Tg = global ? a.g_T : (float)a.T;
            float pm;
            if (global) {
                pm = a.g_psum[tid] / Tg;
            } else if (a.fused_scan) {
                pm = reinterpret_cast<const float *>(Fp + 11 * N)[tid];
            } else {
                pm = a.pmean[tid];
            }
            const float routed = (float)(global ? a.g_routed[tid] : routed_of[tid]);
            f0 = (routed / (Tg * (float)k)) * pm;
            f1 = (pm - invN) * (pm - invN);
        }
        const float s0 = block_sum(f0, shf);
        const float s1 = block_sum(f1, shf);
        if (tid == 0) {
            a.aux[0] = (float)N * s0;
            a.aux[1] = s1 * invN;
        }
    }
    if (tile == 0 && a.z_out && tid == 0) {
        float z = 0.0f;  // tile sums in tile order
        for (int tl = 0; tl < a.tiles; ++tl) z += a.zpart[tl];
        a.z_out[0] = z / (float)a.T;
    }

    for (int s = tid; s < a.TT * 8; s += nt) {
        const int tok = s >> 3, j = s & 7;
        const int t = t0 + tok;
        int e = (t < a.T && j < k) ? a.topk_idx[(size_t)t * k + j] : -1;
        if (t < a.T && j < k && (e < 0 || e >= N)) {
            record_error(a.err, kErrFault);
            e = -2;  // matches no expert: neither kept nor counted
        }
        Is[s] = e;
        Ks[s] = 0;
    }
    for (int i = tid; i < 9 * N; i += nt) Cs[i] = 0;
    __syncthreads();

    // Keep or drop each slot: its priority is the expert's selections before this tile
    // in slot j (pre) plus this tile's earlier tokens that chose the same expert in slot
    // j. Warp j ranks slot j's selections in token order, 32 tokens at a time: lanes with
    // equal experts are matched, a lane's rank among them is the count of lower lanes,
    // and a per-(slot, expert) counter carries the earlier chunks.
    const int warp = tid >> 5, lane = tid & 31;
    const unsigned lower = (1u << lane) - 1u;
    if (warp < k) {
        const int j = warp;
        int *cj = Cs + (size_t)j * N;
        for (int base = 0; base < a.TT; base += 32) {
            const int tok = base + lane;
            const int e = tok < a.TT ? Is[tok * 8 + j] : -2;
            const unsigned peers = __match_any_sync(0xffffffffu, e);
            const int before = e >= 0 ? cj[e] : 0;
            __syncwarp();
            if (e >= 0) {
                const int r = pre_of(e, j) + before + __popc(peers & lower);
                Ks[tok * 8 + j] = r < C;
                if ((peers & lower) == 0) cj[e] = before + __popc(peers);  // the group's lowest lane
            }
            __syncwarp();
        }
    }
    __syncthreads();

    // Rows: a kept slot's row is its expert's offset, plus the expert's kept slots of
    // earlier tiles (kpre), plus this tile's kept slots of the expert in earlier tokens
    // (a token selects an expert at most once, so earlier (token, slot) entries in
    // token-major order). Warp 0 ranks the tile's entries 32 at a time as above.
    if (warp == 0) {
        int *ce = Cs + (size_t)8 * N;
        const int n = a.TT * k;
        for (int base = 0; base < n; base += 32) {
            const int i = base + lane;
            const int tok = i / k, j = i - tok * k, t = t0 + tok;
            const bool live = i < n && t < a.T;
            const int e = live ? Is[tok * 8 + j] : -2;
            const bool kept = e >= 0 && Ks[tok * 8 + j];
            const unsigned peers = __match_any_sync(0xffffffffu, kept ? e : -1);
            const int before = kept ? ce[e] : 0;
            __syncwarp();
            int row = -1;
            if (kept) {
                row = offs[e] + kpre_of(e) + before + __popc(peers & lower);
                if (row < 0 || row >= a.rmax) {
                    record_error(a.err, kErrFault);
                    row = -1;
                } else {
                    a.perm_token[row] = t;
                }
                if ((peers & lower) == 0) ce[e] = before + __popc(peers);
            }
            __syncwarp();
            if (live) a.slot_row[(size_t)t * k + j] = row;
        }
    }
}

// 2D map of the token activations [T][d], box 256 features x `rows` tokens.
template <typename XT>
bool token_map(CUtensorMap *m, const XT *x, int T, int d, int rows) {
    const uint64_t dims[2] = {(uint64_t)d, (uint64_t)T};
    const uint64_t strides[1] = {(uint64_t)d * sizeof(XT)};
    const uint32_t box[2] = {256u, (uint32_t)rows};
    const CUtensorMapDataType dt =
        sizeof(XT) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    return encode_tmap(m, dt, 2, x, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

template <typename XT, int NP>
cudaError_t launch_small(const moe_config &c, const XT *x, const float *w_t, const float *b_r, RouterArgs ra,
                         cudaStream_t s) {
    constexpr int TT = 4 * (32 / NP);
    CUtensorMap tmx;
    if (!token_map<XT>(&tmx, x, c.T, c.d, TT)) return cudaErrorInvalidValue;
    const size_t stage = ((size_t)TT * 256 * sizeof(XT) + (size_t)NP * 256 * 4 + 1023) & ~(size_t)1023;
    const size_t gate = ((size_t)TT * c.N + (size_t)TT * 8) * sizeof(float);
    const size_t bytes = std::max(6 * stage, gate) + 1024;
    auto kern = k_router_small<XT, NP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3(ra.tiles), dim3(160), bytes, s, tmx, w_t, b_r, ra);
}

// Router weight -> expert-pair layout of k_logits_large (N rounded up to even).
cudaError_t launch_transpose_paired(const moe_config &c, const float *w_r, float *w_t, cudaStream_t s) {
    const int n_even = (c.N + 1) & ~1;
    return launch_pdl(k_transpose_wr<true>, dim3((c.d + 31) / 32, (n_even + 31) / 32), dim3(256), 0, s, w_r, w_t, c.d,
                      c.N);
}

template <typename XT, int TO, int EO, int TG, int EG>
cudaError_t launch_logits_tile(const moe_config &c, const XT *x, const float *w_t, const float *b_r, int has_bias,
                               float *logits, uint32_t *err, cudaStream_t s) {
    constexpr int TOK = TG * TO, EXP = EG * EO;
    CUtensorMap tmx;
    if (!token_map<XT>(&tmx, x, c.T, c.d, TOK)) return cudaErrorInvalidValue;
    LogitsArgs la{c.T, c.d, c.N, has_bias, logits, err};
    const size_t stage = ((size_t)TOK * 256 * sizeof(XT) + (size_t)EXP * 256 * 4 + 1023) & ~(size_t)1023;
    const size_t lbytes = 4 * stage + 1024;
    auto kern = k_logits_large<XT, TO, EO, TG, EG>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lbytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, dim3((c.N + EXP - 1) / EXP, (c.T + TOK - 1) / TOK), dim3((TG * EG + 1) * 32), lbytes, s,
                      tmx, w_t, b_r, la);
}

template <typename XT>
cudaError_t launch_logits_only(const moe_config &c, const XT *x, const float *w_t, const float *b_r, int has_bias,
                               float *logits, uint32_t *err, cudaStream_t s) {
    // At most 8 experts (the Expert Choice router of the Mixtral-shaped layer, the
    // backward's recomputed logits): 4 warps of 4 tokens x 8 experts, tile 16 x 8, so no
    // warp works on absent experts and twice as many CTAs share the tokens.
    if (c.N <= 8) return launch_logits_tile<XT, 4, 8, 4, 1>(c, x, w_t, b_r, has_bias, logits, err, s);
    // Otherwise warps of 8 tokens x 8 experts (0.75 bytes of shared memory read per FMA).
    // With 8 warps (tile 32 x 16) this took 902 us for the DeepSeek-shaped router
    // (T = 8192, d = 7168, N = 256) against 995 us with 16 warps of 4 x 8 (1.25 bytes per
    // FMA) and 982-1001 us for 6 x 8, 8 x 4 and 4 x 8 warp tiles; packed fp32x2 FMAs over
    // expert pairs then took it to 890 us. One CTA fits per SM, so its consumer warps are
    // all the SM has: for bf16 tokens 12 warps (tile 48 tokens x 16 experts; 13 warps hold
    // at most 128 registers a thread, a few bytes spill) run the whole router call in
    // 795 us against 832 us with 8 (and 840 us with a 32 x 24 tile); identical logits.
    // fp32 tokens keep 8 warps: a 48-token ring of fp32 rows does not fit in shared memory.
    if constexpr (sizeof(XT) == 2)
        return launch_logits_tile<XT, 8, 8, 6, 2>(c, x, w_t, b_r, has_bias, logits, err, s);
    else
        return launch_logits_tile<XT, 8, 8, 4, 2>(c, x, w_t, b_r, has_bias, logits, err, s);
}

template <typename XT>
cudaError_t launch_large(const moe_config &c, const XT *x, const float *w_t, const float *b_r, RouterArgs ra,
                         float *logits, cudaStream_t s) {
    cudaError_t e = launch_logits_only<XT>(c, x, w_t, b_r, ra.has_bias, logits, ra.err, s);
    if (e != cudaSuccess) return e;
    const size_t gbytes = ((size_t)64 * c.N + 64 * 8) * sizeof(float);
    e = cudaFuncSetAttribute(k_gate, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gbytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(k_gate, dim3(ra.tiles), dim3(kGateThreads), gbytes, s, logits, ra);
}

template <typename XT>
cudaError_t launch_logits_gate(const moe_config &c, const XT *x, const float *w_r, const float *b_r, RouterArgs ra,
                               float *logits, float *w_t, cudaStream_t s) {
    cudaError_t e = c.N > 32 ? launch_transpose_paired(c, w_r, w_t, s)
                             : launch_pdl(k_transpose_wr<false>, dim3((c.d + 31) / 32, (c.N + 31) / 32), dim3(256), 0,
                                          s, w_r, w_t, c.d, c.N);
    if (e != cudaSuccess) return e;
    if (c.N <= 4) return launch_small<XT, 4>(c, x, w_t, b_r, ra, s);
    if (c.N <= 8) return launch_small<XT, 8>(c, x, w_t, b_r, ra, s);
    if (c.N <= 16) return launch_small<XT, 16>(c, x, w_t, b_r, ra, s);
    if (c.N <= 32) return launch_small<XT, 32>(c, x, w_t, b_r, ra, s);
    return launch_large<XT>(c, x, w_t, b_r, ra, logits, s);
}

}  // namespace

cudaError_t launch_router_logits(const moe_config &c, const void *x, const float *w_r, const float *b_r,
                                 float *logits, uint8_t *ws, cudaStream_t s) {
    const WsLayout L = ws_layout(c);
    uint32_t *err = reinterpret_cast<uint32_t *>(ws + L.err);
    float *w_t = reinterpret_cast<float *>(ws + L.w_t);
    cudaError_t e = launch_transpose_paired(c, w_r, w_t, s);
    if (e != cudaSuccess) return e;
    const int hb = c.has_router_bias && b_r ? 1 : 0;
    if (c.dtype == MOE_BF16)
        return launch_logits_only<__nv_bfloat16>(c, static_cast<const __nv_bfloat16 *>(x), w_t, b_r, hb, logits, err, s);
    return launch_logits_only<float>(c, static_cast<const float *>(x), w_t, b_r, hb, logits, err, s);
}

cudaError_t launch_router_stats(const moe_config &c, const void *x, const float *w_r, const float *b_r,
                                int32_t *topk_idx, float *topk_gate, int32_t *slot_counts, float *prob_sums,
                                uint8_t *ws, cudaStream_t s) {
    const WsLayout L = ws_layout(c);
    const int tiles = router_tiles(c);
    uint32_t *err = reinterpret_cast<uint32_t *>(ws + L.err);
    int32_t *cnt = reinterpret_cast<int32_t *>(ws + L.cnt);
    float *psum = reinterpret_cast<float *>(ws + L.psum);
    RouterArgs ra{c.T, c.d, c.N, c.k, c.gating, tiles, c.has_router_bias ? 1 : 0, topk_idx, topk_gate, cnt, psum, err};
    cudaError_t e;
    float *logits = reinterpret_cast<float *>(ws + L.logits);
    float *w_t = reinterpret_cast<float *>(ws + L.w_t);
    if (c.dtype == MOE_BF16)
        e = launch_logits_gate<__nv_bfloat16>(c, static_cast<const __nv_bfloat16 *>(x), w_r, b_r, ra, logits, w_t, s);
    else
        e = launch_logits_gate<float>(c, static_cast<const float *>(x), w_r, b_r, ra, logits, w_t, s);
    if (e != cudaSuccess) return e;
    ScanArgs sa{c.T, c.N, c.k, tiles, 0, cnt, reinterpret_cast<int32_t *>(ws + L.pre),
                reinterpret_cast<int32_t *>(ws + L.kpre), psum, reinterpret_cast<float *>(ws + L.pmean),
                reinterpret_cast<int32_t *>(ws + L.routed), reinterpret_cast<int32_t *>(ws + L.kept)};
    sa.stats_only = 1;
    sa.slot_counts = slot_counts;
    sa.prob_sums = prob_sums;
    return launch_pdl(k_expert_scan, dim3(c.N), dim3(256), 0, s, sa);
}

cudaError_t launch_router_assign(const moe_config &c, const int32_t *topk_idx, const int32_t *slot_base, int32_t cap,
                                 const int32_t *g_routed, const float *g_psum, float g_T, int32_t *counts_kept,
                                 int32_t *expert_offsets, int32_t *slot_row, int32_t *perm_token, float *aux,
                                 uint8_t *ws, cudaStream_t s) {
    const WsLayout L = ws_layout(c);
    const int tiles = router_tiles(c);
    uint32_t *err = reinterpret_cast<uint32_t *>(ws + L.err);
    int32_t *cnt = reinterpret_cast<int32_t *>(ws + L.cnt);
    int32_t *pre = reinterpret_cast<int32_t *>(ws + L.pre);
    int32_t *kpre = reinterpret_cast<int32_t *>(ws + L.kpre);
    float *psum = reinterpret_cast<float *>(ws + L.psum);
    float *pmean = reinterpret_cast<float *>(ws + L.pmean);
    int32_t *routed = reinterpret_cast<int32_t *>(ws + L.routed);
    int32_t *kept = counts_kept ? counts_kept : reinterpret_cast<int32_t *>(ws + L.kept);
    ScanArgs sa{c.T, c.N, c.k, tiles, cap, cnt, pre, kpre, psum, pmean, routed, kept};
    sa.slot_base = slot_base;
    cudaError_t e = launch_pdl(k_expert_scan, dim3(c.N), dim3(256), 0, s, sa);
    if (e != cudaSuccess) return e;
    const int TT = router_tile_tokens(c);
    AssignArgs aa{c.T, c.N, c.k, tiles, TT, cap, max_rows(c), topk_idx, pre, kpre, routed, kept,
                  pmean, expert_offsets, slot_row, perm_token, aux, err};
    aa.g_routed = g_routed;
    aa.g_psum = g_psum;
    aa.g_T = g_T;
    const size_t sbytes = (size_t)(c.N + 1 + 2 * TT * 8 + 9 * c.N) * sizeof(int);
    return launch_pdl(k_assign, dim3(tiles), dim3(256), sbytes, s, aa);
}

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

    float *zpart = o.z_loss ? reinterpret_cast<float *>(ws + L.zpart) : nullptr;
    RouterArgs ra{c.T, c.d, c.N, c.k, c.gating, tiles, c.has_router_bias ? 1 : 0,
                  o.topk_idx, o.topk_gate, cnt, psum, err, o.noise, o.noise_w, zpart};
    ra.stall = (c.debug_flags & MOE_DEBUG_ROUTER_STALL) ? 1 : 0;
    cudaError_t e;
    if (c.dtype == MOE_BF16)
        e = launch_logits_gate<__nv_bfloat16>(c, static_cast<const __nv_bfloat16 *>(x), w_r, b_r, ra, logits, w_t, s);
    else
        e = launch_logits_gate<float>(c, static_cast<const float *>(x), w_r, b_r, ra, logits, w_t, s);
    if (e != cudaSuccess) return e;

    const int cap = capacity_of(c);
    // every CTA scans all the counts again: worth a launch only with few tiles (measured:
    // tiny and decode layers 1-2.5 us faster, 256-tile Switch and Mixtral routers 3 and 15 us
    // slower)
    const bool fused = tiles <= kFusedScanTiles && (int64_t)c.N * c.k * tiles <= kFusedScanMax;
    if (!fused) {
        ScanArgs sa{c.T, c.N, c.k, tiles, cap, cnt, pre, kpre, psum, pmean, routed, kept};
        if ((e = launch_pdl(k_expert_scan, dim3(c.N), dim3(256), 0, s, sa)) != cudaSuccess) return e;
    }

    const int TT = router_tile_tokens(c);
    AssignArgs aa{c.T, c.N, c.k, tiles, TT, cap, max_rows(c), o.topk_idx, pre, kpre, routed, kept,
                  pmean, o.expert_offsets, o.slot_row, o.perm_token, o.aux, err, zpart, o.z_loss};
    if (fused) {
        aa.fused_scan = 1;
        aa.cnt = cnt;
        aa.psum = psum;
        aa.routed_out = routed;
        aa.kept_out = kept;
    }
    const size_t sbytes =
        (size_t)(c.N + 1 + 2 * TT * 8 + 9 * c.N + (fused ? 12 * c.N + c.N * c.k * tiles : 0)) * sizeof(int);
    return launch_pdl(k_assign, dim3(tiles), dim3(256), sbytes, s, aa);
}

}  // namespace moe
