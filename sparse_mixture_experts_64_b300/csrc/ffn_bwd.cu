// Backward building blocks on the GPU: the weight-gradient GEMM of the experts and
// the transposes that feed the K-major tensor-core kernels.
//
// The experts' weight gradients reduce over each expert's rows: dW_out[e] =
// dO_eᵀ H_e, dW_a[e] = dA_eᵀ X_e, dW_b[e] = dB_eᵀ X_e (the chain rule through
// O = H W_outᵀ, H = act(X W_aᵀ) (⊙ X W_bᵀ)). K is an expert's row count, so it varies
// per expert. The activations are transposed into [M][Kall] with expert e's rows in
// columns k0_e .. k0_e + R_e - 1, zero up to kp_e = R_e rounded up to 64, so that a
// 64-wide K tile never reads another expert's rows (k_transpose_rows_padded). The
// weight-gradient kernel (k_wgrad_tc) is the single-CTA tcgen05 structure of
// ffn_tc.cu — TMA producer warp, one MMA-issuing thread, four epilogue warps, two
// TMEM accumulators of 128 x 256 fp32 — with tiles (expert, m, n), K from the
// expert's column range, and an all-zero tile for an expert without rows.
#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"
#include "tc_sync.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4;
constexpr uint32_t A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2, STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int NUM_THREADS = 192;
constexpr int MAX_SEG = 257;
constexpr size_t SMEM_BYTES = (size_t)STAGES * STAGE_BYTES + 1024;

struct WgParams {
    CUtensorMap tmA, tmB;        // At [M][Kall] (box 64 x 128), Bt [Nn][Kall] (box 64 x 256)
    CUtensorMap tmA_sh, tmB_sh;  // shared segment: [M][K_sh], [Nn][K_sh]
    CUtensorMap tmC, tmC_sh;     // outputs for the pair kernel's stores: [n_seg][M][Nn], [1][M][Nn], box of
                                 // 32 rows x 128 bytes (64 bf16 or 32 fp32 columns)
    const int32_t *offsets;      // [n_seg + 1] rows of each expert
    int n_seg, has_sh;
    int a_rows;                  // offsets are clamped to it
    int M, Nn, K_sh;
    void *C, *C_sh;              // [n_seg][M][Nn], [M][Nn]: bf16, or fp32 in the kernels' F32 form
    uint32_t *err;
};

struct WgSmem {
    uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], drain;
    uint32_t tmem_base;
    int abort_flag;
    int k0[MAX_SEG], kp[MAX_SEG];  // first column and padded width of each segment's K range
};

// F32: the output is fp32 (general products of the router gradient), else bf16.
template <bool F32>
__global__ void __launch_bounds__(NUM_THREADS, 1) k_wgrad_tc(const __grid_constant__ WgParams p) {
    __shared__ WgSmem s;
    extern __shared__ uint8_t dyn_smem[];
    const uint32_t dyn_base = smem_u32(dyn_smem);
    uint8_t *tiles = dyn_smem + (((dyn_base + 1023u) & ~1023u) - dyn_base);
    auto smA = [&](int st) { return tiles + (size_t)st * STAGE_BYTES; };
    auto smB = [&](int st) { return tiles + (size_t)st * STAGE_BYTES + A_BYTES; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nseg = p.n_seg + p.has_sh;
    const int mt = (p.M + BM - 1) / BM, nt = (p.Nn + BN - 1) / BN;
    const int per_seg = mt * nt;
    const int total = nseg * per_seg;

    if (warp == 0) {
        // K ranges: kp = rows rounded up to 64, k0 = exclusive scan (routed segments)
        constexpr int PER = (MAX_SEG + 31) / 32;
        int kp[PER];
        int sum = 0;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int g = lane * PER + i;
            int v = 0;
            if (g < p.n_seg) {
                const int r0 = min(max(p.offsets[g], 0), p.a_rows);
                const int r1 = min(max(p.offsets[g + 1], r0), p.a_rows);
                v = (r1 - r0 + BK - 1) / BK * BK;
            }
            kp[i] = v;
            sum += v;
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        int run = incl - sum;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int g = lane * PER + i;
            if (g < p.n_seg) {
                s.k0[g] = run;
                s.kp[g] = kp[i];
            }
            run += kp[i];
        }
        if (lane == 0 && p.has_sh) {
            s.k0[p.n_seg] = 0;
            s.kp[p.n_seg] = p.K_sh;
        }
        if (lane == 0) {
            for (int i = 0; i < STAGES; ++i) {
                mbar_init(&s.full[i], 1);
                mbar_init(&s.empty[i], 1);
            }
            for (int i = 0; i < 2; ++i) {
                mbar_init(&s.tfull[i], 1);
                mbar_init(&s.tempty[i], 128);
            }
            mbar_init(&s.drain, 1);
            s.abort_flag = 0;
            fence_mbar_init();
        }
    }
    if (warp == 1) {
        tmem_alloc(&s.tmem_base, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = s.tmem_base;
    volatile int *abort_flag = &s.abort_flag;

    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            int st = 0;
            uint32_t ph = 0;
            bool ok = true;
            uint32_t issued_mask = 0, issued_par = 0;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const int g = tile / per_seg, local = tile - g * per_seg;
                const int m = local % mt, n = local / mt;
                const bool sh = g >= p.n_seg;
                const CUtensorMap *ta = sh ? &p.tmA_sh : &p.tmA;
                const CUtensorMap *tb = sh ? &p.tmB_sh : &p.tmB;
                const int k0 = s.k0[g];
                for (int kb = 0; kb < s.kp[g] / BK; ++kb) {
                    if (!wait_bar(&s.empty[st], ph ^ 1, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&s.full[st], STAGE_BYTES);
                    tma_load_2d(smA(st), ta, k0 + kb * BK, m * BM, &s.full[st]);
                    tma_load_2d(smB(st), tb, k0 + kb * BK, n * BN, &s.full[st]);
                    issued_mask |= 1u << st;
                    issued_par = (issued_par & ~(1u << st)) | (ph << st);
                    if (++st == STAGES) {
                        st = 0;
                        ph ^= 1;
                    }
                }
            }
            for (int i = 0; i < STAGES; ++i)
                if (issued_mask & (1u << i)) drain_bar(&s.full[i], (issued_par >> i) & 1u);
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);
            int st = 0, acc = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const int g = tile / per_seg;
                if (!wait_bar(&s.tempty[acc], aph ^ 1, abort_flag, p.err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < s.kp[g] / BK; ++kb) {
                    if (!wait_bar(&s.full[st], ph, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = desc_sw128(smem_u32(smA(st)));
                    const uint64_t bd = desc_sw128(smem_u32(smB(st)));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_bf16(d_tmem, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), IDESC,
                                  (kb | kk) != 0 ? 1u : 0u);
                    umma_commit(&s.empty[st]);
                    if (++st == STAGES) {
                        st = 0;
                        ph ^= 1;
                    }
                }
                if (!ok) break;
                umma_commit(&s.tfull[acc]);  // no MMA for an empty segment: the epilogue writes zeros
                if (++acc == 2) {
                    acc = 0;
                    aph ^= 1;
                }
            }
            umma_commit(&s.drain);
            drain_bar(&s.drain, 0);
        }
    } else {
        // ================= epilogue (warps 2..5) =================
        const int quarter = warp & 3;
        const int r_in_tile = quarter * 32 + lane;
        int acc = 0;
        uint32_t aph = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            const int g = tile / per_seg, local = tile - g * per_seg;
            const int m = local % mt, n = local / mt;
            const bool sh = g >= p.n_seg;
            if (!wait_bar(&s.tfull[acc], aph, abort_flag, p.err)) break;
            tc_fence_after();
            const int row = m * BM + r_in_tile;
            const bool empty_seg = s.kp[g] == 0;
            const size_t crow = ((sh ? 0 : (size_t)g * p.M) + (size_t)row) * p.Nn;  // element offset of the row
            const uint32_t tbase = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quarter * 32) << 16);
#pragma unroll 1
            for (int c = 0; c < BN; c += 32) {
                uint32_t v[32];
                tmem_ld32(tbase + c, v);
                tmem_ld_wait();
                const int col = n * BN + c;
                if (F32 && row < p.M && col < p.Nn) {
                    float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(sh ? p.C_sh : p.C) + crow + col);
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        dst[q] = empty_seg ? make_float4(0.0f, 0.0f, 0.0f, 0.0f)
                                           : make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                                         __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
                } else if (!F32 && row < p.M && col < p.Nn) {
                    uint32_t packed[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float f0 = empty_seg ? 0.0f : __uint_as_float(v[2 * i]);
                        const float f1 = empty_seg ? 0.0f : __uint_as_float(v[2 * i + 1]);
                        __nv_bfloat162 b = __floats2bfloat162_rn(f0, f1);
                        packed[i] = *reinterpret_cast<uint32_t *>(&b);
                    }
                    uint4 *dst =
                        reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(sh ? p.C_sh : p.C) + crow + col);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
                }
            }
            tc_fence_before();
            mbar_arrive_relaxed(&s.tempty[acc]);
            if (++acc == 2) {
                acc = 0;
                aph ^= 1;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, 512);
    }
}

// ------------------------------------------------------------------ CTA-pair version
//
// The same tiles with 2-CTA (cta_group::2) MMAs, as the forward's pair kernel in
// ffn_tc.cu: a cluster of two CTAs computes a 256 x 256 output tile per MMA
// 256x256x16; each CTA stages 128 rows of At and 128 of the 256 rows of Bt per
// k-block (a third less operand data per FLOP than the single-CTA kernel), both
// halves complete on the even CTA's stage barrier, the even CTA issues the MMAs and
// its commits arrive on both CTAs' barriers; each CTA's epilogue stores its 128 rows.
// The epilogue writes through shared memory: each warp converts 32 rows x 64 columns
// to bf16 (32 columns in the fp32 form) into one of two 4 KB boxes laid out as the
// output map's 128-byte swizzle and stores the box with one TMA tensor store, so whole
// 128-byte lines reach L2. With an
// expert's few hundred rows as K, a tile's MMAs are short next to its 128 KB of
// gradient, and per-thread 16-byte row stores (32 rows per instruction) kept L2 busy
// with partial-line write requests.
constexpr int STAGES2 = 5;
constexpr uint32_t HALF_BYTES = 128 * BK * 2;
constexpr uint32_t STAGE2_BYTES = 2 * HALF_BYTES;
constexpr uint32_t OUT_BOX_BYTES = 32 * 64 * 2;  // 32 rows x 64 bf16
constexpr size_t SMEM2_BYTES = (size_t)STAGES2 * STAGE2_BYTES + 4 * 2 * OUT_BOX_BYTES + 1024;

struct WgSmem2 {
    uint64_t full[STAGES2], empty[STAGES2], tfull[2], tempty[2], drain;
    uint32_t tmem_base;
    int abort_flag;
    int k0[MAX_SEG], kp[MAX_SEG];
};
static_assert(SMEM2_BYTES + sizeof(WgSmem2) <= 232448, "shared memory budget of one CTA");
static_assert(STAGE2_BYTES % 1024 == 0 && OUT_BOX_BYTES % 1024 == 0, "swizzled boxes stay 1024-byte aligned");

// Tensor maps as in WgParams but with 128-row boxes for Bt (each CTA loads half).
template <bool F32>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    k_wgrad_tc2(const __grid_constant__ WgParams p) {
    __shared__ WgSmem2 s;
    extern __shared__ uint8_t dyn_smem[];
    const uint32_t dyn_base = smem_u32(dyn_smem);
    uint8_t *tiles = dyn_smem + (((dyn_base + 1023u) & ~1023u) - dyn_base);
    auto smA = [&](int st) { return tiles + (size_t)st * STAGE2_BYTES; };
    auto smB = [&](int st) { return tiles + (size_t)st * STAGE2_BYTES + HALF_BYTES; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    const int nseg = p.n_seg + p.has_sh;
    const int mt = (p.M + 2 * BM - 1) / (2 * BM), nt = (p.Nn + BN - 1) / BN;
    const int per_seg = mt * nt;
    const int total = nseg * per_seg;

    if (warp == 0) {
        constexpr int PER = (MAX_SEG + 31) / 32;
        int kp[PER];
        int sum = 0;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int g = lane * PER + i;
            int v = 0;
            if (g < p.n_seg) {
                const int r0 = min(max(p.offsets[g], 0), p.a_rows);
                const int r1 = min(max(p.offsets[g + 1], r0), p.a_rows);
                v = (r1 - r0 + BK - 1) / BK * BK;
            }
            kp[i] = v;
            sum += v;
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += u;
        }
        int run = incl - sum;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int g = lane * PER + i;
            if (g < p.n_seg) {
                s.k0[g] = run;
                s.kp[g] = kp[i];
            }
            run += kp[i];
        }
        if (lane == 0 && p.has_sh) {
            s.k0[p.n_seg] = 0;
            s.kp[p.n_seg] = p.K_sh;
        }
        if (lane == 0) {
            for (int i = 0; i < STAGES2; ++i) {
                mbar_init(&s.full[i], 1);
                mbar_init(&s.empty[i], 1);
            }
            for (int i = 0; i < 2; ++i) {
                mbar_init(&s.tfull[i], 1);
                mbar_init(&s.tempty[i], 8);  // 4 epilogue warps of each CTA
            }
            mbar_init(&s.drain, 1);
            s.abort_flag = 0;
            fence_mbar_init();
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(&s.tmem_base, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after();
    const uint32_t tmem_base = s.tmem_base;
    if (tid == 0) {
        // the pair MMA writes the same TMEM address in both CTAs
        const uint32_t other = ld_shared_cluster_u32(map_to_rank(smem_u32(&s.tmem_base), rank ^ 1u));
        if (other != tmem_base) {
            s.abort_flag = 1;
            record_error(p.err, kErrFault);
        }
    }
    __syncthreads();
    const bool run = s.abort_flag == 0;
    volatile int *abort_flag = &s.abort_flag;
    const uint32_t lead_tempty = map_to_rank(smem_u32(&s.tempty[0]), 0);

    if (warp == 0) {
        // ================= TMA producer (both CTAs) =================
        if (lane == 0 && run) {
            int st = 0;
            uint32_t ph = 0;
            bool ok = true;
            uint32_t issued_mask = 0, issued_par = 0;
            const uint32_t lead_full = map_to_rank(smem_u32(&s.full[0]), 0);
            for (int tile = cluster; tile < total && ok; tile += nclusters) {
                const int g = tile / per_seg, local = tile - g * per_seg;
                const int m = local % mt, n = local / mt;
                const bool sh = g >= p.n_seg;
                const CUtensorMap *ta = sh ? &p.tmA_sh : &p.tmA;
                const CUtensorMap *tb = sh ? &p.tmB_sh : &p.tmB;
                const int k0 = s.k0[g];
                const int arow = m * 2 * BM + (int)rank * BM, brow = n * BN + (int)rank * (BN / 2);
                for (int kb = 0; kb < s.kp[g] / BK; ++kb) {
                    if (!wait_bar(&s.empty[st], ph ^ 1, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = lead_full + 8u * (uint32_t)st;
                    if (leader) mbar_arrive_expect_tx(&s.full[st], 2 * STAGE2_BYTES);
                    tma_load_2d_pair(smA(st), ta, k0 + kb * BK, arow, fb);
                    tma_load_2d_pair(smB(st), tb, k0 + kb * BK, brow, fb);
                    issued_mask |= 1u << st;
                    issued_par = (issued_par & ~(1u << st)) | (ph << st);
                    if (++st == STAGES2) {
                        st = 0;
                        ph ^= 1;
                    }
                }
            }
            // loads in flight land before the CTA exits (the even CTA waits for both halves)
            if (leader)
                for (int i = 0; i < STAGES2; ++i)
                    if (issued_mask & (1u << i)) drain_bar(&s.full[i], (issued_par >> i) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0 && run && leader) {
            // ================= MMA issuer (even CTA) =================
            constexpr uint32_t IDESC = idesc_bf16_f32(2 * BM, BN);
            int st = 0, acc = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            for (int tile = cluster; tile < total && ok; tile += nclusters) {
                const int g = tile / per_seg;
                if (!wait_bar(&s.tempty[acc], aph ^ 1, abort_flag, p.err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < s.kp[g] / BK; ++kb) {
                    if (!wait_bar(&s.full[st], ph, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = desc_sw128(smem_u32(smA(st)));
                    const uint64_t bd = desc_sw128(smem_u32(smB(st)));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_bf16_pair(d_tmem, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), IDESC,
                                       (kb | kk) != 0 ? 1u : 0u);
                    umma_commit_pair_mc(&s.empty[st], 0x3);
                    if (++st == STAGES2) {
                        st = 0;
                        ph ^= 1;
                    }
                }
                if (!ok) break;
                umma_commit_pair_mc(&s.tfull[acc], 0x3);  // no MMA for an empty segment: zeros stored
                if (++acc == 2) {
                    acc = 0;
                    aph ^= 1;
                }
            }
            umma_commit_pair_mc(&s.drain, 0x1);
            drain_bar(&s.drain, 0);
        }
    } else if (run) {
        // ================= epilogue (warps 2..5 of both CTAs) =================
        const int quarter = warp & 3;
        uint8_t *boxes = tiles + (size_t)STAGES2 * STAGE2_BYTES + (size_t)quarter * 2 * OUT_BOX_BYTES;
        const uint32_t swz = (uint32_t)(lane & 7);  // 128-byte swizzle: 16-byte unit j of row r at j ^ (r % 8)
        uint32_t nbox = 0;
        int acc = 0;
        uint32_t aph = 0;
        for (int tile = cluster; tile < total; tile += nclusters) {
            const int g = tile / per_seg, local = tile - g * per_seg;
            const int m = local % mt, n = local / mt;
            const bool sh = g >= p.n_seg;
            if (!wait_bar(&s.tfull[acc], aph, abort_flag, p.err)) break;
            tc_fence_after();
            const int row0 = m * 2 * BM + (int)rank * BM + quarter * 32;  // this warp's 32 rows
            const bool empty_seg = s.kp[g] == 0;
            const CUtensorMap *cmap = sh ? &p.tmC_sh : &p.tmC;
            const int gz = sh ? 0 : g;
            const uint32_t tbase = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quarter * 32) << 16);
            constexpr int CW = F32 ? 32 : 64;  // columns per 128-byte box row
#pragma unroll 1
            for (int c = 0; c < BN; c += CW) {
                uint32_t v[64];
                tmem_ld32(tbase + c, v);
                if (!F32) tmem_ld32(tbase + c + 32, v + 32);
                tmem_ld_wait();
                const int col = n * BN + c;
                // Nn is a multiple of 64: a box's columns lie wholly inside the output or outside;
                // rows past M (a box straddling it) are clipped by the tensor store
                if (row0 < p.M && col < p.Nn) {
                    uint8_t *box = boxes + (nbox & 1u) * OUT_BOX_BYTES;
                    if (lane == 0) bulk_wait_group_read<1>();  // the store of two boxes ago has read this box
                    __syncwarp();
                    uint8_t *rowp = box + lane * 128;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        uint32_t w[4];
#pragma unroll
                        for (int t = 0; t < 4; ++t) {
                            if constexpr (F32) {
                                w[t] = empty_seg ? 0u : v[4 * j + t];
                            } else {
                                const float f0 = empty_seg ? 0.0f : __uint_as_float(v[8 * j + 2 * t]);
                                const float f1 = empty_seg ? 0.0f : __uint_as_float(v[8 * j + 2 * t + 1]);
                                __nv_bfloat162 b = __floats2bfloat162_rn(f0, f1);
                                w[t] = *reinterpret_cast<uint32_t *>(&b);
                            }
                        }
                        *reinterpret_cast<uint4 *>(rowp + ((j ^ swz) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(cmap, box, col, row0, gz);
                        bulk_commit_group();
                    }
                    ++nbox;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader) mbar_arrive_relaxed(&s.tempty[acc]);
                else mbar_arrive_remote_relaxed(lead_tempty + 8u * (uint32_t)acc);
            }
            if (++acc == 2) {
                acc = 0;
                aph ^= 1;
            }
        }
        if (lane == 0) bulk_wait_group<0>();  // every store of this warp done before the CTA exits
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the pair's MMAs and both epilogues are done with TMEM
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, 512);
    }
}

// kpre[g] = sum over segments g' < g of R_g' rounded up to 64 (g = 0 .. n_seg), one CTA.
__global__ void __launch_bounds__(256) k_pad_prefix(const int32_t *__restrict__ offsets, int n_seg, int rows,
                                                    int32_t *__restrict__ kpre) {
    __shared__ int w[MAX_SEG];
    for (int g = threadIdx.x; g < n_seg; g += blockDim.x) {
        const int a = min(max(offsets[g], 0), rows);
        const int e = min(max(offsets[g + 1], a), rows);
        w[g] = (e - a + 63) / 64 * 64;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int run = 0;
        for (int g = 0; g < n_seg; ++g) {
            kpre[g] = run;
            run += w[g];
        }
        kpre[n_seg] = run;
    }
}

// Activation rows [rows][C] (row stride C) into the padded transposed layout
// [C][Kall]: column kpre[g] + i holds row offsets[g] + i for i < R_g, zero up to
// kpre[g + 1]; 64-column blocks from kpre[n_seg] on are left unwritten (no product reads
// them). offsets null: one segment of `rows` rows, zero up to Kall.
// 64 x 64 tiles, 16-byte loads and stores (C and Kall multiples of 8).
__global__ void __launch_bounds__(256) k_transpose_rows_padded(const __nv_bfloat16 *__restrict__ src, int C,
                                                               const int32_t *__restrict__ offsets,
                                                               const int32_t *__restrict__ kpre, int n_seg,
                                                               int rows, int64_t Kall,
                                                               __nv_bfloat16 *__restrict__ dst) {
    __shared__ __nv_bfloat16 tile[64][64 + 2];
    __shared__ int srow[64];
    const int64_t k0 = (int64_t)blockIdx.x * 64;
    const int c0 = blockIdx.y * 64;
    if (offsets && k0 >= kpre[n_seg]) return;  // past the last segment: never read
    if (threadIdx.x < 64) {
        // source row of padded column k0 + threadIdx.x (-1: padding), by binary search on kpre
        const int64_t kc = k0 + threadIdx.x;
        int r = -1;
        if (!offsets) {
            r = kc < rows ? (int)kc : -1;
        } else if (kc < kpre[n_seg]) {
            int lo = 0, hi = n_seg - 1;  // largest g with kpre[g] <= kc
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (kpre[mid] <= kc) lo = mid;
                else hi = mid - 1;
            }
            const int a = min(max(offsets[lo], 0), rows);
            const int e = min(max(offsets[lo + 1], a), rows);
            const int64_t i = kc - kpre[lo];
            r = i < e - a ? (int)(a + i) : -1;
        }
        srow[threadIdx.x] = r;
    }
    __syncthreads();
    for (int v = threadIdx.x; v < 64 * 8; v += 256) {
        const int i = v >> 3, j = (v & 7) * 8;  // padded column k0 + i, source columns c0 + j .. + 7
        const int r = srow[i];
        uint4 q = make_uint4(0, 0, 0, 0);
        if (r >= 0 && c0 + j < C) q = *reinterpret_cast<const uint4 *>(src + (size_t)r * C + c0 + j);
        const __nv_bfloat16 *e = reinterpret_cast<const __nv_bfloat16 *>(&q);
#pragma unroll
        for (int u = 0; u < 8; ++u) tile[i][j + u] = e[u];
    }
    __syncthreads();
    for (int v = threadIdx.x; v < 64 * 8; v += 256) {
        const int i = v >> 3, j = (v & 7) * 8;  // destination row c0 + i, padded columns k0 + j .. + 7
        if (c0 + i < C && k0 + j < Kall) {
            __align__(16) __nv_bfloat16 e[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) e[u] = tile[j + u][i];
            *reinterpret_cast<uint4 *>(dst + (size_t)(c0 + i) * Kall + k0 + j) = *reinterpret_cast<const uint4 *>(e);
        }
    }
}

}  // namespace

int64_t wgrad_kall_bound(const moe_config &c) { return (max_rows(c) + 64LL * c.N + 63) / 64 * 64; }

// Output map of the pair kernel's tensor stores: [n][M][Nn] of bf16 or fp32, box of 32
// rows x 128 bytes, 128-byte swizzle.
static bool encode_out_map(CUtensorMap *m, void *base, int Nn, int M, int n, bool f32) {
    const uint64_t es = f32 ? 4 : 2;
    const uint64_t dims[3] = {(uint64_t)Nn, (uint64_t)M, (uint64_t)n};
    const uint64_t strides[2] = {(uint64_t)Nn * es, (uint64_t)Nn * M * es};
    const uint32_t box[3] = {(uint32_t)(128 / es), 32u, 1u};
    return encode_tmap(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims,
                       strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <typename Kern> static cudaError_t smem_attr_once(Kern kern, size_t bytes, bool &done) {
    if (done) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) done = true;
    return e;
}

cudaError_t launch_wgrad(const int32_t *offsets, int n_seg, int64_t a_rows, const void *At, const void *Bt,
                         int64_t Kall, int M, int Nn, void *out, const void *At_sh, const void *Bt_sh, int K_sh,
                         void *out_sh, uint32_t *err, cudaStream_t s, bool allow_pair, bool f32_out) {
    // CTA pairs once a 256-row output tile is not mostly empty
    const bool pair = allow_pair && M >= 2 * BM;
    const uint32_t box_b = pair ? BN / 2 : BN;
    if (Nn % 64 != 0) return cudaErrorInvalidValue;
    WgParams p;
    memset(&p, 0, sizeof(p));
    p.offsets = offsets;
    p.n_seg = n_seg;
    p.has_sh = At_sh ? 1 : 0;
    p.a_rows = (int)a_rows;
    p.M = M;
    p.Nn = Nn;
    p.K_sh = K_sh;
    p.C = out;
    p.C_sh = out_sh;
    p.err = err;
    if (n_seg > 0) {
        if (!encode_bf16_2d(&p.tmA, At, (uint64_t)Kall, (uint64_t)M, BM)) return cudaErrorInvalidValue;
        if (!encode_bf16_2d(&p.tmB, Bt, (uint64_t)Kall, (uint64_t)Nn, box_b)) return cudaErrorInvalidValue;
        if (pair && !encode_out_map(&p.tmC, out, Nn, M, n_seg, f32_out)) return cudaErrorInvalidValue;
    }
    if (p.has_sh) {
        if (!encode_bf16_2d(&p.tmA_sh, At_sh, (uint64_t)K_sh, (uint64_t)M, BM)) return cudaErrorInvalidValue;
        if (!encode_bf16_2d(&p.tmB_sh, Bt_sh, (uint64_t)K_sh, (uint64_t)Nn, box_b)) return cudaErrorInvalidValue;
        if (pair && !encode_out_map(&p.tmC_sh, out_sh, Nn, M, 1, f32_out)) return cudaErrorInvalidValue;
    }
    cudaError_t e;
    if (pair) {
        const int64_t tiles2 = (int64_t)(n_seg + p.has_sh) * ((M + 2 * BM - 1) / (2 * BM)) * ((Nn + BN - 1) / BN);
        if (tiles2 == 0) return cudaSuccess;
        static bool done_h = false, done_f = false;
        if ((e = f32_out ? smem_attr_once(k_wgrad_tc2<true>, SMEM2_BYTES, done_f)
                         : smem_attr_once(k_wgrad_tc2<false>, SMEM2_BYTES, done_h)) != cudaSuccess)
            return e;
        const int clusters = (int)std::max<int64_t>(1, std::min<int64_t>(tiles2, device_sm_count() / 2));
        if (f32_out) k_wgrad_tc2<true><<<2 * clusters, NUM_THREADS, SMEM2_BYTES, s>>>(p);
        else k_wgrad_tc2<false><<<2 * clusters, NUM_THREADS, SMEM2_BYTES, s>>>(p);
        return cudaGetLastError();
    }
    const int64_t tiles = (int64_t)(n_seg + p.has_sh) * ((M + BM - 1) / BM) * ((Nn + BN - 1) / BN);
    if (tiles == 0) return cudaSuccess;
    static bool done1_h = false, done1_f = false;
    if ((e = f32_out ? smem_attr_once(k_wgrad_tc<true>, SMEM_BYTES, done1_f)
                     : smem_attr_once(k_wgrad_tc<false>, SMEM_BYTES, done1_h)) != cudaSuccess)
        return e;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, device_sm_count()));
    if (f32_out) k_wgrad_tc<true><<<grid, NUM_THREADS, SMEM_BYTES, s>>>(p);
    else k_wgrad_tc<false><<<grid, NUM_THREADS, SMEM_BYTES, s>>>(p);
    return cudaGetLastError();
}

cudaError_t launch_pad_prefix(const int32_t *offsets, int n_seg, int rows, int32_t *kpre, cudaStream_t s) {
    k_pad_prefix<<<1, 256, 0, s>>>(offsets, n_seg, rows, kpre);
    return cudaGetLastError();
}

cudaError_t launch_transpose_rows_padded(const void *src, int C, const int32_t *offsets, const int32_t *kpre,
                                         int n_seg, int rows, int64_t Kall, void *dst, cudaStream_t s) {
    dim3 grid((unsigned)((Kall + 63) / 64), (unsigned)((C + 63) / 64));
    k_transpose_rows_padded<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(src), C, offsets, kpre, n_seg,
                                                 rows, Kall, static_cast<__nv_bfloat16 *>(dst));
    return cudaGetLastError();
}

}  // namespace moe
