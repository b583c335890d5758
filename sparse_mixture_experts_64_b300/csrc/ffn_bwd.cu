// Weight-gradient GEMM of the experts on the tensor cores.
//
// The experts' weight gradients reduce over each expert's rows: dW_out[e] =
// dO_eᵀ H_e, dW_a[e] = dA_eᵀ X_e, dW_b[e] = dB_eᵀ X_e (the chain rule through
// O = H W_outᵀ, H = act(X W_aᵀ) (⊙ X W_bᵀ)). K is an expert's row count, so it varies
// per expert. Both operands are read where the forward and the row products left them,
// [rows][columns] with the rows grouped by expert: for these products that is the
// MN-major layout (M or N contiguous), staged as 64-column chunks of 64 K-rows under the
// 128-byte swizzle. Expert e's k-blocks start at its first row; when its row count is
// not a multiple of 64 its last k-block reaches into the next expert's rows (or past the
// rows in use), and those K-rows are zeroed in shared memory before the MMAs read the
// stage: in this layout K-row i of a chunk is its 128-byte line i, so that is the tail of
// each 8 KB chunk. The kernels — a TMA producer warp, an MMA-issuing warp, four epilogue
// warps, a fixup warp that does that zeroing as soon as such a stage lands, two TMEM
// accumulators — take tiles (expert, m, n) and store an all-zero tile for an expert
// without rows. An optional shared segment (the shared expert, or with no
// routed segment a plain product such as the router's gradients) reduces over K_sh,
// with either operand MN-major ([rows][..], K-rows past its rows read as zero by the
// copy) or K-major ([M|Nn][K_sh], zero-padded to a multiple of 64).
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
constexpr uint32_t CHUNK_BYTES = 64 * BK * 2;  // MN-major: 64 columns x 64 K-rows
constexpr int NUM_THREADS = 224;  // 7 warps (roles below)
constexpr int MAX_SEG = 257;
constexpr size_t SMEM_BYTES = (size_t)STAGES * STAGE_BYTES + 1024;

struct WgParams {
    CUtensorMap tmA, tmB;        // routed segments: MN-major maps over [a_rows][M], [a_rows][Nn] seen as
                                 // (64 columns, rows, 64-column chunks): one box stages a CTA's chunks
    CUtensorMap tmA_sh, tmB_sh;  // shared segment: MN-major as above over K_sh rows, or K-major over
                                 // [M|Nn][K_sh] with a box of 64 x the rows one CTA stages
    CUtensorMap tmC, tmC_sh;     // outputs for the pair kernel's stores: [n_seg][M][Nn], [1][M][Nn], box of
                                 // 32 rows x 128 bytes (64 bf16 or 32 fp32 columns)
    const int32_t *offsets;      // [n_seg + 1] rows of each expert
    int n_seg, has_sh;
    int a_rows;                  // offsets are clamped to it
    int M, Nn, K_sh;
    int a_mn_sh, b_mn_sh;        // the shared segment's operands MN-major (routed ones always are)
    void *C, *C_sh;              // [n_seg][M][Nn], [M][Nn]: bf16, or fp32 in the kernels' F32 form
    uint32_t *err;
};

// Per segment: first K-row, k-blocks, and the valid rows of a partial last k-block (0: none).
struct SegK {
    int k0[MAX_SEG], nk[MAX_SEG], kv[MAX_SEG];
};

__device__ __forceinline__ void seg_k_ranges(const WgParams &p, SegK &s, int lane) {
    for (int g = lane; g < p.n_seg; g += 32) {
        const int r0 = min(max(p.offsets[g], 0), p.a_rows);
        const int r1 = min(max(p.offsets[g + 1], r0), p.a_rows);
        s.k0[g] = r0;
        s.nk[g] = (r1 - r0 + BK - 1) / BK;
        s.kv[g] = (r1 - r0) % BK;
    }
    if (lane == 0 && p.has_sh) {
        s.k0[p.n_seg] = 0;
        s.nk[p.n_seg] = (p.K_sh + BK - 1) / BK;
        s.kv[p.n_seg] = 0;  // MN-major: K-rows past the operand's rows are outside its map (zero);
                            // K-major: zero-padded
    }
}

// Zero K-rows kv .. 63 of `chunks` consecutive MN-major chunks (lines kv .. 63 of each
// 8 KB chunk; a line keeps its 16-byte units whatever the swizzle). One warp.
__device__ __forceinline__ void zero_k_tail(uint8_t *base, int chunks, int kv, int lane) {
    for (int c = 0; c < chunks; ++c) {
        uint4 *q = reinterpret_cast<uint4 *>(base + (size_t)c * CHUNK_BYTES);
        for (int u = kv * 8 + lane; u < (int)(CHUNK_BYTES / 16); u += 32) q[u] = make_uint4(0u, 0u, 0u, 0u);
    }
}

// Instruction-descriptor bits and descriptor steps (16-byte units per K step of 16) of a
// segment's operands.
struct SegMajor {
    bool a_mn, b_mn;
    __device__ uint32_t idesc_bits() const { return (a_mn ? kIdescAMajorMN : 0u) | (b_mn ? kIdescBMajorMN : 0u); }
    __device__ uint64_t a_step() const { return a_mn ? 128u : 2u; }  // MN-major: 16 K-rows of 128 bytes
    __device__ uint64_t b_step() const { return b_mn ? 128u : 2u; }
    __device__ uint64_t a_desc(uint32_t addr) const { return a_mn ? desc_sw128_mn(addr) : desc_sw128(addr); }
    __device__ uint64_t b_desc(uint32_t addr) const { return b_mn ? desc_sw128_mn(addr) : desc_sw128(addr); }
};
__device__ __forceinline__ SegMajor seg_major(const WgParams &p, int g) {
    const bool sh = g >= p.n_seg;
    return {!sh || p.a_mn_sh != 0, !sh || p.b_mn_sh != 0};
}

struct WgSmem {
    uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], drain;
    uint64_t bfull[STAGES];  // a segment's partial last k-block landed (only those complete it)
    uint64_t fixed[STAGES];  // ... and the fixup warp zeroed its rows past the segment
    uint32_t tmem_base;
    int abort_flag;
    SegK seg;
};

// Warp roles of both kernels: 0 TMA producer, 1 MMA issuer (one thread), 2-5 epilogue,
// 6 fixup (zeroes the rows past a segment in a partial last k-block as soon as it lands,
// beside the MMAs of the stages before it).
constexpr int FIXUP_WARP = 6;

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
        seg_k_ranges(p, s.seg, lane);
        if (lane == 0) {
            for (int i = 0; i < STAGES; ++i) {
                mbar_init(&s.full[i], 1);
                mbar_init(&s.empty[i], 1);
                mbar_init(&s.bfull[i], 1);
                mbar_init(&s.fixed[i], 1);
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
        // A stage completes full[], or bfull[] when it is a segment's partial last k-block.
        if (lane == 0) {
            int st = 0;
            uint32_t ph = 0;
            bool ok = true;
            uint32_t issued_mask = 0, issued_par = 0, fcount = 0;    // full[]: parity of each stage's uses
            uint32_t bissued_mask = 0, bissued_par = 0, bcount = 0;  // bfull[]
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const int g = tile / per_seg, local = tile - g * per_seg;
                const int m = local % mt, n = local / mt;
                const bool sh = g >= p.n_seg;
                const SegMajor mj = seg_major(p, g);
                const CUtensorMap *ta = sh ? &p.tmA_sh : &p.tmA;
                const CUtensorMap *tb = sh ? &p.tmB_sh : &p.tmB;
                const int k0 = s.seg.k0[g], nk = s.seg.nk[g], kv = s.seg.kv[g];
                for (int kb = 0; kb < nk; ++kb) {
                    if (!wait_bar(&s.empty[st], ph ^ 1, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bit = 1u << st;
                    const bool edge = kb == nk - 1 && kv != 0;
                    uint64_t *bar = edge ? &s.bfull[st] : &s.full[st];
                    mbar_arrive_expect_tx(bar, STAGE_BYTES);
                    const int kc = k0 + kb * BK;
                    if (mj.a_mn) tma_load_3d(smA(st), ta, 0, kc, m * (BM / 64), bar);
                    else tma_load_2d(smA(st), ta, kc, m * BM, bar);
                    if (mj.b_mn) tma_load_3d(smB(st), tb, 0, kc, n * (BN / 64), bar);
                    else tma_load_2d(smB(st), tb, kc, n * BN, bar);
                    if (edge) {
                        bissued_mask |= bit;
                        bissued_par = (bissued_par & ~bit) | (bcount & bit);
                        bcount ^= bit;
                    } else {
                        issued_mask |= bit;
                        issued_par = (issued_par & ~bit) | (fcount & bit);
                        fcount ^= bit;
                    }
                    if (++st == STAGES) {
                        st = 0;
                        ph ^= 1;
                    }
                }
            }
            for (int i = 0; i < STAGES; ++i) {
                if (issued_mask & (1u << i)) drain_bar(&s.full[i], (issued_par >> i) & 1u);
                if (bissued_mask & (1u << i)) drain_bar(&s.bfull[i], (bissued_par >> i) & 1u);
            }
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            int st = 0, acc = 0;
            uint32_t aph = 0, fpar = 0, xpar = 0;  // per-stage parities of full[] and fixed[] uses
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const int g = tile / per_seg;
                const SegMajor mj = seg_major(p, g);
                const uint32_t idesc = idesc_bf16_f32(BM, BN) | mj.idesc_bits();
                if (!wait_bar(&s.tempty[acc], aph ^ 1, abort_flag, p.err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                const int nk = s.seg.nk[g], kv = s.seg.kv[g];
                for (int kb = 0; kb < nk; ++kb) {
                    const uint32_t bit = 1u << st;
                    const bool edge = kb == nk - 1 && kv != 0;
                    if (!(edge ? wait_bar(&s.fixed[st], (xpar >> st) & 1u, abort_flag, p.err)
                               : wait_bar(&s.full[st], (fpar >> st) & 1u, abort_flag, p.err))) {
                        ok = false;
                        break;
                    }
                    if (edge) xpar ^= bit;
                    else fpar ^= bit;
                    tc_fence_after();
                    const uint64_t ad = mj.a_desc(smem_u32(smA(st))), bd = mj.b_desc(smem_u32(smB(st)));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_bf16(d_tmem, ad + mj.a_step() * kk, bd + mj.b_step() * kk, idesc, (kb | kk) != 0 ? 1u : 0u);
                    umma_commit(&s.empty[st]);
                    if (++st == STAGES) st = 0;
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
    } else if (warp == FIXUP_WARP) {
        // ================= fixup: rows past a segment in its partial last k-block =================
        int st = 0;
        uint32_t bpar = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
            const int g = tile / per_seg;
            const int nk = s.seg.nk[g], kv = s.seg.kv[g];
            for (int kb = 0; kb < nk; ++kb) {
                if (kb == nk - 1 && kv != 0) {
                    if (!__all_sync(0xffffffffu, wait_bar(&s.bfull[st], (bpar >> st) & 1u, abort_flag, p.err))) {
                        ok = false;
                        break;
                    }
                    bpar ^= 1u << st;
                    zero_k_tail(smA(st), BM / 64, kv, lane);  // routed segments: both operands MN-major
                    zero_k_tail(smB(st), BN / 64, kv, lane);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&s.fixed[st]);
                }
                if (++st == STAGES) st = 0;
            }
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
            const bool empty_seg = s.seg.nk[g] == 0;
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
// 256x256x16; each CTA stages 128 of the 256 A columns (M) and 128 of the 256 B columns
// (N) per k-block (a third less operand data per FLOP than the single-CTA kernel), both
// halves complete on the even CTA's stage barrier, the even CTA issues the MMAs and
// its commits arrive on both CTAs' barriers; each CTA's epilogue stores its 128 rows.
// A segment's partial last k-block is the exception: each CTA's half lands on that CTA's
// own bfull[] barrier, each CTA's fixup warp zeroes the rows past the segment in its half
// and arrives on the even CTA's fixed[] barrier (two arrivals), and the MMA issuer waits
// for fixed[] instead of full[] before that k-block's MMAs.
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
    uint64_t bfull[STAGES2];  // this CTA's half of a partial last k-block landed
    uint64_t fixed[STAGES2];  // even CTA: both halves of that k-block zeroed past the segment
    uint32_t tmem_base;
    int abort_flag;
    SegK seg;
};
static_assert(SMEM2_BYTES + sizeof(WgSmem2) <= 232448, "shared memory budget of one CTA");
static_assert(STAGE2_BYTES % 1024 == 0 && OUT_BOX_BYTES % 1024 == 0, "swizzled boxes stay 1024-byte aligned");

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
        seg_k_ranges(p, s.seg, lane);
        if (lane == 0) {
            for (int i = 0; i < STAGES2; ++i) {
                mbar_init(&s.full[i], 1);
                mbar_init(&s.empty[i], 1);
                mbar_init(&s.bfull[i], 1);
                mbar_init(&s.fixed[i], 2);  // the fixup warps of both CTAs
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
    const uint32_t lead_fixed = map_to_rank(smem_u32(&s.fixed[0]), 0);

    if (warp == 0) {
        // ================= TMA producer (both CTAs) =================
        // Both CTAs' loads complete on the even CTA's full[] barrier, which the even
        // CTA's producer arms with the bytes of both halves; in a partial last k-block
        // each CTA's half lands on its own bfull[] instead.
        if (lane == 0 && run) {
            int st = 0;
            uint32_t ph = 0;
            bool ok = true;
            uint32_t issued_mask = 0, issued_par = 0, fcount = 0;    // full[] (even CTA)
            uint32_t bissued_mask = 0, bissued_par = 0, bcount = 0;  // bfull[] (each CTA)
            const uint32_t lead_full = map_to_rank(smem_u32(&s.full[0]), 0);
            for (int tile = cluster; tile < total && ok; tile += nclusters) {
                const int g = tile / per_seg, local = tile - g * per_seg;
                const int m = local % mt, n = local / mt;
                const bool sh = g >= p.n_seg;
                const SegMajor mj = seg_major(p, g);
                const CUtensorMap *ta = sh ? &p.tmA_sh : &p.tmA;
                const CUtensorMap *tb = sh ? &p.tmB_sh : &p.tmB;
                const int k0 = s.seg.k0[g], nk = s.seg.nk[g], kv = s.seg.kv[g];
                const int acol = m * 2 * BM + (int)rank * BM, bcol = n * BN + (int)rank * (BN / 2);
                for (int kb = 0; kb < nk; ++kb) {
                    if (!wait_bar(&s.empty[st], ph ^ 1, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t bit = 1u << st;
                    const bool edge = kb == nk - 1 && kv != 0;
                    const int kc = k0 + kb * BK;
                    if (edge) {
                        // routed segment (MN-major): this CTA's half, plain copies into its own stage
                        mbar_arrive_expect_tx(&s.bfull[st], STAGE2_BYTES);
                        tma_load_3d(smA(st), ta, 0, kc, acol / 64, &s.bfull[st]);
                        tma_load_3d(smB(st), tb, 0, kc, bcol / 64, &s.bfull[st]);
                        bissued_mask |= bit;
                        bissued_par = (bissued_par & ~bit) | (bcount & bit);
                        bcount ^= bit;
                    } else {
                        const uint32_t fb = lead_full + 8u * (uint32_t)st;
                        if (leader) mbar_arrive_expect_tx(&s.full[st], 2 * STAGE2_BYTES);
                        if (mj.a_mn) tma_load_3d_pair(smA(st), ta, 0, kc, acol / 64, fb);
                        else tma_load_2d_pair(smA(st), ta, kc, acol, fb);
                        if (mj.b_mn) tma_load_3d_pair(smB(st), tb, 0, kc, bcol / 64, fb);
                        else tma_load_2d_pair(smB(st), tb, kc, bcol, fb);
                        issued_mask |= bit;
                        issued_par = (issued_par & ~bit) | (fcount & bit);
                        fcount ^= bit;
                    }
                    if (++st == STAGES2) {
                        st = 0;
                        ph ^= 1;
                    }
                }
            }
            // loads in flight land before the CTA exits (the even CTA waits for both halves
            // on full[], each CTA for its own half on bfull[])
            for (int i = 0; i < STAGES2; ++i) {
                if (leader && (issued_mask & (1u << i))) drain_bar(&s.full[i], (issued_par >> i) & 1u);
                if (bissued_mask & (1u << i)) drain_bar(&s.bfull[i], (bissued_par >> i) & 1u);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && run && leader) {
            // ================= MMA issuer (even CTA) =================
            int st = 0, acc = 0;
            uint32_t aph = 0, fpar = 0, xpar = 0;  // per-stage parities of full[] and fixed[] uses
            bool ok = true;
            for (int tile = cluster; tile < total && ok; tile += nclusters) {
                const int g = tile / per_seg;
                const SegMajor mj = seg_major(p, g);
                const uint32_t idesc = idesc_bf16_f32(2 * BM, BN) | mj.idesc_bits();
                if (!wait_bar(&s.tempty[acc], aph ^ 1, abort_flag, p.err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                const int nk = s.seg.nk[g], kv = s.seg.kv[g];
                for (int kb = 0; kb < nk; ++kb) {
                    const uint32_t bit = 1u << st;
                    const bool edge = kb == nk - 1 && kv != 0;
                    // fixed[] gets the odd CTA's fixup arrival from across the cluster
                    if (!(edge ? wait_bar_cluster(&s.fixed[st], (xpar >> st) & 1u, abort_flag, p.err)
                               : wait_bar(&s.full[st], (fpar >> st) & 1u, abort_flag, p.err))) {
                        ok = false;
                        break;
                    }
                    if (edge) xpar ^= bit;
                    else fpar ^= bit;
                    tc_fence_after();
                    const uint64_t ad = mj.a_desc(smem_u32(smA(st))), bd = mj.b_desc(smem_u32(smB(st)));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_bf16_pair(d_tmem, ad + mj.a_step() * kk, bd + mj.b_step() * kk, idesc,
                                       (kb | kk) != 0 ? 1u : 0u);
                    umma_commit_pair_mc(&s.empty[st], 0x3);
                    if (++st == STAGES2) st = 0;
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
    } else if (warp == FIXUP_WARP) {
        if (run) {
            // ================= fixup (both CTAs): rows past a segment in this CTA's half ==========
            int st = 0;
            uint32_t bpar = 0;
            bool ok = true;
            for (int tile = cluster; tile < total && ok; tile += nclusters) {
                const int g = tile / per_seg;
                const int nk = s.seg.nk[g], kv = s.seg.kv[g];
                for (int kb = 0; kb < nk; ++kb) {
                    if (kb == nk - 1 && kv != 0) {
                        if (!__all_sync(0xffffffffu, wait_bar(&s.bfull[st], (bpar >> st) & 1u, abort_flag, p.err))) {
                            ok = false;
                            break;
                        }
                        bpar ^= 1u << st;
                        zero_k_tail(smA(st), 2, kv, lane);
                        zero_k_tail(smB(st), 2, kv, lane);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            if (leader) mbar_arrive(&s.fixed[st]);
                            else mbar_arrive_remote(lead_fixed + 8u * (uint32_t)st);
                        }
                    }
                    if (++st == STAGES2) st = 0;
                }
            }
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
            const bool empty_seg = s.seg.nk[g] == 0;
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

}  // namespace

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

// An operand's map. MN-major: [o.rows][o.ld] (cols columns used, a multiple of 64) seen
// as (64 columns, rows, cols / 64 chunks) with the chunks 128 bytes apart, box 64 x 64 x
// box_k / 64: one copy stages box_k columns of 64 K-rows as consecutive 8 KB chunks (K-rows
// past o.rows read as zero). K-major: [cols][o.ld] (K = o.ld), box 64 x box_k.
static bool encode_operand(CUtensorMap *m, const WgOperand &o, uint64_t cols, uint32_t box_k) {
    if (!o.p || o.ld <= 0 || (o.ld * 2) % 16 != 0 || box_k % 64 != 0 ||
        (o.mn && (o.rows <= 0 || cols % 64 != 0 || cols > (uint64_t)o.ld)))
        return false;
    if (o.mn) {
        const uint64_t dims[3] = {64u, (uint64_t)o.rows, cols / 64};
        const uint64_t strides[2] = {(uint64_t)o.ld * 2, 128u};
        const uint32_t box[3] = {64u, 64u, box_k / 64};
        return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, o.p, dims, strides, box,
                           CU_TENSOR_MAP_SWIZZLE_128B);
    }
    const uint64_t dims[2] = {(uint64_t)o.ld, cols};
    const uint64_t strides[1] = {(uint64_t)o.ld * 2};
    const uint32_t box[2] = {64u, box_k};
    return encode_tmap(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, o.p, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
}

template <typename Kern> static cudaError_t smem_attr_once(Kern kern, size_t bytes, bool &done) {
    if (done) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) done = true;
    return e;
}

cudaError_t launch_wgrad(const int32_t *offsets, int n_seg, int64_t a_rows, WgOperand A, WgOperand B, int M, int Nn,
                         void *out, WgOperand A_sh, WgOperand B_sh, int K_sh, void *out_sh, uint32_t *err,
                         cudaStream_t s, bool allow_pair, bool f32_out) {
    // CTA pairs once a 256-row output tile is not mostly empty
    const bool pair = allow_pair && M >= 2 * BM;
    if (Nn % 64 != 0 || M <= 0 || n_seg < 0 || n_seg >= MAX_SEG) return cudaErrorInvalidValue;
    WgParams p;
    memset(&p, 0, sizeof(p));
    p.offsets = offsets;
    p.n_seg = n_seg;
    p.has_sh = A_sh.p ? 1 : 0;
    p.a_rows = (int)a_rows;
    p.M = M;
    p.Nn = Nn;
    p.K_sh = K_sh;
    p.a_mn_sh = A_sh.mn ? 1 : 0;
    p.b_mn_sh = B_sh.mn ? 1 : 0;
    p.C = out;
    p.C_sh = out_sh;
    p.err = err;
    if (n_seg > 0) {
        // the routed segments' operands are the activations in their own layout
        if (!A.mn || !B.mn || !offsets) return cudaErrorInvalidValue;
        if (A.rows != a_rows || B.rows != a_rows || !encode_operand(&p.tmA, A, (uint64_t)M, BM) ||
            !encode_operand(&p.tmB, B, (uint64_t)Nn, pair ? BN / 2 : BN))
            return cudaErrorInvalidValue;
        if (pair && !encode_out_map(&p.tmC, out, Nn, M, n_seg, f32_out)) return cudaErrorInvalidValue;
    }
    if (p.has_sh) {
        // K-major operands hold K_sh (zero-padded to a multiple of 64) per row
        if ((!A_sh.mn && (A_sh.ld != K_sh || K_sh % BK)) || (!B_sh.mn && (B_sh.ld != K_sh || K_sh % BK)))
            return cudaErrorInvalidValue;
        if (K_sh <= 0 || !encode_operand(&p.tmA_sh, A_sh, (uint64_t)M, BM) ||
            !encode_operand(&p.tmB_sh, B_sh, (uint64_t)Nn, pair ? BN / 2 : BN))
            return cudaErrorInvalidValue;
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

}  // namespace moe
