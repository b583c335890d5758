// Grouped expert FFN on tcgen05 tensor cores (bf16 in, fp32 accumulate in TMEM).
//
// Each expert is an independent FFN applied to the rows dispatched to it
// ("Mixture of Experts (MoE)" glossary; "MoE: Choosing Which MLPs to Use for Each
// Token", sections "Dense MLP and MoE" and "From Router to Combine"; DeepSeekMoE
// layer equation, FFN_i). Product 1 computes the hidden activation — for gated
// experts SiLU(X W_gateᵀ) ⊙ (X W_upᵀ) fused in the epilogue from two accumulators
// of one MMA, for ReLU experts max(0, X W1ᵀ) — and product 2 the output H W_downᵀ.
// A shared expert ("Shared Expert" section, Figure 4) is one more segment of the
// same launch, with its own operands.
//
// Kernel structure (one persistent CTA per SM, 192 threads):
//   warp 0   TMA producer: A tile 128x64 and B tile 256x64 (bf16, 128-byte
//            swizzle) per k-block into a 4-stage shared-memory ring;
//   warp 1   owns the TMEM allocation (2 accumulators x 256 fp32 columns) and
//            issues tcgen05.mma 128x256x16 from one thread;
//   warps 2-5 epilogue: tcgen05.ld of the accumulator, activation, bf16 rows
//            stored straight to global memory; overlaps the next tile's MMAs.
// Tiles are enumerated on the device from the expert offsets (segment, then
// n-tile, then m-tile fastest, so CTAs running together share weight tiles in
// L2); row counts never travel to the host. Rows past a segment's end are
// computed on whatever the A rows hold and never stored. Every wait is bounded:
// after kTimeoutNs the kernel records MOE_ERR_TIMEOUT, drains its own copies and
// MMAs, frees TMEM and returns. The CTA-pair kernel further down has the same roles
// with 2-SM MMAs (256 x 256 tiles) and computes a segment's last partial row block
// with the tokens on the MMA's N side.
#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"
#include "tc_sync.cuh"

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128, BK = 64, STAGES = 4;
constexpr int BN_MMA = 256;
constexpr uint32_t A_BYTES = BM * BK * 2;
constexpr uint32_t B_BYTES = BN_MMA * BK * 2;
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int ACC_COLS = 256;
constexpr uint32_t TMEM_COLS = 512;
constexpr int NUM_THREADS = 192;
constexpr int MAX_SEG = 257;
constexpr size_t SMEM_BYTES = (size_t)STAGES * STAGE_BYTES + 1024;

// KIND_PREACT: the gated product's two accumulators stored raw (no activation), gate
// pre-activations in columns [0, n_out) and up pre-activations in [n_out, 2 n_out) of
// a 2 n_out-wide output (the backward recomputes them).
enum { KIND_GATED = 0, KIND_RELU = 1, KIND_PLAIN = 2, KIND_PREACT = 3 };
template <int KIND> constexpr bool kGatedLayout = KIND == KIND_GATED || KIND == KIND_PREACT;
template <int KIND> constexpr int kOutLd = KIND == KIND_PREACT ? 2 : 1;  // output row stride / n_out

struct TcParams {
    CUtensorMap tmA, tmA_sh;       // [rows][K], box 64 x 128
    CUtensorMap tmA64, tmA64_sh;   // the same arrays, box 64 x 64 (single-CTA half tiles)
    CUtensorMap tmB0, tmB1;        // routed weights [n_seg][n_out][K], box 64 x (128|256) x 1
    CUtensorMap tmB0_sh, tmB1_sh;  // shared weights [n_out_sh][K_sh], box 64 x (128|256)
    // Plain products only: weights MN-major, maps over [n_seg][K][n_out] and [K_sh][n_out_sh]
    // (box 64 x 64), for k < k_split from tmB0 and beyond from tmB1 at k - k_split
    // (k_split 0: tmB0 only); likewise k_split_sh for the shared segment.
    int b_mn, k_split, k_split_sh;
    const int32_t *offsets;
    int n_seg, sh_rows;
    int a_rows;                    // rows of the routed buffers; offsets are clamped to it
    int n_out, K, n_out_sh, K_sh;
    __nv_bfloat16 *C, *C_sh;
    // Gated and ReLU products: null, or where the raw pre-activations are stored too
    // (gated: gate in columns [0, n_out), up in [n_out, 2 n_out) of 2 n_out-wide rows)
    __nv_bfloat16 *P, *P_sh;
    uint32_t *err;
    // Which routed segments this launch covers: all (0); those whose last 256-row
    // block holds more than 128 rows or is full (1: the pair kernel); those whose
    // last 256-row block holds 1 to 128 rows, whole (2: the single-CTA kernel, in
    // 128-row tiles).
    int tail_mode;
};

// The rows of a routed segment a launch covers under its tail mode (all or none).
__device__ __forceinline__ void apply_tail_mode(int mode, int &rows) {
    const int tail = rows & 255;
    const bool short_tail = tail > 0 && tail <= 128;
    if ((mode == 1 && short_tail) || (mode == 2 && !short_tail)) rows = 0;
}


struct Smem {
    uint64_t full[STAGES], empty[STAGES], tfull[2], tempty[2], drain;
    uint32_t tmem_base;
    int abort_flag;
    int base[MAX_SEG + 1];  // first tile of each segment; base[nseg] = total
    int mt[MAX_SEG];        // m-tiles per segment
    int row0[MAX_SEG];      // first A row of each segment
    int rows[MAX_SEG];      // rows per segment
};

struct TileInfo {
    int seg, m, n;
    bool shared;
};

template <typename S>
__device__ __forceinline__ TileInfo decode_tile(const S &s, int nseg, int tile) {
    int lo = 0, hi = nseg - 1;  // largest g with base[g] <= tile
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s.base[mid] <= tile) lo = mid;
        else hi = mid - 1;
    }
    TileInfo ti;
    ti.seg = lo;
    const int local = tile - s.base[lo];
    ti.m = local % s.mt[lo];
    ti.n = local / s.mt[lo];
    return ti;
}

// Epilogue of one accumulator row (this thread's TMEM lane): activation, bf16,
// 16-byte stores of the output columns [col0, col0 + BN_OUT) when row_ok.
__device__ __forceinline__ void store_bf16x32(__nv_bfloat16 *dst, const uint32_t *v) {
    uint32_t packed[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        __nv_bfloat162 b = __floats2bfloat162_rn(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
        packed[i] = *reinterpret_cast<uint32_t *>(&b);
    }
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) d4[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
}

// Gated layouts: SPLIT64 = false (single-CTA kernel): accumulator columns 0-127 gate,
// 128-255 up of the tile's 128 hidden units; SPLIT64 = true (pair kernel): columns
// 0-63 gate and 64-127 up of hidden units 0-63, 128-191 gate and 192-255 up of 64-127.
template <bool SPLIT64> __device__ __forceinline__ int gate_col(int c) { return SPLIT64 ? (c >> 6) * 128 + (c & 63) : c; }
template <bool SPLIT64> __device__ __forceinline__ int up_col(int c) { return gate_col<SPLIT64>(c) + (SPLIT64 ? 64 : 128); }

// prow (gated and ReLU products): null, or the row of the pre-activation output, where
// the raw accumulators are stored as well (gated: gate at col, up at n_out + col).
template <int KIND, bool SPLIT64 = false>
__device__ __forceinline__ void epilogue_row(uint32_t tbase, __nv_bfloat16 *crow, int col0, int n_out, bool row_ok,
                                             __nv_bfloat16 *prow = nullptr) {
    if constexpr (KIND == KIND_PREACT) {
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
            uint32_t g[32], u[32];
            tmem_ld32(tbase + gate_col<SPLIT64>(c), g);
            tmem_ld32(tbase + up_col<SPLIT64>(c), u);
            tmem_ld_wait();
            const int col = col0 + c;
            if (row_ok && col < n_out) {
                store_bf16x32(crow + col, g);
                store_bf16x32(crow + n_out + col, u);
            }
        }
    } else if constexpr (KIND == KIND_GATED) {
#pragma unroll 1
        for (int c = 0; c < 128; c += 32) {
            uint32_t g[32], u[32];
            tmem_ld32(tbase + gate_col<SPLIT64>(c), g);
            tmem_ld32(tbase + up_col<SPLIT64>(c), u);
            tmem_ld_wait();
            const int col = col0 + c;
            if (prow && row_ok && col < n_out) {
                store_bf16x32(prow + col, g);
                store_bf16x32(prow + n_out + col, u);
            }
            if (row_ok && col < n_out) {
                uint32_t packed[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const float h0 = silu_f32(__uint_as_float(g[2 * i])) * __uint_as_float(u[2 * i]);
                    const float h1 = silu_f32(__uint_as_float(g[2 * i + 1])) * __uint_as_float(u[2 * i + 1]);
                    __nv_bfloat162 b = __floats2bfloat162_rn(h0, h1);
                    packed[i] = *reinterpret_cast<uint32_t *>(&b);
                }
                uint4 *dst = reinterpret_cast<uint4 *>(crow + col);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
            }
        }
    } else {
#pragma unroll 1
        for (int c = 0; c < 256; c += 32) {
            uint32_t v[32];
            tmem_ld32(tbase + c, v);
            tmem_ld_wait();
            const int col = col0 + c;
            if (KIND == KIND_RELU && prow && row_ok && col < n_out) store_bf16x32(prow + col, v);
            if (row_ok && col < n_out) {
                uint32_t packed[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    float h0 = __uint_as_float(v[2 * i]), h1 = __uint_as_float(v[2 * i + 1]);
                    if (KIND == KIND_RELU) {
                        h0 = fmaxf(h0, 0.0f);
                        h1 = fmaxf(h1, 0.0f);
                    }
                    __nv_bfloat162 b = __floats2bfloat162_rn(h0, h1);
                    packed[i] = *reinterpret_cast<uint32_t *>(&b);
                }
                uint4 *dst = reinterpret_cast<uint4 *>(crow + col);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    dst[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2], packed[4 * q + 3]);
            }
        }
    }
}

// A single-CTA tile whose 128-row block holds at most 64 rows of its segment (a segment's
// last block) runs one M = 64 MMA per k-step on a 64-row A tile: half the tensor work and
// half the A bytes. The M = 64 accumulator puts row r in TMEM lane 32 (r / 16) + r % 16,
// so epilogue warp q holds rows 16 q .. 16 q + 15 in its lanes 0-15.
__device__ __forceinline__ bool half_tile(int rows_left) { return rows_left <= BM / 2; }

template <int KIND>
__global__ void __launch_bounds__(NUM_THREADS, 1) k_ffn_tc(const __grid_constant__ TcParams p) {
    constexpr int BN_OUT = kGatedLayout<KIND> ? 128 : 256;
    __shared__ Smem s;
    extern __shared__ uint8_t dyn_smem[];
    const uint32_t dyn_base = smem_u32(dyn_smem);
    uint8_t *tiles = dyn_smem + (((dyn_base + 1023u) & ~1023u) - dyn_base);
    auto smA = [&](int st) { return tiles + (size_t)st * STAGE_BYTES; };
    auto smB = [&](int st) { return tiles + (size_t)st * STAGE_BYTES + A_BYTES; };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nseg = p.n_seg + (p.sh_rows > 0 ? 1 : 0);
    const int nt_routed = (p.n_out + BN_OUT - 1) / BN_OUT;
    const int nt_sh = (p.n_out_sh + BN_OUT - 1) / BN_OUT;

    // ---- tile table (warp 0) and barriers (thread 0) ----
    if (warp == 0) {
        pdl_wait();  // the offsets come from the router
        constexpr int PER = (MAX_SEG + 31) / 32;
        int cnt[PER];
        int sum = 0;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int g = lane * PER + i;
            int tiles_g = 0;
            if (g < nseg) {
                int r0, rows, nt;
                if (g < p.n_seg) {
                    r0 = min(max(p.offsets[g], 0), p.a_rows);
                    rows = min(max(p.offsets[g + 1], r0), p.a_rows) - r0;
                    apply_tail_mode(p.tail_mode, rows);
                    nt = nt_routed;
                } else {
                    r0 = 0;
                    rows = p.tail_mode == 2 ? 0 : p.sh_rows;
                    nt = nt_sh;
                }
                rows = max(rows, 0);
                const int mt = (rows + BM - 1) / BM;
                s.mt[g] = max(mt, 1);
                s.row0[g] = r0;
                s.rows[g] = rows;
                tiles_g = mt * nt;
            }
            cnt[i] = tiles_g;
            sum += tiles_g;
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
            if (g < nseg) s.base[g] = run;
            run += cnt[i];
        }
        if (lane == 31) s.base[nseg] = incl;
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
        tmem_alloc(&s.tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_enter();
    const uint32_t tmem_base = s.tmem_base;
    const int total = s.base[nseg];
    volatile int *abort_flag = &s.abort_flag;

    if (warp == 0) {
        // ================= TMA producer =================
        if (lane == 0) {
            int st = 0;
            uint32_t ph = 0;
            bool ok = true;
            uint32_t issued_mask = 0, issued_par = 0;  // last issue per stage
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const TileInfo ti = decode_tile(s, nseg, tile);
                const bool sh = ti.seg >= p.n_seg;
                const int K = sh ? p.K_sh : p.K;
                const int arow = s.row0[ti.seg] + ti.m * BM;
                const bool half = half_tile(s.rows[ti.seg] - ti.m * BM);
                const CUtensorMap *ta = half ? (sh ? &p.tmA64_sh : &p.tmA64) : (sh ? &p.tmA_sh : &p.tmA);
                const uint32_t tx = (half ? A_BYTES / 2 : A_BYTES) + B_BYTES;
                for (int kb = 0; kb < K / BK; ++kb) {
                    if (!wait_bar(&s.empty[st], ph ^ 1, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&s.full[st], tx);
                    const int kc = kb * BK;
                    tma_load_2d(smA(st), ta, kc, arow, &s.full[st]);
                    if (kGatedLayout<KIND>) {
                        if (sh) {
                            tma_load_2d(smB(st), &p.tmB0_sh, kc, ti.n * 128, &s.full[st]);
                            tma_load_2d(smB(st) + B_BYTES / 2, &p.tmB1_sh, kc, ti.n * 128, &s.full[st]);
                        } else {
                            tma_load_3d(smB(st), &p.tmB0, kc, ti.n * 128, ti.seg, &s.full[st]);
                            tma_load_3d(smB(st) + B_BYTES / 2, &p.tmB1, kc, ti.n * 128, ti.seg, &s.full[st]);
                        }
                    } else if (p.b_mn) {
                        // MN-major weights: four 64-column chunks of 64 K-rows
                        const int ks = sh ? p.k_split_sh : p.k_split;
                        const bool hi = ks > 0 && kc >= ks;
                        const int kq = hi ? kc - ks : kc;
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            if (sh) tma_load_2d(smB(st) + j * 8192, hi ? &p.tmB1_sh : &p.tmB0_sh, ti.n * 256 + 64 * j, kq,
                                                &s.full[st]);
                            else tma_load_3d(smB(st) + j * 8192, hi ? &p.tmB1 : &p.tmB0, ti.n * 256 + 64 * j, kq, ti.seg,
                                             &s.full[st]);
                        }
                    } else {
                        if (sh) tma_load_2d(smB(st), &p.tmB0_sh, kc, ti.n * 256, &s.full[st]);
                        else tma_load_3d(smB(st), &p.tmB0, kc, ti.n * 256, ti.seg, &s.full[st]);
                    }
                    issued_mask |= 1u << st;
                    issued_par = (issued_par & ~(1u << st)) | (ph << st);
                    if (++st == STAGES) {
                        st = 0;
                        ph ^= 1;
                    }
                }
            }
            // every load issued has landed before the CTA exits (immediate unless aborted)
            for (int i = 0; i < STAGES; ++i)
                if (issued_mask & (1u << i)) drain_bar(&s.full[i], (issued_par >> i) & 1u);
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN_MMA);
            constexpr uint32_t IDESC64 = idesc_bf16_f32(BM / 2, BN_MMA);
            int st = 0, acc = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < total && ok; tile += gridDim.x) {
                const TileInfo ti = decode_tile(s, nseg, tile);
                const int K = ti.seg >= p.n_seg ? p.K_sh : p.K;
                const uint32_t idesc =
                    (half_tile(s.rows[ti.seg] - ti.m * BM) ? IDESC64 : IDESC) | (p.b_mn ? kIdescBMajorMN : 0u);
                const uint64_t bstep = p.b_mn ? 128u : 2u;  // descriptor units (16 B) per K step of 16
                if (!wait_bar(&s.tempty[acc], aph ^ 1, abort_flag, p.err)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * ACC_COLS);
                for (int kb = 0; kb < K / BK; ++kb) {
                    if (!wait_bar(&s.full[st], ph, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = desc_sw128(smem_u32(smA(st)));
                    const uint64_t bd = p.b_mn ? desc_sw128_mn(smem_u32(smB(st))) : desc_sw128(smem_u32(smB(st)));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_bf16(d_tmem, ad + (uint64_t)(2 * kk), bd + bstep * (uint64_t)kk, idesc,
                                  (kb | kk) != 0 ? 1u : 0u);
                    umma_commit(&s.empty[st]);
                    if (++st == STAGES) {
                        st = 0;
                        ph ^= 1;
                    }
                }
                if (!ok) break;
                umma_commit(&s.tfull[acc]);
                if (++acc == 2) {
                    acc = 0;
                    aph ^= 1;
                }
            }
            // all MMAs issued by this thread complete before TMEM is released
            umma_commit(&s.drain);
            drain_bar(&s.drain, 0);
        }
    } else {
        // ================= epilogue (warps 2..5) =================
        const int quarter = warp & 3;  // TMEM lanes this warp may access
        int acc = 0;
        uint32_t aph = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            const TileInfo ti = decode_tile(s, nseg, tile);
            const bool sh = ti.seg >= p.n_seg;
            if (!wait_bar(&s.tfull[acc], aph, abort_flag, p.err)) break;
            tc_fence_after();
            const int rows = s.rows[ti.seg] - ti.m * BM;
            const bool half = half_tile(rows);
            const int r_in_tile = half ? quarter * 16 + lane : quarter * 32 + lane;
            const bool row_ok = (!half || lane < 16) && r_in_tile < rows;
            const int64_t orow = (int64_t)s.row0[ti.seg] + ti.m * BM + r_in_tile;
            const int n_out = sh ? p.n_out_sh : p.n_out;
            __nv_bfloat16 *crow = (sh ? p.C_sh : p.C) + orow * n_out * kOutLd<KIND>;
            __nv_bfloat16 *P = sh ? p.P_sh : p.P;
            __nv_bfloat16 *prow = P ? P + orow * n_out * (KIND == KIND_GATED ? 2 : 1) : nullptr;
            const uint32_t tbase = tmem_base + (uint32_t)(acc * ACC_COLS) + ((uint32_t)(quarter * 32) << 16);
            epilogue_row<KIND>(tbase, crow, ti.n * BN_OUT, n_out, row_ok, prow);
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
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ CTA-pair kernel
//
// Same computation with 2-CTA (cta_group::2) MMAs: a cluster of two CTAs on two
// SMs computes a 256 x 256 tile per MMA 256x256x16. Each CTA stages its own 128
// rows of A and 128 of the 256 B rows, so each SM moves a third less operand data
// per FLOP than the single-CTA kernel. Gated experts: CTA r stages the gate rows and
// then the up rows of hidden units 64r .. 64r+63 of the tile's 128, so accumulator
// columns 0-63 / 64-127 are gate / up of units 0-63 and 128-191 / 192-255 those of
// 64-127. Both CTAs' loads complete on the even CTA's stage barrier, the even CTA
// issues the MMAs and its commits arrive on both CTAs' barriers (multicast); each
// CTA's TMEM holds its own 128 accumulator rows and its epilogue stores them.
//
// Last blocks. A segment of r = 256 q + t rows has q full 256-row blocks and t rows
// left. With 0 < t < 256 those t rows are not a partly empty 256-row tile but a tile
// with the weights on the MMA's M side and the tokens on its N side,
//   D[256 weight rows][t' tokens] = W[256][64] · X_tail[t'][64]ᵀ,  t' = t rounded up to 16,
// whose MMAs cost t'/256 of a row tile's; the tokens are staged where a row tile's
// token rows go (t'/2 per CTA) and the weights as for a row tile, so the tile follows
// the segment's full blocks in the tile order and finds their weights in L2. Its
// epilogue turns the transposed result (one lane per weight row, one column per token)
// back into rows (gated: the up lanes hand their values to the gate lanes of the same
// units through shared memory, bounded mbarrier handshakes).
constexpr int STAGES2 = 6;
constexpr uint32_t HALF_BYTES = 128 * BK * 2;            // 16 KB: 128 rows x 64 bf16
constexpr uint32_t STAGE2_BYTES = 2 * HALF_BYTES;
constexpr int XSTRIDE2 = 33;                              // exchange buffer row stride (fp32)
constexpr uint32_t XBUF2_BYTES = 32 * XSTRIDE2 * 4;       // one warp's 32 lanes x 32 tokens
constexpr size_t SMEM2_BYTES = 1024 + (size_t)STAGES2 * STAGE2_BYTES + 2 * XBUF2_BYTES;

enum { TILE_ROW = 0, TILE_TAIL = 1 };

struct Smem2 {
    uint64_t full[STAGES2], empty[STAGES2], tfull[2], tempty[2], drain;
    uint64_t xfull[2], xempty[2];  // gated tail exchange, per (gate warp, up warp) pair
    uint32_t tmem_base;
    int abort_flag;
    int base[MAX_SEG + 1];
    int mt[MAX_SEG];
    int row0[MAX_SEG];
    int rows[MAX_SEG];
};
static_assert(SMEM2_BYTES + sizeof(Smem2) <= 232448, "shared memory budget of one CTA");

struct Tile2 {
    int seg, m, n;
    int type;   // TILE_ROW: rows [256 m, 256 m + 256); TILE_TAIL: rows [256 q, 256 q + tail)
    int tail;   // tail rows (TILE_TAIL)
    int tpad;   // tail rounded up to 16: the tail MMA's N (t'/2 rows per CTA, whole 8-row groups)
};

// Tiles per n-tile of a segment of `rows` rows: its full blocks and a tail tile.
__device__ __forceinline__ int pair_tiles(int rows) { return (rows >> 8) + ((rows & 255) ? 1 : 0); }

__device__ __forceinline__ Tile2 decode_tile2(const Smem2 &s, int nseg, int tile) {
    const TileInfo ti = decode_tile(s, nseg, tile);
    Tile2 t2;
    t2.seg = ti.seg;
    t2.m = ti.m;
    t2.n = ti.n;
    const int rows = s.rows[ti.seg];
    t2.type = ti.m == (rows >> 8) ? TILE_TAIL : TILE_ROW;
    t2.tail = t2.type == TILE_TAIL ? rows & 255 : 0;
    t2.tpad = (t2.tail + 15) & ~15;
    return t2;
}

// Tail epilogue of one warp (TMEM lane quarter q of CTA `rank`): the accumulator holds
// one weight row per lane and one tail token per column (tokens [0, tpad)).
// pre (gated and ReLU products): null, or the pre-activation output, where the raw
// accumulators are stored as well (gated rows 2 n_out wide: gate, then up).
template <int KIND>
__device__ __forceinline__ bool epilogue_tail(Smem2 &s, uint8_t *xbufs, uint32_t tbase, const Tile2 &t,
                                              int64_t row_tail0, __nv_bfloat16 *out, int n_out, uint32_t rank,
                                              int q, int lane, uint32_t &xcount, volatile int *abort_flag,
                                              uint32_t *err, __nv_bfloat16 *pre = nullptr) {
    const int nchunks = (t.tpad + 31) >> 5;  // the last chunk's columns past t' are never stored
    if constexpr (KIND == KIND_GATED || KIND == KIND_PREACT) {
        // lanes of quarters 0-1: gate rows, 2-3: up rows of hidden units 64 rank + 32 (q & 1) + lane
        const bool is_gate = q < 2;
        const int pidx = q & 1;
        const int hcol = t.n * 128 + (int)rank * 64 + pidx * 32 + lane;
        const bool col_ok = hcol < n_out;
        float *xb = reinterpret_cast<float *>(xbufs + (size_t)pidx * XBUF2_BYTES);
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
            uint32_t v[32];
            tmem_ld32(tbase + (uint32_t)(c * 32), v);
            tmem_ld_wait();
            if constexpr (KIND == KIND_PREACT) {
                // raw pre-activations: gate in columns [0, n_out), up in [n_out, 2 n_out)
                const int col = hcol + (is_gate ? 0 : n_out);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int j = c * 32 + i;
                    if (col_ok && j < t.tail)
                        out[(row_tail0 + j) * (2 * (int64_t)n_out) + col] = __float2bfloat16_rn(__uint_as_float(v[i]));
                }
            } else {
                if (pre) {
                    // raw gate (quarters 0-1) or up (quarters 2-3) pre-activations of unit hcol
                    const int col = hcol + (is_gate ? 0 : n_out);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int j = c * 32 + i;
                        if (col_ok && j < t.tail)
                            pre[(row_tail0 + j) * (2 * (int64_t)n_out) + col] = __float2bfloat16_rn(__uint_as_float(v[i]));
                    }
                }
                const uint32_t ph = xcount & 1u;
                ++xcount;
                if (!is_gate) {
                    // up warp: hand this chunk's values to the gate warp of the same units
                    if (!wait_bar(&s.xempty[pidx], ph ^ 1u, abort_flag, err)) return false;
#pragma unroll
                    for (int i = 0; i < 32; ++i) xb[lane * XSTRIDE2 + i] = __uint_as_float(v[i]);
                    mbar_arrive(&s.xfull[pidx]);
                } else {
                    if (!wait_bar(&s.xfull[pidx], ph, abort_flag, err)) return false;
                    float u[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) u[i] = xb[lane * XSTRIDE2 + i];
                    mbar_arrive(&s.xempty[pidx]);
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int j = c * 32 + i;
                        if (col_ok && j < t.tail)
                            out[(row_tail0 + j) * (int64_t)n_out + hcol] =
                                __float2bfloat16_rn(silu_f32(__uint_as_float(v[i])) * u[i]);
                    }
                }
            }
        }
    } else {
        // one output column per lane: 256 n + 128 rank + 32 q + lane
        const int ocol = t.n * 256 + (int)rank * 128 + q * 32 + lane;
        const bool col_ok = ocol < n_out;
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
            uint32_t v[32];
            tmem_ld32(tbase + (uint32_t)(c * 32), v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int j = c * 32 + i;
                float x = __uint_as_float(v[i]);
                if (KIND == KIND_RELU && pre && col_ok && j < t.tail)
                    pre[(row_tail0 + j) * (int64_t)n_out + ocol] = __float2bfloat16_rn(x);
                if (KIND == KIND_RELU) x = fmaxf(x, 0.0f);
                if (col_ok && j < t.tail) out[(row_tail0 + j) * (int64_t)n_out + ocol] = __float2bfloat16_rn(x);
            }
        }
    }
    return true;
}

template <int KIND>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    k_ffn_tc2(const __grid_constant__ TcParams p) {
    constexpr int BN_OUT = kGatedLayout<KIND> ? 128 : 256;
    __shared__ Smem2 s;
    extern __shared__ uint8_t dyn_smem[];
    const uint32_t dyn_base = smem_u32(dyn_smem);
    uint8_t *tiles = dyn_smem + (((dyn_base + 1023u) & ~1023u) - dyn_base);
    auto smA = [&](int st) { return tiles + (size_t)st * STAGE2_BYTES; };
    auto smB = [&](int st) { return tiles + (size_t)st * STAGE2_BYTES + HALF_BYTES; };
    uint8_t *xbufs = tiles + (size_t)STAGES2 * STAGE2_BYTES;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    const int nseg = p.n_seg + (p.sh_rows > 0 ? 1 : 0);
    const int nt_routed = (p.n_out + BN_OUT - 1) / BN_OUT;
    const int nt_sh = (p.n_out_sh + BN_OUT - 1) / BN_OUT;

    // ---- tile table and barriers ----
    if (warp == 0) {
        pdl_wait();  // the offsets come from the router
        constexpr int PER = (MAX_SEG + 31) / 32;
        int cnt[PER];
        int sum = 0;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int g = lane * PER + i;
            int tiles_g = 0;
            if (g < nseg) {
                int r0, rows, nt;
                if (g < p.n_seg) {
                    r0 = min(max(p.offsets[g], 0), p.a_rows);
                    rows = min(max(p.offsets[g + 1], r0), p.a_rows) - r0;
                    apply_tail_mode(p.tail_mode, rows);
                    nt = nt_routed;
                } else {
                    r0 = 0;
                    rows = p.tail_mode == 2 ? 0 : p.sh_rows;
                    nt = nt_sh;
                }
                rows = max(rows, 0);
                const int mt = pair_tiles(rows);
                s.mt[g] = max(mt, 1);
                s.row0[g] = r0;
                s.rows[g] = rows;
                tiles_g = mt * nt;
            }
            cnt[i] = tiles_g;
            sum += tiles_g;
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
            if (g < nseg) s.base[g] = run;
            run += cnt[i];
        }
        if (lane == 31) s.base[nseg] = incl;
        if (lane == 0) {
            for (int i = 0; i < STAGES2; ++i) {
                mbar_init(&s.full[i], 1);
                mbar_init(&s.empty[i], 1);
            }
            for (int i = 0; i < 2; ++i) {
                mbar_init(&s.tfull[i], 1);
                mbar_init(&s.tempty[i], 8);  // 4 epilogue warps of each CTA
                mbar_init(&s.xfull[i], 32);  // the 32 lanes of an up warp
                mbar_init(&s.xempty[i], 32); // the 32 lanes of a gate warp
            }
            mbar_init(&s.drain, 1);
            s.abort_flag = 0;
            fence_mbar_init();
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(&s.tmem_base, 2 * ACC_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after();
    pdl_enter();
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
    const int total = s.base[nseg];
    volatile int *abort_flag = &s.abort_flag;
    const uint32_t lead_tempty = map_to_rank(smem_u32(&s.tempty[0]), 0);

    if (warp == 0) {
        // ================= TMA producer (both CTAs) =================
        // Both CTAs' loads complete on the even CTA's full[] barrier, which the even
        // CTA's producer arms with the bytes of both halves.
        if (lane == 0 && run) {
            int st = 0;
            uint32_t ph = 0;
            bool ok = true;
            uint32_t issued_mask = 0, issued_par = 0;
            const uint32_t lead_full = map_to_rank(smem_u32(&s.full[0]), 0);
            for (int tile = cluster; tile < total && ok; tile += nclusters) {
                const Tile2 t = decode_tile2(s, nseg, tile);
                const bool sh = t.seg >= p.n_seg;
                const int K = sh ? p.K_sh : p.K;
                // token rows of this CTA: 128 of a row tile, or t'/2 of the tail (the box
                // loads 128; the MMA reads the first t'/2)
                const int arow = s.row0[t.seg] + t.m * 2 * BM +
                                 (int)rank * (t.type == TILE_TAIL ? (t.tpad >> 1) : BM);
                const CUtensorMap *ta = sh ? &p.tmA_sh : &p.tmA;
                for (int kb = 0; kb < K / BK; ++kb) {
                    if (!wait_bar(&s.empty[st], ph ^ 1, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = lead_full + 8u * (uint32_t)st;
                    if (leader) mbar_arrive_expect_tx(&s.full[st], 2 * STAGE2_BYTES);
                    const int kc = kb * BK;
                    tma_load_2d_pair(smA(st), ta, kc, arow, fb);
                    if (kGatedLayout<KIND>) {
                        // gate rows then up rows of hidden units 128 n + 64 rank .. + 63
                        const int wrow = t.n * 128 + (int)rank * 64;
                        if (sh) {
                            tma_load_2d_pair(smB(st), &p.tmB0_sh, kc, wrow, fb);
                            tma_load_2d_pair(smB(st) + HALF_BYTES / 2, &p.tmB1_sh, kc, wrow, fb);
                        } else {
                            tma_load_3d_pair(smB(st), &p.tmB0, kc, wrow, t.seg, fb);
                            tma_load_3d_pair(smB(st) + HALF_BYTES / 2, &p.tmB1, kc, wrow, t.seg, fb);
                        }
                    } else if (p.b_mn) {
                        // MN-major weights: this CTA's 128 columns as two chunks of 64 K-rows
                        const int brow = t.n * 256 + (int)rank * 128;
                        const int ks = sh ? p.k_split_sh : p.k_split;
                        const bool hi = ks > 0 && kc >= ks;
                        const int kq = hi ? kc - ks : kc;
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            if (sh) tma_load_2d_pair(smB(st) + j * 8192, hi ? &p.tmB1_sh : &p.tmB0_sh, brow + 64 * j, kq,
                                                     fb);
                            else tma_load_3d_pair(smB(st) + j * 8192, hi ? &p.tmB1 : &p.tmB0, brow + 64 * j, kq, t.seg,
                                                  fb);
                        }
                    } else {
                        const int brow = t.n * 256 + (int)rank * 128;
                        if (sh) tma_load_2d_pair(smB(st), &p.tmB0_sh, kc, brow, fb);
                        else tma_load_3d_pair(smB(st), &p.tmB0, kc, brow, t.seg, fb);
                    }
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
            constexpr uint32_t IDESC = idesc_bf16_f32(2 * BM, BN_MMA);
            int st = 0, acc = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            for (int tile = cluster; tile < total && ok; tile += nclusters) {
                const Tile2 t = decode_tile2(s, nseg, tile);
                const int K = t.seg >= p.n_seg ? p.K_sh : p.K;
                const bool tail = t.type == TILE_TAIL;
                // a tail tile: the weights (B stage) as the M side, the tokens as N; MN-major
                // weights mark that side of the MMA as MN-major
                const uint32_t idesc = (tail ? idesc_bf16_f32(2 * BM, t.tpad) : IDESC) |
                                       (p.b_mn ? (tail ? kIdescAMajorMN : kIdescBMajorMN) : 0u);
                const uint64_t wstep = p.b_mn ? 128u : 2u;  // descriptor units per K step of 16 (weights)
                if (!wait_bar(&s.tempty[acc], aph ^ 1, abort_flag, p.err)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * ACC_COLS);
                for (int kb = 0; kb < K / BK; ++kb) {
                    if (!wait_bar(&s.full[st], ph, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = desc_sw128(smem_u32(smA(st)));
                    const uint64_t bd = p.b_mn ? desc_sw128_mn(smem_u32(smB(st))) : desc_sw128(smem_u32(smB(st)));
                    const uint64_t m_side = tail ? bd : ad, n_side = tail ? ad : bd;
                    const uint64_t m_step = tail ? wstep : 2u, n_step = tail ? 2u : wstep;
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_bf16_pair(d_tmem, m_side + m_step * (uint64_t)kk, n_side + n_step * (uint64_t)kk, idesc,
                                       (kb | kk) != 0 ? 1u : 0u);
                    umma_commit_pair_mc(&s.empty[st], 0x3);
                    if (++st == STAGES2) {
                        st = 0;
                        ph ^= 1;
                    }
                }
                if (!ok) break;
                umma_commit_pair_mc(&s.tfull[acc], 0x3);
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
        const int r_in_tile = quarter * 32 + lane;
        int acc = 0;
        uint32_t aph = 0, xcount = 0;
        for (int tile = cluster; tile < total; tile += nclusters) {
            const Tile2 t = decode_tile2(s, nseg, tile);
            const bool sh = t.seg >= p.n_seg;
            const int n_out = sh ? p.n_out_sh : p.n_out;
            __nv_bfloat16 *C = sh ? p.C_sh : p.C;
            __nv_bfloat16 *P = sh ? p.P_sh : p.P;
            if (!wait_bar(&s.tfull[acc], aph, abort_flag, p.err)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (uint32_t)(acc * ACC_COLS) + ((uint32_t)(quarter * 32) << 16);
            if (t.type == TILE_ROW) {
                const int r_seg = t.m * 2 * BM + (int)rank * BM + r_in_tile;  // row within the segment
                const bool row_ok = r_seg < s.rows[t.seg];
                const int64_t orow = (int64_t)s.row0[t.seg] + r_seg;
                __nv_bfloat16 *prow = P ? P + orow * n_out * (KIND == KIND_GATED ? 2 : 1) : nullptr;
                epilogue_row<KIND, true>(tbase, C + orow * n_out * kOutLd<KIND>, t.n * BN_OUT, n_out, row_ok, prow);
            } else {
                const int64_t row_tail0 = (int64_t)s.row0[t.seg] + t.m * 2 * BM;
                if (!epilogue_tail<KIND>(s, xbufs, tbase, t, row_tail0, C, n_out, rank, quarter, lane, xcount,
                                         abort_flag, p.err, P))
                    break;
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
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the pair's MMAs and both epilogues are done with TMEM
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, 2 * ACC_COLS);
    }
}

// ------------------------------------------------------------------ host side

template <int KIND>
cudaError_t launch_kind(const TcParams &p, int64_t max_tiles, cudaStream_t s) {
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e =
            cudaFuncSetAttribute(k_ffn_tc<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(max_tiles, device_sm_count()));
    return launch_pdl(k_ffn_tc<KIND>, dim3(grid), dim3(NUM_THREADS), SMEM_BYTES, s, p);
}

template <int KIND>
cudaError_t launch_kind2(const TcParams &p, int64_t max_tiles, cudaStream_t s) {
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e =
            cudaFuncSetAttribute(k_ffn_tc2<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM2_BYTES);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    const int clusters = (int)std::max<int64_t>(1, std::min<int64_t>(max_tiles, device_sm_count() / 2));
    return launch_pdl(k_ffn_tc2<KIND>, dim3(2 * clusters), dim3(NUM_THREADS), SMEM2_BYTES, s, p);
}

// One product over the routed segments and/or the shared segment.
//   a / a_sh: A operands ([a_rows][K] / [sh_rows][K_sh]);
//   b0,b1 / b0_sh,b1_sh: weights ([n_seg][n_out][K] / [n_out_sh][K_sh]);
//   out / out_sh: outputs ([a_rows][n_out] / [sh_rows][n_out_sh]).
// pair: run the CTA-pair kernel (256-row tiles) instead of the single-CTA one.
//   b_mn (plain products only): the weights are MN-major, b0 [n_seg][K or k_split][n_out]
//   and, with k_split > 0, b1 [n_seg][K - k_split][n_out] for k >= k_split (likewise
//   b0_sh / b1_sh with k_split_sh).
template <int KIND>
cudaError_t product(const int32_t *offsets, int n_seg, int64_t a_rows, const void *a, const void *b0,
                    const void *b1, int K, int n_out, void *out, int sh_rows, const void *a_sh,
                    const void *b0_sh, const void *b1_sh, int K_sh, int n_out_sh, void *out_sh,
                    uint32_t *err, cudaStream_t s, bool pair, bool b_mn = false, int k_split = 0,
                    int k_split_sh = 0, void *pre = nullptr, void *pre_sh = nullptr) {
    if (b_mn && KIND != KIND_PLAIN) return cudaErrorInvalidValue;
    if ((pre || pre_sh) && KIND != KIND_GATED && KIND != KIND_RELU) return cudaErrorInvalidValue;
    constexpr int BN_OUT = kGatedLayout<KIND> ? 128 : 256;
    // weight rows per TMA box: the single-CTA kernel stages 256 rows (gated: 128 gate +
    // 128 up), the pair kernel 128 per CTA (gated: 64 gate + 64 up)
    const uint32_t box_b = kGatedLayout<KIND> ? (pair ? 64 : 128) : (pair ? 128 : 256);
    const int64_t tm = pair ? 2 * BM : BM;
    TcParams p;
    memset(&p, 0, sizeof(p));
    p.offsets = offsets;
    p.n_seg = n_seg;
    p.sh_rows = sh_rows;
    p.a_rows = (int)a_rows;
    p.n_out = n_out;
    p.K = K;
    p.n_out_sh = n_out_sh;
    p.K_sh = K_sh;
    p.C = static_cast<__nv_bfloat16 *>(out);
    p.C_sh = static_cast<__nv_bfloat16 *>(out_sh);
    p.P = static_cast<__nv_bfloat16 *>(pre);
    p.P_sh = static_cast<__nv_bfloat16 *>(pre_sh);
    p.err = err;
    p.b_mn = b_mn ? 1 : 0;
    p.k_split = b_mn ? k_split : 0;
    p.k_split_sh = b_mn ? k_split_sh : 0;
    if (b_mn && (k_split < 0 || k_split % BK || k_split >= K || k_split_sh < 0 || k_split_sh % BK ||
                 (sh_rows > 0 && k_split_sh >= K_sh)))
        return cudaErrorInvalidValue;
    // MN-major weight maps: [n_exp][rows of K][n_out], box 64 columns x 64 K-rows
    auto mn_maps = [&](CUtensorMap *m0, CUtensorMap *m1, const void *w0, const void *w1, int Kt, int ks, int no,
                       int nexp) {
        const int k0 = ks > 0 ? ks : Kt;
        if (nexp > 0) {
            if (!encode_bf16_3d(m0, w0, no, k0, nexp, BK)) return false;
            if (ks > 0 && !encode_bf16_3d(m1, w1, no, Kt - ks, nexp, BK)) return false;
        } else {
            if (!encode_bf16_2d(m0, w0, no, k0, BK)) return false;
            if (ks > 0 && !encode_bf16_2d(m1, w1, no, Kt - ks, BK)) return false;
        }
        return true;
    };
    int64_t max_tiles = 0;
    if (n_seg > 0) {
        if (!encode_bf16_2d(&p.tmA, a, K, a_rows, BM)) return cudaErrorInvalidValue;
        if (!encode_bf16_2d(&p.tmA64, a, K, a_rows, BM / 2)) return cudaErrorInvalidValue;
        if (b_mn) {
            if (!mn_maps(&p.tmB0, &p.tmB1, b0, b1, K, k_split, n_out, n_seg)) return cudaErrorInvalidValue;
        } else {
            if (!encode_bf16_3d(&p.tmB0, b0, K, n_out, n_seg, box_b)) return cudaErrorInvalidValue;
            if (kGatedLayout<KIND> && !encode_bf16_3d(&p.tmB1, b1, K, n_out, n_seg, box_b))
                return cudaErrorInvalidValue;
        }
        max_tiles += ((a_rows + tm - 1) / tm + n_seg) * ((n_out + BN_OUT - 1) / BN_OUT);
    }
    if (sh_rows > 0) {
        if (!encode_bf16_2d(&p.tmA_sh, a_sh, K_sh, sh_rows, BM)) return cudaErrorInvalidValue;
        if (!encode_bf16_2d(&p.tmA64_sh, a_sh, K_sh, sh_rows, BM / 2)) return cudaErrorInvalidValue;
        if (b_mn) {
            if (!mn_maps(&p.tmB0_sh, &p.tmB1_sh, b0_sh, b1_sh, K_sh, k_split_sh, n_out_sh, 0))
                return cudaErrorInvalidValue;
        } else {
            if (!encode_bf16_2d(&p.tmB0_sh, b0_sh, K_sh, n_out_sh, box_b)) return cudaErrorInvalidValue;
            if (kGatedLayout<KIND> && !encode_bf16_2d(&p.tmB1_sh, b1_sh, K_sh, n_out_sh, box_b))
                return cudaErrorInvalidValue;
        }
        max_tiles += ((int64_t)(sh_rows + tm - 1) / tm) * ((n_out_sh + BN_OUT - 1) / BN_OUT);
    }
    if (max_tiles == 0) return cudaSuccess;
    if (!pair) return launch_kind<KIND>(p, max_tiles, s);
    // With few rows per expert (under 512 on average) a short last block is a large
    // share of the work: an expert whose last 256-row block holds at most 128 rows then
    // runs whole on the single-CTA kernel (128-row tiles), the others on the pair kernel,
    // so that no expert's weights are streamed by both launches (measured on the
    // DeepSeek-shaped layer against the pair kernel's tail tiles alone: 7.97-8.03 vs
    // 8.17-8.23 ms per forward).
    const bool split = n_seg > 0 && a_rows < 512LL * n_seg;
    p.tail_mode = split ? 1 : 0;
    cudaError_t e = launch_kind2<KIND>(p, max_tiles, s);
    if (e != cudaSuccess || !split) return e;
    TcParams q = p;
    q.tail_mode = 2;
    q.sh_rows = 0;
    if (!b_mn) {  // the single-CTA kernel stages 256 weight rows per K-major box (MN-major maps serve both)
        if (!encode_bf16_3d(&q.tmB0, b0, K, n_out, n_seg, kGatedLayout<KIND> ? 128 : 256))
            return cudaErrorInvalidValue;
        if (kGatedLayout<KIND> && !encode_bf16_3d(&q.tmB1, b1, K, n_out, n_seg, 128)) return cudaErrorInvalidValue;
    }
    return launch_kind<KIND>(q, ((a_rows + BM - 1) / BM + n_seg) * ((n_out + BN_OUT - 1) / BN_OUT), s);
}

}  // namespace

cudaError_t launch_gemm_rows(const moe_config &c, bool preact, const int32_t *offsets, int n_seg, int64_t a_rows,
                             const void *a, const void *b0, const void *b1, int K, int n_out, void *out, int sh_rows,
                             const void *a_sh, const void *b0_sh, const void *b1_sh, int K_sh, int n_out_sh,
                             void *out_sh, uint32_t *err, cudaStream_t s, bool b_mn, int k_split, int k_split_sh) {
    bool pair = n_seg > 0 && a_rows >= 224LL * n_seg;
    if (c.debug_flags & MOE_DEBUG_FFN_PAIR) pair = true;
    if (c.debug_flags & MOE_DEBUG_FFN_SINGLE) pair = false;
    if (preact) {
        if (b_mn) return cudaErrorInvalidValue;
        return product<KIND_PREACT>(offsets, n_seg, a_rows, a, b0, b1, K, n_out, out, sh_rows, a_sh, b0_sh, b1_sh,
                                    K_sh, n_out_sh, out_sh, err, s, pair);
    }
    return product<KIND_PLAIN>(offsets, n_seg, a_rows, a, b0, b1, K, n_out, out, sh_rows, a_sh, b0_sh, b1_sh, K_sh,
                               n_out_sh, out_sh, err, s, pair, b_mn, k_split, k_split_sh);
}

cudaError_t launch_ffn_tc(const moe_config &c, const FfnGroup &g, uint32_t *err, cudaStream_t s) {
    if (c.debug_flags & MOE_DEBUG_FFN_SWAP) return launch_ffn_sw(c, g, err, s);
    // CTA-pair tiles hold 256 rows of one segment. Measured on B300, the pair
    // kernel wins from about 256 rows per expert on average (DeepSeek-shaped
    // layer: 8.70 vs 9.27 ms per forward, even with half of its last tiles
    // empty); with a few rows per expert the single-CTA kernel's 128-row tiles
    // waste less.
    bool pair = g.n_seg > 0 && g.a_rows >= 224LL * g.n_seg;
    if (c.debug_flags & MOE_DEBUG_FFN_PAIR) pair = true;
    if (c.debug_flags & MOE_DEBUG_FFN_SINGLE) pair = false;
    cudaError_t e;
    // product 1: hidden activations
    if (g.act == MOE_ACT_SILU_GATED) {
        e = product<KIND_GATED>(g.offsets, g.n_seg, g.a_rows, g.a, g.w_a, g.w_b, c.d, g.h, g.hid, g.sh_rows,
                                g.sh_a, g.sh_w_gate, g.sh_w_up, c.d, g.h_sh, g.sh_hid, err, s, pair, false, 0, 0,
                                g.pre, g.sh_pre);
    } else {
        e = product<KIND_RELU>(g.offsets, g.n_seg, g.a_rows, g.a, g.w_a, nullptr, c.d, g.h, g.hid, 0, nullptr,
                               nullptr, nullptr, 0, 0, nullptr, err, s, pair, false, 0, 0, g.pre, nullptr);
        if (e == cudaSuccess && g.sh_rows > 0)
            e = product<KIND_GATED>(nullptr, 0, 0, nullptr, nullptr, nullptr, 0, 0, nullptr, g.sh_rows, g.sh_a,
                                    g.sh_w_gate, g.sh_w_up, c.d, g.h_sh, g.sh_hid, err, s, false, false, 0, 0,
                                    nullptr, g.sh_pre);
    }
    if (e != cudaSuccess) return e;
    if (g.mid_event && (e = cudaEventRecordWithFlags(g.mid_event, s, g.event_flags)) != cudaSuccess) return e;
    // product 2: outputs
    return product<KIND_PLAIN>(g.offsets, g.n_seg, g.a_rows, g.hid, g.w_out, nullptr, g.h, c.d, g.out,
                               g.sh_rows, g.sh_hid, g.sh_w_down, nullptr, g.h_sh, c.d, g.sh_out, err, s, pair);
}

}  // namespace moe
