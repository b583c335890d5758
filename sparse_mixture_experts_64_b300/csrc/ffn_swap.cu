// Grouped expert FFN with the weights on the MMA's M side (CTA pair, tcgen05
// cta_group::2, bf16 in, fp32 accumulate in TMEM).
//
// The products are those of ffn_tc.cu ("MoE: Choosing Which MLPs to Use for Each
// Token", sections "Dense MLP and MoE" and "From Router to Combine"; DeepSeekMoE
// layer equation, FFN_i; "Shared Expert" section, Figure 4): product 1 gives the
// hidden activation SiLU(X W_gateᵀ) ⊙ (X W_upᵀ) (ReLU experts: max(0, X W1ᵀ)) and
// product 2 the output H W_downᵀ. Here each MMA computes a transposed tile:
//
//   D[256 weight rows][N tokens] = W[256][K] · X[N][K]ᵀ,  N = 32 .. 256, step 32.
//
// The weight rows are the M side (128 per CTA of the pair) and one expert's tokens
// are the N side (N/2 per CTA), so a tile holds any multiple of 32 tokens: an
// expert with r rows is covered by ceil(r/256) tiles of equal size and wastes
// fewer than 32 token columns per tile, where fixed 128- or 256-row token tiles
// waste up to a whole tile (a quarter of the MMA work at 256 rows per expert).
//
//   gated  : CTA r holds gate rows and up rows of the same 64 hidden units
//            h0 + 64r .. h0 + 64r + 63 as its 128 M rows (TMEM lanes 0-63 gate,
//            64-127 up); the epilogue warps of lanes 0-63 and 64-127 swap half of
//            their token columns through shared memory, so each computes
//            SiLU(gate)·up for 16 of every 32 tokens.
//   plain  : CTA r holds 128 output rows o0 + 128r .. o0 + 128r + 127.
//
// Warp roles per CTA (192 threads): warp 0 TMA producer (both CTAs load their own
// halves; the loads complete on the even CTA's stage barrier), warp 1 TMEM owner
// and, in the even CTA, the MMA issuer; warps 2-5 epilogue. The epilogue turns a
// 32 x 32 block of the accumulator (rows x tokens) around in shared memory so that
// each token's 32 outputs (64 bytes) are stored contiguously.
//
// Tiles are enumerated on the device from the expert offsets: segment, then weight
// block, then token tile fastest, so the clusters running together read the same
// weight block. Every wait is bounded (tc_sync.cuh); after a timeout the kernel
// records MOE_ERR_TIMEOUT, drains its copies and MMAs, frees TMEM and returns.
#include <algorithm>
#include <cstring>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"
#include "tc_sync.cuh"

namespace moe {
namespace {

using namespace tc;

enum { KIND_GATED = 0, KIND_RELU = 1, KIND_PLAIN = 2 };

constexpr int BK = 64;
constexpr int STAGES = 6;
constexpr int NUM_THREADS = 192;
constexpr int MAX_SEG = 257;
constexpr int TOK_TILE = 256;                        // tokens per tile at most (MMA N)
constexpr int TOK_BOX = 64;                          // token rows per TMA box
constexpr uint32_t TOK_BOX_BYTES = TOK_BOX * BK * 2;  // 8 KB
constexpr uint32_t A_BYTES = 128 * BK * 2;           // 16 KB: this CTA's 128 weight rows
constexpr uint32_t B_BYTES = 2 * TOK_BOX_BYTES;      // 16 KB: up to 128 token rows
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int ACC_COLS = 256;
constexpr int NACC = 2;
constexpr uint32_t TMEM_COLS = NACC * ACC_COLS;
// epilogue scratch of one epilogue warp: two exchange buffers [32 lanes][16 + 1
// pad] fp32 (alternating chunks) and one [32 tokens][32 rows] bf16 transpose tile
constexpr int XSTRIDE = 17;
constexpr uint32_t XBUF_BYTES = 32 * XSTRIDE * 4;
constexpr uint32_t TBUF_BYTES = 32 * 32 * 2;
constexpr uint32_t EPI_WARP_BYTES = 2 * XBUF_BYTES + TBUF_BYTES;
constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + 4 * EPI_WARP_BYTES;

struct SwParams {
    CUtensorMap tmX, tmX_sh;       // tokens [rows][K], box 64 x 64
    CUtensorMap tmW0, tmW1;        // routed weights [n_seg][n_out][K], box 64 x (64 gated | 128) x 1
    CUtensorMap tmW0_sh, tmW1_sh;  // shared weights [n_out_sh][K_sh]
    const int32_t *offsets;
    int n_seg, sh_rows;
    int a_rows;                    // rows of the routed buffers; offsets are clamped to it
    int n_out, K, n_out_sh, K_sh;
    __nv_bfloat16 *C, *C_sh;       // outputs [rows][n_out] / [sh_rows][n_out_sh]
    uint32_t *err;
};

struct Smem {
    uint64_t full[STAGES], empty[STAGES], tfull[NACC], tempty[NACC], drain;
    uint64_t xbar[2][2];  // gated exchange: [warp pair][chunk parity], 64 arrivals
    uint32_t tmem_base;
    int abort_flag;
    int base[MAX_SEG + 1];  // first tile of each segment; base[nseg] = total
    int nt[MAX_SEG];        // token tiles per segment
    int ttok[MAX_SEG];      // tokens per tile (a multiple of 32)
    int row0[MAX_SEG];      // first row of the segment in its buffers
    int rows[MAX_SEG];      // rows of the segment
};
static_assert(SMEM_BYTES + sizeof(Smem) <= 232448, "shared memory budget of one CTA");

struct Tile {
    int seg, blk, t0, ntok, nmma;
};

__device__ __forceinline__ Tile decode(const Smem &s, int nseg, int tile) {
    int lo = 0, hi = nseg - 1;  // largest g with base[g] <= tile
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s.base[mid] <= tile) lo = mid;
        else hi = mid - 1;
    }
    Tile t;
    t.seg = lo;
    const int local = tile - s.base[lo];
    const int i = local % s.nt[lo];
    t.blk = local / s.nt[lo];
    t.t0 = i * s.ttok[lo];
    t.ntok = min(s.ttok[lo], s.rows[lo] - t.t0);
    t.nmma = (t.ntok + 31) & ~31;
    return t;
}

// Epilogue of one tile in one epilogue warp (TMEM lane quarter q of CTA `rank`).
// Returns false if an exchange wait gave up.
template <int KIND>
__device__ __forceinline__ bool epilogue_tile(Smem &s, uint8_t *scratch, uint32_t tbase, const Tile &t,
                                              const SwParams &p, uint32_t rank, int q, int lane,
                                              uint32_t &xcount, volatile int *abort_flag) {
    const bool sh = t.seg >= p.n_seg;
    const int n_out = sh ? p.n_out_sh : p.n_out;
    __nv_bfloat16 *out = sh ? p.C_sh : p.C;
    const int64_t row_base = (int64_t)s.row0[t.seg] + t.t0;  // output row of token 0 of the tile
    uint8_t *mine = scratch + (size_t)q * EPI_WARP_BYTES;
    __nv_bfloat16 *tb = reinterpret_cast<__nv_bfloat16 *>(mine + 2 * XBUF_BYTES);
    const int nchunks = (t.ntok + 31) >> 5;
    const int piece = lane & 3;  // 16-byte piece of a token's 64-byte output run
    if constexpr (KIND == KIND_GATED) {
        const bool is_gate = q < 2;
        const int pidx = q & 1;
        // hidden units of this warp: 32 consecutive, the same for gate and up warps
        const int hcol = t.blk * 128 + (int)rank * 64 + pidx * 32;
        const bool cols_ok = hcol < n_out;
        uint8_t *partner = scratch + (size_t)(q ^ 2) * EPI_WARP_BYTES;
        const int keep = is_gate ? 0 : 16;  // this warp's tokens: 16 of every 32, the rest go to the partner
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
            uint32_t v[32];
            tmem_ld32(tbase + (uint32_t)(c * 32), v);
            tmem_ld_wait();
            const uint32_t par = xcount & 1u, ph = (xcount >> 1) & 1u;
            ++xcount;
            float *xo = reinterpret_cast<float *>(mine + par * XBUF_BYTES);
            const float *xi = reinterpret_cast<const float *>(partner + par * XBUF_BYTES);
            if (is_gate) {
#pragma unroll
                for (int i = 0; i < 16; ++i) xo[lane * XSTRIDE + i] = __uint_as_float(v[16 + i]);
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) xo[lane * XSTRIDE + i] = __uint_as_float(v[i]);
            }
            mbar_arrive(&s.xbar[pidx][par]);
            if (!wait_bar(&s.xbar[pidx][par], ph, abort_flag, p.err)) return false;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float other = xi[lane * XSTRIDE + i];
                const float mineval = __uint_as_float(is_gate ? v[i] : v[16 + i]);
                const float g = is_gate ? mineval : other;
                const float u = is_gate ? other : mineval;
                tb[i * 32 + lane] = __float2bfloat16_rn(silu_f32(g) * u);
            }
            __syncwarp();
            // tokens c*32 + keep + [0, 16): 16 tokens x 64 bytes, 8 tokens per pass
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int tk = half * 8 + (lane >> 2);
                const int j = c * 32 + keep + tk;
                if (cols_ok && j < t.ntok) {
                    const uint4 val = *reinterpret_cast<const uint4 *>(tb + tk * 32 + piece * 8);
                    *reinterpret_cast<uint4 *>(out + (row_base + j) * n_out + hcol + piece * 8) = val;
                }
            }
            __syncwarp();
        }
    } else {
        const int ocol = t.blk * 256 + (int)rank * 128 + q * 32;
        const bool cols_ok = ocol < n_out;
#pragma unroll 1
        for (int c = 0; c < nchunks; ++c) {
            uint32_t v[32];
            tmem_ld32(tbase + (uint32_t)(c * 32), v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                float x = __uint_as_float(v[i]);
                if (KIND == KIND_RELU) x = fmaxf(x, 0.0f);
                tb[i * 32 + lane] = __float2bfloat16_rn(x);
            }
            __syncwarp();
#pragma unroll
            for (int part = 0; part < 4; ++part) {
                const int tk = part * 8 + (lane >> 2);
                const int j = c * 32 + tk;
                if (cols_ok && j < t.ntok) {
                    const uint4 val = *reinterpret_cast<const uint4 *>(tb + tk * 32 + piece * 8);
                    *reinterpret_cast<uint4 *>(out + (row_base + j) * n_out + ocol + piece * 8) = val;
                }
            }
            __syncwarp();
        }
    }
    return true;
}

template <int KIND>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1) k_ffn_sw2(const __grid_constant__ SwParams p) {
    constexpr int WROWS = KIND == KIND_GATED ? 64 : 128;  // weight rows per TMA box
    constexpr int BLK = KIND == KIND_GATED ? 128 : 256;   // output columns per weight block
    __shared__ Smem s;
    extern __shared__ uint8_t dyn_smem[];
    const uint32_t dyn_base = smem_u32(dyn_smem);
    uint8_t *tiles = dyn_smem + (((dyn_base + 1023u) & ~1023u) - dyn_base);
    auto smA = [&](int st) { return tiles + (size_t)st * STAGE_BYTES; };
    auto smB = [&](int st) { return tiles + (size_t)st * STAGE_BYTES + A_BYTES; };
    uint8_t *scratch = tiles + (size_t)STAGES * STAGE_BYTES;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int cluster = blockIdx.x >> 1, nclusters = gridDim.x >> 1;
    const int nseg = p.n_seg + (p.sh_rows > 0 ? 1 : 0);
    const int nb_routed = (p.n_out + BLK - 1) / BLK;
    const int nb_sh = (p.n_out_sh + BLK - 1) / BLK;

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
                int r0, rows, nb;
                if (g < p.n_seg) {
                    r0 = min(max(p.offsets[g], 0), p.a_rows);
                    rows = min(max(p.offsets[g + 1], r0), p.a_rows) - r0;
                    nb = nb_routed;
                } else {
                    r0 = 0;
                    rows = p.sh_rows;
                    nb = nb_sh;
                }
                rows = max(rows, 0);
                const int nt = (rows + TOK_TILE - 1) / TOK_TILE;
                const int per_tile = nt > 0 ? (rows + nt - 1) / nt : 0;
                s.nt[g] = max(nt, 1);
                s.ttok[g] = (per_tile + 31) & ~31;
                s.row0[g] = r0;
                s.rows[g] = rows;
                tiles_g = nt * nb;
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
            for (int i = 0; i < NACC; ++i) {
                mbar_init(&s.tfull[i], 1);
                mbar_init(&s.tempty[i], 8);  // 4 epilogue warps of each CTA
            }
            for (int i = 0; i < 2; ++i)
                for (int j = 0; j < 2; ++j) mbar_init(&s.xbar[i][j], 64);
            mbar_init(&s.drain, 1);
            s.abort_flag = 0;
            fence_mbar_init();
        }
    }
    if (warp == 1) {
        tmem_alloc_pair(&s.tmem_base, TMEM_COLS);
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
        if (lane == 0 && run) {
            int st = 0;
            uint32_t ph = 0;
            bool ok = true;
            uint32_t issued_mask = 0, issued_par = 0;
            const uint32_t lead_full = map_to_rank(smem_u32(&s.full[0]), 0);
            for (int tile = cluster; tile < total && ok; tile += nclusters) {
                const Tile t = decode(s, nseg, tile);
                const bool sh = t.seg >= p.n_seg;
                const int K = sh ? p.K_sh : p.K;
                const int half = t.nmma >> 1;                              // token rows per CTA
                const int trow = s.row0[t.seg] + t.t0 + (int)rank * half;  // first token row loaded here
                const int nbox = (half + TOK_BOX - 1) / TOK_BOX;
                const uint32_t tx = 2u * (A_BYTES + (uint32_t)nbox * TOK_BOX_BYTES);
                const int wrow = t.blk * BLK + (int)rank * WROWS;  // first weight row loaded here
                const CUtensorMap *tx_map = sh ? &p.tmX_sh : &p.tmX;
                for (int kb = 0; kb < K / BK; ++kb) {
                    if (!wait_bar(&s.empty[st], ph ^ 1, abort_flag, p.err)) {
                        ok = false;
                        break;
                    }
                    const uint32_t fb = lead_full + 8u * (uint32_t)st;
                    if (leader) mbar_arrive_expect_tx(&s.full[st], tx);
                    const int kc = kb * BK;
                    if (KIND == KIND_GATED) {
                        // 64 gate rows then the 64 up rows of the same hidden units
                        if (sh) {
                            tma_load_2d_pair(smA(st), &p.tmW0_sh, kc, wrow, fb);
                            tma_load_2d_pair(smA(st) + A_BYTES / 2, &p.tmW1_sh, kc, wrow, fb);
                        } else {
                            tma_load_3d_pair(smA(st), &p.tmW0, kc, wrow, t.seg, fb);
                            tma_load_3d_pair(smA(st) + A_BYTES / 2, &p.tmW1, kc, wrow, t.seg, fb);
                        }
                    } else {
                        if (sh) tma_load_2d_pair(smA(st), &p.tmW0_sh, kc, wrow, fb);
                        else tma_load_3d_pair(smA(st), &p.tmW0, kc, wrow, t.seg, fb);
                    }
                    for (int bx = 0; bx < nbox; ++bx)
                        tma_load_2d_pair(smB(st) + bx * TOK_BOX_BYTES, tx_map, kc, trow + bx * TOK_BOX, fb);
                    issued_mask |= 1u << st;
                    issued_par = (issued_par & ~(1u << st)) | (ph << st);
                    if (++st == STAGES) {
                        st = 0;
                        ph ^= 1;
                    }
                }
            }
            // loads in flight land before the CTA exits (the even CTA waits for both halves)
            if (leader)
                for (int i = 0; i < STAGES; ++i)
                    if (issued_mask & (1u << i)) drain_bar(&s.full[i], (issued_par >> i) & 1u);
        }
    } else if (warp == 1) {
        if (lane == 0 && run && leader) {
            // ================= MMA issuer (even CTA) =================
            int st = 0, acc = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            for (int tile = cluster; tile < total && ok; tile += nclusters) {
                const Tile t = decode(s, nseg, tile);
                const int K = t.seg >= p.n_seg ? p.K_sh : p.K;
                const uint32_t idesc = idesc_bf16_f32(256, t.nmma);
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
                    const uint64_t bd = desc_sw128(smem_u32(smB(st)));
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk)
                        umma_bf16_pair(d_tmem, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), idesc,
                                       (kb | kk) != 0 ? 1u : 0u);
                    umma_commit_pair_mc(&s.empty[st], 0x3);
                    if (++st == STAGES) {
                        st = 0;
                        ph ^= 1;
                    }
                }
                if (!ok) break;
                umma_commit_pair_mc(&s.tfull[acc], 0x3);
                if (++acc == NACC) {
                    acc = 0;
                    aph ^= 1;
                }
            }
            umma_commit_pair_mc(&s.drain, 0x1);
            drain_bar(&s.drain, 0);
        }
    } else if (run) {
        // ================= epilogue (warps 2..5 of both CTAs) =================
        const int q = warp & 3;
        int acc = 0;
        uint32_t aph = 0, xcount = 0;
        for (int tile = cluster; tile < total; tile += nclusters) {
            const Tile t = decode(s, nseg, tile);
            if (!wait_bar(&s.tfull[acc], aph, abort_flag, p.err)) break;
            tc_fence_after();
            const uint32_t tbase = tmem_base + (uint32_t)(acc * ACC_COLS) + ((uint32_t)(q * 32) << 16);
            if (!epilogue_tile<KIND>(s, scratch, tbase, t, p, rank, q, lane, xcount, abort_flag)) break;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader) mbar_arrive_relaxed(&s.tempty[acc]);
                else mbar_arrive_remote_relaxed(lead_tempty + 8u * (uint32_t)acc);
            }
            if (++acc == NACC) {
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
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host side

template <int KIND>
cudaError_t launch_kind(const SwParams &p, int64_t max_tiles, cudaStream_t s) {
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e =
            cudaFuncSetAttribute(k_ffn_sw2<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    const int clusters = (int)std::max<int64_t>(1, std::min<int64_t>(max_tiles, device_sm_count() / 2));
    return launch_pdl(k_ffn_sw2<KIND>, dim3(2 * clusters), dim3(NUM_THREADS), SMEM_BYTES, s, p);
}

// One product over the routed segments and/or the shared segment.
//   x / x_sh: token rows ([a_rows][K] / [sh_rows][K_sh]);
//   w0,w1 / w0_sh,w1_sh: weights ([n_seg][n_out][K] / [n_out_sh][K_sh]), w1 = up (gated only);
//   out / out_sh: outputs ([a_rows][n_out] / [sh_rows][n_out_sh]).
template <int KIND>
cudaError_t product(const int32_t *offsets, int n_seg, int64_t a_rows, const void *x, const void *w0,
                    const void *w1, int K, int n_out, void *out, int sh_rows, const void *x_sh, const void *w0_sh,
                    const void *w1_sh, int K_sh, int n_out_sh, void *out_sh, uint32_t *err, cudaStream_t s) {
    constexpr int BLK = KIND == KIND_GATED ? 128 : 256;
    constexpr uint32_t WROWS = KIND == KIND_GATED ? 64 : 128;
    SwParams p;
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
    p.err = err;
    int64_t max_tiles = 0;
    if (n_seg > 0) {
        if (!encode_bf16_2d(&p.tmX, x, K, a_rows, TOK_BOX)) return cudaErrorInvalidValue;
        if (!encode_bf16_3d(&p.tmW0, w0, K, n_out, n_seg, WROWS)) return cudaErrorInvalidValue;
        if (KIND == KIND_GATED && !encode_bf16_3d(&p.tmW1, w1, K, n_out, n_seg, WROWS)) return cudaErrorInvalidValue;
        max_tiles += ((a_rows + TOK_TILE - 1) / TOK_TILE + n_seg) * ((n_out + BLK - 1) / BLK);
    }
    if (sh_rows > 0) {
        if (!encode_bf16_2d(&p.tmX_sh, x_sh, K_sh, sh_rows, TOK_BOX)) return cudaErrorInvalidValue;
        if (!encode_bf16_2d(&p.tmW0_sh, w0_sh, K_sh, n_out_sh, WROWS)) return cudaErrorInvalidValue;
        if (KIND == KIND_GATED && !encode_bf16_2d(&p.tmW1_sh, w1_sh, K_sh, n_out_sh, WROWS))
            return cudaErrorInvalidValue;
        max_tiles += ((int64_t)(sh_rows + TOK_TILE - 1) / TOK_TILE) * ((n_out_sh + BLK - 1) / BLK);
    }
    if (max_tiles == 0) return cudaSuccess;
    return launch_kind<KIND>(p, max_tiles, s);
}

}  // namespace

cudaError_t launch_ffn_sw(const moe_config &c, const FfnGroup &g, uint32_t *err, cudaStream_t s) {
    cudaError_t e;
    // product 1: hidden activations
    if (g.act == MOE_ACT_SILU_GATED) {
        e = product<KIND_GATED>(g.offsets, g.n_seg, g.a_rows, g.a, g.w_a, g.w_b, c.d, g.h, g.hid, g.sh_rows, g.sh_a,
                                g.sh_w_gate, g.sh_w_up, c.d, g.h_sh, g.sh_hid, err, s);
    } else {
        e = product<KIND_RELU>(g.offsets, g.n_seg, g.a_rows, g.a, g.w_a, nullptr, c.d, g.h, g.hid, 0, nullptr, nullptr,
                               nullptr, 0, 0, nullptr, err, s);
        if (e == cudaSuccess && g.sh_rows > 0)
            e = product<KIND_GATED>(nullptr, 0, 0, nullptr, nullptr, nullptr, 0, 0, nullptr, g.sh_rows, g.sh_a,
                                    g.sh_w_gate, g.sh_w_up, c.d, g.h_sh, g.sh_hid, err, s);
    }
    if (e != cudaSuccess) return e;
    if (g.mid_event && (e = cudaEventRecordWithFlags(g.mid_event, s, g.event_flags)) != cudaSuccess) return e;
    // product 2: outputs
    return product<KIND_PLAIN>(g.offsets, g.n_seg, g.a_rows, g.hid, g.w_out, nullptr, g.h, c.d, g.out, g.sh_rows,
                               g.sh_hid, g.sh_w_down, nullptr, g.h_sh, c.d, g.sh_out, err, s);
}

}  // namespace moe
