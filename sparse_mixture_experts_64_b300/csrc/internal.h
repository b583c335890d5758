// Host-side internals shared by the translation units of libmoe.so:
// workspace layout, launcher declarations and tiling constants.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime_api.h>
#include "../../include/moe.h"

namespace moe {

// Device error word bits (the word lives at the start of the workspace).
constexpr uint32_t kErrFault = 1u;    // an out-of-range index was seen and skipped
constexpr uint32_t kErrTimeout = 2u;  // a bounded wait gave up

// Expert Choice selects each expert's tokens by sorting all T scores of its column
// in shared memory (8-byte keys, T rounded up to a power of two).
constexpr int kMaxExpertChoiceTokens = 16384;

// The router writes its per-expert statistics per tile of router_tile_tokens(cfg)
// tokens; the tile is a pure function of the config (no device query), so the
// workspace size can be computed without a GPU.
int router_tile_tokens(const moe_config &c);
inline int router_tiles(const moe_config &c) {
    const int tt = router_tile_tokens(c);
    return (c.T + tt - 1) / tt;
}

int64_t max_rows(const moe_config &c);     // R_max
int32_t capacity_of(const moe_config &c);  // C, 0 = no limit
size_t dtype_size(const moe_config &c);

// Byte offsets of every workspace region (each 256-byte aligned).
struct WsLayout {
    size_t err;                  // uint32 error word
    size_t cnt, pre;             // int32 [N][k][tiles]
    size_t kpre;                 // int32 [N][tiles]
    size_t psum;                 // f32   [N][tiles]
    size_t pmean;                // f32   [N]
    size_t zpart;                // f32   [tiles] per-tile sums of the z-loss terms
    size_t routed, kept;         // int32 [N] (used when the caller passes NULL)
    size_t logits;               // f32   [T][N]  (N > 32 only)
    size_t w_t;                  // f32   [ceil(d/256)][N even][256]  router weight, re-laid out
    size_t offsets;              // int32 [N+1]
    size_t topk_idx, topk_gate;  // [T][k]
    size_t slot_row;             // int32 [T][k]
    size_t perm_token;           // int32 [R_max]
    size_t aux;                  // f32 [2]
    size_t x_perm, y_perm;       // [R_max][d]
    // Expert Choice: scores [N][T] f32, row of (expert, token) [N][T] int32 (-1: not
    // chosen), per-token row counts [T], list offsets [T+1], row lists [R_max] and
    // row gates [R_max] (used by moe_forward)
    size_t ec_scores, ec_row, ec_tok_cnt, ec_tok_ptr, ec_tok_rows, ec_row_gate;
    size_t hid;                  // [R_max][h]
    size_t hid_sh;               // [T][h_shared]
    size_t s_out;                // [T][d]  shared expert output
    // pre-activations kept by moe_forward for moe_backward (saves_preact): bf16 [R_max][W]
    // (gated: gate in columns [0, h), up in [h, 2h); ReLU: W = h) and [T][2 h_shared]
    size_t preact, preact_sh;
    size_t total;
};
WsLayout ws_layout(const moe_config &c);
// moe_forward keeps the pre-activations (cfg.save_preact on the bf16 token-choice
// tensor-core path; not with the forced CUDA-core or weights-as-M kernels).
bool saves_preact(const moe_config &c);

// Byte offsets of the backward workspace regions (each 256-byte aligned). W = 2h for
// SiLU-gated experts ([A | B] pre-activations), h for ReLU experts.
struct BwdLayout {
    size_t dO;                   // bf16 [R_max][d]  gate-scaled dy per row
    size_t dgate;                // f32  [T][k]      gate gradients
    size_t AB, dH, dAB;          // bf16 [R_max][W], [R_max][h], [R_max][W]
    size_t dX;                   // bf16 [R_max][d]
    size_t AB_sh, dH_sh, dAB_sh, dX_sh;  // shared expert, rows = T
    size_t logits, routed, dL, dxr;  // router: f32 [T][N] (N <= 32: recomputed), int32 [N], f32 [T][N], f32 [T][d]
    size_t rA, rB, dLt, wrC;         // router-gradient split operands: bf16 [T][Kr], [d][Kr] (Kr = 3N
                                     // rounded up to 64), [2N][ceil64(T)]; f32 [2N][d] dW_rᵀ halves
    size_t total;
};
BwdLayout bwd_layout(const moe_config &c);

// ---- launchers (return cudaGetLastError() after the launch) ----
struct RouterOut {
    int32_t *topk_idx;
    float *topk_gate;
    int32_t *counts_routed, *counts_kept, *expert_offsets, *slot_row, *perm_token;
    float *aux;
    // training-time router (null / 0 for inference): noise draws [T][N] and their
    // weight (noisy top-k), and the z-loss output [1]
    const float *noise = nullptr;
    float noise_w = 0.0f;
    float *z_loss = nullptr;
};
cudaError_t launch_router(const moe_config &c, const void *x, const float *w_r, const float *b_r,
                          const RouterOut &o, uint8_t *ws, cudaStream_t s);
// Router logits [T][N] fp32 alone (the blocked summation order of every router
// path), for any N; used by Expert Choice.
cudaError_t launch_router_logits(const moe_config &c, const void *x, const float *w_r, const float *b_r,
                                 float *logits, uint8_t *ws, cudaStream_t s);
// Expert Choice: scores, per-expert selection (expert_offsets, perm_token,
// row_gate) and per-token row lists (tok_ptr, tok_rows) from the logits.
cudaError_t launch_expert_choice(const moe_config &c, const float *logits, int32_t *expert_offsets,
                                 int32_t *perm_token, float *row_gate, int32_t *tok_ptr, int32_t *tok_rows,
                                 uint8_t *ws, cudaStream_t s);
// Expert Choice combine: y = x + [s_out] + sum over each token's rows of gate * y_perm.
cudaError_t launch_combine_ec(const moe_config &c, const void *x, const void *y_perm, const void *s_out,
                              const int32_t *tok_ptr, const int32_t *tok_rows, const float *row_gate, void *y,
                              uint32_t *err, cudaStream_t s);
// Backward pieces (backward.cu).
cudaError_t launch_bwd_slots(const moe_config &c, const void *dy, const void *y_perm, const int32_t *slot_row,
                             const float *gate, void *dO, float *dgate, uint32_t *err, cudaStream_t s);
cudaError_t launch_act_bwd(bool gated, const void *AB, const void *dH, int64_t rows, int h, void *dAB,
                           cudaStream_t s);
// Router backward from the fp32 logits [T][N]: dL, then dx_router (into L.dxr) and dW_r
// on the tensor cores from bf16-split operands and the tokens x [T][d].
cudaError_t launch_router_bwd(const moe_config &c, const void *x, const float *w_r, const float *logits,
                              const int32_t *topk_idx, const float *topk_gate, const BwdLayout &L, uint8_t *bw,
                              float aux_coef, float z_coef, float *dw_r, float *db_r, uint32_t *err, bool allow_pair,
                              cudaStream_t s);
cudaError_t launch_bwd_dx(const moe_config &c, const void *dy, const void *dX, const int32_t *slot_row,
                          const void *dX_sh, const float *dxr, void *dx, uint32_t *err, cudaStream_t s);
// Token-sharded router, phase 1: routing of this shard and the statistics the
// shards exchange (selections per expert and slot, sums of the softmax).
cudaError_t launch_router_stats(const moe_config &c, const void *x, const float *w_r, const float *b_r,
                                int32_t *topk_idx, float *topk_gate, int32_t *slot_counts, float *prob_sums,
                                uint8_t *ws, cudaStream_t s);
// Phase 2: capacity decisions at global priorities, dispatch order, global aux.
cudaError_t launch_router_assign(const moe_config &c, const int32_t *topk_idx, const int32_t *slot_base, int32_t cap,
                                 const int32_t *g_routed, const float *g_psum, float g_T, int32_t *counts_kept,
                                 int32_t *expert_offsets, int32_t *slot_row, int32_t *perm_token, float *aux,
                                 uint8_t *ws, cudaStream_t s);

cudaError_t launch_dispatch(const moe_config &c, const void *x, const int32_t *perm_token,
                            const int32_t *offsets, void *x_perm, uint32_t *err, cudaStream_t s);
// Dispatch in token order from slot_row [T][k] (each token read once).
cudaError_t launch_dispatch_tokens(const moe_config &c, const void *x, const int32_t *slot_row, void *x_perm,
                                   uint32_t *err, cudaStream_t s);

cudaError_t launch_combine(const moe_config &c, const void *x, const void *y_perm,
                           const void *s_out, const int32_t *slot_row, const float *gate,
                           void *y, uint32_t *err, cudaStream_t s);

// One grouped FFN problem: routed segments given by offsets (n_seg experts,
// rows [offsets[e], offsets[e+1]) of A) plus an optional shared segment of
// sh_rows rows with its own A and weights.
struct FfnGroup {
    const int32_t *offsets;  // device, [n_seg + 1]; may be null when n_seg == 0
    int n_seg;
    int64_t a_rows;          // rows allocated in the routed A / hidden / output buffers
    const void *a;           // routed A [a_rows][d]
    const void *w_a, *w_b, *w_out;  // routed weights (w_b null for ReLU)
    void *hid;               // routed hidden [a_rows][h]
    void *out;               // routed output [a_rows][d]
    int h;
    int act;
    int sh_rows;             // 0: no shared segment
    const void *sh_a;        // [sh_rows][d]
    const void *sh_w_gate, *sh_w_up, *sh_w_down;
    void *sh_hid;            // [sh_rows][h_shared]
    void *sh_out;            // [sh_rows][d]
    void *pre, *sh_pre;      // null, or where product 1 also stores its raw pre-activations
                             // ([a_rows][2h] gated / [a_rows][h] ReLU; [sh_rows][2 h_sh])
    int h_sh;
    cudaEvent_t mid_event;   // if set: recorded between the two products
    unsigned event_flags;    // cudaEventRecordExternal while a graph is being captured
};
cudaError_t launch_ffn_simt(const moe_config &c, const FfnGroup &g, uint32_t *err, cudaStream_t s);
cudaError_t launch_ffn_tc(const moe_config &c, const FfnGroup &g, uint32_t *err, cudaStream_t s);
cudaError_t launch_ffn_sw(const moe_config &c, const FfnGroup &g, uint32_t *err, cudaStream_t s);
// One grouped product on the tensor cores (bf16): out[rows of segment g] = a[rows][K]
// · b0[g][n_out][K]ᵀ, plain, or with preact the gated pair (b0, b1) stored raw as
// [gate | up] rows of width 2 n_out; an optional shared segment with its own operands.
// b_mn (plain only): the weights are MN-major instead, out = a · b0[g] with b0[g]
// [K][n_out]; with k_split > 0 the K rows are b0[g] [k_split][n_out] followed by b1[g]
// [K - k_split][n_out] (likewise b0_sh / b1_sh with k_split_sh), so [W_gate; W_up] need
// not be stacked.
cudaError_t launch_gemm_rows(const moe_config &c, bool preact, const int32_t *offsets, int n_seg, int64_t a_rows,
                             const void *a, const void *b0, const void *b1, int K, int n_out, void *out, int sh_rows,
                             const void *a_sh, const void *b0_sh, const void *b1_sh, int K_sh, int n_out_sh,
                             void *out_sh, uint32_t *err, cudaStream_t s, bool b_mn = false, int k_split = 0,
                             int k_split_sh = 0);
// An operand of the weight-gradient GEMM. MN-major (mn): an activation array
// [rows][ld] whose first M (or Nn) columns are the operand, its rows the reduction
// index; K-rows at or past `rows` read as zero. K-major: [M|Nn][ld] with K = ld along
// each row (zero-padded to a multiple of 64).
struct WgOperand {
    const void *p;
    int64_t ld, rows;
    bool mn;
};
// Weight-gradient GEMM with K running over each expert's rows: for expert e with rows
// [r0, r1) of `offsets` (clamped to a_rows), out[e] [M][Nn] = A[r0:r1]ᵀ · B[r0:r1] with A
// and B MN-major over the a_rows rows of the routed buffers. An optional shared segment:
// out_sh [M][Nn] = Aᵀ B over K_sh K-rows, either operand MN-major or K-major (then ld =
// K_sh, a multiple of 64); with n_seg = 0 that is a plain product. Outputs are bf16, or
// fp32 with f32_out. Nn must be a multiple of 64; M is any row count; ld × 2 bytes and
// the operand addresses must be multiples of 16.
cudaError_t launch_wgrad(const int32_t *offsets, int n_seg, int64_t a_rows, WgOperand A, WgOperand B, int M, int Nn,
                         void *out, WgOperand A_sh, WgOperand B_sh, int K_sh, void *out_sh, uint32_t *err,
                         cudaStream_t s, bool allow_pair = true, bool f32_out = false);

int device_sm_count();

// TMA tensor map of a `rank`-dimensional array (dims innermost first, strides in
// bytes for dims 1..rank-1, box in elements). false if the driver refuses it.
bool encode_tmap(CUtensorMap *m, CUtensorMapDataType dt, int rank, const void *base, const uint64_t *dims,
                 const uint64_t *strides_bytes, const uint32_t *box, CUtensorMapSwizzle swizzle);
// bf16 K-major operand maps: [outer][inner] and [n_exp][outer][inner], box 64
// (inner) x box_outer (x 1), 128-byte swizzle.
bool encode_bf16_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint32_t box_outer);
bool encode_bf16_3d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t n_exp,
                    uint32_t box_outer);

}  // namespace moe
