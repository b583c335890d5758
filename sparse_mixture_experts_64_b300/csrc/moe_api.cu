// C ABI of libmoe.so: host-side validation, workspace layout and the launch
// sequence of the sparse MoE layer forward (router -> dispatch -> experts ->
// combine). The calls and their order follow "MoE: Choosing Which MLPs to Use for
// Each Token", section "From Router to Combine"; see include/moe.h for each
// call's contract.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>

#include "common.cuh"
#include "internal.h"

namespace moe {

thread_local bool g_no_pdl = false;

// Programmatic launches off for one call (MOE_DEBUG_NO_PDL), restored on return.
struct PdlScope {
    bool saved;
    explicit PdlScope(const moe_config *c) : saved(g_no_pdl) {
        if (c && (c->debug_flags & MOE_DEBUG_NO_PDL)) g_no_pdl = true;
    }
    ~PdlScope() { g_no_pdl = saved; }
};

int64_t max_rows(const moe_config &c) {
    const int32_t C = capacity_of(c);
    if (c.routing == MOE_ROUTING_EXPERT_CHOICE) return (int64_t)c.N * std::min<int64_t>(C, c.T);
    const int64_t tk = (int64_t)c.T * c.k;
    return C > 0 ? std::min<int64_t>(tk, (int64_t)c.N * C) : tk;
}

int32_t capacity_of(const moe_config &c) {
    if (c.cap_num <= 0 || c.cap_den <= 0) return 0;
    const int64_t num = (int64_t)c.T * c.cap_num, den = (int64_t)c.N * c.cap_den;
    const int64_t C = (num + den - 1) / den;
    return (int32_t)std::min<int64_t>(C, INT32_MAX);
}

size_t dtype_size(const moe_config &c) { return c.dtype == MOE_BF16 ? 2 : 4; }

static size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

WsLayout ws_layout(const moe_config &c) {
    WsLayout L;
    const size_t tiles = (size_t)router_tiles(c);
    const size_t N = c.N, k = c.k, T = c.T, es = dtype_size(c);
    const size_t rmax = (size_t)max_rows(c);
    size_t o = 0;
    auto take = [&](size_t bytes) {
        const size_t at = o;
        o = align256(o + std::max<size_t>(bytes, 1));
        return at;
    };
    // router scratch first: moe_router_topk needs only this prefix
    L.err = take(4);
    L.cnt = take(N * k * tiles * 4);
    L.pre = take(N * k * tiles * 4);
    L.kpre = take(N * tiles * 4);
    L.psum = take(N * tiles * 4);
    L.pmean = take(N * 4);
    L.zpart = take(tiles * 4);
    L.routed = take(N * 4);
    L.kept = take(N * 4);
    const bool ec = c.routing == MOE_ROUTING_EXPERT_CHOICE;
    L.logits = take(c.N > 32 || ec ? T * N * 4 : 0);
    L.w_t = take((size_t)((c.d + 255) / 256) * 256 * ((N + 1) & ~(size_t)1) * 4);  // N rounded up to even
    // expert / shared-expert buffers
    L.hid = take(rmax * c.h * es);
    L.hid_sh = take(c.h_shared ? T * c.h_shared * es : 0);
    L.s_out = take(c.h_shared ? T * c.d * es : 0);
    // moe_forward only
    L.offsets = take((N + 1) * 4);
    L.topk_idx = take(T * k * 4);
    L.topk_gate = take(T * k * 4);
    L.slot_row = take(T * k * 4);
    L.perm_token = take(rmax * 4);
    L.aux = take(2 * 4);
    L.x_perm = take(rmax * c.d * es);
    L.y_perm = take(rmax * c.d * es);
    // Expert Choice only
    L.ec_scores = take(ec ? N * T * 4 : 0);
    L.ec_row = take(ec ? N * T * 4 : 0);
    L.ec_tok_cnt = take(ec ? T * 4 : 0);
    L.ec_tok_ptr = take(ec ? (T + 1) * 4 : 0);
    L.ec_tok_rows = take(ec ? rmax * 4 : 0);
    L.ec_row_gate = take(ec ? rmax * 4 : 0);
    const bool keep = saves_preact(c);
    const size_t W = c.act == MOE_ACT_SILU_GATED ? 2 * (size_t)c.h : (size_t)c.h;
    L.preact = take(keep ? rmax * W * 2 : 0);
    L.preact_sh = take(keep && c.h_shared ? T * 2 * (size_t)c.h_shared * 2 : 0);
    L.total = o;
    return L;
}

bool saves_preact(const moe_config &c) {
    return c.save_preact == 1 && c.dtype == MOE_BF16 && c.routing == MOE_ROUTING_TOKEN_CHOICE &&
           !(c.debug_flags & (MOE_DEBUG_FORCE_SIMT_FFN | MOE_DEBUG_FFN_SWAP));
}

int device_sm_count() {
    static int count = 0;
    if (count == 0) {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) == cudaSuccess &&
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess && v > 0)
            count = v;
        else
            return 148;  // B300
    }
    return count;
}

static bool dim_ok(int32_t v, int dtype) {
    if (v < 8 || v > 65536) return false;
    return dtype == MOE_BF16 ? v % 64 == 0 : v % 8 == 0;
}

static moe_status validate(const moe_config *c) {
    if (!c) return MOE_ERR_INVALID_ARG;
    if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (c->gating != MOE_SOFTMAX_THEN_TOPK && c->gating != MOE_TOPK_THEN_SOFTMAX) return MOE_ERR_INVALID_ARG;
    if (c->act != MOE_ACT_SILU_GATED && c->act != MOE_ACT_RELU) return MOE_ERR_INVALID_ARG;
    if (c->T < 1 || c->T > 65536) return MOE_ERR_INVALID_ARG;
    if (c->N < 1 || c->N > 256) return MOE_ERR_INVALID_ARG;
    if (c->k < 1 || c->k > c->N || c->k > 8) return MOE_ERR_INVALID_ARG;
    if (c->d < 1 || c->h < 1 || c->h_shared < 0) return MOE_ERR_INVALID_ARG;
    if ((c->cap_num == 0) != (c->cap_den == 0) || c->cap_num < 0 || c->cap_den < 0) return MOE_ERR_INVALID_ARG;
    if (c->has_router_bias != 0 && c->has_router_bias != 1) return MOE_ERR_INVALID_ARG;
    if (!dim_ok(c->d, c->dtype) || !dim_ok(c->h, c->dtype)) return MOE_ERR_UNSUPPORTED;
    if (c->h_shared && !dim_ok(c->h_shared, c->dtype)) return MOE_ERR_UNSUPPORTED;
    if (c->routing != MOE_ROUTING_TOKEN_CHOICE && c->routing != MOE_ROUTING_EXPERT_CHOICE) return MOE_ERR_INVALID_ARG;
    if (c->save_preact != 0 && c->save_preact != 1) return MOE_ERR_INVALID_ARG;
    if (c->routing == MOE_ROUTING_EXPERT_CHOICE) {
        if (c->cap_num == 0) return MOE_ERR_INVALID_ARG;  // the experts' capacity is the routing
        if (c->T > kMaxExpertChoiceTokens) return MOE_ERR_UNSUPPORTED;
    }
    return MOE_OK;
}

static moe_status check_ws(const void *ws, size_t ws_bytes, size_t need) {
    if (!ws) return MOE_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(ws) % 256 != 0) return MOE_ERR_WORKSPACE;
    if (ws_bytes < need) return MOE_ERR_WORKSPACE;
    return MOE_OK;
}

static bool aligned16(const void *p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; }

static moe_status to_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

static cudaError_t run_ffn(const moe_config &c, const FfnGroup &g, uint32_t *err, cudaStream_t s) {
    const bool simt = c.dtype == MOE_F32 || (c.debug_flags & MOE_DEBUG_FORCE_SIMT_FFN);
    return simt ? launch_ffn_simt(c, g, err, s) : launch_ffn_tc(c, g, err, s);
}

// The shared expert S(x) of every token into the workspace (hidden and output).
static cudaError_t run_shared_expert(const moe_config &c, const void *x, const void *sw_gate, const void *sw_up,
                                     const void *sw_down, uint8_t *w, const WsLayout &L, uint32_t *err,
                                     cudaStream_t s) {
    FfnGroup g{};
    g.n_seg = 0;
    g.act = MOE_ACT_SILU_GATED;
    g.h = c.h;
    g.sh_rows = c.T;
    g.sh_a = x;
    g.sh_w_gate = sw_gate;
    g.sh_w_up = sw_up;
    g.sh_w_down = sw_down;
    g.sh_hid = w + L.hid_sh;
    g.sh_out = w + L.s_out;
    g.h_sh = c.h_shared;
    return run_ffn(c, g, err, s);
}

}  // namespace moe

using namespace moe;

extern "C" {

moe_status moe_validate_config(const moe_config *cfg) { return validate(cfg); }

size_t moe_workspace_size(const moe_config *cfg) {
    if (validate(cfg) != MOE_OK) return 0;
    return ws_layout(*cfg).total;
}

size_t moe_router_workspace_size(const moe_config *cfg) {
    if (validate(cfg) != MOE_OK || cfg->routing != MOE_ROUTING_TOKEN_CHOICE) return 0;
    return ws_layout(*cfg).hid;
}

size_t moe_preact_offset(const moe_config *cfg, int32_t shared) {
    if (validate(cfg) != MOE_OK || !saves_preact(*cfg)) return SIZE_MAX;
    if (shared && !cfg->h_shared) return SIZE_MAX;
    const WsLayout L = ws_layout(*cfg);
    return shared ? L.preact_sh : L.preact;
}

int64_t moe_max_rows(const moe_config *cfg) {
    if (validate(cfg) != MOE_OK) return 0;
    return max_rows(*cfg);
}

int32_t moe_capacity(const moe_config *cfg) {
    if (validate(cfg) != MOE_OK) return 0;
    return capacity_of(*cfg);
}

moe_status moe_router_topk(const moe_config *cfg, const void *x, const float *w_r, const float *b_r,
                           int32_t *topk_idx, float *topk_gate, int32_t *counts_routed,
                           int32_t *counts_kept, int32_t *expert_offsets, int32_t *slot_row,
                           int32_t *perm_token, float *aux, void *ws, size_t ws_bytes,
                           cudaStream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    const moe_config &c = *cfg;
    if (c.routing != MOE_ROUTING_TOKEN_CHOICE) return MOE_ERR_UNSUPPORTED;
    if (!x || !w_r || !topk_idx || !topk_gate || !expert_offsets || !slot_row || !perm_token)
        return MOE_ERR_INVALID_ARG;
    if (c.has_router_bias && !b_r) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_r)) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(c);
    if ((st = check_ws(ws, ws_bytes, L.hid)) != MOE_OK) return st;
    RouterOut o{topk_idx, topk_gate, counts_routed, counts_kept, expert_offsets, slot_row, perm_token, aux};
    return to_status(launch_router(c, x, w_r, c.has_router_bias ? b_r : nullptr, o,
                                   static_cast<uint8_t *>(ws), stream));
}

moe_status moe_router_topk_train(const moe_config *cfg, const void *x, const float *w_r, const float *b_r,
                                 const float *noise, float noise_weight, int32_t *topk_idx, float *topk_gate,
                                 int32_t *counts_routed, int32_t *counts_kept, int32_t *expert_offsets,
                                 int32_t *slot_row, int32_t *perm_token, float *aux, float *z_loss, void *ws,
                                 size_t ws_bytes, cudaStream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    const moe_config &c = *cfg;
    if (c.routing != MOE_ROUTING_TOKEN_CHOICE) return MOE_ERR_UNSUPPORTED;
    if (!x || !w_r || !topk_idx || !topk_gate || !expert_offsets || !slot_row || !perm_token)
        return MOE_ERR_INVALID_ARG;
    if (c.has_router_bias && !b_r) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_r)) return MOE_ERR_INVALID_ARG;
    if (noise && !std::isfinite(noise_weight)) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(c);
    if ((st = check_ws(ws, ws_bytes, L.hid)) != MOE_OK) return st;
    RouterOut o{topk_idx, topk_gate, counts_routed, counts_kept, expert_offsets, slot_row, perm_token, aux};
    o.noise = noise;
    o.noise_w = noise ? noise_weight : 0.0f;
    o.z_loss = z_loss;
    return to_status(launch_router(c, x, w_r, c.has_router_bias ? b_r : nullptr, o,
                                   static_cast<uint8_t *>(ws), stream));
}

moe_status moe_router_shard_stats(const moe_config *cfg, const void *x, const float *w_r, const float *b_r,
                                  int32_t *topk_idx, float *topk_gate, int32_t *slot_counts, float *prob_sums,
                                  void *ws, size_t ws_bytes, cudaStream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    const moe_config &c = *cfg;
    if (c.routing != MOE_ROUTING_TOKEN_CHOICE) return MOE_ERR_UNSUPPORTED;
    if (c.cap_num != 0 || c.cap_den != 0) return MOE_ERR_INVALID_ARG;  // the capacity is global
    if (!x || !w_r || !topk_idx || !topk_gate || !slot_counts) return MOE_ERR_INVALID_ARG;
    if (c.has_router_bias && !b_r) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_r)) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(c);
    if ((st = check_ws(ws, ws_bytes, L.hid)) != MOE_OK) return st;
    return to_status(launch_router_stats(c, x, w_r, c.has_router_bias ? b_r : nullptr, topk_idx, topk_gate,
                                         slot_counts, prob_sums, static_cast<uint8_t *>(ws), stream));
}

moe_status moe_router_shard_assign(const moe_config *cfg, const int32_t *topk_idx, const int32_t *slot_base,
                                   int32_t capacity, const int32_t *global_routed, const float *global_prob_sums,
                                   int64_t global_T, int32_t *counts_kept, int32_t *expert_offsets,
                                   int32_t *slot_row, int32_t *perm_token, float *aux, void *ws,
                                   size_t ws_bytes, cudaStream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    const moe_config &c = *cfg;
    if (c.routing != MOE_ROUTING_TOKEN_CHOICE) return MOE_ERR_UNSUPPORTED;
    if (c.cap_num != 0 || c.cap_den != 0) return MOE_ERR_INVALID_ARG;
    if (!topk_idx || !slot_base || !expert_offsets || !slot_row || !perm_token) return MOE_ERR_INVALID_ARG;
    if (capacity < 0 || global_T < c.T) return MOE_ERR_INVALID_ARG;
    if (aux && (!global_routed || !global_prob_sums)) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(c);
    if ((st = check_ws(ws, ws_bytes, L.hid)) != MOE_OK) return st;
    return to_status(launch_router_assign(c, topk_idx, slot_base, capacity, aux ? global_routed : nullptr,
                                          aux ? global_prob_sums : nullptr, (float)global_T, counts_kept,
                                          expert_offsets, slot_row, perm_token, aux, static_cast<uint8_t *>(ws),
                                          stream));
}

moe_status moe_router_expert_choice(const moe_config *cfg, const void *x, const float *w_r, const float *b_r,
                                   int32_t *expert_offsets, int32_t *perm_token, float *row_gate,
                                   int32_t *token_ptr, int32_t *token_rows, void *ws, size_t ws_bytes,
                                   cudaStream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    const moe_config &c = *cfg;
    if (c.routing != MOE_ROUTING_EXPERT_CHOICE) return MOE_ERR_UNSUPPORTED;
    if (!x || !w_r || !expert_offsets || !perm_token || !row_gate || !token_ptr || !token_rows)
        return MOE_ERR_INVALID_ARG;
    if (c.has_router_bias && !b_r) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_r)) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(c);
    if ((st = check_ws(ws, ws_bytes, L.total)) != MOE_OK) return st;
    uint8_t *w = static_cast<uint8_t *>(ws);
    float *logits = reinterpret_cast<float *>(w + L.logits);
    cudaError_t e = launch_router_logits(c, x, w_r, c.has_router_bias ? b_r : nullptr, logits, w, stream);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    return to_status(launch_expert_choice(c, logits, expert_offsets, perm_token, row_gate, token_ptr, token_rows,
                                          w, stream));
}

moe_status moe_combine_expert_choice(const moe_config *cfg, const void *x, const void *y_perm,
                                     const int32_t *token_ptr, const int32_t *token_rows, const float *row_gate,
                                     const void *shared_w_gate, const void *shared_w_up,
                                     const void *shared_w_down, void *y, void *ws, size_t ws_bytes,
                                     cudaStream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    const moe_config &c = *cfg;
    if (c.routing != MOE_ROUTING_EXPERT_CHOICE) return MOE_ERR_UNSUPPORTED;
    if (!x || !y_perm || !token_ptr || !token_rows || !row_gate || !y) return MOE_ERR_INVALID_ARG;
    if (c.h_shared && (!shared_w_gate || !shared_w_up || !shared_w_down)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y_perm) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(c);
    if ((st = check_ws(ws, ws_bytes, L.offsets)) != MOE_OK) return st;
    uint8_t *w = static_cast<uint8_t *>(ws);
    uint32_t *err = reinterpret_cast<uint32_t *>(w + L.err);
    const void *s_out = nullptr;
    if (c.h_shared) {
        cudaError_t e = run_shared_expert(c, x, shared_w_gate, shared_w_up, shared_w_down, w, L, err, stream);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
        s_out = w + L.s_out;
    }
    return to_status(launch_combine_ec(c, x, y_perm, s_out, token_ptr, token_rows, row_gate, y, err, stream));
}

size_t moe_backward_workspace_size(const moe_config *cfg) {
    if (validate(cfg) != MOE_OK) return 0;
    return bwd_layout(*cfg).total;
}

moe_status moe_backward(const moe_config *cfg, const void *x, const float *w_r, const float *b_r,
                        const void *w_gate_or_w1, const void *w_up, const void *w_down, const void *shared_w_gate,
                        const void *shared_w_up, const void *shared_w_down, const int32_t *topk_idx,
                        const float *topk_gate, const void *dy, float aux_coef, float z_coef, void *dx, float *dw_r,
                        float *db_r, void *dw_gate_or_w1, void *dw_up, void *dw_down, void *dshared_w_gate,
                        void *dshared_w_up, void *dshared_w_down, void *ws, size_t ws_bytes, void *bws,
                        size_t bws_bytes, cudaStream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    const moe_config &c = *cfg;
    if (c.routing != MOE_ROUTING_TOKEN_CHOICE || c.dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    const bool gated = c.act == MOE_ACT_SILU_GATED;
    if (!x || !w_r || !w_gate_or_w1 || !w_down || !dy || !dx || !dw_r || !dw_gate_or_w1 || !dw_down)
        return MOE_ERR_INVALID_ARG;
    if (gated && (!w_up || !dw_up)) return MOE_ERR_INVALID_ARG;
    if (c.has_router_bias && !b_r) return MOE_ERR_INVALID_ARG;
    if (c.h_shared && (!shared_w_gate || !shared_w_up || !shared_w_down || !dshared_w_gate || !dshared_w_up ||
                       !dshared_w_down))
        return MOE_ERR_INVALID_ARG;
    if (!std::isfinite(aux_coef) || !std::isfinite(z_coef)) return MOE_ERR_INVALID_ARG;
    const void *must_align[] = {x, w_r, w_gate_or_w1, w_down, dy, dx, dw_gate_or_w1, dw_down};
    for (const void *q : must_align)
        if (!aligned16(q)) return MOE_ERR_INVALID_ARG;
    if ((w_up && !aligned16(w_up)) || (dw_up && !aligned16(dw_up))) return MOE_ERR_INVALID_ARG;
    if (c.h_shared && (!aligned16(shared_w_gate) || !aligned16(shared_w_up) || !aligned16(shared_w_down) ||
                       !aligned16(dshared_w_gate) || !aligned16(dshared_w_up) || !aligned16(dshared_w_down)))
        return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(c);
    if ((st = check_ws(ws, ws_bytes, L.total)) != MOE_OK) return st;
    const BwdLayout B = bwd_layout(c);
    if ((st = check_ws(bws, bws_bytes, B.total)) != MOE_OK) return st;

    uint8_t *w = static_cast<uint8_t *>(ws), *bw = static_cast<uint8_t *>(bws);
    uint32_t *err = reinterpret_cast<uint32_t *>(w + L.err);
    const int32_t *idx = topk_idx ? topk_idx : reinterpret_cast<const int32_t *>(w + L.topk_idx);
    const float *gate = topk_gate ? topk_gate : reinterpret_cast<const float *>(w + L.topk_gate);
    const int32_t *offsets = reinterpret_cast<const int32_t *>(w + L.offsets);
    const int32_t *slot_row = reinterpret_cast<const int32_t *>(w + L.slot_row);
    const void *x_perm = w + L.x_perm, *y_perm = w + L.y_perm, *hid = w + L.hid, *hid_sh = w + L.hid_sh;
    const int64_t R = max_rows(c);
    const int N = c.N, d = c.d, h = c.h, hs = c.h_shared, Wd = gated ? 2 * h : h;
    // pre-activations: kept by moe_forward (save_preact), else recomputed into the scratch
    const bool kept_pre = saves_preact(c);
    void *AB = kept_pre ? w + L.preact : bw + B.AB, *AB_sh = kept_pre ? w + L.preact_sh : bw + B.AB_sh;
    void *dO = bw + B.dO, *dH = bw + B.dH, *dAB = bw + B.dAB, *dX = bw + B.dX;
    float *dgate = reinterpret_cast<float *>(bw + B.dgate);
    cudaError_t e = cudaSuccess;
    auto ok = [&](cudaError_t r) {
        if (e == cudaSuccess) e = r;
        return e == cudaSuccess;
    };

    // For N <= 32 the router logits are recomputed on an auxiliary stream beside the
    // expert products (FMA-bound beside tensor-bound work), joined before the router
    // backward; without the stream (creation failed) they run in order on `stream`. For
    // N > 32 the forward left them in its workspace. Every other operand is read where
    // the forward and the earlier steps left it: the row products take the expert weights
    // and the weight gradients the activations in their own layouts (MN-major operands).
    const bool fwd_logits = N > 32;
    const float *logits = reinterpret_cast<const float *>(fwd_logits ? w + L.logits : bw + B.logits);
    cudaStream_t aux = nullptr;
    cudaEvent_t ev[2] = {nullptr, nullptr};  // fork, logits done
    bool two = !fwd_logits && cudaStreamCreateWithFlags(&aux, cudaStreamNonBlocking) == cudaSuccess;
    for (int i = 0; i < 2 && two; ++i) two = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming) == cudaSuccess;
    if (two) two = cudaEventRecord(ev[0], stream) == cudaSuccess && cudaStreamWaitEvent(aux, ev[0], 0) == cudaSuccess;
    const cudaStream_t sa = two ? aux : stream;
    if (!fwd_logits) {
        ok(launch_router_logits(c, x, w_r, c.has_router_bias ? b_r : nullptr, reinterpret_cast<float *>(bw + B.logits),
                                w, sa));
        if (two) ok(cudaEventRecord(ev[1], sa));
    }

    // gate-scaled dy per row and the gate gradients
    ok(launch_bwd_slots(c, dy, y_perm, slot_row, gate, dO, dgate, err, stream));
    // pre-activations, recomputed unless the forward kept them: [A | B] (gated) or A (ReLU)
    if (!kept_pre) {
        ok(launch_gemm_rows(c, gated, offsets, N, R, x_perm, w_gate_or_w1, w_up, d, h, AB, 0, nullptr, nullptr,
                            nullptr, 0, 0, nullptr, err, stream));
        if (hs)
            ok(launch_gemm_rows(c, true, nullptr, 0, 0, nullptr, nullptr, nullptr, 0, 0, nullptr, c.T, x,
                                shared_w_gate, shared_w_up, d, hs, AB_sh, err, stream));
    }
    // dH = dO W_out (W_out [d][h] per expert: MN-major, K = d)
    ok(launch_gemm_rows(c, false, offsets, N, R, dO, w_down, nullptr, d, h, dH, hs ? c.T : 0, dy, shared_w_down,
                        nullptr, d, hs, bw + B.dH_sh, err, stream, true, 0, 0));
    // [dA | dB] from the pre-activations
    ok(launch_act_bwd(gated, AB, dH, R, h, dAB, stream));
    if (hs) ok(launch_act_bwd(true, AB_sh, bw + B.dH_sh, c.T, hs, bw + B.dAB_sh, stream));
    // dX = [dA | dB] [W_a ; W_b] (W_a, W_b [h][d] per expert: MN-major, K = Wd split at h)
    ok(launch_gemm_rows(c, false, offsets, N, R, dAB, w_gate_or_w1, gated ? w_up : nullptr, Wd, d, dX, hs ? c.T : 0,
                        bw + B.dAB_sh, shared_w_gate, shared_w_up, 2 * hs, d, bw + B.dX_sh, err, stream, true,
                        gated ? h : 0, hs));
    // weight gradients over each expert's rows, the activations [rows][..] as MN-major operands
    const bool pair_ok = !(c.debug_flags & MOE_DEBUG_FFN_SINGLE);
    const auto rows_op = [&](const void *q, int64_t ld) { return WgOperand{q, ld, R, true}; };
    const auto tok_op = [&](const void *q, int64_t ld) { return WgOperand{q, ld, c.T, true}; };
    const WgOperand none{nullptr, 0, 0, false};
    const char *dAB_up = static_cast<const char *>(dAB) + (size_t)h * 2;
    ok(launch_wgrad(offsets, N, R, rows_op(dO, d), rows_op(hid, h), d, h, dw_down, none, none, 0, nullptr, err,
                    stream, pair_ok));
    ok(launch_wgrad(offsets, N, R, rows_op(dAB, Wd), rows_op(x_perm, d), h, d, dw_gate_or_w1, none, none, 0, nullptr,
                    err, stream, pair_ok));
    if (gated)
        ok(launch_wgrad(offsets, N, R, rows_op(dAB_up, Wd), rows_op(x_perm, d), h, d, dw_up, none, none, 0, nullptr,
                        err, stream, pair_ok));
    if (hs) {
        const char *dABsh = reinterpret_cast<const char *>(bw + B.dAB_sh);
        ok(launch_wgrad(nullptr, 0, 0, none, none, d, hs, nullptr, tok_op(dy, d), tok_op(hid_sh, hs), c.T,
                        dshared_w_down, err, stream, pair_ok));
        ok(launch_wgrad(nullptr, 0, 0, none, none, hs, d, nullptr, tok_op(dABsh, 2 * hs), tok_op(x, d), c.T,
                        dshared_w_gate, err, stream, pair_ok));
        ok(launch_wgrad(nullptr, 0, 0, none, none, hs, d, nullptr, tok_op(dABsh + (size_t)hs * 2, 2 * hs),
                        tok_op(x, d), c.T, dshared_w_up, err, stream, pair_ok));
    }
    // router: dL, dx_router, dW_r, db
    if (two) ok(cudaStreamWaitEvent(stream, ev[1], 0));
    ok(launch_router_bwd(c, x, w_r, logits, idx, gate, B, bw, aux_coef, z_coef, dw_r, c.has_router_bias ? db_r : nullptr,
                         err, pair_ok, stream));
    // dx = dy + sum_j dX_r + dX_shared + dx_router
    ok(launch_bwd_dx(c, dy, dX, slot_row, hs ? bw + B.dX_sh : nullptr, reinterpret_cast<const float *>(bw + B.dxr), dx,
                     err, stream));
    // the stream and events are released once their work completes
    for (cudaEvent_t q : ev)
        if (q) cudaEventDestroy(q);
    if (aux) cudaStreamDestroy(aux);
    return to_status(e);
}

moe_status moe_dispatch(const moe_config *cfg, const void *x, const int32_t *perm_token,
                        const int32_t *expert_offsets, void *x_perm, void *ws, size_t ws_bytes,
                        cudaStream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    if (!x || !perm_token || !expert_offsets || !x_perm) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(x_perm)) return MOE_ERR_INVALID_ARG;
    uint32_t *err = nullptr;
    if (ws) {
        if ((st = check_ws(ws, ws_bytes, 4)) != MOE_OK) return st;
        err = static_cast<uint32_t *>(ws);
    }
    return to_status(launch_dispatch(*cfg, x, perm_token, expert_offsets, x_perm, err, stream));
}

moe_status moe_grouped_ffn(const moe_config *cfg, const void *x_perm, const int32_t *expert_offsets,
                           const void *w_gate_or_w1, const void *w_up, const void *w_down, void *y_perm,
                           void *ws, size_t ws_bytes, cudaStream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    const moe_config &c = *cfg;
    if (!x_perm || !expert_offsets || !w_gate_or_w1 || !w_down || !y_perm) return MOE_ERR_INVALID_ARG;
    if (c.act == MOE_ACT_SILU_GATED && !w_up) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x_perm) || !aligned16(w_gate_or_w1) || !aligned16(w_down) || !aligned16(y_perm) ||
        (w_up && !aligned16(w_up)))
        return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(c);
    if ((st = check_ws(ws, ws_bytes, L.hid_sh)) != MOE_OK) return st;
    uint8_t *w = static_cast<uint8_t *>(ws);
    FfnGroup g{};
    g.offsets = expert_offsets;
    g.n_seg = c.N;
    g.a_rows = max_rows(c);
    g.a = x_perm;
    g.w_a = w_gate_or_w1;
    g.w_b = c.act == MOE_ACT_SILU_GATED ? w_up : nullptr;
    g.w_out = w_down;
    g.hid = w + L.hid;
    g.out = y_perm;
    g.h = c.h;
    g.act = c.act;
    return to_status(run_ffn(c, g, reinterpret_cast<uint32_t *>(w + L.err), stream));
}

moe_status moe_combine(const moe_config *cfg, const void *x, const void *y_perm, const int32_t *slot_row,
                       const float *topk_gate, const void *shared_w_gate, const void *shared_w_up,
                       const void *shared_w_down, void *y, void *ws, size_t ws_bytes, cudaStream_t stream) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    const moe_config &c = *cfg;
    if (c.routing != MOE_ROUTING_TOKEN_CHOICE) return MOE_ERR_UNSUPPORTED;
    if (!x || !y_perm || !slot_row || !topk_gate || !y) return MOE_ERR_INVALID_ARG;
    if (c.h_shared && (!shared_w_gate || !shared_w_up || !shared_w_down)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y_perm) || !aligned16(y)) return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(c);
    if ((st = check_ws(ws, ws_bytes, L.offsets)) != MOE_OK) return st;
    uint8_t *w = static_cast<uint8_t *>(ws);
    uint32_t *err = reinterpret_cast<uint32_t *>(w + L.err);
    const void *s_out = nullptr;
    if (c.h_shared) {
        cudaError_t e = run_shared_expert(c, x, shared_w_gate, shared_w_up, shared_w_down, w, L, err, stream);
        if (e != cudaSuccess) return MOE_ERR_CUDA;
        s_out = w + L.s_out;
    }
    return to_status(launch_combine(c, x, y_perm, s_out, slot_row, topk_gate, y, err, stream));
}

// Expert Choice: every expert takes Ce = min(C, T) tokens.
__global__ void k_fill_counts(int32_t *a, int32_t *b, int n, int32_t v) {
    moe::pdl_enter();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n) {
        if (a) a[i] = v;
        if (b) b[i] = v;
    }
}

static cudaError_t fill_counts(const moe_config &c, int32_t *routed, int32_t *kept, cudaStream_t s) {
    return moe::launch_pdl(k_fill_counts, dim3((c.N + 255) / 256), dim3(256), 0, s, routed, kept, c.N,
                      (int32_t)(max_rows(c) / c.N));
}

static moe_status forward_impl(const moe_config *cfg, const void *x, const float *w_r, const float *b_r,
                               const void *w_gate_or_w1, const void *w_up, const void *w_down,
                               const void *shared_w_gate, const void *shared_w_up,
                               const void *shared_w_down, void *y, int32_t *topk_idx, float *topk_gate,
                               int32_t *counts_routed, int32_t *counts_kept, float *aux, void *ws,
                               size_t ws_bytes, cudaStream_t stream, cudaEvent_t *ev,
                               unsigned ev_flags = cudaEventRecordDefault) {
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    const moe_config &c = *cfg;
    const PdlScope pdl(cfg);
    if (!x || !w_r || !w_gate_or_w1 || !w_down || !y) return MOE_ERR_INVALID_ARG;
    if (c.act == MOE_ACT_SILU_GATED && !w_up) return MOE_ERR_INVALID_ARG;
    if (c.has_router_bias && !b_r) return MOE_ERR_INVALID_ARG;
    if (c.h_shared && (!shared_w_gate || !shared_w_up || !shared_w_down)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_r) || !aligned16(w_gate_or_w1) || !aligned16(w_down) ||
        !aligned16(y) || (w_up && !aligned16(w_up)))
        return MOE_ERR_INVALID_ARG;
    const WsLayout L = ws_layout(c);
    if ((st = check_ws(ws, ws_bytes, L.total)) != MOE_OK) return st;
    uint8_t *w = static_cast<uint8_t *>(ws);
    uint32_t *err = reinterpret_cast<uint32_t *>(w + L.err);
    // Under stream capture an event record only orders the capture unless it is
    // external; external records become graph nodes that record on every launch.
    auto mark = [&](int i) { return ev ? cudaEventRecordWithFlags(ev[i], stream, ev_flags) : cudaSuccess; };

    const bool ec = c.routing == MOE_ROUTING_EXPERT_CHOICE;
    if (ec && (topk_idx || topk_gate || aux)) return MOE_ERR_INVALID_ARG;  // token-choice outputs
    RouterOut o;
    o.topk_idx = topk_idx ? topk_idx : reinterpret_cast<int32_t *>(w + L.topk_idx);
    o.topk_gate = topk_gate ? topk_gate : reinterpret_cast<float *>(w + L.topk_gate);
    o.counts_routed = counts_routed;
    o.counts_kept = counts_kept;
    o.expert_offsets = reinterpret_cast<int32_t *>(w + L.offsets);
    o.slot_row = reinterpret_cast<int32_t *>(w + L.slot_row);
    o.perm_token = reinterpret_cast<int32_t *>(w + L.perm_token);
    o.aux = aux ? aux : reinterpret_cast<float *>(w + L.aux);
    int32_t *ec_tok_ptr = reinterpret_cast<int32_t *>(w + L.ec_tok_ptr);
    int32_t *ec_tok_rows = reinterpret_cast<int32_t *>(w + L.ec_tok_rows);
    float *ec_row_gate = reinterpret_cast<float *>(w + L.ec_row_gate);
    if (mark(0) != cudaSuccess) return MOE_ERR_CUDA;
    cudaError_t e;
    if (ec) {
        float *logits = reinterpret_cast<float *>(w + L.logits);
        e = launch_router_logits(c, x, w_r, c.has_router_bias ? b_r : nullptr, logits, w, stream);
        if (e == cudaSuccess)
            e = launch_expert_choice(c, logits, o.expert_offsets, o.perm_token, ec_row_gate, ec_tok_ptr, ec_tok_rows,
                                     w, stream);
        if (e == cudaSuccess && (counts_routed || counts_kept))
            e = fill_counts(c, counts_routed, counts_kept, stream);
    } else {
        e = launch_router(c, x, w_r, c.has_router_bias ? b_r : nullptr, o, w, stream);
    }
    if (e != cudaSuccess || mark(1) != cudaSuccess) return MOE_ERR_CUDA;

    void *x_perm = w + L.x_perm, *y_perm = w + L.y_perm;
    e = ec ? launch_dispatch(c, x, o.perm_token, o.expert_offsets, x_perm, err, stream)
           : launch_dispatch_tokens(c, x, o.slot_row, x_perm, err, stream);
    if (e != cudaSuccess || mark(2) != cudaSuccess) return MOE_ERR_CUDA;

    FfnGroup g{};
    g.offsets = o.expert_offsets;
    g.n_seg = c.N;
    g.a_rows = max_rows(c);
    g.a = x_perm;
    g.w_a = w_gate_or_w1;
    g.w_b = c.act == MOE_ACT_SILU_GATED ? w_up : nullptr;
    g.w_out = w_down;
    g.hid = w + L.hid;
    g.out = y_perm;
    g.h = c.h;
    g.act = c.act;
    g.mid_event = ev ? ev[3] : nullptr;
    g.event_flags = ev_flags;
    const bool keep = saves_preact(c);
    g.pre = keep ? w + L.preact : nullptr;
    if (c.h_shared) {
        g.sh_rows = c.T;
        g.sh_a = x;
        g.sh_w_gate = shared_w_gate;
        g.sh_w_up = shared_w_up;
        g.sh_w_down = shared_w_down;
        g.sh_hid = w + L.hid_sh;
        g.sh_out = w + L.s_out;
        g.h_sh = c.h_shared;
        g.sh_pre = keep ? w + L.preact_sh : nullptr;
    }
    e = run_ffn(c, g, err, stream);
    if (e != cudaSuccess || mark(4) != cudaSuccess) return MOE_ERR_CUDA;

    if (ec)
        e = launch_combine_ec(c, x, y_perm, c.h_shared ? w + L.s_out : nullptr, ec_tok_ptr, ec_tok_rows, ec_row_gate,
                              y, err, stream);
    else
        e = launch_combine(c, x, y_perm, c.h_shared ? w + L.s_out : nullptr, o.slot_row, o.topk_gate, y, err,
                           stream);
    if (e != cudaSuccess || mark(5) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

moe_status moe_forward(const moe_config *cfg, const void *x, const float *w_r, const float *b_r,
                       const void *w_gate_or_w1, const void *w_up, const void *w_down,
                       const void *shared_w_gate, const void *shared_w_up, const void *shared_w_down,
                       void *y, int32_t *topk_idx, float *topk_gate, int32_t *counts_routed,
                       int32_t *counts_kept, float *aux, void *ws, size_t ws_bytes, cudaStream_t stream) {
    return forward_impl(cfg, x, w_r, b_r, w_gate_or_w1, w_up, w_down, shared_w_gate, shared_w_up,
                        shared_w_down, y, topk_idx, topk_gate, counts_routed, counts_kept, aux, ws, ws_bytes,
                        stream, nullptr);
}

moe_status moe_forward_profiled(const moe_config *cfg, const void *x, const float *w_r, const float *b_r,
                                const void *w_gate_or_w1, const void *w_up, const void *w_down,
                                const void *shared_w_gate, const void *shared_w_up,
                                const void *shared_w_down, void *y, int32_t *topk_idx, float *topk_gate,
                                int32_t *counts_routed, int32_t *counts_kept, float *aux, void *ws,
                                size_t ws_bytes, cudaStream_t stream, cudaEvent_t *events, int32_t n_events) {
    if (!events || n_events != 6) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < 6; ++i)
        if (!events[i]) return MOE_ERR_INVALID_ARG;
    return forward_impl(cfg, x, w_r, b_r, w_gate_or_w1, w_up, w_down, shared_w_gate, shared_w_up,
                        shared_w_down, y, topk_idx, topk_gate, counts_routed, counts_kept, aux, ws, ws_bytes,
                        stream, events);
}

struct moe_forward_graph_s {
    cudaGraph_t graph;
    cudaGraphExec_t exec;
};

moe_status moe_forward_graph_create(const moe_config *cfg, const void *x, const float *w_r, const float *b_r,
                                    const void *w_gate_or_w1, const void *w_up, const void *w_down,
                                    const void *shared_w_gate, const void *shared_w_up,
                                    const void *shared_w_down, void *y, int32_t *topk_idx, float *topk_gate,
                                    int32_t *counts_routed, int32_t *counts_kept, float *aux, void *ws,
                                    size_t ws_bytes, cudaEvent_t *events, int32_t n_events,
                                    moe_forward_graph *out) {
    if (!out) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    if (n_events != 0 && (n_events != 6 || !events)) return MOE_ERR_INVALID_ARG;
    for (int i = 0; i < n_events; ++i)
        if (!events[i]) return MOE_ERR_INVALID_ARG;
    // Config and workspace are checked before a stream or a capture exists; the pointer
    // checks run inside forward_impl, which returns before its first launch on an error.
    moe_status st = validate(cfg);
    if (st != MOE_OK) return st;
    if ((st = check_ws(ws, ws_bytes, ws_layout(*cfg).total)) != MOE_OK) return st;
    cudaStream_t cs;
    if (cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess) return MOE_ERR_CUDA;
    cudaGraph_t graph = nullptr;
    if (cudaStreamBeginCapture(cs, cudaStreamCaptureModeRelaxed) != cudaSuccess) {
        cudaStreamDestroy(cs);
        return MOE_ERR_CUDA;
    }
    st = forward_impl(cfg, x, w_r, b_r, w_gate_or_w1, w_up, w_down, shared_w_gate, shared_w_up, shared_w_down, y,
                      topk_idx, topk_gate, counts_routed, counts_kept, aux, ws, ws_bytes, cs,
                      n_events ? events : nullptr, cudaEventRecordExternal);
    const cudaError_t ce = cudaStreamEndCapture(cs, &graph);
    cudaStreamDestroy(cs);
    if (st == MOE_OK && ce != cudaSuccess) st = MOE_ERR_CUDA;
    if (st != MOE_OK) {
        if (graph) cudaGraphDestroy(graph);
        return st;
    }
    cudaGraphExec_t exec = nullptr;
    if (cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess) {
        cudaGraphDestroy(graph);
        return MOE_ERR_CUDA;
    }
    auto *g = new (std::nothrow) moe_forward_graph_s{graph, exec};
    if (!g) {
        cudaGraphExecDestroy(exec);
        cudaGraphDestroy(graph);
        return MOE_ERR_CUDA;
    }
    *out = g;
    return MOE_OK;
}

moe_status moe_forward_graph_launch(moe_forward_graph graph, cudaStream_t stream) {
    if (!graph) return MOE_ERR_INVALID_ARG;
    return cudaGraphLaunch(graph->exec, stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_forward_graph_destroy(moe_forward_graph graph) {
    if (!graph) return MOE_OK;
    const bool ok = cudaGraphExecDestroy(graph->exec) == cudaSuccess && cudaGraphDestroy(graph->graph) == cudaSuccess;
    delete graph;
    return ok ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_check_error(void *ws, cudaStream_t stream) {
    if (!ws) return MOE_ERR_WORKSPACE;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_ERR_CUDA;
    uint32_t word = 0;
    if (cudaMemcpy(&word, ws, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (word && cudaMemset(ws, 0, sizeof(word)) != cudaSuccess) return MOE_ERR_CUDA;
    if (word & kErrTimeout) return MOE_ERR_TIMEOUT;
    if (word & kErrFault) return MOE_ERR_DEVICE_FAULT;
    return MOE_OK;
}

const char *moe_status_str(moe_status s) {
    switch (s) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_WORKSPACE: return "MOE_ERR_WORKSPACE";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_TIMEOUT: return "MOE_ERR_TIMEOUT";
        case MOE_ERR_DEVICE_FAULT: return "MOE_ERR_DEVICE_FAULT";
    }
    return "MOE_ERR_UNKNOWN";
}

}  // extern "C"
