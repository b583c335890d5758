/*
 * moe.h — C ABI of libmoe.so: the forward pass of one sparse Mixture-of-Experts
 * layer on one B300 GPU (sm_103a).
 *
 * The layer computes, for every token t with hidden state x_t (the pages' u_t):
 *
 *     y_t = x_t + S(x_t) + sum_{j < k, slot j kept} g_{t,j} * FFN_{e_{t,j}}(x_t)
 *
 * "Mixture-of-Experts (MoE)" ml-notes page (DeepSeekMoE layer equation: a sum of
 * gated expert FFNs plus the residual, with s = softmax over all N affinities and
 * Topk); "MoE: Choosing Which MLPs to Use for Each Token" (sections "Router:
 * Selecting Experts and Computing Weights", "From Router to Combine", "Shared
 * Expert"); "Mixture of Experts (MoE)" glossary (top-k gating, expert capacity
 * with residual bypass of overflow, auxiliary load-balancing loss); "Switch
 * Transformers ... explained" (top-1 routing, capacity, router in higher
 * precision).
 *
 * The calls follow the pages' Router -> Dispatch -> Expert computation ->
 * Combine sequence; moe_forward runs all of them.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Every pointer argument is a DEVICE pointer unless stated otherwise; the
 *    config is a HOST pointer. The caller owns all memory. The library never
 *    allocates device memory and never synchronises (moe_check_error excepted):
 *    every call enqueues kernels on `stream` and returns. Two calls hold other CUDA
 *    objects: moe_forward_graph_create (a graph, captured on a private stream) and
 *    moe_backward (an auxiliary stream and events for the duration of the call).
 *  - Layouts are row-major. Activations x, x_perm, y_perm, y: [rows][d].
 *    Router weight w_r: [d][N] fp32; router bias b_r: [N] fp32.
 *    Expert weights use the [out][in] (nn.Linear) layout:
 *      SiLU-gated experts: w_gate, w_up [N][h][d], w_down [N][d][h];
 *      ReLU experts:       w1 (passed as w_gate) [N][h][d], w_up NULL, w2 (as w_down) [N][d][h];
 *      shared expert:      shared_w_gate, shared_w_up [h_shared][d], shared_w_down [d][h_shared].
 *  - Element type of activations and expert weights: cfg->dtype (fp32 or bf16).
 *    Router math is fp32 in both cases; gates are fp32.
 *  - Worst-case row count of the dispatched buffers x_perm / y_perm:
 *      R_max = T*k                      without a capacity limit,
 *      R_max = min(T*k, N*C)            with capacity C = ceil(T*cap_num / (N*cap_den)).
 *    The actual row count R = expert_offsets[N] stays on the device.
 *  - Workspace: `ws` is a device buffer of at least moe_workspace_size(cfg)
 *    bytes, 256-byte aligned, owned by the caller, reused across calls. It holds
 *    intermediate arrays and the device error word. Concurrent calls on different
 *    streams must use different workspaces.
 *  - Errors: host-side validation returns a status before anything is enqueued.
 *    A failed launch returns MOE_ERR_CUDA. Faults detected on the device (index
 *    out of range, bounded waits that ran out) are recorded in the workspace's
 *    error word and reported by moe_check_error.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,   /* null pointer, size out of range, bad enum value      */
    MOE_ERR_UNSUPPORTED = 2,   /* valid layer, but a shape/dtype this build does not run */
    MOE_ERR_WORKSPACE = 3,     /* workspace missing, too small or misaligned            */
    MOE_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed           */
    MOE_ERR_TIMEOUT = 5,       /* a bounded wait inside a kernel ran out                */
    MOE_ERR_DEVICE_FAULT = 6   /* a kernel saw an out-of-range index and skipped it     */
} moe_status;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;

/* Gating convention.
 * MOE_SOFTMAX_THEN_TOPK: softmax over all N logits, keep the top-k probabilities
 *   as gates without renormalising (DeepSeekMoE layer equation; glossary's
 *   gating-network paragraph; Switch top-1 uses this with k = 1).
 * MOE_TOPK_THEN_SOFTMAX: keep the k largest logits, softmax over those k only
 *   (the worked example in "Router: Selecting Experts and Computing Weights"). */
typedef enum { MOE_SOFTMAX_THEN_TOPK = 0, MOE_TOPK_THEN_SOFTMAX = 1 } moe_gating;

/* Expert FFN. SILU_GATED: W_down (SiLU(W_gate x) * (W_up x)); RELU: W2 max(0, W1 x). */
typedef enum { MOE_ACT_SILU_GATED = 0, MOE_ACT_RELU = 1 } moe_act;

/* Who chooses: every token its top-k experts, or every expert its top tokens
 * ("Mixture of Experts (MoE)" glossary, sparse-MoE list: Expert Choice inverts the
 * routing). Expert Choice needs a capacity factor cap_num/cap_den > 0 (the average
 * number of experts per token): each expert takes min(C, T) tokens, C =
 * ceil(T * cap_num / (N * cap_den)); k and gating are not used; T <= 16384. */
typedef enum { MOE_ROUTING_TOKEN_CHOICE = 0, MOE_ROUTING_EXPERT_CHOICE = 1 } moe_routing;

typedef struct {
    int32_t T;                /* tokens, 1..65536                                    */
    int32_t d;                /* model dim: multiple of 8 (fp32) or of 64 (bf16)    */
    int32_t N;                /* routed experts, 1..256                              */
    int32_t k;                /* experts per token, 1..min(N, 8)                     */
    int32_t h;                /* routed expert hidden size, same multiple rule as d  */
    int32_t h_shared;         /* shared expert hidden size, 0 = no shared expert     */
    int32_t dtype;            /* moe_dtype                                           */
    int32_t gating;           /* moe_gating                                          */
    int32_t act;              /* moe_act (the shared expert is always SiLU-gated)    */
    int32_t cap_num, cap_den; /* capacity factor cap_num/cap_den; 0/0 = no limit     */
    int32_t has_router_bias;  /* 1: b_r is read and added to the logits              */
    int32_t debug_flags;      /* MOE_DEBUG_* bits, 0 in normal use                   */
    int32_t routing;          /* moe_routing: token choice (top-k) or Expert Choice  */
    int32_t save_preact;      /* 1: moe_forward also keeps the experts' pre-activations
                                 in the workspace and moe_backward reads them instead of
                                 recomputing them (see moe_backward); 0 or 1          */
} moe_config;

/* debug_flags bits */
#define MOE_DEBUG_FORCE_SIMT_FFN 1u  /* run the expert FFN on the CUDA-core kernel even for bf16 */
#define MOE_DEBUG_FFN_PAIR 2u        /* bf16: always use the row-tile CTA-pair kernel (256-row tiles)  */
#define MOE_DEBUG_FFN_SINGLE 4u      /* bf16: always use the row-tile single-CTA kernel (128-row tiles),
                                        in moe_backward also for the weight gradients */
#define MOE_DEBUG_FFN_SWAP 8u        /* bf16: use the weights-as-M CTA-pair kernel (token tiles 32..256) */
#define MOE_DEBUG_NO_PDL 16u         /* moe_forward: launch every kernel only after its predecessor has
                                        completed (no programmatic dependent launch)             */
#define MOE_DEBUG_ROUTER_STALL 32u   /* exercises the timeout path of the bounded waits: the router
                                        kernel for N <= 32 (token choice) copies nothing into its
                                        staging ring and its waits give up after about 1 ms, so the
                                        call records MOE_ERR_TIMEOUT (read by moe_check_error) with
                                        no copy in flight. Every output of the call is then
                                        meaningless (later kernels of the call still check every
                                        index they read). Ignored for N > 32.                      */
/* Without these flags bf16 experts run on the row-tile pair kernel when the row buffers hold at
   least 224 rows per expert, else on the row-tile single-CTA kernel; the backward's weight
   gradients run on CTA pairs when the gradient has at least 256 rows. */

/* Validate a config on the host. No CUDA call is made. */
moe_status moe_validate_config(const moe_config *cfg);

/* Bytes of workspace every call below needs for `cfg` (the maximum over calls);
 * 0 when the config is invalid. No CUDA call is made. */
size_t moe_workspace_size(const moe_config *cfg);

/* Bytes of workspace the router calls need for `cfg` (moe_router_topk,
 * moe_router_topk_train, moe_router_shard_stats / _assign): the leading part of
 * the full workspace, smaller than moe_workspace_size(cfg). 0 when the config is
 * invalid or uses Expert Choice routing. No CUDA call is made. */
size_t moe_router_workspace_size(const moe_config *cfg);

/* Byte offset in the workspace of the pre-activations moe_forward keeps when
 * cfg->save_preact = 1 for the backward (router and experts learn together by
 * backpropagation, "Mixture of Experts (MoE)" glossary; the expert products of "MoE:
 * Choosing Which MLPs to Use for Each Token", "Dense MLP and MoE"; see moe_backward):
 * shared = 0, the routed experts' rows
 * [R_max][W] bf16 in dispatch order (row r of expert e's range holds the token
 * perm_token[r]; W = 2h with X W_gateᵀ in columns [0, h) and X W_upᵀ in [h, 2h), or
 * W = h with X W1ᵀ for ReLU experts); shared = 1, the shared expert's [T][2 h_shared].
 * Rows past the kept row count are not written. SIZE_MAX when the config keeps none
 * (or has no shared expert). No CUDA call is made. */
size_t moe_preact_offset(const moe_config *cfg, int32_t shared);

/* Worst-case dispatched row count R_max for `cfg` (see above); 0 if invalid. */
int64_t moe_max_rows(const moe_config *cfg);

/* Expert capacity C for `cfg`, or 0 when no capacity limit is set / invalid. */
int32_t moe_capacity(const moe_config *cfg);

/*
 * Router: logits, gating, counts, capacity and dispatch order.
 *
 * logits L[t][e] = sum_i x[t][i] * w_r[i][e] (+ b_r[e]) in fp32 ("Noise Top-k
 * Gating" router paragraph; "Router: Selecting Experts ..." Figure 2; Switch
 * explainer "Making it work" for the fp32 router), summed in one fixed order so
 * that the routing is reproducible bit for bit:
 *   - the features are taken in blocks of 8 (block b = features 8b .. 8b+7);
 *   - partial sum l (l = 0 .. 31) starts at 0 and takes every block b with
 *     b mod 32 = l, in increasing b, with one correctly rounded fused
 *     multiply-add per feature in increasing feature order;
 *   - the 32 partials are combined by five pairwise rounds
 *     p_l <- p_l + p_(l xor o) for o = 16, 8, 4, 2, 1 (each sum rounded to fp32),
 *     and the logit is p_0;
 *   - the bias, when present, is added last (one fp32 addition).
 * Top-k by logit, largest first, lower expert index first on equal logits (-0 and
 * +0 are equal); a NaN logit ranks below every number and is chosen only when
 * fewer than k experts have a numeric logit. Gates per cfg->gating.
 * Capacity (glossary capacity paragraph; Switch "Making it work"): when set, an
 * expert keeps at most C slots, chosen slot-major (every token's first choice in
 * token order, then every second choice, ...); dropped slots get slot_row = -1
 * and contribute nothing (the token keeps its residual).
 * Kept rows are grouped by expert ascending, token ascending within an expert
 * ("From Router to Combine", Figure 3).
 *
 * Inputs:  x [T][d] (cfg->dtype), w_r [d][N] fp32, b_r [N] fp32 (NULL unless
 *          cfg->has_router_bias).
 * Outputs (device, caller-owned):
 *   topk_idx       int32 [T][k]   selected experts, slot order = descending logit
 *   topk_gate      fp32  [T][k]   gate of each slot
 *   counts_routed  int32 [N]      selections per expert before capacity
 *   counts_kept    int32 [N]      kept slots per expert (= min(routed, C))
 *   expert_offsets int32 [N+1]    exclusive scan of counts_kept; R = offsets[N]
 *   slot_row       int32 [T][k]   row of each slot in the dispatched order, -1 if dropped
 *   perm_token     int32 [R_max]  token of each dispatched row (rows >= R untouched)
 *   aux            fp32  [2]      aux[0] = N * sum_e f_e P_e, aux[1] = mean_e (P_e - 1/N)^2
 *                                 with P_e = mean_t softmax_e, f_e = routed_e / (T k).
 * Any output pointer except topk_idx, topk_gate, slot_row, perm_token and
 * expert_offsets may be NULL (not written).
 */
moe_status moe_router_topk(const moe_config *cfg, const void *x, const float *w_r,
                           const float *b_r, int32_t *topk_idx, float *topk_gate,
                           int32_t *counts_routed, int32_t *counts_kept,
                           int32_t *expert_offsets, int32_t *slot_row, int32_t *perm_token,
                           float *aux, void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Training-time router: moe_router_topk with noisy top-k gating and the router
 * z-loss ("Noise Top-k Gating" page: standard-normal noise, scaled by one scalar
 * noise weight, is added to the raw logits before the top-k choice and is off at
 * inference; "Mixture of Experts (MoE)" glossary: a z-loss penalises large router
 * logits).
 *   noise        fp32 [T][N] standard-normal draws n (sampled by the caller), or NULL
 *                for no noise. The router then works on H = fl(L + fl(w * n)) (the
 *                product and the sum each rounded to fp32): selection, gates,
 *                counts, capacity and aux all use H.
 *   noise_weight the scalar w; must be finite when noise is given.
 *   z_loss       fp32 [1] or NULL: (1/T) sum_t (log sum_e exp L[t,e])^2 on the
 *                noiseless logits L (bias included). The pages print no formula;
 *                this is the reading used.
 * Every other argument, output and error as moe_router_topk. With noise == NULL
 * and z_loss == NULL the results are those of moe_router_topk, bit for bit.
 */
moe_status moe_router_topk_train(const moe_config *cfg, const void *x, const float *w_r,
                                 const float *b_r, const float *noise, float noise_weight,
                                 int32_t *topk_idx, float *topk_gate, int32_t *counts_routed,
                                 int32_t *counts_kept, int32_t *expert_offsets, int32_t *slot_row,
                                 int32_t *perm_token, float *aux, float *z_loss, void *ws,
                                 size_t ws_bytes, cudaStream_t stream);

/*
 * Token-sharded router (one batch split over R ranks in token order: rank 0 holds
 * the first tokens). The capacity rule is global ("Mixture of Experts (MoE)"
 * glossary, capacity-factor paragraph; GShard top-2 in its sparse-MoE list): the
 * first C selections of each expert in priority order are kept, priority being
 * slot-major over the whole batch (every token's first choice in token order, then
 * every second choice, ...). Each rank runs the two phases below on its own tokens
 * with its own workspace; between them the ranks exchange, per expert and slot,
 * their selection counts (and, for the aux loss, per expert the sums of the
 * softmax). cfg describes this rank's shard: T = its tokens, cap_num = cap_den = 0
 * (the global capacity is an argument of phase 2), everything else as for the
 * whole batch.
 *
 * Phase 1: logits, gating (topk_idx, topk_gate as in moe_router_topk) and
 *   slot_counts int32 [N][k]  selections of expert e in slot j on this rank;
 *   prob_sums   fp32  [N]     sum over this rank's tokens of softmax_e, or NULL.
 * The workspace keeps per-tile counts that phase 2 reads: pass the same ws.
 */
moe_status moe_router_shard_stats(const moe_config *cfg, const void *x, const float *w_r,
                                  const float *b_r, int32_t *topk_idx, float *topk_gate,
                                  int32_t *slot_counts, float *prob_sums, void *ws,
                                  size_t ws_bytes, cudaStream_t stream);

/*
 * Phase 2: capacity decisions and dispatch order of this rank's selections.
 *   slot_base        int32 [N][k] (device) global priority of this rank's first
 *                    selection of (e, j): sum over slots j' < j of all ranks' counts
 *                    of (e, j'), plus the counts of (e, j) on ranks before this one;
 *   capacity         global C (0: no limit), e.g. ceil(T_global * cf / N);
 *   global_routed    int32 [N], global_prob_sums fp32 [N], global_T: the sums over all
 *                    ranks, for aux (both may be NULL when aux is NULL);
 *   topk_idx         this rank's selections from phase 1.
 * Outputs as in moe_router_topk for this rank's tokens: counts_kept (may be NULL),
 * expert_offsets, slot_row, perm_token, and aux [2] (or NULL) computed from the
 * global statistics, so every rank gets the batch's aux loss.
 */
moe_status moe_router_shard_assign(const moe_config *cfg, const int32_t *topk_idx,
                                   const int32_t *slot_base, int32_t capacity,
                                   const int32_t *global_routed, const float *global_prob_sums,
                                   int64_t global_T, int32_t *counts_kept, int32_t *expert_offsets,
                                   int32_t *slot_row, int32_t *perm_token, float *aux, void *ws,
                                   size_t ws_bytes, cudaStream_t stream);

/*
 * Expert Choice router (cfg->routing == MOE_ROUTING_EXPERT_CHOICE): every expert
 * picks its top tokens ("Mixture of Experts (MoE)" glossary, sparse-MoE list).
 * Scores S[t][e] = softmax over experts of the fp32 logits (the router's probability
 * distribution), computed in fixed fp32 steps (max, an exponential from Cody-Waite
 * reduction and a degree-7 Taylor series, sum over experts ascending, division) so
 * that the choice is reproducible bit for bit. Expert e keeps the Ce = min(C, T)
 * tokens of largest S[t][e] (lower token first on equal scores), C =
 * ceil(T * cap_num / (N * cap_den)): every expert is full, a token may be chosen by
 * several experts or by none. Outputs (R = N * Ce rows, moe_max_rows(cfg)):
 *   expert_offsets int32 [N+1]  e * Ce
 *   perm_token     int32 [R]    rows e*Ce .. e*Ce+Ce-1: expert e's tokens, ascending
 *   row_gate       fp32  [R]    S[token][e] of each row
 *   token_ptr      int32 [T+1]  token t's rows are token_rows[token_ptr[t] .. token_ptr[t+1])
 *   token_rows     int32 [R]    in expert order
 * Feed perm_token and expert_offsets to moe_dispatch and moe_grouped_ffn as usual,
 * then moe_combine_expert_choice. The workspace must hold moe_workspace_size(cfg).
 */
moe_status moe_router_expert_choice(const moe_config *cfg, const void *x, const float *w_r,
                                   const float *b_r, int32_t *expert_offsets, int32_t *perm_token,
                                   float *row_gate, int32_t *token_ptr, int32_t *token_rows,
                                   void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Expert Choice combine: y_t = x_t + S(x_t) + sum over token t's rows r (expert
 * order) of row_gate[r] * y_perm[r], fp32 accumulation; a token no expert chose
 * gets x_t (+ S(x_t)). Shared expert as in moe_combine.
 */
moe_status moe_combine_expert_choice(const moe_config *cfg, const void *x, const void *y_perm,
                                     const int32_t *token_ptr, const int32_t *token_rows,
                                     const float *row_gate, const void *shared_w_gate,
                                     const void *shared_w_up, const void *shared_w_down, void *y,
                                     void *ws, size_t ws_bytes, cudaStream_t stream);

/*
 * moe_router_topk for callers that cannot allocate device memory. The pages
 * describe no such call; it exists for hosts that forbid allocation after
 * start-up (engines that plan all device memory ahead and call plugins from an
 * enqueue path, services with a fixed memory budget), which cannot hand over a
 * workspace on demand.
 * Same computation, arguments and outputs as moe_router_topk, without the
 * workspace: the router's scratch lives in one static 32 MiB device array of the
 * library, held by every GPU that loads it until the process exits. Configs whose
 * router scratch (moe_router_workspace_size) exceeds 32 MiB are rejected with
 * MOE_ERR_UNSUPPORTED before anything is enqueued (the tiny, Switch, Mixtral and
 * DeepSeekMoE-shaped layers all fit). Nothing is allocated and no allocating
 * routine is called.
 * The first call on a device looks up the array's device address (make that first
 * call before any stream capture). All calls share the array: the error word in
 * it is cleared at the start of each call and is read with
 * moe_router_noalloc_check_error, not moe_check_error; calls that overlap on the
 * GPU race on the array and must be serialised by the caller.
 */
moe_status moe_router_topk_noalloc(const moe_config *cfg, const void *x, const float *w_r,
                                   const float *b_r, int32_t *topk_idx, float *topk_gate,
                                   int32_t *counts_routed, int32_t *counts_kept,
                                   int32_t *expert_offsets, int32_t *slot_row,
                                   int32_t *perm_token, float *aux, cudaStream_t stream);

/*
 * Device error word of moe_router_topk_noalloc on the current device: synchronises
 * `stream`, reads and clears the word, and returns MOE_OK, MOE_ERR_TIMEOUT (a bounded
 * wait ran out: that call's outputs are not written), MOE_ERR_DEVICE_FAULT or
 * MOE_ERR_CUDA. The word covers the calls made since the last call started (each
 * call clears it first), so read it after the call it is meant to check.
 */
moe_status moe_router_noalloc_check_error(cudaStream_t stream);

/*
 * Dispatch: x_perm[r] = x[perm_token[r]] for r < expert_offsets[N]
 * ("From Router to Combine": the original token vectors are sent to the experts
 * that chose them). x [T][d], x_perm [R_max][d] in cfg->dtype. Rows r >= R are
 * not written. A perm_token entry outside [0, T) is skipped and recorded as
 * MOE_ERR_DEVICE_FAULT in the error word (ws may be NULL: no record).
 */
moe_status moe_dispatch(const moe_config *cfg, const void *x, const int32_t *perm_token,
                        const int32_t *expert_offsets, void *x_perm, void *ws,
                        size_t ws_bytes, cudaStream_t stream);

/*
 * Expert computation: each expert e applies its FFN to its rows
 * [expert_offsets[e], expert_offsets[e+1]) of x_perm, independently per row
 * ("From Router to Combine"; glossary: experts are independent FFNs):
 *   SILU_GATED: y_perm[r] = W_down[e] (SiLU(W_gate[e] x_perm[r]) * (W_up[e] x_perm[r]))
 *   RELU:       y_perm[r] = W2[e] max(0, W1[e] x_perm[r])
 * fp32 accumulation; for bf16 the hidden activation is rounded to bf16 between
 * the two products and y_perm is bf16. Rows >= R are not written. The bf16 path
 * runs on tcgen05 tensor cores; fp32 runs on CUDA cores.
 */
moe_status moe_grouped_ffn(const moe_config *cfg, const void *x_perm,
                           const int32_t *expert_offsets, const void *w_gate_or_w1,
                           const void *w_up, const void *w_down, void *y_perm, void *ws,
                           size_t ws_bytes, cudaStream_t stream);

/*
 * Combine: y[t] = x[t] + S(x[t]) + sum_{j: slot_row[t][j] >= 0} topk_gate[t][j] * y_perm[slot_row[t][j]]
 * ("From Router to Combine": weighted sum per original token; "Shared Expert":
 * y = S(x) + R(x); DeepSeekMoE equation: + u_t). The expert terms are summed in
 * fp32 in slot order, then S, then x. S is computed here (SiLU-gated, hidden
 * cfg->h_shared) when cfg->h_shared > 0; the shared_* pointers are then required.
 * A token whose slots were all dropped gets y = x + S(x) (exactly x without a
 * shared expert). y [T][d] in cfg->dtype.
 */
moe_status moe_combine(const moe_config *cfg, const void *x, const void *y_perm,
                       const int32_t *slot_row, const float *topk_gate,
                       const void *shared_w_gate, const void *shared_w_up,
                       const void *shared_w_down, void *y, void *ws, size_t ws_bytes,
                       cudaStream_t stream);

/*
 * Whole layer: router -> dispatch -> experts (+ shared expert) -> combine.
 * With cfg->routing == MOE_ROUTING_EXPERT_CHOICE the router and the combine are the
 * Expert Choice ones; topk_idx, topk_gate and aux must then be NULL and
 * counts_routed / counts_kept (when given) receive Ce for every expert.
 * Same inputs as above; outputs y [T][d] and, when non-NULL, topk_idx, topk_gate,
 * counts_routed, counts_kept (as in moe_router_topk) and aux [2]. The dispatch
 * order, x_perm, hidden activations and y_perm live in the workspace.
 */
moe_status moe_forward(const moe_config *cfg, const void *x, const float *w_r,
                       const float *b_r, const void *w_gate_or_w1, const void *w_up,
                       const void *w_down, const void *shared_w_gate,
                       const void *shared_w_up, const void *shared_w_down, void *y,
                       int32_t *topk_idx, float *topk_gate, int32_t *counts_routed,
                       int32_t *counts_kept, float *aux, void *ws, size_t ws_bytes,
                       cudaStream_t stream);

/*
 * Backward of the layer (token choice, bf16): the gradients of
 *   Loss = sum(dy * y) + aux_coef * aux[0] + z_coef * z
 * with the routing of the preceding moe_forward held fixed (selections and capacity
 * are piecewise constant; f_e of the aux loss is held fixed too). Chain rule through
 * the combine ("From Router to Combine"), the experts (O = H W_outᵀ with H =
 * SiLU(X W_gateᵀ) ⊙ X W_upᵀ, or max(0, X W1ᵀ)), the shared expert and the router
 * (gates from the fp32 logits; aux N sum_e f_e P_e; z = mean_t (log sum_e exp L)²).
 * Call it after moe_forward with the same inputs and the same workspace ws (it
 * reads the saved dispatch order, rows, expert outputs and hidden activations, and
 * for N > 32 the router logits);
 * topk_idx / topk_gate: the buffers given to that moe_forward, or NULL if it was
 * given NULL. bws: backward scratch of moe_backward_workspace_size(cfg) bytes.
 *   dy [T][d] bf16 in;  dx [T][d] bf16, dw_r [d][N] fp32, db_r [N] fp32 (NULL or
 *   ignored without a router bias), dw_gate_or_w1 / dw_up [N][h][d], dw_down
 *   [N][d][h], dshared_* shaped like the shared weights — all bf16 outputs.
 * x, w_r, dy, dx, the expert and shared-expert weights and their gradients must be
 * 16-byte aligned (MOE_ERR_INVALID_ARG otherwise).
 * The backward needs the experts' pre-activations (X W_gateᵀ and X W_upᵀ, or X W1ᵀ, and
 * the shared expert's): with cfg->save_preact = 1, moe_forward stores them in ws as its
 * first product computes them (bf16 token choice on the tensor-core kernels; not with
 * MOE_DEBUG_FORCE_SIMT_FFN or MOE_DEBUG_FFN_SWAP) and moe_backward reads them, else
 * moe_backward recomputes them; moe_forward and moe_backward must then get the same
 * cfg. The row products read the expert weights, and the weight gradients (which
 * reduce over each expert's rows on the tensor cores) the activations, in their own
 * layouts: nothing is transposed or copied. For N <= 32 the router logits are
 * recomputed on a non-blocking auxiliary stream that the call creates, joins to
 * `stream` with an event before the router's backward, and releases before returning
 * (its work completes asynchronously, ordered before the work enqueued on `stream`
 * after the call); if the stream cannot be created, everything runs on `stream`. fp32 and
 * Expert Choice configs return MOE_ERR_UNSUPPORTED.
 */
size_t moe_backward_workspace_size(const moe_config *cfg);
moe_status moe_backward(const moe_config *cfg, const void *x, const float *w_r, const float *b_r,
                        const void *w_gate_or_w1, const void *w_up, const void *w_down,
                        const void *shared_w_gate, const void *shared_w_up,
                        const void *shared_w_down, const int32_t *topk_idx,
                        const float *topk_gate, const void *dy, float aux_coef, float z_coef,
                        void *dx, float *dw_r, float *db_r, void *dw_gate_or_w1, void *dw_up,
                        void *dw_down, void *dshared_w_gate, void *dshared_w_up,
                        void *dshared_w_down, void *ws, size_t ws_bytes, void *bws,
                        size_t bws_bytes, cudaStream_t stream);

/*
 * moe_forward with timing instrumentation: the same launches and results, plus
 * events[0..5] recorded on `stream` before the router, after the router, after
 * dispatch, after the first expert product (hidden activations), after the second
 * expert product (expert outputs) and after combine. `events` is a host array of
 * n_events == 6 caller-created CUDA events. Not part of the layer's math.
 */
moe_status moe_forward_profiled(const moe_config *cfg, const void *x, const float *w_r,
                                const float *b_r, const void *w_gate_or_w1, const void *w_up,
                                const void *w_down, const void *shared_w_gate,
                                const void *shared_w_up, const void *shared_w_down, void *y,
                                int32_t *topk_idx, float *topk_gate, int32_t *counts_routed,
                                int32_t *counts_kept, float *aux, void *ws, size_t ws_bytes,
                                cudaStream_t stream, cudaEvent_t *events, int32_t n_events);

/*
 * The whole forward captured once as a CUDA graph and replayed (the layer's steps as
 * in moe_forward; for small layers the host's launch work, not the GPU, bounds a
 * stream of moe_forward calls, and one graph launch replaces its seven to ten kernel
 * launches).
 *
 * moe_forward_graph_create validates its arguments exactly as moe_forward does and
 * returns that status without capturing anything on an error; otherwise it captures
 * one moe_forward with these arguments on a private stream and instantiates it into
 * *out. Nothing runs on the GPU during create. Every pointer is baked into the graph:
 * the caller keeps all buffers alive and in place until moe_forward_graph_destroy and
 * changes inputs (x, weights) by writing into the same buffers; each launch then
 * computes the layer from their current contents, routing included (all
 * data-dependent sizes stay on the device). `events` is NULL (n_events 0) or six
 * caller-created events recorded at the stages of moe_forward_profiled on every
 * launch.
 *
 * moe_forward_graph_launch enqueues one forward on `stream` (any stream of the device
 * the graph was created on); launches on one stream run in order, and two launches of
 * one graph must not overlap (they share the workspace). Device errors go to the
 * error word of ws as for moe_forward. moe_forward_graph_destroy frees the graph
 * (NULL is a no-op) after the caller has synchronised with its last launch.
 * Errors: MOE_ERR_INVALID_ARG (NULL out or graph, n_events not 0 or 6), the statuses
 * of moe_forward, MOE_ERR_CUDA if capture or instantiation fails.
 */
typedef struct moe_forward_graph_s *moe_forward_graph;
moe_status moe_forward_graph_create(const moe_config *cfg, const void *x, const float *w_r,
                                    const float *b_r, const void *w_gate_or_w1, const void *w_up,
                                    const void *w_down, const void *shared_w_gate,
                                    const void *shared_w_up, const void *shared_w_down, void *y,
                                    int32_t *topk_idx, float *topk_gate, int32_t *counts_routed,
                                    int32_t *counts_kept, float *aux, void *ws, size_t ws_bytes,
                                    cudaEvent_t *events, int32_t n_events, moe_forward_graph *out);
moe_status moe_forward_graph_launch(moe_forward_graph graph, cudaStream_t stream);
moe_status moe_forward_graph_destroy(moe_forward_graph graph);

/* Synchronise `stream`, read and clear the device error word in `ws`.
 * Returns MOE_OK, MOE_ERR_TIMEOUT, MOE_ERR_DEVICE_FAULT or MOE_ERR_CUDA. */
moe_status moe_check_error(void *ws, cudaStream_t stream);

/* Static string naming a status. */
const char *moe_status_str(moe_status s);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
