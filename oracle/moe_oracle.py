"""Plain CPU oracle for the forward pass of one sparse Mixture-of-Experts layer.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import this
module. The CUDA product path never imports, calls or links anything here, and
nothing here imports the product package.

Every step follows the pages literally, in their order, and is written for a
reader to check by eye rather than for speed:

  router logits -> softmax / top-k gates -> counts, capacity, aux loss
  -> dispatch (group rows by expert) -> expert FFN per group
  -> combine (gate-weighted sum per token) + shared expert + residual.

Precision. The router logits are fp32 with one fixed summation order (see
``router_logits.c``: 32 blocked fma partials and a pairwise combine), because the top-k decision is an integer result that the
CUDA router must reproduce bit for bit; the decision is therefore taken in the
kernel's precision on identical values. Everything after the logits (softmax,
gates, aux loss, expert FFNs, combine) is float64 on the exact values of the
(bf16 or fp32) inputs.

Page references used below:
  [MoE glossary]   "Mixture of Experts (MoE)" glossary page (inferensys.com)
  [Switch]         "Switch Transformers: Mixture of Experts explained" (thelatentdaily.com)
  [Noisy top-k]    "Noise Top-k Gating" glossary page (inferensys.com)
  [Choosing MLPs]  "MoE: Choosing Which MLPs to Use for Each Token" (llm-systems-engineering)
  [DeepSeekMoE eq] "Mixture-of-Experts (MoE)" ml-notes page, the MoE-layer equation
                   h_t = sum_i g_{i,t} FFN_i(u_t) + u_t quoted from DeepSeekMoE.

Readings where the pages are silent:
  * top-k selects by logit, descending, lower expert index first on equal values;
  * softmax-then-top-k gates are not renormalised (DeepSeekMoE eq.);
  * capacity C = ceil(T * cf / N); priority is slot-major (all first choices in
    token order, then all second choices, ...); a dropped slot contributes 0 and
    the remaining gates are not renormalised;
  * kept rows are grouped by expert ascending, token ascending inside a group;
  * aux loss is reported in two forms (Switch form and the variance form);
  * expert FFNs have no biases; SiLU(z) = z / (1 + exp(-z));
  * noisy top-k: H = fl(L + fl(w n)) drives everything after the logits; the z-loss
    is mean_t (log sum_e exp L)^2 on the noiseless logits;
  * Expert Choice: scores = the softmax over experts in fixed fp32 steps
    (expert_choice.c); expert e keeps the min(C, T) highest-scoring tokens, lower
    index first on ties, C = ceil(T cf / N); gates are the scores; rows are grouped
    by expert, tokens ascending; a token no expert chose keeps its residual.

Parity pins: the aux-loss *form* has no printed formula on the pages, so which
of the two values "the" auxiliary loss is stays parity unpinned; the
arithmetic of both forms is pinned by closed-form cases in tests/test_oracle.py.
"""
from __future__ import annotations

import ctypes
import pathlib
import subprocess

import numpy as np

_HERE = pathlib.Path(__file__).resolve().parent
_SO = _HERE / "_liboracle.so"
_SRCS = (_HERE / "router_logits.c", _HERE / "expert_choice.c")
_lib = None

GATING_SOFTMAX_THEN_TOPK = "softmax_then_topk"
GATING_TOPK_THEN_SOFTMAX = "topk_then_softmax"


def build(force: bool = False) -> pathlib.Path:
    """Compile the C part of the oracle (plain gcc, no GPU headers)."""
    if force or not _SO.exists() or any(_SO.stat().st_mtime < s.stat().st_mtime for s in _SRCS):
        # -mfma makes fmaf a single instruction; its result is the correctly
        # rounded fused multiply-add either way (libm's fmaf is exact too).
        cmd = ["gcc", "-O3", "-mfma", "-fno-fast-math", "-ffp-contract=off",
               "-shared", "-fPIC", "-o", str(_SO), *map(str, _SRCS), "-lm"]
        subprocess.run(cmd, check=True)
    return _SO


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(str(_SO))
        lib.oracle_router_logits.restype = None
        lib.oracle_router_logits.argtypes = [ctypes.c_long] * 3 + [ctypes.c_void_p] * 4
        lib.oracle_ec_scores.restype = None
        lib.oracle_ec_scores.argtypes = [ctypes.c_long] * 2 + [ctypes.c_void_p] * 2
        lib.oracle_ec_exp_array.restype = None
        lib.oracle_ec_exp_array.argtypes = [ctypes.c_long] + [ctypes.c_void_p] * 2
        _lib = lib
    return _lib


# --------------------------------------------------------------------------- router

def router_logits(x: np.ndarray, w_r: np.ndarray, b: np.ndarray | None = None) -> np.ndarray:
    """fp32 logits L[t, e] = sum_i x[t, i] * W_r[i, e] (+ b[e]).

    [Noisy top-k] router paragraph (one linear layer to one logit per expert);
    [Choosing MLPs] section "Router: Selecting Experts and Computing Weights",
    Figure 2 (W_r is d x N); [DeepSeekMoE eq] the affinity u_t^T e_i; [Switch]
    section "Making it work" (the router runs in higher precision).
    Summation order (C code): 8-feature blocks dealt round-robin to 32 fma partial
    sums, combined by five pairwise rounds (xor distance 16, 8, 4, 2, 1), then + b.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    w_r = np.ascontiguousarray(w_r, dtype=np.float32)
    T, d = x.shape
    d2, N = w_r.shape
    assert d == d2
    assert np.isfinite(x).all() and np.isfinite(w_r).all(), "router inputs must be finite"
    out = np.empty((T, N), dtype=np.float32)
    bp = None
    if b is not None:
        b = np.ascontiguousarray(b, dtype=np.float32)
        assert b.shape == (N,)
        bp = b.ctypes.data
    _load().oracle_router_logits(T, d, N, x.ctypes.data, w_r.ctypes.data, bp, out.ctypes.data)
    return out


def select_topk(logits: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest logits per token, largest first.

    [MoE glossary] top-k gating bullet (the k experts with the highest scores
    process the token); [Choosing MLPs] section "Router: Selecting Experts and
    Computing Weights" (top-2 keeps the two largest scores); [DeepSeekMoE eq]
    the Topk(., K) set. Softmax is monotone, so selecting on logits is
    the same set as selecting on the affinities s in exact arithmetic.
    Equal logits: the lower expert index comes first (a stable sort of -logit;
    -0.0 and +0.0 compare equal).
    """
    order = np.argsort(-logits, axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


def softmax_all(logits: np.ndarray) -> np.ndarray:
    """p[t, e] = exp(L[t, e] - max_e L) / sum_e' exp(L[t, e'] - max_e L), float64.

    [MoE glossary] gating-network paragraph (a softmax turns the router output
    into a probability vector over every expert); [DeepSeekMoE eq]
    s_{i,t} = Softmax_i(u_t^T e_i).
    """
    L = logits.astype(np.float64)
    z = np.exp(L - L.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def gates(logits: np.ndarray, idx: np.ndarray, gating: str) -> np.ndarray:
    """Gate weight per selected slot, float64 [T][k].

    softmax_then_topk: g = s at the selected experts, not renormalised
      ([DeepSeekMoE eq]: g_{i,t} = s_{i,t} if s_{i,t} in Topk, else 0).
    topk_then_softmax: softmax over the k selected logits only
      ([Choosing MLPs] section "Router: Selecting Experts and Computing
      Weights": the softmax runs over the two selected scores only, so the
      weights add up to 1).
    """
    if gating == GATING_SOFTMAX_THEN_TOPK:
        p = softmax_all(logits)
        return np.take_along_axis(p, idx, axis=1)
    if gating == GATING_TOPK_THEN_SOFTMAX:
        sel = np.take_along_axis(logits, idx, axis=1).astype(np.float64)
        z = np.exp(sel - sel.max(axis=1, keepdims=True))
        return z / z.sum(axis=1, keepdims=True)
    raise ValueError(gating)


# --------------------------------------------------------------- counts, capacity, aux

def counts_routed(idx: np.ndarray, N: int) -> np.ndarray:
    """Number of (token, slot) selections per expert, before any capacity drop."""
    return np.bincount(idx.reshape(-1), minlength=N).astype(np.int64)


def capacity(T: int, N: int, capacity_factor) -> int | None:
    """Expert capacity C = (tokens_per_batch / num_experts) * capacity_factor,
    rounded up ([MoE glossary] capacity-factor paragraph). None: no limit."""
    if capacity_factor is None:
        return None
    num, den = capacity_factor
    return (T * num + N * den - 1) // (N * den)


def keep_within_capacity(idx: np.ndarray, N: int, C: int | None) -> np.ndarray:
    """kept[t, j]: slot j of token t is processed by its expert.

    [MoE glossary] capacity-factor paragraph: assignments beyond an expert's
    capacity are dropped and the token passes through the residual; [Switch]
    section "Making it work": tokens over the limit bypass the layer. Priority
    (a reading): slot-major, i.e. every token's first choice in token order,
    then every second choice, and so on.
    """
    T, k = idx.shape
    kept = np.ones((T, k), dtype=bool)
    if C is None:
        return kept
    used = [0] * N
    for j in range(k):
        for t in range(T):
            e = int(idx[t, j])
            if used[e] < C:
                used[e] += 1
            else:
                kept[t, j] = False
    return kept


def group_by_expert(idx: np.ndarray, kept: np.ndarray, N: int):
    """Dispatch: group the kept (token, slot) pairs by expert.

    [Choosing MLPs] section "From Router to Combine", Figure 3: dispatch collects,
    for each expert, the tokens that chose it (E1 gets x1 and x3, E2 gets x2, E3
    gets x1, x2 and x3, E4 gets nothing). Rows are ordered by expert, then by
    token, the order in which the figure lists them.

    Returns counts_kept [N], expert_offsets [N+1], perm_token [R] (token of each
    row), slot_row [T][k] (row of each slot, -1 when dropped).
    """
    T, k = idx.shape
    groups = [[] for _ in range(N)]
    for t in range(T):
        for j in range(k):
            if kept[t, j]:
                groups[int(idx[t, j])].append((t, j))
    counts_kept = np.array([len(g) for g in groups], dtype=np.int64)
    offsets = np.zeros(N + 1, dtype=np.int64)
    offsets[1:] = np.cumsum(counts_kept)
    perm_token = np.empty(int(offsets[-1]), dtype=np.int64)
    slot_row = np.full((T, k), -1, dtype=np.int64)
    for e in range(N):
        for r, (t, j) in enumerate(groups[e]):
            perm_token[offsets[e] + r] = t
            slot_row[t, j] = offsets[e] + r
    return counts_kept, offsets, perm_token, slot_row


def aux_losses(p: np.ndarray, routed: np.ndarray, k: int):
    """Auxiliary load-balancing loss, two forms (the pages print no formula).

    P_e = mean over tokens of the full softmax p[t, e]; f_e = routed_e / (T k)
    (selections before capacity drops).
      form 0 (Switch form):  N * sum_e f_e P_e   ([Switch] section "Making it
              work" names a load-balancing loss that pushes the router toward an
              even spread; the expression itself is a reading, not printed)
      form 1 (variance form): (1/N) sum_e (P_e - 1/N)^2  ([Noisy top-k] load-
              balancing bullets and [MoE glossary] auxiliary-loss paragraph: the
              loss penalises how unevenly the routing probability is spread over
              the experts, measured as a variance)
    """
    T, N = p.shape
    P = p.mean(axis=0)
    f = routed.astype(np.float64) / float(T * k)
    return float(N * np.sum(f * P)), float(np.mean((P - 1.0 / N) ** 2))


# ------------------------------------------------------------------------- experts

def silu(z: np.ndarray) -> np.ndarray:
    """SiLU(z) = z / (1 + exp(-z))."""
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def expert_ffn(xr: np.ndarray, w_a, w_b, w_out, act: str) -> np.ndarray:
    """One expert applied to each row of xr independently, float64.

    act="silu_gated": W_down (SiLU(W_gate x) * (W_up x)) — a gated MLP with
      separate gate, up and down projections per expert ([Choosing MLPs]
      section "Dense MLP and MoE", Figure 1; [MoE glossary]: experts are
      independent feed-forward networks).
    act="relu": W2 max(0, W1 x) — the plain FFN of [DeepSeekMoE eq]'s text.
    Weights use the [out][in] layout: w_a/w_b [h][d], w_out [d][h].
    """
    xr = np.asarray(xr, dtype=np.float64)
    wa = np.asarray(w_a, dtype=np.float64)
    wo = np.asarray(w_out, dtype=np.float64)
    if act == "silu_gated":
        wb = np.asarray(w_b, dtype=np.float64)
        hid = silu(xr @ wa.T) * (xr @ wb.T)
    elif act == "relu":
        hid = np.maximum(xr @ wa.T, 0.0)
    else:
        raise ValueError(act)
    return hid @ wo.T


# ------------------------------------------------------------------------- layer

def route(cfg, x, w_r, b_r=None) -> dict:
    """Router, gates, counts, capacity, aux loss and dispatch order for all tokens."""
    return route_from_logits(cfg, router_logits(x, w_r, b_r))


def route_from_logits(cfg, L: np.ndarray) -> dict:
    """Everything after the router's linear layer, from the fp32 logits L [T][N]."""
    idx = select_topk(L, cfg.k)
    g = gates(L, idx, cfg.gating)
    p = softmax_all(L)
    routed = counts_routed(idx, cfg.N)
    C = capacity(cfg.T, cfg.N, cfg.capacity_factor)
    kept = keep_within_capacity(idx, cfg.N, C)
    counts_kept, offsets, perm_token, slot_row = group_by_expert(idx, kept, cfg.N)
    aux = aux_losses(p, routed, cfg.k)
    return dict(logits=L, topk_idx=idx, topk_gate=g, p=p, counts_routed=routed,
                capacity=C, kept=kept, counts_kept=counts_kept, expert_offsets=offsets,
                perm_token=perm_token, slot_row=slot_row, aux=aux)


# ------------------------------------------------------- training-time router variants

def noisy_logits(logits: np.ndarray, noise: np.ndarray, noise_weight: float) -> np.ndarray:
    """Noisy top-k: H[t, e] = L[t, e] + W_noise * n[t, e], n ~ N(0, 1).

    [Noisy top-k] "Noise Top-k Gating", opening paragraphs and the parameter list:
    Gaussian noise of a standard normal, scaled by one scalar noise weight, is added
    to the raw router logits before the top-k choice; at inference the weight is
    zero. The draws n are an input (the caller samples them). The sum is taken in
    fp32 like the logits, as two correctly rounded steps: the product W_noise * n
    rounded to fp32, then the sum rounded to fp32, so the noisy top-k decision is
    reproducible bit for bit.
    """
    L = np.asarray(logits, dtype=np.float32)
    n = np.asarray(noise, dtype=np.float32)
    prod = (np.float32(noise_weight) * n).astype(np.float32)
    return (L + prod).astype(np.float32)


def z_loss(logits: np.ndarray) -> float:
    """Router z-loss, float64: (1/T) * sum_t (log sum_e exp L[t, e])^2.

    [MoE glossary], load-balancing bullets: the z-loss penalises large router
    logits; the pages print no formula. Reading: the square of each token's
    log-sum-exp of its logits, averaged over tokens. It is taken on the logits of
    the router's linear layer (bias included, noise excluded).
    """
    L = np.asarray(logits, dtype=np.float64)
    m = L.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(L - m).sum(axis=1))
    return float(np.mean(lse * lse))


def route_train(cfg, x, w_r, b_r=None, noise=None, noise_weight: float = 0.0) -> dict:
    """Training-time router: the noisy logits H drive the selection, the gates, the
    counts, the capacity decisions and the aux loss (softmax of H); the z-loss is
    computed on the noiseless logits L. Without noise H = L."""
    L = router_logits(x, w_r, b_r)
    H = L if noise is None else noisy_logits(L, noise, noise_weight)
    rt = route_from_logits(cfg, H)
    rt["raw_logits"] = L
    rt["z_loss"] = z_loss(L)
    return rt


# ------------------------------------------------------------- Expert Choice routing

def ec_exp(x: np.ndarray) -> np.ndarray:
    """The fp32 exponential of the Expert Choice scores (expert_choice.c: Cody-Waite
    reduction, degree-7 Taylor polynomial, exact power-of-two scaling), elementwise."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    y = np.empty_like(x)
    _load().oracle_ec_exp_array(x.size, x.ctypes.data, y.ctypes.data)
    return y


def ec_scores(logits: np.ndarray) -> np.ndarray:
    """Expert Choice scores S[t, e], fp32: the softmax over experts of each token's
    logits, computed in the fixed fp32 steps of expert_choice.c (max, shifted
    exponential, sum over experts ascending, division), because the experts'
    choices compare these values across tokens."""
    L = np.ascontiguousarray(logits, dtype=np.float32)
    T, N = L.shape
    S = np.empty_like(L)
    _load().oracle_ec_scores(T, N, L.ctypes.data, S.ctypes.data)
    return S


def expert_choice_select(S: np.ndarray, C: int) -> np.ndarray:
    """chosen [N][min(C, T)]: the tokens each expert keeps, ascending token index.

    [MoE glossary] sparse-MoE list: Expert Choice lets the experts select their
    top tokens. Expert e keeps the min(C, T) tokens with the largest S[t, e]; on
    equal scores the lower token index wins (a reading). Every expert is full, so
    the load is balanced by construction; a token may be chosen by several experts
    or by none.
    """
    T, N = S.shape
    Ce = min(C, T)
    chosen = np.empty((N, Ce), dtype=np.int64)
    for e in range(N):
        order = np.lexsort((np.arange(T), -S[:, e].astype(np.float64)))   # score desc, t asc
        chosen[e] = np.sort(order[:Ce])
    return chosen


def route_expert_choice(cfg, x, w_r, b_r=None) -> dict:
    """Expert Choice router: logits, scores, per-expert selections, dispatch order.

    Capacity C = ceil(T * cf / N) (cf = the capacity factor, the average number of
    experts per token); expert e owns rows [e * Ce, (e + 1) * Ce), Ce = min(C, T),
    holding its tokens in ascending order. row_gate[r] = S[token, e]. For each
    token its rows in expert order (token_rows, split by token_ptr) drive the
    combine."""
    L = router_logits(x, w_r, b_r)
    S = ec_scores(L)
    T, N = S.shape
    C = capacity(T, N, cfg.capacity_factor)
    assert C is not None and C > 0, "Expert Choice needs a capacity factor"
    chosen = expert_choice_select(S, C)
    Ce = chosen.shape[1]
    perm_token = chosen.reshape(-1)
    expert_of_row = np.repeat(np.arange(N), Ce)
    row_gate = S[perm_token, expert_of_row].astype(np.float32)
    token_rows = [[] for _ in range(T)]
    for r in range(N * Ce):                        # rows in expert order
        token_rows[int(perm_token[r])].append(r)
    token_ptr = np.zeros(T + 1, dtype=np.int64)
    token_ptr[1:] = np.cumsum([len(v) for v in token_rows])
    return dict(logits=L, scores=S, capacity=C, chosen=chosen,
                expert_offsets=np.arange(N + 1, dtype=np.int64) * Ce, perm_token=perm_token,
                row_gate=row_gate, token_ptr=token_ptr,
                token_rows=np.array([r for v in token_rows for r in v], dtype=np.int64))


def layer_output_expert_choice(cfg, x, rt: dict, w_gate, w_up, w_down, sw_gate=None, sw_up=None,
                               sw_down=None, tokens=None) -> np.ndarray:
    """y_t = x_t + S(x_t) + sum over the experts that chose t (ascending) of
    S[t, e] * FFN_e(x_t), float64; a token no expert chose keeps x_t (+ S(x_t))."""
    x = np.asarray(x, dtype=np.float64)
    toks = np.arange(x.shape[0]) if tokens is None else np.asarray(tokens)
    out = np.zeros((len(toks), x.shape[1]))
    Ce = rt["chosen"].shape[1]
    N = rt["chosen"].shape[0]
    for e in range(N):                          # experts ascending = each token's row order
        rows = [(i, r) for i, t in enumerate(toks)
                for r in rt["token_rows"][rt["token_ptr"][t]:rt["token_ptr"][t + 1]] if int(r) // Ce == e]
        if not rows:
            continue
        wu = None if w_up is None else w_up[e]
        f = expert_ffn(x[[toks[i] for i, _ in rows]], w_gate[e], wu, w_down[e], cfg.act)
        for q, (i, r) in enumerate(rows):
            out[i] += float(rt["row_gate"][r]) * f[q]
    xt = x[toks]
    if sw_gate is not None:
        out += shared_expert(xt, sw_gate, sw_up, sw_down)
    return out + xt


def forward_expert_choice(cfg, inp: dict, tokens=None) -> dict:
    rt = route_expert_choice(cfg, inp["x"], inp["w_r"], inp.get("b_r"))
    rt["y"] = layer_output_expert_choice(cfg, inp["x"], rt, inp["w_gate"], inp.get("w_up"),
                                         inp["w_down"], inp.get("shared_w_gate"),
                                         inp.get("shared_w_up"), inp.get("shared_w_down"), tokens)
    return rt


def shared_expert(xr, sw_gate, sw_up, sw_down) -> np.ndarray:
    """Always-on shared expert S(x), a gated MLP applied to every token
    ([Choosing MLPs] "Shared Expert: A Transformation Applied to Every Token",
    Figure 4: y = S(x) + R(x))."""
    return expert_ffn(xr, sw_gate, sw_up, sw_down, "silu_gated")


def layer_output(cfg, x, rt: dict, w_gate, w_up, w_down,
                 sw_gate=None, sw_up=None, sw_down=None, tokens=None) -> np.ndarray:
    """Layer output y for `tokens` (all tokens when None), float64 [len(tokens)][d].

    Dispatch -> expert computation -> combine ([Choosing MLPs] "From Router to
    Combine", Figure 3), then the shared expert ([Choosing MLPs] Figure 4) and the
    residual ([DeepSeekMoE eq]: + u_t; [MoE glossary]: dropped overflow keeps the
    residual). Only the dispatched rows whose token is requested are computed.
    """
    T = cfg.T
    tokens = np.arange(T) if tokens is None else np.asarray(tokens, dtype=np.int64)
    want = np.zeros(T, dtype=bool)
    want[tokens] = True
    perm_token, offsets = rt["perm_token"], rt["expert_offsets"]
    R = len(perm_token)
    y_perm = {}                                    # row -> expert output (float64 [d])
    for e in range(cfg.N):
        rows = [r for r in range(int(offsets[e]), int(offsets[e + 1])) if want[perm_token[r]]]
        if not rows:
            continue
        xe = np.asarray(x[perm_token[rows]], dtype=np.float64)   # dispatch: gather rows
        ye = expert_ffn(xe, w_gate[e], None if w_up is None else w_up[e], w_down[e], cfg.act)
        for i, r in enumerate(rows):
            y_perm[r] = ye[i]
    assert all(0 <= r < R for r in y_perm)
    xt = np.asarray(x[tokens], dtype=np.float64)
    out = np.zeros_like(xt)
    for n, t in enumerate(tokens):                 # combine: weighted sum per token
        for j in range(cfg.k):
            r = int(rt["slot_row"][t, j])
            if r >= 0:
                out[n] += rt["topk_gate"][t, j] * y_perm[r]
    if cfg.h_shared:
        out += shared_expert(xt, sw_gate, sw_up, sw_down)
    return out + xt


def forward(cfg, inp: dict, tokens=None) -> dict:
    """Whole layer: routing for all tokens, outputs for `tokens` (default all)."""
    rt = route(cfg, inp["x"], inp["w_r"], inp.get("b_r"))
    rt["y"] = layer_output(cfg, inp["x"], rt, inp["w_gate"], inp.get("w_up"), inp["w_down"],
                           inp.get("shared_w_gate"), inp.get("shared_w_up"),
                           inp.get("shared_w_down"), tokens)
    return rt


# ------------------------------------------------------------------------- backward

def _silu_parts(A):
    sig = 1.0 / (1.0 + np.exp(-A))
    return A * sig, sig * (1.0 + A * (1.0 - sig))     # SiLU(A) and its derivative


def expert_ffn_backward(X, dO, w_a, w_b, w_out, act: str):
    """One expert's FFN backward on its rows, float64: given dO = dLoss/dO for
    O = FFN(X), returns (dX, dW_a, dW_b, dW_out) by the chain rule through
    O = H W_outᵀ, H = SiLU(X W_aᵀ) ⊙ (X W_bᵀ) (gated) or H = max(0, X W_aᵀ) (ReLU):
      dH = dO W_out,  dW_out = dOᵀ H,
      gated: dA = dH ⊙ B ⊙ SiLU'(A), dB = dH ⊙ SiLU(A), SiLU'(z) = σ(z)(1 + z(1 - σ(z)));
      ReLU:  dA = dH ⊙ [A > 0];
      dW_a = dAᵀ X, dW_b = dBᵀ X, dX = dA W_a + dB W_b.
    """
    X = np.asarray(X, np.float64)
    wa = np.asarray(w_a, np.float64)
    wo = np.asarray(w_out, np.float64)
    A = X @ wa.T
    if act == "silu_gated":
        wb = np.asarray(w_b, np.float64)
        B = X @ wb.T
        sA, dsA = _silu_parts(A)
        H = sA * B
        dH = dO @ wo
        dA = dH * B * dsA
        dB = dH * sA
        return dA @ wa + dB @ wb, dA.T @ X, dB.T @ X, dO.T @ H
    if act == "relu":
        H = np.maximum(A, 0.0)
        dH = dO @ wo
        dA = dH * (A > 0)
        return dA @ wa, dA.T @ X, None, dO.T @ H
    raise ValueError(act)


def backward(cfg, inp: dict, dy, aux_coef: float = 0.0, z_coef: float = 0.0) -> dict:
    """Gradients of  Loss = sum(dy ⊙ y) + aux_coef * aux[0] + z_coef * z  (float64).

    The routing decisions (selections, capacity drops) are held fixed: they are
    piecewise constant in the inputs. With O_r = FFN_e(x_t) the output of row r =
    (t, j) and g_tj its gate:
      dO_r = g_tj dy_t;  dg_tj = <dy_t, O_r> (0 for a dropped slot);
      expert weights and dX_r from expert_ffn_backward; dx_t = dy_t + sum_j dX_r
      + the shared expert's dx + the router's dx;
      router: dL from the gates (softmax over the k selected logits, or the full
      softmax at the selected experts), from the aux loss N sum_e f_e P_e (f held
      fixed, dP_e = N f_e) and from the z-loss (d lse_t / dL = softmax p_t);
      dW_r = xᵀ dL, db = sum_t dL_t, dx += dL W_rᵀ.
    Returns dx [T][d], dw_r [d][N], db_r [N] (or None), dw_gate / dw_up / dw_down as
    lists over experts (None for an expert without rows), shared-expert gradients
    (or None), and the routing it used.
    """
    x32 = np.asarray(inp["x"], np.float32)
    x = x32.astype(np.float64)
    T, d = x.shape
    N, k = cfg.N, cfg.k
    dy = np.asarray(dy, np.float64)
    rt = route(cfg, x32, inp["w_r"], inp.get("b_r"))
    idx, kept, g = rt["topk_idx"], rt["kept"], rt["topk_gate"]
    dx = dy.copy()
    dg = np.zeros((T, k))
    dwa, dwb, dwo = [None] * N, [None] * N, [None] * N
    for e in range(N):
        sel = [(t, j) for t in range(T) for j in range(k) if kept[t, j] and idx[t, j] == e]
        if not sel:
            continue
        ts = np.array([t for t, _ in sel])
        js = np.array([j for _, j in sel])
        wu = None if inp.get("w_up") is None else inp["w_up"][e]
        O = expert_ffn(x[ts], inp["w_gate"][e], wu, inp["w_down"][e], cfg.act)
        dg[ts, js] = np.sum(dy[ts] * O, axis=1)
        dO = g[ts, js][:, None] * dy[ts]
        dX, dwa[e], dwb[e], dwo[e] = expert_ffn_backward(x[ts], dO, inp["w_gate"][e], wu, inp["w_down"][e],
                                                          cfg.act)
        np.add.at(dx, ts, dX)
    sh = None
    if cfg.h_shared:
        dXs, a_, b_, o_ = expert_ffn_backward(x, dy, inp["shared_w_gate"], inp["shared_w_up"],
                                               inp["shared_w_down"], "silu_gated")
        dx += dXs
        sh = dict(dw_gate=a_, dw_up=b_, dw_down=o_)
    # router
    L = rt["logits"].astype(np.float64)
    p = rt["p"]
    dL = np.zeros((T, N))
    for t in range(T):
        sel = idx[t]
        if cfg.gating == GATING_TOPK_THEN_SOFTMAX:
            gt = g[t]
            dL[t, sel] += gt * (dg[t] - np.sum(gt * dg[t]))
        else:
            dp = np.zeros(N)
            dp[sel] = dg[t]
            dL[t] += p[t] * (dp - np.sum(p[t] * dp))
    if aux_coef:
        f = rt["counts_routed"].astype(np.float64) / float(T * k)
        dp = np.broadcast_to(aux_coef * N * f / T, (T, N))
        dL += p * (dp - np.sum(p * dp, axis=1, keepdims=True))
    if z_coef:
        m = L.max(axis=1, keepdims=True)
        lse = m[:, 0] + np.log(np.exp(L - m).sum(axis=1))
        dL += z_coef * (2.0 * lse / T)[:, None] * p
    w_r = np.asarray(inp["w_r"], np.float64)
    dx += dL @ w_r.T
    return dict(dx=dx, dw_r=x.T @ dL, db_r=dL.sum(axis=0) if inp.get("b_r") is not None else None,
                dlogits=dL, dw_gate=dwa, dw_up=dwb, dw_down=dwo, shared=sh, route=rt, dgate=dg)


def forward_dense(cfg, inp: dict) -> np.ndarray:
    """Brute-force dense evaluation of the DeepSeekMoE equation on tiny inputs.

    h_t = sum_{i=1..N} g_{i,t} FFN_i(u_t) + u_t with g the dense N-vector (the
    gate at kept selected experts, 0 elsewhere); every expert is computed for
    every token and then masked. Plus S(u_t) when a shared expert is present.
    """
    rt = route(cfg, inp["x"], inp["w_r"], inp.get("b_r"))
    x = np.asarray(inp["x"], dtype=np.float64)
    G = np.zeros((cfg.T, cfg.N))
    for t in range(cfg.T):
        for j in range(cfg.k):
            if rt["kept"][t, j]:
                G[t, rt["topk_idx"][t, j]] = rt["topk_gate"][t, j]
    y = x.copy()
    for i in range(cfg.N):
        wu = None if inp.get("w_up") is None else inp["w_up"][i]
        y += G[:, i:i + 1] * expert_ffn(x, inp["w_gate"][i], wu, inp["w_down"][i], cfg.act)
    if cfg.h_shared:
        y += shared_expert(x, inp["shared_w_gate"], inp["shared_w_up"], inp["shared_w_down"])
    return y


def config_from(T, d, N, k, h, h_shared=0, gating=GATING_TOPK_THEN_SOFTMAX,
                act="silu_gated", capacity_factor=None):
    """A plain attribute bag with the fields the oracle reads."""
    class _Cfg:
        pass
    c = _Cfg()
    c.T, c.d, c.N, c.k, c.h, c.h_shared = T, d, N, k, h, h_shared
    c.gating, c.act, c.capacity_factor = gating, act, capacity_factor
    return c


def tokens_per_second_sample(cfg, inp: dict, tokens) -> float:
    """Time the oracle on a token sample (routing for all tokens, outputs for the
    sample); returns sample tokens per second."""
    import time
    t0 = time.perf_counter()
    forward(cfg, inp, tokens=tokens)
    return len(tokens) / (time.perf_counter() - t0)


__all__ = [n for n in dir() if not n.startswith("_") and n not in ("ctypes", "np", "pathlib",
                                                                   "subprocess")]
