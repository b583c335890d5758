"""Router selections when a logit is NaN (a NaN in a token or in the router weight).

The oracle takes finite inputs only, so this is the library's own rule, stated in
include/moe.h: a NaN logit ranks below every number and is chosen only when fewer
than k experts have a numeric logit, and every token still gets k distinct, valid
experts. Numeric logits are selected exactly as without the NaN: the oracle's
selection on the same logits with the NaN expert at -inf."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import sparse_mixture_experts_64_b300 as moe
    from moe_harness import TOL_GATE, cfg_of

NAN_EXPERT, NAN_TOKEN = 3, 7

CASES = [
    # k_router_small (N <= 32), top-k then softmax
    W.WORKLOADS["mixtral_prefill"].replace(name="nan_small", T=100, d=256, h=128),
    W.WORKLOADS["mixtral_prefill"].replace(name="nan_small_k4", T=90, d=128, N=16, k=4, h=128),
    # k_logits_large + k_gate (N > 32), both gating conventions
    W.WORKLOADS["deepseek_fine"].replace(name="nan_large", T=130, d=256, N=64, k=6, h=128, h_shared=0),
    W.WORKLOADS["deepseek_fine"].replace(name="nan_large_tks", T=70, d=128, N=40, k=8, h=128, h_shared=0,
                                         gating="topk_then_softmax"),
]


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_nan_logits_give_distinct_valid_experts(w):
    inp = W.make_inputs(w, device="cuda", router_only=True)
    x, w_r = inp["x"].clone(), inp["w_r"].clone()
    w_r[5, NAN_EXPERT] = float("nan")       # expert NAN_EXPERT's logit is NaN for every token
    x[NAN_TOKEN] = 0
    x[NAN_TOKEN, 9] = float("nan")          # every logit of token NAN_TOKEN is NaN
    cfg = cfg_of(w)
    ws = moe.workspace(cfg)
    T, k, N = w.T, w.k, w.N
    i32 = dict(dtype=torch.int32, device="cuda")
    idx, gate = torch.full((T, k), -5, **i32), torch.zeros((T, k), device="cuda")
    cr, ck, off = torch.full((N,), -5, **i32), torch.full((N,), -5, **i32), torch.full((N + 1,), -5, **i32)
    sr, perm = torch.full((T, k), -5, **i32), torch.full((moe.moe_max_rows(cfg),), -5, **i32)
    moe.moe_router_topk(cfg, x, w_r, None, idx, gate, cr, ck, off, sr, perm, None, ws)
    assert moe.moe_check_error(ws) == moe.MOE_OK
    got = idx.cpu().numpy()
    assert ((got >= 0) & (got < N)).all()
    for t in range(T):
        assert len(set(got[t].tolist())) == k, f"token {t}: {got[t]}"
    # all logits NaN: ties among equal keys go to the lower index
    assert got[NAN_TOKEN].tolist() == list(range(k))
    # the other tokens never take the NaN expert, and pick what the oracle picks on
    # the same logits with that expert at -inf
    xf = x.float().cpu().numpy()
    xf[NAN_TOKEN] = 0.0
    wf = w_r.cpu().numpy()
    wf[5, NAN_EXPERT] = 0.0
    L = O.router_logits(xf, wf)
    L[:, NAN_EXPERT] = -np.inf
    ref = O.select_topk(L, k)
    keep = np.arange(T) != NAN_TOKEN
    assert (got[keep] != NAN_EXPERT).all()
    assert np.array_equal(got[keep], ref[keep])
    # every selection counted once, and the dispatch order covers them all
    assert int(cr.sum()) == T * k and int(off[-1]) == T * k
    if w.gating == "topk_then_softmax":
        g = O.gates(L, ref, w.gating)
        assert float(np.max(np.abs(gate.cpu().numpy()[keep] - g[keep]))) <= TOL_GATE
