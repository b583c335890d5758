"""Ties in the router: many experts with exactly the same logit.

Selection takes the k largest logits, and between equal logits the lower expert index
(the top-k of the router in "MoE: Choosing Which MLPs to Use for Each Token", *Router:
Selecting Experts and Computing Weights*, with ties broken towards the lower index).
Random normal inputs almost never tie, so these cases build inputs whose logits are
exact small integers: token features and router weights drawn from {-1, 0, 1}. Every
partial sum is then an exact integer in fp32, whatever the summation order, and most
tokens have several experts on the same logit, at the k-th place as well. The CUDA
router (both its small-N kernel and the logits/gating kernels for N > 32) must pick
exactly the oracle's experts, and the capacity decisions built on them must agree too.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import moe_oracle as O

if torch.cuda.is_available():
    import sparse_mixture_experts_64_b300 as moe
    from moe_harness import cfg_of, check_routing, host


def _case(T, d, N, k, dtype="bf16", gating="softmax_then_topk", capacity_factor=None):
    name = f"ties_T{T}_d{d}_N{N}_k{k}_{dtype}_{gating}" + ("_cap" if capacity_factor else "")
    return W.Workload(name, 5, T=T, d=d, N=N, k=k, h=64, dtype=dtype, gating=gating,
                      capacity_factor=capacity_factor)


CASES = [
    _case(300, 64, 8, 2, gating="topk_then_softmax"),            # k_router_small, NP = 8
    _case(129, 128, 32, 4),                                      # k_router_small, NP = 32
    _case(333, 64, 64, 8),                                       # k_logits_large + k_gate, bf16
    _case(200, 128, 256, 8),                                     # 256 experts, bf16
    _case(97, 64, 100, 6, dtype="f32", gating="topk_then_softmax"),  # fp32 tokens, N > 32
    _case(512, 64, 64, 2, capacity_factor=(1, 1)),               # drops decided among tied tokens
]


def _integer_inputs(w, seed):
    rng = np.random.default_rng(seed)
    x = rng.integers(-1, 2, size=(w.T, w.d)).astype(np.float32)
    w_r = rng.integers(-1, 2, size=(w.d, w.N)).astype(np.float32)
    return x, w_r


def _tie_fraction(x, w_r, k):
    """Fraction of tokens whose k-th largest logit is shared with an expert left out."""
    L = x.astype(np.float64) @ w_r.astype(np.float64)
    srt = -np.sort(-L, axis=1)
    return float(np.mean(srt[:, k - 1] == srt[:, k])) if L.shape[1] > k else 0.0


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_inputs_really_tie(w):
    """The construction gives ties at the selection boundary (CPU only)."""
    x, w_r = _integer_inputs(w, seed=w.T + w.N)
    assert _tie_fraction(x, w_r, w.k) > 0.2


def _router_on_gpu(w, x, w_r):
    cfg = cfg_of(w)
    ws = moe.workspace(cfg)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    xd = torch.from_numpy(x).to("cuda", dt)
    wd = torch.from_numpy(w_r).to("cuda")
    T, k, N = w.T, w.k, w.N
    i32 = dict(dtype=torch.int32, device="cuda")
    o = dict(topk_idx=torch.full((T, k), -7, **i32),
             topk_gate=torch.zeros((T, k), device="cuda"),
             counts_routed=torch.full((N,), -7, **i32),
             counts_kept=torch.full((N,), -7, **i32),
             expert_offsets=torch.full((N + 1,), -7, **i32),
             slot_row=torch.full((T, k), -7, **i32),
             perm_token=torch.full((moe.moe_max_rows(cfg),), -7, **i32),
             aux=torch.zeros(2, device="cuda"))
    moe.moe_router_topk(cfg, xd, wd, None, o["topk_idx"], o["topk_gate"], o["counts_routed"],
                        o["counts_kept"], o["expert_offsets"], o["slot_row"], o["perm_token"],
                        o["aux"], ws)
    assert moe.moe_check_error(ws) == moe.MOE_OK
    return host(o)


@pytest.mark.gpu
@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_ties_pick_the_oracles_experts(w):
    x, w_r = _integer_inputs(w, seed=w.T + w.N)
    g = _router_on_gpu(w, x, w_r)
    rt = O.route(w, x, w_r, None)
    check_routing(g, rt)


@pytest.mark.gpu
@pytest.mark.parametrize("N,k", [(8, 2), (64, 8), (256, 8)])
def test_all_logits_equal(N, k):
    """A zero router weight ties every expert: each token takes experts 0..k-1."""
    w = _case(150, 64, N, k)
    x, _ = _integer_inputs(w, seed=7)
    w_r = np.zeros((w.d, N), np.float32)
    g = _router_on_gpu(w, x, w_r)
    assert (g["topk_idx"] == np.arange(k, dtype=np.int32)[None, :]).all()
    check_routing(g, O.route(w, x, w_r, None))
