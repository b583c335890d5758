"""Parity of the training-time router (noisy top-k gating, router z-loss) with the
oracle, through moe_router_topk_train.

Routing outputs are bit-exact (the noisy logits are formed in fp32 the same way on
both sides from the same draws); gates within 1e-5; aux losses and the z-loss within
1e-4 relative."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import sparse_mixture_experts_64_b300 as moe
    from moe_harness import TOL_AUX, cfg_of, check_routing, host, oracle_inputs


def _w(name, **kw):
    base = W.WORKLOADS[name]
    return base.replace(name=name + "_" + "_".join(f"{a}{b}" for a, b in kw.items()), **kw)


# every router kernel path: N <= 4, 8, 16, 32 (one fused kernel) and N > 32 (logits +
# gating kernels); both gating conventions; bias; capacity with drops; fp32 and bf16
CASES = [
    _w("tiny_fp32", T=77, N=3, k=2),
    _w("tiny_fp32", T=50, N=7, k=3, gating="softmax_then_topk"),
    _w("switch_top1", T=333, d=128, h=128, N=8),
    _w("mixtral_prefill", T=129, d=192, h=128, N=16, k=2),
    _w("mixtral_prefill", T=96, d=256, h=128, N=32, k=4),
    _w("deepseek_fine", T=130, d=128, N=256, k=8, h=128, h_shared=0),
    _w("deepseek_fine", T=200, d=320, N=40, k=6, h=128, h_shared=0, capacity_factor=(1, 1)),
]


def _run(w, noise, noise_weight, want_z=True):
    cfg = cfg_of(w)
    inp = W.make_inputs(w, device="cuda", router_only=True)
    ws = moe.workspace(cfg)
    T, k, N = w.T, w.k, w.N
    i32 = dict(dtype=torch.int32, device="cuda")
    o = dict(topk_idx=torch.full((T, k), -7, **i32), topk_gate=torch.zeros((T, k), device="cuda"),
             counts_routed=torch.full((N,), -7, **i32), counts_kept=torch.full((N,), -7, **i32),
             expert_offsets=torch.full((N + 1,), -7, **i32), slot_row=torch.full((T, k), -7, **i32),
             perm_token=torch.full((moe.moe_max_rows(cfg),), -7, **i32),
             aux=torch.zeros(2, device="cuda"))
    z = torch.full((1,), -1.0, device="cuda") if want_z else None
    moe.moe_router_topk_train(cfg, inp["x"], inp["w_r"], inp["b_r"], noise, noise_weight,
                              o["topk_idx"], o["topk_gate"], o["counts_routed"], o["counts_kept"],
                              o["expert_offsets"], o["slot_row"], o["perm_token"], o["aux"], z, ws)
    assert moe.moe_check_error(ws) == moe.MOE_OK
    if z is not None:
        o["z"] = z
    return cfg, inp, ws, host(o)


def _noise(w, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn((w.T, w.N), device="cuda", generator=g)


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
@pytest.mark.parametrize("noise_weight", [0.7, 3.0])
def test_noisy_router_matches_oracle(w, noise_weight):
    noise = _noise(w, 5)
    cfg, inp, ws, g = _run(w, noise, noise_weight)
    oi = oracle_inputs(inp)
    rt = O.route_train(w, oi["x"], oi["w_r"], oi["b_r"], noise.cpu().numpy(), noise_weight)
    check_routing(g, rt, sep=True)
    z = float(g["z"][0])
    assert abs(z - rt["z_loss"]) <= TOL_AUX * abs(rt["z_loss"]), (z, rt["z_loss"])
    # the noise changed the routing somewhere (else the test would not see it)
    plain = O.route(w, oi["x"], oi["w_r"], oi["b_r"])
    assert not np.array_equal(plain["topk_idx"], rt["topk_idx"])


@pytest.mark.parametrize("w", CASES[:4] + CASES[5:6], ids=[c.name for c in CASES[:4] + CASES[5:6]])
def test_without_noise_is_the_inference_router(w):
    """noise NULL and z_loss NULL: the same bits as moe_router_topk."""
    _, inp, ws, g = _run(w, None, 0.0, want_z=False)
    cfg = cfg_of(w)
    T, k, N = w.T, w.k, w.N
    i32 = dict(dtype=torch.int32, device="cuda")
    o = dict(topk_idx=torch.empty((T, k), **i32), topk_gate=torch.empty((T, k), device="cuda"),
             counts_routed=torch.empty((N,), **i32), counts_kept=torch.empty((N,), **i32),
             expert_offsets=torch.empty((N + 1,), **i32), slot_row=torch.empty((T, k), **i32),
             perm_token=torch.full((moe.moe_max_rows(cfg),), -7, **i32),
             aux=torch.empty(2, device="cuda"))
    moe.moe_router_topk(cfg, inp["x"], inp["w_r"], inp["b_r"], o["topk_idx"], o["topk_gate"],
                        o["counts_routed"], o["counts_kept"], o["expert_offsets"], o["slot_row"],
                        o["perm_token"], o["aux"], ws)
    ref = host(o)
    for key in ref:
        assert np.array_equal(g[key], ref[key]), key


def test_zero_noise_weight_keeps_routing_and_reports_z():
    w = CASES[3]
    _, inp, _, g = _run(w, _noise(w, 9), 0.0)
    oi = oracle_inputs(inp)
    rt = O.route_train(w, oi["x"], oi["w_r"], oi["b_r"])
    check_routing(g, rt, sep=True)
    assert abs(float(g["z"][0]) - rt["z_loss"]) <= TOL_AUX * rt["z_loss"]


FULL = ["switch_top1", "mixtral_prefill", "deepseek_fine"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_noisy_routing(name):
    """Full-size router with noise: routing for all tokens bit-exact, aux and z."""
    w = W.WORKLOADS[name]
    noise = _noise(w, 21)
    _, inp, _, g = _run(w, noise, 1.0)
    oi = oracle_inputs(inp)
    rt = O.route_train(w, oi["x"], oi["w_r"], oi["b_r"], noise.cpu().numpy(), 1.0)
    check_routing(g, rt, sep=True)
    assert abs(float(g["z"][0]) - rt["z_loss"]) <= TOL_AUX * abs(rt["z_loss"])
