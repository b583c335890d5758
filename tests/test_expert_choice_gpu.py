"""Expert Choice routing on the GPU against the oracle.

The router's outputs are compared bit for bit — including the row gates, which are
the fp32 scores both sides compute in the same fixed steps — and the layer output
within the usual tolerance. The step-by-step calls (router, dispatch, grouped FFN,
Expert Choice combine) must give the same bits as moe_forward."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import sparse_mixture_experts_64_b300 as moe
    from moe_harness import cfg_of, check_output, host, oracle_inputs


def _ec(name, **kw):
    base = W.WORKLOADS[name].replace(routing="expert_choice")
    kw.setdefault("capacity_factor", (2, 1))
    return base.replace(name="ec_" + name + "_" + "_".join(f"{a}{b}" for a, b in kw.items()), **kw)


CASES = [
    _ec("tiny_fp32", T=77, N=5),
    _ec("mixtral_prefill", T=300, d=256, h=384),
    _ec("mixtral_prefill", T=129, d=192, h=320, N=3, capacity_factor=(5, 4)),
    _ec("deepseek_fine", T=200, d=256, N=64, h=128, h_shared=128, capacity_factor=(3, 1)),
    _ec("deepseek_fine", T=130, d=128, N=256, h=128, h_shared=0, capacity_factor=(8, 1)),
    _ec("switch_top1", T=333, d=128, h=256, capacity_factor=(1, 1)),        # ReLU experts, bias
    _ec("mixtral_prefill", T=40, d=128, h=128, N=4, capacity_factor=(9, 1)),  # C >= T
    _ec("tiny_fp32", T=1, N=4),
]


def _router(cfg, w, inp, ws):
    R = moe.moe_max_rows(cfg)
    i32 = dict(dtype=torch.int32, device="cuda")
    o = dict(expert_offsets=torch.full((w.N + 1,), -7, **i32), perm_token=torch.full((R,), -7, **i32),
             row_gate=torch.full((R,), -1.0, device="cuda"), token_ptr=torch.full((w.T + 1,), -7, **i32),
             token_rows=torch.full((R,), -7, **i32))
    moe.moe_router_expert_choice(cfg, inp["x"], inp["w_r"], inp["b_r"], o["expert_offsets"], o["perm_token"],
                                 o["row_gate"], o["token_ptr"], o["token_rows"], ws)
    return o


def _check_router(g, rt):
    assert np.array_equal(g["expert_offsets"], rt["expert_offsets"]), "expert_offsets"
    assert np.array_equal(g["perm_token"], rt["perm_token"]), "perm_token"
    assert np.array_equal(g["row_gate"], rt["row_gate"]), "row_gate (fp32 scores) not bit-exact"
    assert np.array_equal(g["token_ptr"], rt["token_ptr"]), "token_ptr"
    assert np.array_equal(g["token_rows"], rt["token_rows"]), "token_rows"


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_expert_choice_matches_oracle(w):
    cfg = cfg_of(w)
    inp = W.make_inputs(w, device="cuda")
    ws = moe.workspace(cfg)
    g = host(_router(cfg, w, inp, ws))
    oi = oracle_inputs(inp)
    rt = O.forward_expert_choice(w, oi)
    _check_router(g, rt)
    # whole layer through moe_forward
    y = torch.empty((w.T, w.d), dtype=inp["x"].dtype, device="cuda")
    kept = torch.empty(w.N, dtype=torch.int32, device="cuda")
    moe.moe_forward(cfg, inp["x"], inp["w_r"], inp["b_r"], inp["w_gate"], inp["w_up"], inp["w_down"],
                    inp["shared_w_gate"], inp["shared_w_up"], inp["shared_w_down"], y, None, None, None,
                    kept, None, ws)
    assert moe.moe_check_error(ws) == moe.MOE_OK
    assert kept.cpu().tolist() == [int(rt["expert_offsets"][1])] * w.N
    yf = y.float().cpu().numpy()
    check_output(yf, rt["y"], w.dtype)
    # the same through the step-by-step calls
    o = _router(cfg, w, inp, ws)
    R = moe.moe_max_rows(cfg)
    x_perm = torch.zeros((R, w.d), dtype=inp["x"].dtype, device="cuda")
    moe.moe_dispatch(cfg, inp["x"], o["perm_token"], o["expert_offsets"], x_perm, ws)
    y_perm = torch.zeros((R, w.d), dtype=inp["x"].dtype, device="cuda")
    moe.moe_grouped_ffn(cfg, x_perm, o["expert_offsets"], inp["w_gate"], inp["w_up"], inp["w_down"], y_perm, ws)
    y2 = torch.empty_like(y)
    moe.moe_combine_expert_choice(cfg, inp["x"], y_perm, o["token_ptr"], o["token_rows"], o["row_gate"],
                                  inp["shared_w_gate"], inp["shared_w_up"], inp["shared_w_down"], y2, ws)
    assert moe.moe_check_error(ws) == moe.MOE_OK
    assert torch.equal(y, y2)
    # tokens no expert chose keep their residual exactly (no shared expert)
    unchosen = rt["token_ptr"][1:] == rt["token_ptr"][:-1]
    if unchosen.any() and not w.h_shared:
        assert np.array_equal(yf[unchosen], inp["x"].float().cpu().numpy()[unchosen])


def test_all_scores_equal_take_the_first_tokens():
    """A zero router weight makes every score 1/N: each expert keeps tokens 0..Ce-1."""
    w = _ec("mixtral_prefill", T=50, d=128, h=128, N=4, capacity_factor=(1, 1))
    cfg = cfg_of(w)
    inp = W.make_inputs(w, device="cuda")
    inp["w_r"] = torch.zeros_like(inp["w_r"])
    ws = moe.workspace(cfg)
    g = host(_router(cfg, w, inp, ws))
    Ce = 13
    assert g["perm_token"].tolist() == list(range(Ce)) * 4
    assert np.all(g["row_gate"] == np.float32(0.25))


def test_full_size_expert_choice():
    """The Mixtral-shaped prefill layer with Expert Choice (two experts per token on
    average): routing bit-exact for all 4096 tokens, outputs on a token sample."""
    w = W.WORKLOADS["mixtral_expert_choice"]
    cfg = cfg_of(w)
    inp = W.make_inputs(w, device="cuda")
    ws = moe.workspace(cfg)
    g = host(_router(cfg, w, inp, ws))
    oi = oracle_inputs(inp)
    rt = O.route_expert_choice(w, oi["x"], oi["w_r"], oi["b_r"])
    _check_router(g, rt)
    y = torch.empty((w.T, w.d), dtype=inp["x"].dtype, device="cuda")
    moe.moe_forward(cfg, inp["x"], inp["w_r"], inp["b_r"], inp["w_gate"], inp["w_up"], inp["w_down"],
                    None, None, None, y, None, None, None, None, None, ws)
    assert moe.moe_check_error(ws) == moe.MOE_OK
    tokens = np.sort(np.random.default_rng(5).choice(w.T, size=12, replace=False))
    ref = O.layer_output_expert_choice(w, oi["x"], rt, oi["w_gate"], oi["w_up"], oi["w_down"], tokens=tokens)
    check_output(y.float().cpu().numpy()[tokens], ref, w.dtype)


def test_largest_expert_choice_batch():
    """T = 16384, the largest batch the Expert Choice selection sorts in shared memory,
    over 64 experts: routing bit-exact for all tokens, outputs on a sample."""
    w = _ec("deepseek_fine", T=16384, d=128, N=64, h=128, h_shared=0, capacity_factor=(2, 1))
    cfg = cfg_of(w)
    inp = W.make_inputs(w, device="cuda")
    ws = moe.workspace(cfg)
    g = host(_router(cfg, w, inp, ws))
    oi = oracle_inputs(inp)
    rt = O.route_expert_choice(w, oi["x"], oi["w_r"], oi["b_r"])
    _check_router(g, rt)
    y = torch.empty((w.T, w.d), dtype=inp["x"].dtype, device="cuda")
    moe.moe_forward(cfg, inp["x"], inp["w_r"], inp["b_r"], inp["w_gate"], inp["w_up"], inp["w_down"],
                    None, None, None, y, None, None, None, None, None, ws)
    assert moe.moe_check_error(ws) == moe.MOE_OK
    tokens = np.sort(np.random.default_rng(6).choice(w.T, size=16, replace=False))
    ref = O.layer_output_expert_choice(w, oi["x"], rt, oi["w_gate"], oi["w_up"], oi["w_down"], tokens=tokens)
    check_output(y.float().cpu().numpy()[tokens], ref, w.dtype)
