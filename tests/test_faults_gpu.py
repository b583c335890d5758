"""Failure detection on the GPU without a GPU fault.

A bounded wait is made to run out (MOE_DEBUG_ROUTER_STALL: the router kernel for
N <= 32 stages nothing into its ring, so its consumers' first wait on the ring's
barrier gives up after about 1 ms with no copy in flight). The call must record
MOE_ERR_TIMEOUT in the workspace's error word, moe_check_error must report it and
clear it, and the next normal call on the same workspace must route bit-exactly
like the oracle: the context stays usable."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import sparse_mixture_experts_64_b300 as moe
    from moe_harness import TOL_GATE, cfg_of

CASES = [
    W.WORKLOADS["mixtral_prefill"].replace(name="stall_mixtral", T=64, d=256, h=128),
    W.WORKLOADS["switch_top1"].replace(name="stall_switch", T=100, d=128, h=128),
]


def _outputs(cfg, dev="cuda"):
    T, k, N = cfg.T, cfg.k, cfg.N
    i32 = dict(dtype=torch.int32, device=dev)
    return dict(topk_idx=torch.full((T, k), -5, **i32),
                topk_gate=torch.zeros((T, k), dtype=torch.float32, device=dev),
                counts_routed=torch.full((N,), -5, **i32), counts_kept=torch.full((N,), -5, **i32),
                expert_offsets=torch.full((N + 1,), -5, **i32), slot_row=torch.full((T, k), -5, **i32),
                perm_token=torch.full((moe.moe_max_rows(cfg),), -5, **i32),
                aux=torch.zeros(2, dtype=torch.float32, device=dev))


def _router(cfg, inp, o, ws):
    moe.moe_router_topk(cfg, inp["x"], inp["w_r"], inp["b_r"], o["topk_idx"], o["topk_gate"],
                        o["counts_routed"], o["counts_kept"], o["expert_offsets"], o["slot_row"],
                        o["perm_token"], o["aux"], ws)


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_router_wait_timeout_is_reported_and_the_next_call_is_clean(w):
    inp = W.make_inputs(w, device="cuda", router_only=True)
    cfg = cfg_of(w)
    ws = moe.workspace(cfg)
    stalled = _outputs(cfg)
    _router(cfg_of(w, debug_flags=moe.MOE_DEBUG_ROUTER_STALL), inp, stalled, ws)
    assert moe.moe_check_error(ws) == moe.MOE_ERR_TIMEOUT
    assert moe.moe_check_error(ws) == moe.MOE_OK          # read and cleared

    o = _outputs(cfg)
    _router(cfg, inp, o, ws)
    assert moe.moe_check_error(ws) == moe.MOE_OK
    rt = O.route(w, inp["x"].float().cpu().numpy(), inp["w_r"].cpu().numpy(),
                 None if inp["b_r"] is None else inp["b_r"].cpu().numpy())
    assert np.array_equal(o["topk_idx"].cpu().numpy(), rt["topk_idx"])
    assert np.array_equal(o["counts_kept"].cpu().numpy(), rt["counts_kept"])
    assert np.array_equal(o["expert_offsets"].cpu().numpy(), rt["expert_offsets"])
    assert np.array_equal(o["slot_row"].cpu().numpy(), rt["slot_row"])
    R = int(rt["expert_offsets"][-1])
    assert np.array_equal(o["perm_token"].cpu().numpy()[:R], rt["perm_token"])
    assert float(np.max(np.abs(o["topk_gate"].cpu().numpy() - rt["topk_gate"]))) <= TOL_GATE


def test_stall_flag_is_ignored_by_the_large_router():
    """N > 32 routes through the logits and gating kernels, which do not honour the
    flag: the call is a normal one."""
    w = W.WORKLOADS["deepseek_fine"].replace(name="stall_large", T=70, d=128, N=40, k=4, h=128,
                                             h_shared=0)
    inp = W.make_inputs(w, device="cuda", router_only=True)
    cfg = cfg_of(w, debug_flags=moe.MOE_DEBUG_ROUTER_STALL)
    ws = moe.workspace(cfg)
    o = _outputs(cfg)
    _router(cfg, inp, o, ws)
    assert moe.moe_check_error(ws) == moe.MOE_OK
    rt = O.route(w, inp["x"].float().cpu().numpy(), inp["w_r"].cpu().numpy())
    assert np.array_equal(o["topk_idx"].cpu().numpy(), rt["topk_idx"])
