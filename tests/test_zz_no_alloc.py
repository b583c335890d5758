"""moe_router_topk_noalloc: the router for callers that cannot allocate device
memory (hosts that plan all device memory at start-up and forbid allocation in
their enqueue path, or run inside a fixed budget). It must give the same routing
as moe_router_topk with a caller workspace, call after call, although its
scratch is a static array shared by every call.

This file is collected last on purpose, so a failure here leaves every other
test already run."""
import numpy as np
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import sparse_mixture_experts_64_b300 as moe
    from moe_harness import TOL_AUX, TOL_GATE, cfg_of

CASES = [
    W.WORKLOADS["mixtral_prefill"].replace(name="nx_mixtral", T=333, d=256, h=128),
    W.WORKLOADS["switch_top1"].replace(name="nx_switch", T=640, d=256, h=128),
    W.WORKLOADS["deepseek_fine"].replace(name="nx_deepseek", T=200, d=256, N=64, k=4, h=128,
                                         h_shared=128),
]


def _outputs(cfg, dev="cuda"):
    T, k, N = cfg.T, cfg.k, cfg.N
    rmax = moe.moe_max_rows(cfg)
    return dict(topk_idx=torch.full((T, k), -5, dtype=torch.int32, device=dev),
                topk_gate=torch.zeros((T, k), dtype=torch.float32, device=dev),
                counts_routed=torch.full((N,), -5, dtype=torch.int32, device=dev),
                counts_kept=torch.full((N,), -5, dtype=torch.int32, device=dev),
                expert_offsets=torch.full((N + 1,), -5, dtype=torch.int32, device=dev),
                slot_row=torch.full((T, k), -5, dtype=torch.int32, device=dev),
                perm_token=torch.full((rmax,), -5, dtype=torch.int32, device=dev),
                aux=torch.zeros(2, dtype=torch.float32, device=dev))


def _args(o):
    return (o["topk_idx"], o["topk_gate"], o["counts_routed"], o["counts_kept"],
            o["expert_offsets"], o["slot_row"], o["perm_token"], o["aux"])


def _compare(ref, got):
    for name in ("topk_idx", "counts_routed", "counts_kept", "expert_offsets", "slot_row"):
        assert torch.equal(ref[name], got[name]), name
    R = int(ref["expert_offsets"][-1])
    assert torch.equal(ref["perm_token"][:R], got["perm_token"][:R])
    assert float((ref["topk_gate"] - got["topk_gate"]).abs().max()) <= TOL_GATE
    a, b = ref["aux"].cpu().numpy(), got["aux"].cpu().numpy()
    assert np.all(np.abs(a - b) <= TOL_AUX * np.maximum(np.abs(a), 1e-6))


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_noalloc_router_matches_workspace_router(w):
    inp = W.make_inputs(w, device="cuda")
    cfg = cfg_of(w)
    ws = moe.workspace(cfg)
    ref = _outputs(cfg)
    moe.moe_router_topk(cfg, inp["x"], inp["w_r"], inp["b_r"], *_args(ref), ws)
    for _ in range(2):                       # two calls in a row share the static scratch
        got = _outputs(cfg)
        moe.moe_router_topk_noalloc(cfg, inp["x"], inp["w_r"], inp["b_r"], *_args(got))
        torch.cuda.synchronize()
        _compare(ref, got)
    assert moe.moe_check_error(ws) == moe.MOE_OK


def test_noalloc_router_rejects_configs_beyond_its_scratch():
    big = moe.make_config(T=65536, d=256, N=256, k=8, h=128)
    x = torch.zeros((1, 8), device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_router_topk_noalloc(big, x, x, None, x, x, None, None, x, x, x, None)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
