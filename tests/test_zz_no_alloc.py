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

LIMIT = 32 << 20          # bytes of the static scratch array

CASES = [
    W.WORKLOADS["mixtral_prefill"].replace(name="nx_mixtral", T=333, d=256, h=128),
    W.WORKLOADS["switch_top1"].replace(name="nx_switch", T=640, d=256, h=128),
    W.WORKLOADS["deepseek_fine"].replace(name="nx_deepseek", T=200, d=256, N=64, k=4, h=128,
                                         h_shared=128),
    # the router of the DeepSeekMoE-shaped layer itself (T = 8192, d = 7168, N = 256, top-8)
    W.WORKLOADS["deepseek_fine"],
]


def _largest_fitting_T(N, k, d):
    """The largest T (a multiple of 64) whose router scratch fits the static array."""
    def fits(u):
        return moe.moe_router_workspace_size(moe.make_config(T=64 * u, d=d, N=N, k=k, h=128)) <= LIMIT
    lo, hi = 1, 1024                          # in units of 64 tokens: lo fits, hi does not
    assert fits(lo) and not fits(hi)
    while hi - lo > 1:
        mid = (lo + hi) // 2
        lo, hi = (mid, hi) if fits(mid) else (lo, mid)
    return 64 * lo


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
    inp = W.make_inputs(w, device="cuda", router_only=True)
    cfg = cfg_of(w)
    assert moe.moe_router_workspace_size(cfg) <= LIMIT
    ws = moe.workspace(cfg)
    ref = _outputs(cfg)
    moe.moe_router_topk(cfg, inp["x"], inp["w_r"], inp["b_r"], *_args(ref), ws)
    for _ in range(2):                       # two calls in a row share the static scratch
        got = _outputs(cfg)
        moe.moe_router_topk_noalloc(cfg, inp["x"], inp["w_r"], inp["b_r"], *_args(got))
        assert moe.moe_router_noalloc_check_error() == moe.MOE_OK
        _compare(ref, got)
    assert moe.moe_check_error(ws) == moe.MOE_OK


def test_noalloc_router_at_the_size_limit():
    """The largest top-8 router over 256 experts that fits the array runs and matches
    the workspace router; 64 more tokens are rejected before anything is enqueued."""
    N, k, d = 256, 8, 256
    T = _largest_fitting_T(N, k, d)
    w = W.WORKLOADS["deepseek_fine"].replace(name="nx_limit", T=T, d=d, h=128, h_shared=0)
    cfg = cfg_of(w)
    assert moe.moe_router_workspace_size(cfg) <= LIMIT
    over = cfg_of(w.replace(T=T + 64))
    assert moe.moe_router_workspace_size(over) > LIMIT
    inp = W.make_inputs(w, device="cuda", router_only=True)
    ws = moe.workspace(cfg)
    ref = _outputs(cfg)
    moe.moe_router_topk(cfg, inp["x"], inp["w_r"], inp["b_r"], *_args(ref), ws)
    got = _outputs(cfg)
    moe.moe_router_topk_noalloc(cfg, inp["x"], inp["w_r"], inp["b_r"], *_args(got))
    assert moe.moe_router_noalloc_check_error() == moe.MOE_OK
    _compare(ref, got)
    x = torch.zeros((T + 64, d), dtype=torch.bfloat16, device="cuda")
    big = _outputs(over)
    with pytest.raises(moe.MoeError) as e:
        moe.moe_router_topk_noalloc(over, x, inp["w_r"], None, *_args(big))
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED


def test_noalloc_router_reports_a_wait_that_ran_out():
    """A bounded wait made to run out (MOE_DEBUG_ROUTER_STALL) shows up through the
    no-allocation router's own error accessor; the next call is clean and exact."""
    w = CASES[0]
    inp = W.make_inputs(w, device="cuda", router_only=True)
    cfg = cfg_of(w)
    ws = moe.workspace(cfg)
    ref = _outputs(cfg)
    moe.moe_router_topk(cfg, inp["x"], inp["w_r"], inp["b_r"], *_args(ref), ws)
    stalled = _outputs(cfg)
    moe.moe_router_topk_noalloc(cfg_of(w, debug_flags=moe.MOE_DEBUG_ROUTER_STALL), inp["x"], inp["w_r"],
                                inp["b_r"], *_args(stalled))
    assert moe.moe_router_noalloc_check_error() == moe.MOE_ERR_TIMEOUT
    assert moe.moe_router_noalloc_check_error() == moe.MOE_OK
    got = _outputs(cfg)
    moe.moe_router_topk_noalloc(cfg, inp["x"], inp["w_r"], inp["b_r"], *_args(got))
    assert moe.moe_router_noalloc_check_error() == moe.MOE_OK
    _compare(ref, got)
    assert moe.moe_check_error(ws) == moe.MOE_OK


def test_noalloc_router_rejects_configs_beyond_its_scratch():
    big = moe.make_config(T=65536, d=256, N=256, k=8, h=128)
    x = torch.zeros((1, 8), device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.moe_router_topk_noalloc(big, x, x, None, x, x, None, None, x, x, x, None)
    assert e.value.status == moe.MOE_ERR_UNSUPPORTED
