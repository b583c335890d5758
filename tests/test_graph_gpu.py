"""The forward captured as a CUDA graph (moe_forward_graph_*) against moe_forward and
the oracle: a launch gives the same bits as moe_forward on the same buffers, a launch
after the inputs were overwritten in place routes and computes the new inputs (every
data-dependent size stays on the device), and the six stage events captured into the
graph time every launch."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import sparse_mixture_experts_64_b300 as moe
    from moe_harness import cfg_of, check_output, check_routing, host, oracle_inputs


def _w(name, **kw):
    return W.WORKLOADS[name].replace(name="graph_" + name + "_" + "_".join(f"{a}{b}" for a, b in kw.items()), **kw)


CASES = [
    _w("switch_top1", T=333, d=128, h=256),                                   # ReLU, bias, drops
    _w("deepseek_fine", T=200, d=256, N=16, k=4, h=128, h_shared=128),       # shared expert
    _w("mixtral_prefill", T=1024, d=512, h=1024),                             # CTA-pair kernels
    _w("tiny_fp32", T=100),                                                   # fp32 SIMT path
    _w("mixtral_prefill", T=300, d=256, h=384, routing="expert_choice", capacity_factor=(2, 1)),
]


def _outputs(w, dev="cuda"):
    ec = w.routing == "expert_choice"
    i32 = dict(dtype=torch.int32, device=dev)
    return dict(y=torch.empty((w.T, w.d), dtype=torch.float32 if w.dtype == "f32" else torch.bfloat16, device=dev),
                topk_idx=None if ec else torch.full((w.T, w.k), -7, **i32),
                topk_gate=None if ec else torch.zeros((w.T, w.k), device=dev),
                counts_routed=torch.full((w.N,), -7, **i32), counts_kept=torch.full((w.N,), -7, **i32),
                aux=None if ec else torch.zeros(2, device=dev))


def _args(inp, o):
    return (inp["x"], inp["w_r"], inp["b_r"], inp["w_gate"], inp["w_up"], inp["w_down"], inp["shared_w_gate"],
            inp["shared_w_up"], inp["shared_w_down"], o["y"], o["topk_idx"], o["topk_gate"], o["counts_routed"],
            o["counts_kept"], o["aux"])


def _equal(a, b):
    for key in a:
        if a[key] is not None:
            assert torch.equal(a[key], b[key]), key


@pytest.mark.parametrize("w", CASES, ids=[c.name for c in CASES])
def test_graph_matches_forward_and_follows_new_inputs(w):
    cfg = cfg_of(w)
    inp = W.make_inputs(w, device="cuda")
    ws_a, ws_b = moe.workspace(cfg), moe.workspace(cfg)
    ref, got = _outputs(w), _outputs(w)
    moe.moe_forward(cfg, *_args(inp, ref), ws_a)
    graph = moe.moe_forward_graph_create(cfg, *_args(inp, got), ws_b)
    graph.launch()
    assert moe.moe_check_error(ws_b) == moe.MOE_OK
    _equal(ref, got)
    # new inputs written into the same buffers: the next launch routes them afresh
    g = torch.Generator(device="cuda").manual_seed(11)
    inp["x"].copy_(torch.randn(inp["x"].shape, device="cuda", generator=g).to(inp["x"].dtype))
    for _ in range(2):
        graph.launch()
    moe.moe_forward(cfg, *_args(inp, ref), ws_a)
    assert moe.moe_check_error(ws_b) == moe.MOE_OK and moe.moe_check_error(ws_a) == moe.MOE_OK
    _equal(ref, got)
    oi = oracle_inputs(inp)
    h = host({k: v for k, v in got.items() if v is not None})
    if w.routing == "expert_choice":
        rt = O.forward_expert_choice(w, oi)
        assert h["counts_kept"].tolist() == [int(rt["expert_offsets"][1])] * w.N
    else:
        rt = O.forward(w, oi)
        check_routing(h, rt, sep=False)
    check_output(h["y"], rt["y"], w.dtype)
    graph.destroy()


def test_graph_stage_events_time_every_launch():
    w = CASES[2]
    cfg = cfg_of(w)
    inp = W.make_inputs(w, device="cuda")
    ws = moe.workspace(cfg)
    o = _outputs(w)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    for e in evs:
        e.record()
    graph = moe.moe_forward_graph_create(cfg, *_args(inp, o), ws, events=evs)
    totals = []
    for _ in range(3):
        graph.launch()
        evs[5].synchronize()
        stages = [evs[j].elapsed_time(evs[j + 1]) for j in range(5)]
        total = evs[0].elapsed_time(evs[5])
        assert all(s >= 0 for s in stages) and total > 0
        assert abs(sum(stages) - total) <= 1e-3 * total + 1e-3
        totals.append(total)
    assert moe.moe_check_error(ws) == moe.MOE_OK
    graph.destroy()
