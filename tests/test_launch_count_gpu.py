"""The kernel count bench.py reports (`gpu_launches`, from `launches_per_forward`)
against the kernels one moe_forward really enqueues: the call is captured into a
CUDA graph and its kernel nodes are counted."""
import pytest
import torch

import workloads as W

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    from cuda.bindings import runtime as rt

    import bench
    import sparse_mixture_experts_64_b300 as moe
    from moe_harness import cfg_of


def _small(name, **kw):
    return W.WORKLOADS[name].replace(name=name + "_" + "_".join(f"{a}{b}" for a, b in kw.items()), **kw)


CASES = [
    W.WORKLOADS["tiny_fp32"],                                           # fp32, scan folded into the assignment
    W.WORKLOADS["switch_top1"],                                         # 256 router tiles: separate scan
    _small("mixtral_decode_16", d=512, h=1024),                         # one router tile
    _small("mixtral_prefill", T=4096, d=256, h=512),                    # 1024 rows per expert: one launch per product
    _small("deepseek_fine", T=1024, d=256, N=64, k=6, h=256, h_shared=256),   # N > 32, few rows per expert
    _small("deepseek_fine", T=2048, d=256, N=64, k=8, h=256, h_shared=256),   # 256 rows per expert: split products
    _small("switch_top1", T=512, d=256, h=256, N=4, k=2, h_shared=256, capacity_factor=None),  # ReLU + shared
    _small("mixtral_prefill", T=512, d=256, h=512, N=8, k=2, capacity_factor=(2, 1),
           routing="expert_choice"),                                    # Expert Choice
]


def _check(r):
    err = r[0] if isinstance(r, tuple) else r
    assert err == rt.cudaError_t.cudaSuccess, err
    return r[1:] if isinstance(r, tuple) else ()


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_kernels_per_forward(w):
    inp = W.make_inputs(w, device="cuda")
    cfg = cfg_of(w)
    ws = moe.workspace(cfg)
    T, d, k = w.T, w.d, w.k
    y = torch.empty((T, d), dtype=inp["x"].dtype, device="cuda")
    ec = w.routing == "expert_choice"
    idx = None if ec else torch.empty((T, k), dtype=torch.int32, device="cuda")
    gate = None if ec else torch.empty((T, k), device="cuda")
    # the outputs the benchmark asks for: per-expert counts too
    routed = torch.empty(w.N, dtype=torch.int32, device="cuda")
    kept = torch.empty(w.N, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()

    def fwd():
        moe.moe_forward(cfg, inp["x"], inp["w_r"], inp["b_r"], inp["w_gate"], inp["w_up"], inp["w_down"],
                        inp["shared_w_gate"], inp["shared_w_up"], inp["shared_w_down"], y, idx, gate, routed, kept,
                        None, ws, s)
    fwd()  # first call: one-time kernel attributes outside the capture
    torch.cuda.synchronize()
    cs = rt.cudaStream_t(s.cuda_stream)
    _check(rt.cudaStreamBeginCapture(cs, rt.cudaStreamCaptureMode.cudaStreamCaptureModeRelaxed))
    fwd()
    (graph,) = _check(rt.cudaStreamEndCapture(cs))
    try:
        _, n = _check(rt.cudaGraphGetNodes(graph, 0))
        nodes, _ = _check(rt.cudaGraphGetNodes(graph, n))
        kinds = [_check(rt.cudaGraphNodeGetType(node))[0] for node in nodes]
        kernels = sum(1 for t in kinds if t == rt.cudaGraphNodeType.cudaGraphNodeTypeKernel)
    finally:
        _check(rt.cudaGraphDestroy(graph))
    assert kernels == bench.launches_per_forward(w), (kernels, kinds)
    assert moe.moe_check_error(ws) == moe.MOE_OK
