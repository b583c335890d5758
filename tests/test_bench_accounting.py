"""Host-side checks of bench.py's accounting (no GPU): the algorithmic FLOPs and bytes
behind the roofline fractions, recomputed here by hand from the layer shapes, and the
kernels per forward that `gpu_launches` counts, against the launch lists ncu recorded
(every forward of a workload launches the same kernels; tests/test_launch_count_gpu.py
checks the same function against captured CUDA graphs on a GPU)."""
import pytest

import bench
import workloads as W


def test_mixtral_prefill_floor():
    w = W.WORKLOADS["mixtral_prefill"]
    R = w.T * w.k                                  # every token kept (no capacity)
    a = bench.algorithmic(w, R)
    # gate and up (2 matrices) then down: 2 FLOP per multiply-add
    assert a["flops_p1"] == 2 * 2 * R * 4096 * 14336
    assert a["flops_p2"] == 2 * R * 4096 * 14336
    assert a["flops"] == 6 * R * 4096 * 14336 == 2_886_218_022_912
    # weights of the 8 experts (3 matrices of d x h bf16), the router weight, x and y
    assert a["bytes"] == 8 * 3 * 4096 * 14336 * 2 + 4 * 4096 * 8 + 2 * 4096 * 4096 * 2
    peaks = {"bf16": 1811.4, "hbm": 6497.4}
    ms = max(a["flops"] / (peaks["bf16"] * 1e12), a["bytes"] / (peaks["hbm"] * 1e9)) * 1e3
    assert ms == pytest.approx(1.5934, abs=1e-3)   # tensor-bound: 2.886 TFLOP at the bf16 peak


def test_deepseek_floor_is_near_the_ridge():
    w = W.WORKLOADS["deepseek_fine"]
    R = w.T * w.k
    a = bench.algorithmic(w, R)
    routed = 6 * R * 7168 * 2048
    shared = 6 * 8192 * 7168 * 2048
    assert a["flops"] == routed + shared
    assert a["flops"] == pytest.approx(6.494e12, rel=1e-3)
    assert a["bytes"] == pytest.approx(22.87e9, rel=1e-3)
    # arithmetic intensity within 10 % of the B300's measured ridge (FLOP per byte)
    ridge = 1811.4e12 / 6497.4e9
    assert abs(a["flops"] / a["bytes"] / ridge - 1) < 0.1
    # product 1 streams gate and up weights of every expert and the shared expert,
    # reads the dispatched rows and x, and writes the hidden rows
    assert a["bytes_p1"] == (2 * 7168 * 2048 * 256 + 2 * 7168 * 2048) * 2 + (R * 7168 + R * 2048) * 2 \
        + (8192 * 7168 + 8192 * 2048) * 2


def test_switch_and_decode_bytes():
    sw = W.WORKLOADS["switch_top1"]
    a = bench.algorithmic(sw, sw.T)                # at most T rows survive capacity
    assert a["flops"] == 4 * 4096 * 768 * 3072      # two ReLU products
    dec = W.WORKLOADS["mixtral_decode_16"]
    assert bench.weight_bytes_hit(dec) == 8 * 3 * 4096 * 14336 * 2 + 4 * 4096 * 8
    # an expert that receives no row is not read
    assert bench.weight_bytes_hit(dec, [1, 0, 2, 0, 0, 3, 1, 1]) == 5 * 3 * 4096 * 14336 * 2 + 4 * 4096 * 8


# kernels per forward in the ncu launch lists of the benchmark commands
# (profiles/launch_list__*.md, profiles/expert_choice__*.md)
LAUNCHES = {"tiny_fp32": 7, "switch_top1": 8, "mixtral_prefill": 8, "mixtral_decode_16": 7,
            "deepseek_fine": 11, "mixtral_expert_choice": 11}


@pytest.mark.parametrize("name", sorted(LAUNCHES))
def test_kernels_per_forward(name):
    assert bench.launches_per_forward(W.WORKLOADS[name]) == LAUNCHES[name]
