"""Seeded synthetic workloads for the sparse MoE layer forward.

This module only names workload shapes and draws their random inputs. It holds
none of the layer's arithmetic, so both the CUDA path's tests/benchmark and the
CPU oracle may take their inputs from it without sharing any computation.

Shapes follow the five workloads the layer is measured on:

* ``tiny_fp32``       T=256,  d=64,   N=4,   h=128,   top-2, top-k then softmax, fp32.
* ``switch_top1``     T=4096, d=768,  N=8,   h=3072,  top-1, softmax over all N then top-1,
                      ReLU (non-gated) experts, capacity factor 1.25, per-expert router bias.
* ``mixtral_prefill`` T=4096, d=4096, N=8,   h=14336, top-2, top-k then softmax, SiLU-gated.
* ``mixtral_decode_{16,64,128}``  the same layer with T in {16, 64, 128}.
* ``deepseek_fine``   T=8192, d=7168, N=256, h=2048,  top-8, softmax over all N then top-8
                      (gates not renormalised), one always-on shared expert of hidden 2048.

Distributions: x ~ N(0, 1); every weight ~ N(0, 1/d_in) (d_in = d for the router,
gate, up and W1 projections; d_in = h for the down and W2 projections); the
Switch router bias ~ N(0, 0.5), read as a variance like the N(0, 1/d) notation,
so its standard deviation is sqrt(0.5).

Seeds: workload number c (1..5) uses seed 1000*c + j for tensor j:
0 x, 1 W_r, 2 router bias, 3 W_gate (or W1), 4 W_up, 5 W_down (or W2),
6 shared W_gate, 7 shared W_up, 8 shared W_down.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    number: int           # seed family (1..5)
    T: int                # tokens
    d: int                # model dimension
    N: int                # routed experts
    k: int                # experts per token
    h: int                # routed expert hidden size
    h_shared: int = 0     # shared expert hidden size (0: no shared expert)
    dtype: str = "bf16"   # "f32" or "bf16": activations and expert weights
    gating: str = "topk_then_softmax"   # or "softmax_then_topk"
    act: str = "silu_gated"             # or "relu"
    capacity_factor: tuple | None = None  # (num, den) or None for no limit
    router_bias: bool = False
    routing: str = "token_choice"       # or "expert_choice" (capacity_factor = experts per token)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    "tiny_fp32": Workload("tiny_fp32", 1, T=256, d=64, N=4, k=2, h=128, dtype="f32",
                          gating="topk_then_softmax", act="silu_gated"),
    "switch_top1": Workload("switch_top1", 2, T=4096, d=768, N=8, k=1, h=3072,
                            gating="softmax_then_topk", act="relu",
                            capacity_factor=(5, 4), router_bias=True),
    "mixtral_prefill": Workload("mixtral_prefill", 3, T=4096, d=4096, N=8, k=2, h=14336,
                                gating="topk_then_softmax", act="silu_gated"),
    "mixtral_decode_16": Workload("mixtral_decode_16", 4, T=16, d=4096, N=8, k=2, h=14336),
    "mixtral_decode_64": Workload("mixtral_decode_64", 4, T=64, d=4096, N=8, k=2, h=14336),
    "mixtral_decode_128": Workload("mixtral_decode_128", 4, T=128, d=4096, N=8, k=2, h=14336),
    "deepseek_fine": Workload("deepseek_fine", 5, T=8192, d=7168, N=256, k=8, h=2048,
                              h_shared=2048, gating="softmax_then_topk", act="silu_gated"),
    # Expert Choice on the Mixtral prefill layer (same seeds, so the same inputs):
    # every expert takes C = T * 2 / N tokens, two experts per token on average
    "mixtral_expert_choice": Workload("mixtral_expert_choice", 3, T=4096, d=4096, N=8, k=2,
                                      h=14336, act="silu_gated", capacity_factor=(2, 1),
                                      routing="expert_choice"),
}


def torch_dtype(w: Workload) -> torch.dtype:
    return torch.float32 if w.dtype == "f32" else torch.bfloat16


def _normal(shape, std, seed, device, out_dtype, chunk_dim0=False):
    """N(0, std^2) drawn in fp32 from a generator seeded with `seed`, then cast.

    With chunk_dim0 the leading dimension is drawn one slice at a time from the
    same generator, which bounds the fp32 temporary for the big expert stacks."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    out = torch.empty(shape, dtype=out_dtype, device=device)
    if chunk_dim0:
        tmp = torch.empty(shape[1:], dtype=torch.float32, device=device)
        for i in range(shape[0]):
            tmp.normal_(0.0, std, generator=g)
            out[i].copy_(tmp)
        del tmp
    else:
        tmp = torch.empty(shape, dtype=torch.float32, device=device)
        tmp.normal_(0.0, std, generator=g)
        out.copy_(tmp)
    return out


def make_inputs(w: Workload, device="cpu", seed_family: int | None = None,
                router_only: bool = False) -> dict:
    """All inputs of one layer forward for workload `w`, on `device`.
    router_only: only x, w_r and b_r (the same values); the weight entries are None.

    Returns a dict of torch tensors:
      x [T][d] (dtype of w), w_r [d][N] fp32, b_r [N] fp32 or None,
      w_gate/w_up [N][h][d] and w_down [N][d][h] (SiLU-gated), or
      w1 [N][h][d] (as "w_gate"), w_up None, w2 [N][d][h] (as "w_down") for ReLU,
      shared_w_gate/shared_w_up [h_s][d], shared_w_down [d][h_s] or None.
    """
    c = w.number if seed_family is None else seed_family
    s = 1000 * c
    dt = torch_dtype(w)
    inp = {}
    inp["x"] = _normal((w.T, w.d), 1.0, s + 0, device, dt)
    inp["w_r"] = _normal((w.d, w.N), 1.0 / math.sqrt(w.d), s + 1, device, torch.float32)
    inp["b_r"] = (_normal((w.N,), math.sqrt(0.5), s + 2, device, torch.float32)
                  if w.router_bias else None)
    if router_only:
        for n in ("w_gate", "w_up", "w_down", "shared_w_gate", "shared_w_up", "shared_w_down"):
            inp[n] = None
        return inp
    inp["w_gate"] = _normal((w.N, w.h, w.d), 1.0 / math.sqrt(w.d), s + 3, device, dt, True)
    inp["w_up"] = (_normal((w.N, w.h, w.d), 1.0 / math.sqrt(w.d), s + 4, device, dt, True)
                   if w.act == "silu_gated" else None)
    inp["w_down"] = _normal((w.N, w.d, w.h), 1.0 / math.sqrt(w.h), s + 5, device, dt, True)
    if w.h_shared:
        hs = w.h_shared
        inp["shared_w_gate"] = _normal((hs, w.d), 1.0 / math.sqrt(w.d), s + 6, device, dt)
        inp["shared_w_up"] = _normal((hs, w.d), 1.0 / math.sqrt(w.d), s + 7, device, dt)
        inp["shared_w_down"] = _normal((w.d, hs), 1.0 / math.sqrt(hs), s + 8, device, dt)
    else:
        inp["shared_w_gate"] = inp["shared_w_up"] = inp["shared_w_down"] = None
    return inp


def small_variant(w: Workload, **kw) -> Workload:
    """A reduced copy of workload `w` (same gating, activation, dtype, capacity)."""
    return w.replace(name=w.name + "_small", **kw)
