"""Small launch sequences of the C-ABI calls for profiling single kernels under ncu.

Usage: python sparse_mixture_experts_64_b300/profile_cases.py CASE [--config NAME] [--reps N]

  router  moe_router_topk alone (router logits, gating, expert scan, slot assignment);
  memory  moe_router_topk, moe_dispatch and moe_combine (no shared expert) with the
          config's activation sizes: the HBM-bound kernels without the expert weights,
          so a DeepSeek-shaped case (0.94 GB of dispatched rows) holds about 2 GB;
  backward  one moe_forward, then moe_backward --reps times (the full layer: expert
          weights, their gradients and the backward scratch are all on the device);
  forward  moe_forward --reps times on the config's full layer.

Inputs are seeded synthetic tensors of the config's shapes (x ~ N(0,1), router
weight ~ N(0, 1/d), y_perm ~ N(0,1)); every launch goes through the library.
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import sparse_mixture_experts_64_b300 as moe  # noqa: E402
import workloads as W  # noqa: E402


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=("router", "memory", "backward", "forward"))
    ap.add_argument("--config", default="deepseek_fine", choices=sorted(W.WORKLOADS))
    ap.add_argument("--reps", type=int, default=4)
    ap.add_argument("--tokens", type=int, default=None, help="override T (smaller cases)")
    ap.add_argument("--experts", type=int, default=None, help="override N")
    ap.add_argument("--hidden", type=int, default=None, help="override h")
    a = ap.parse_args()
    w = W.WORKLOADS[a.config]
    over = {k: v for k, v in (("T", a.tokens), ("N", a.experts), ("h", a.hidden)) if v}
    if over:
        w = w.replace(name=w.name + "_" + "_".join(f"{k}{v}" for k, v in over.items()), **over)
    if a.case == "backward":
        return backward_case(w, a.reps)
    if a.case == "forward":
        return forward_case(w, a.reps)
    if a.case == "memory":
        w = w.replace(h_shared=0)
    dt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    g = torch.Generator(device="cuda").manual_seed(1)
    x = torch.randn((w.T, w.d), device="cuda", generator=g).to(dt)
    w_r = torch.randn((w.d, w.N), device="cuda", generator=g) / w.d ** 0.5
    b_r = torch.randn(w.N, device="cuda", generator=g) * 0.5 ** 0.5 if w.router_bias else None
    cfg = moe.make_config(T=w.T, d=w.d, N=w.N, k=w.k, h=w.h, h_shared=w.h_shared, dtype=w.dtype,
                          gating=w.gating, act=w.act, capacity_factor=w.capacity_factor,
                          router_bias=w.router_bias)
    ws = moe.workspace(cfg)
    T, k, N, R = w.T, w.k, w.N, moe.moe_max_rows(cfg)
    i32 = dict(dtype=torch.int32, device="cuda")
    idx, slot_row = torch.empty((T, k), **i32), torch.empty((T, k), **i32)
    gate = torch.empty((T, k), device="cuda")
    routed, kept, offsets = torch.empty(N, **i32), torch.empty(N, **i32), torch.empty(N + 1, **i32)
    perm, aux = torch.empty(R, **i32), torch.empty(2, device="cuda")
    if a.case == "memory":
        x_perm = torch.empty((R, w.d), dtype=dt, device="cuda")
        y_perm = torch.randn((R, w.d), device="cuda", generator=g).to(dt)
        y = torch.empty((T, w.d), dtype=dt, device="cuda")
    for _ in range(a.reps):
        moe.moe_router_topk(cfg, x, w_r, b_r, idx, gate, routed, kept, offsets, slot_row, perm, aux, ws)
        if a.case == "memory":
            moe.moe_dispatch(cfg, x, perm, offsets, x_perm, ws)
            moe.moe_combine(cfg, x, y_perm, slot_row, gate, None, None, None, y, ws)
    st = moe.moe_check_error(ws)
    print(f"{a.case} {w.name}: status {moe.status_str(st)}, "
          f"{torch.cuda.max_memory_allocated() / 1e9:.2f} GB allocated")
    if st != moe.MOE_OK:
        sys.exit(1)


def _layer_config(w):
    return moe.make_config(T=w.T, d=w.d, N=w.N, k=w.k, h=w.h, h_shared=w.h_shared, dtype=w.dtype,
                           gating=w.gating, act=w.act, capacity_factor=w.capacity_factor,
                           router_bias=w.router_bias, routing=w.routing)


def forward_case(w, reps: int) -> None:
    cfg = _layer_config(w)
    inp = W.make_inputs(w, device="cuda")
    ws = moe.workspace(cfg)
    y = torch.empty((w.T, w.d), dtype=inp["x"].dtype, device="cuda")
    for _ in range(reps):
        moe.moe_forward(cfg, inp["x"], inp["w_r"], inp["b_r"], inp["w_gate"], inp["w_up"], inp["w_down"],
                        inp["shared_w_gate"], inp["shared_w_up"], inp["shared_w_down"], y, None, None, None,
                        None, None, ws)
    st = moe.moe_check_error(ws)
    print(f"forward {w.name}: status {moe.status_str(st)}, "
          f"{torch.cuda.max_memory_allocated() / 1e9:.2f} GB allocated")
    if st != moe.MOE_OK:
        sys.exit(1)


def backward_case(w, reps: int) -> None:
    cfg = moe.make_config(T=w.T, d=w.d, N=w.N, k=w.k, h=w.h, h_shared=w.h_shared, dtype=w.dtype,
                          gating=w.gating, act=w.act, capacity_factor=w.capacity_factor,
                          router_bias=w.router_bias)
    inp = W.make_inputs(w, device="cuda")
    ws, bws = moe.workspace(cfg), moe.backward_workspace(cfg)
    T, d, k = w.T, w.d, w.k
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, k), device="cuda")
    y = torch.empty((T, d), dtype=inp["x"].dtype, device="cuda")
    moe.moe_forward(cfg, inp["x"], inp["w_r"], inp["b_r"], inp["w_gate"], inp["w_up"], inp["w_down"],
                    inp["shared_w_gate"], inp["shared_w_up"], inp["shared_w_down"], y, idx, gate, None, None,
                    None, ws)
    g = torch.Generator(device="cuda").manual_seed(2)
    dy = torch.randn((T, d), device="cuda", generator=g).to(inp["x"].dtype)
    e = lambda t: None if t is None else torch.empty_like(t)  # noqa: E731
    out = [e(inp[n]) for n in ("x", "w_r", "b_r", "w_gate", "w_up", "w_down", "shared_w_gate", "shared_w_up",
                               "shared_w_down")]
    for _ in range(reps):
        moe.moe_backward(cfg, inp["x"], inp["w_r"], inp["b_r"], inp["w_gate"], inp["w_up"], inp["w_down"],
                         inp["shared_w_gate"], inp["shared_w_up"], inp["shared_w_down"], idx, gate, dy, 0.01,
                         0.001, *out, ws, bws)
    st = moe.moe_check_error(ws)
    print(f"backward {w.name}: status {moe.status_str(st)}, "
          f"{torch.cuda.max_memory_allocated() / 1e9:.2f} GB allocated")
    if st != moe.MOE_OK:
        sys.exit(1)


if __name__ == "__main__":
    main()
