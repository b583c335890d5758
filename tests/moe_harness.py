"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
and the oracle on the same seeded inputs, and compare.

Comparison rules:
  * routing, counts, offsets, dispatch order, slot rows and the drop set: bit-exact;
  * gates: |gpu - oracle| <= 1e-5;
  * aux losses: relative error <= 1e-4;
  * layer output: max |y_gpu - y_oracle| / RMS(y_oracle) <= 2e-2 (bf16) or 1e-4 (fp32).
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

import sparse_mixture_experts_64_b300 as moe
from oracle import moe_oracle as O

TOL_Y = {"bf16": 2e-2, "f32": 1e-4}
TOL_GATE = 1e-5
TOL_AUX = 1e-4


def cfg_of(w, debug_flags=0, save_preact=False):
    f = dataclasses.asdict(w)
    return moe.make_config(**f, debug_flags=debug_flags, save_preact=save_preact)


class _ExpertsView:
    """Per-expert host copies of a [N][...] device tensor, fetched on demand."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, e):
        return self.t[e].float().cpu().numpy()


def oracle_inputs(inp: dict) -> dict:
    """Host views of the device inputs for the oracle (exact values, fp32/fp64)."""
    out = {"x": inp["x"].float().cpu().numpy(), "w_r": inp["w_r"].cpu().numpy(),
           "b_r": None if inp["b_r"] is None else inp["b_r"].cpu().numpy()}
    for n in ("w_gate", "w_up", "w_down"):
        out[n] = None if inp[n] is None else _ExpertsView(inp[n])
    for n in ("shared_w_gate", "shared_w_up", "shared_w_down"):
        out[n] = None if inp[n] is None else inp[n].float().cpu().numpy()
    return out


def run_separate(cfg, inp, ws, dev="cuda"):
    """router -> dispatch -> grouped FFN -> combine through the four ABI calls."""
    T, k, N, d = cfg.T, cfg.k, cfg.N, cfg.d
    dt = inp["x"].dtype
    rmax = moe.moe_max_rows(cfg)
    o = dict(
        topk_idx=torch.full((T, k), -7, dtype=torch.int32, device=dev),
        topk_gate=torch.zeros((T, k), dtype=torch.float32, device=dev),
        counts_routed=torch.full((N,), -7, dtype=torch.int32, device=dev),
        counts_kept=torch.full((N,), -7, dtype=torch.int32, device=dev),
        expert_offsets=torch.full((N + 1,), -7, dtype=torch.int32, device=dev),
        slot_row=torch.full((T, k), -7, dtype=torch.int32, device=dev),
        perm_token=torch.full((rmax,), -7, dtype=torch.int32, device=dev),
        aux=torch.zeros(2, dtype=torch.float32, device=dev),
    )
    moe.moe_router_topk(cfg, inp["x"], inp["w_r"], inp["b_r"], o["topk_idx"], o["topk_gate"],
                        o["counts_routed"], o["counts_kept"], o["expert_offsets"], o["slot_row"],
                        o["perm_token"], o["aux"], ws)
    x_perm = torch.zeros((rmax, d), dtype=dt, device=dev)
    moe.moe_dispatch(cfg, inp["x"], o["perm_token"], o["expert_offsets"], x_perm, ws)
    y_perm = torch.zeros((rmax, d), dtype=dt, device=dev)
    moe.moe_grouped_ffn(cfg, x_perm, o["expert_offsets"], inp["w_gate"], inp["w_up"],
                        inp["w_down"], y_perm, ws)
    y = torch.empty((T, d), dtype=dt, device=dev)
    moe.moe_combine(cfg, inp["x"], y_perm, o["slot_row"], o["topk_gate"], inp["shared_w_gate"],
                    inp["shared_w_up"], inp["shared_w_down"], y, ws)
    o.update(x_perm=x_perm, y_perm=y_perm, y=y)
    return o


def run_forward(cfg, inp, ws, dev="cuda"):
    T, k, N, d = cfg.T, cfg.k, cfg.N, cfg.d
    o = dict(
        y=torch.empty((T, d), dtype=inp["x"].dtype, device=dev),
        topk_idx=torch.full((T, k), -7, dtype=torch.int32, device=dev),
        topk_gate=torch.zeros((T, k), dtype=torch.float32, device=dev),
        counts_routed=torch.full((N,), -7, dtype=torch.int32, device=dev),
        counts_kept=torch.full((N,), -7, dtype=torch.int32, device=dev),
        aux=torch.zeros(2, dtype=torch.float32, device=dev),
    )
    moe.moe_forward(cfg, inp["x"], inp["w_r"], inp["b_r"], inp["w_gate"], inp["w_up"],
                    inp["w_down"], inp["shared_w_gate"], inp["shared_w_up"],
                    inp["shared_w_down"], o["y"], o["topk_idx"], o["topk_gate"],
                    o["counts_routed"], o["counts_kept"], o["aux"], ws)
    return o


def host(o: dict) -> dict:
    return {k: v.float().cpu().numpy() if v.dtype in (torch.bfloat16, torch.float16)
            else v.cpu().numpy() for k, v in o.items()}


def rel_max_err(y, ref):
    ref = np.asarray(ref, np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(np.max(np.abs(np.asarray(y, np.float64) - ref))) / max(rms, 1e-30)


def check_routing(g: dict, rt: dict, sep: bool = True):
    """Bit-exact routing outputs and toleranced gates/aux against the oracle."""
    assert np.array_equal(g["topk_idx"], rt["topk_idx"]), "topk_idx differs"
    assert np.array_equal(g["counts_routed"], rt["counts_routed"]), "counts_routed differs"
    assert np.array_equal(g["counts_kept"], rt["counts_kept"]), "counts_kept differs"
    gate_err = float(np.max(np.abs(g["topk_gate"] - rt["topk_gate"])))
    assert gate_err <= TOL_GATE, f"gate error {gate_err}"
    for i in range(2):
        ref = rt["aux"][i]
        err = abs(float(g["aux"][i]) - ref)
        assert err <= TOL_AUX * max(abs(ref), 1e-6), f"aux[{i}] {g['aux'][i]} vs {ref}"
    if sep:
        assert np.array_equal(g["expert_offsets"], rt["expert_offsets"]), "expert_offsets differ"
        R = int(rt["expert_offsets"][-1])
        assert np.array_equal(g["perm_token"][:R], rt["perm_token"]), "perm_token differs"
        assert np.array_equal(g["slot_row"], rt["slot_row"]), "slot_row (drop set) differs"


def check_output(y, ref, dtype):
    err = rel_max_err(y, ref)
    assert err <= TOL_Y[dtype], f"output error {err} > {TOL_Y[dtype]}"
    return err
