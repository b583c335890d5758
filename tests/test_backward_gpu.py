"""Backward of the layer on the GPU against the oracle's backward (float64, pinned
against torch autograd and finite differences).

The GPU keeps dy, the gate-scaled rows dO, the hidden activations H, the recomputed
pre-activations A and B, dH and [dA | dB] in bf16 and accumulates in fp32 (the
router's gradients are fp32; its two contractions multiply bf16 hi/lo splits of the
fp32 operands, whose products the fp32 accumulator holds exactly, within 2^-15 of the
fp32 products). Each of those roundings is relative
(2^-9), so a gradient element's error is proportional to its own size, and the
gradients are heavy-tailed (elements 10-20 times their RMS occur). A float64
simulation of exactly those roundings (and of the bf16 outputs) on these shapes gives
an RMS-relative error of 0.3-0.5 %, and an elementwise error |Δ| / (|oracle| + RMS)
up to 2 % with ~50 rows per expert and up to 4.7 % with ~9 rows per expert (N = 64,
top-6 on 96 tokens: a weight-gradient element is then a sum of a few products and
cancels). Every gradient is therefore held to
    RMS(gpu - oracle) / RMS(oracle) <= 1e-2      (a wrong term, sign or row: O(1))
    max |gpu - oracle| / (|oracle| + RMS(oracle)) <= 6e-2   (elementwise)."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import sparse_mixture_experts_64_b300 as moe
    from moe_harness import cfg_of, oracle_inputs

TOL_RMS, TOL_ELEM = 1e-2, 6e-2


def _errs(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = max(float(np.sqrt(np.mean(ref * ref))), 1e-30)
    return (float(np.sqrt(np.mean((got - ref) ** 2))) / rms,
            float(np.max(np.abs(got - ref) / (np.abs(ref) + rms))))


def _w(name, **kw):
    return W.WORKLOADS[name].replace(name="bwd_" + name + "_" + "_".join(f"{a}{b}" for a, b in kw.items()), **kw)


CASES = [
    (_w("mixtral_prefill", T=300, d=256, h=384), 0.01, 0.001),
    (_w("deepseek_fine", T=200, d=256, N=16, k=4, h=128, h_shared=128), 0.02, 0.0),
    (_w("switch_top1", T=333, d=128, h=256), 0.01, 0.001),                       # ReLU, bias, drops
    (_w("switch_top1", T=150, d=192, h=128, N=4, k=2, h_shared=192, capacity_factor=None), 0.0, 0.01),
    (_w("mixtral_prefill", T=1024, d=512, h=1024, N=8, k=2), 0.0, 0.0),          # pair kernels
    (_w("deepseek_fine", T=96, d=128, N=64, k=6, h=192, h_shared=0), 0.05, 0.0),  # N > 32 router
    (_w("deepseek_fine", T=600, d=64, N=4, k=2, h=64, h_shared=64), 0.01, 0.001),  # smallest tiles, pair
    # 128 routed rows over 64 experts: many experts without rows on the pair
    # weight-gradient kernel (their gradients are stored as zero boxes)
    (_w("deepseek_fine", T=64, d=256, N=64, k=2, h=256, h_shared=256), 0.01, 0.0),
    # N = 128: both router-gradient products on CTA pairs (2N = 256 and T = 320 rows)
    (_w("deepseek_fine", T=320, d=256, N=128, k=4, h=128, h_shared=0), 0.01, 0.001),
    # the DeepSeekMoE structure: 256 experts, top-8 and a shared expert (257 segments in
    # the row products, about 16 rows per expert, partial k-blocks everywhere)
    (_w("deepseek_fine", T=512, d=128, N=256, k=8, h=128, h_shared=128), 0.01, 0.001),
]


def _run(w, aux_coef, z_coef, seed=3, debug_flags=0, save_preact=False, stale=False):
    cfg = cfg_of(w, debug_flags=debug_flags, save_preact=save_preact)
    inp = W.make_inputs(w, device="cuda")
    ws = moe.workspace(cfg)
    bws = moe.backward_workspace(cfg)
    if stale:
        # every byte 0xFF (NaN in bf16 and fp32) but the error word's region
        ws.fill_(255)
        ws[:256] = 0
        bws.fill_(255)
    T, d, N, k = w.T, w.d, w.N, w.k
    y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, k), device="cuda")
    moe.moe_forward(cfg, inp["x"], inp["w_r"], inp["b_r"], inp["w_gate"], inp["w_up"], inp["w_down"],
                    inp["shared_w_gate"], inp["shared_w_up"], inp["shared_w_down"], y, idx, gate, None, None,
                    None, ws)
    g = torch.Generator(device="cuda").manual_seed(seed)
    dy = torch.randn((T, d), device="cuda", generator=g).to(torch.bfloat16)
    out = dict(dx=torch.empty_like(inp["x"]), dw_r=torch.empty_like(inp["w_r"]),
               db_r=torch.empty(N, device="cuda") if w.router_bias else None,
               dw_gate=torch.empty_like(inp["w_gate"]),
               dw_up=torch.empty_like(inp["w_up"]) if inp["w_up"] is not None else None,
               dw_down=torch.empty_like(inp["w_down"]))
    for n in ("shared_w_gate", "shared_w_up", "shared_w_down"):
        out["d" + n] = torch.empty_like(inp[n]) if inp[n] is not None else None
    moe.moe_backward(cfg, inp["x"], inp["w_r"], inp["b_r"], inp["w_gate"], inp["w_up"], inp["w_down"],
                     inp["shared_w_gate"], inp["shared_w_up"], inp["shared_w_down"], idx, gate, dy, aux_coef,
                     z_coef, out["dx"], out["dw_r"], out["db_r"], out["dw_gate"], out["dw_up"], out["dw_down"],
                     out["dshared_w_gate"], out["dshared_w_up"], out["dshared_w_down"], ws, bws)
    assert moe.moe_check_error(ws) == moe.MOE_OK
    return inp, dy, out


def _f(t):
    return None if t is None else t.float().cpu().numpy()




@pytest.mark.parametrize("w,aux,z", CASES, ids=[c[0].name for c in CASES])
def test_backward_matches_oracle(w, aux, z):
    _check(w, aux, z, 0)


# gated with a shared expert, ReLU with bias and drops, ReLU with a shared expert, the
# pair kernels (with a split), the smallest tiles, and ReLU experts on the pair kernel
# with tail tiles
KEPT = [CASES[i] for i in (1, 2, 3, 4, 6)] + [
    (_w("switch_top1", T=1100, d=128, h=256, N=2, capacity_factor=None), 0.01, 0.001),
    # the shared expert as a segment of the forward's pair launch, its 1100 rows ending
    # in a tail tile
    (_w("deepseek_fine", T=1100, d=256, N=8, k=2, h=128, h_shared=128), 0.01, 0.001)]


@pytest.mark.parametrize("w,aux,z", KEPT, ids=[c[0].name for c in KEPT])
def test_backward_with_kept_preactivations(w, aux, z):
    """save_preact: the forward keeps the pre-activations and the backward reads them;
    the gradients match the oracle, and match bit for bit those of the backward that
    recomputes them (the same products on the same kernels)."""
    out = _check(w, aux, z, 0, save_preact=True)
    _, _, ref = _run(w, aux, z)
    for key, t in out.items():
        if t is not None:
            assert torch.equal(t, ref[key]), key


def test_kept_preactivations_on_single_cta_kernels():
    """The pair-kernel shape with every product on the single-CTA kernel, whose row
    epilogue (half tiles included) then keeps the pre-activations."""
    w, aux, z = CASES[4]
    _check(w, aux, z, moe.MOE_DEBUG_FFN_SINGLE, save_preact=True)


def test_kept_preactivations_through_the_forward_graph():
    """A keeping forward captured as a CUDA graph leaves what moe_backward reads: the
    gradients equal bit for bit those after the stream-launched keeping forward."""
    w, aux, z = CASES[1]
    _, _, ref = _run(w, aux, z, save_preact=True)
    cfg = cfg_of(w, save_preact=True)
    inp = W.make_inputs(w, device="cuda")
    ws = moe.workspace(cfg)
    bws = moe.backward_workspace(cfg)
    T, d, k = w.T, w.d, w.k
    y = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    idx = torch.empty((T, k), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, k), device="cuda")
    g = moe.moe_forward_graph_create(cfg, inp["x"], inp["w_r"], inp["b_r"], inp["w_gate"], inp["w_up"],
                                     inp["w_down"], inp["shared_w_gate"], inp["shared_w_up"],
                                     inp["shared_w_down"], y, idx, gate, None, None, None, ws)
    try:
        g.launch()
    finally:
        g.destroy()
    gen = torch.Generator(device="cuda").manual_seed(3)
    dy = torch.randn((T, d), device="cuda", generator=gen).to(torch.bfloat16)
    out = {key: None if t is None else torch.empty_like(t) for key, t in ref.items()}
    moe.moe_backward(cfg, inp["x"], inp["w_r"], inp["b_r"], inp["w_gate"], inp["w_up"], inp["w_down"],
                     inp["shared_w_gate"], inp["shared_w_up"], inp["shared_w_down"], idx, gate, dy, aux, z,
                     out["dx"], out["dw_r"], out["db_r"], out["dw_gate"], out["dw_up"], out["dw_down"],
                     out["dshared_w_gate"], out["dshared_w_up"], out["dshared_w_down"], ws, bws)
    assert moe.moe_check_error(ws) == moe.MOE_OK
    for key, t in ref.items():
        if t is not None:
            assert torch.equal(out[key], t), key


def test_backward_single_cta_kernels():
    """The pair-kernel shape once more with every expert product and weight gradient
    on the single-CTA kernels."""
    w, aux, z = CASES[4]
    _check(w, aux, z, moe.MOE_DEBUG_FFN_SINGLE)


# every row product over several rounds of the persistent schedule (each CTA or CTA
# pair takes several tiles in turn): 128-256 tiles on the 74 CTA pairs, 256-512 on the
# 148 single CTAs
ROUNDS = (_w("mixtral_prefill", T=2048, d=2048, h=2048, N=8, k=2), 0.01, 0.001)


@pytest.mark.parametrize("kernel", ["pair", "single", "pair_kept"])
def test_backward_over_several_rounds(kernel):
    w, aux, z = ROUNDS
    flags = moe.MOE_DEBUG_FFN_SINGLE if kernel == "single" else 0
    out = _check(w, aux, z, flags, save_preact=kernel == "pair_kept")
    if kernel == "pair_kept":
        _, _, ref = _run(w, aux, z)
        for key, t in out.items():
            if t is not None:
                assert torch.equal(t, ref[key]), key


# capacity limits: the row buffers (N x capacity rows) are longer than the rows kept
STALE = [(_w("switch_top1", T=333, d=128, h=256), 0.01, 0.001),
         (_w("mixtral_prefill", T=600, d=256, h=384, N=8, k=2, capacity_factor=(5, 4)), 0.01, 0.001)]


@pytest.mark.parametrize("kernel", ["pair", "single"])
@pytest.mark.parametrize("w,aux,z", STALE, ids=[c[0].name for c in STALE])
def test_backward_with_stale_workspaces(w, aux, z, kernel):
    """Workspaces left with NaN bit patterns (every byte 0xFF but the error word): the
    rows past the kept ones, which an expert's partial last k-block of the weight
    gradients reaches into, then hold NaN unless zeroed on the way to the MMAs. The
    forward and the gradients still match the oracle and hold no NaN."""
    flags = moe.MOE_DEBUG_FFN_SINGLE if kernel == "single" else 0
    out = _check(w, aux, z, flags, stale=True)
    for key, t in out.items():
        if t is not None:
            assert not torch.isnan(t.float()).any(), key


def _check(w, aux, z, flags, save_preact=False, stale=False):
    inp, dy, out = _run(w, aux, z, debug_flags=flags, save_preact=save_preact, stale=stale)
    ref = O.backward(w, oracle_inputs(inp), _f(dy), aux_coef=aux, z_coef=z)
    errs = {"dx": _errs(_f(out["dx"]), ref["dx"]), "dw_r": _errs(_f(out["dw_r"]), ref["dw_r"])}
    if out["db_r"] is not None:
        errs["db_r"] = _errs(_f(out["db_r"]), ref["db_r"])
    for key in ("dw_gate", "dw_up", "dw_down"):
        if out[key] is None:
            continue
        got = _f(out[key])
        want = np.stack([np.zeros_like(got[e]) if ref[key][e] is None else ref[key][e] for e in range(w.N)])
        errs[key] = _errs(got, want)
        # experts without rows get exactly zero
        for e in range(w.N):
            if ref[key][e] is None:
                assert not np.any(got[e]), (key, e)
    if w.h_shared:
        for key, rk in (("dshared_w_gate", "dw_gate"), ("dshared_w_up", "dw_up"), ("dshared_w_down", "dw_down")):
            errs[key] = _errs(_f(out[key]), ref["shared"][rk])
    print({k_: (round(a, 5), round(b, 4)) for k_, (a, b) in errs.items()})
    bad = {k_: v for k_, v in errs.items() if not (v[0] <= TOL_RMS and v[1] <= TOL_ELEM)}
    assert not bad, errs
    return out


def test_backward_is_deterministic():
    w = CASES[1][0]
    _, _, a = _run(w, 0.02, 0.01)
    _, _, b = _run(w, 0.02, 0.01)
    for key in a:
        if a[key] is not None:
            assert torch.equal(a[key], b[key]), key
