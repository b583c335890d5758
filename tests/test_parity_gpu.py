"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Small and ragged shapes are compared element by element on every output; the
full-size workloads are compared bit-exactly on all routing outputs, on the layer
output of a seeded token sample, and on the expert outputs of rows drawn from every
128-row block of every expert."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import sparse_mixture_experts_64_b300 as moe
    from moe_harness import (cfg_of, check_output, check_routing, host, oracle_inputs,
                             rel_max_err, run_forward, run_separate)


def _small(name, **kw):
    return W.WORKLOADS[name].replace(name=name + "_" + "_".join(f"{a}{b}" for a, b in kw.items()),
                                     **kw)


SMALL = [
    W.WORKLOADS["tiny_fp32"],
    _small("tiny_fp32", T=77),
    _small("tiny_fp32", T=33, N=1, k=1, d=16, h=24),
    _small("tiny_fp32", T=50, N=5, k=5, d=24, h=40, h_shared=16,
           gating="softmax_then_topk"),
    _small("switch_top1", T=640, d=256, h=512),
    W.WORKLOADS["switch_top1"],
    _small("switch_top1", T=333, d=128, h=256, k=2, capacity_factor=(1, 2), act="silu_gated"),
    _small("mixtral_prefill", T=300, d=256, h=384),
    _small("mixtral_prefill", T=1, d=128, h=128),
    _small("mixtral_prefill", T=129, d=192, h=320, N=3, k=3),
    # 256 rows per expert on average: pair kernel for some experts, single-CTA for the
    # experts whose last 256-row block holds at most 128 rows
    _small("mixtral_prefill", T=1024, d=256, h=256),
    _small("deepseek_fine", T=200, d=256, N=16, k=4, h=128, h_shared=128),
    _small("deepseek_fine", T=130, d=128, N=256, k=8, h=128, h_shared=192),
    _small("deepseek_fine", T=96, d=128, N=100, k=6, h=192, h_shared=0,
           gating="topk_then_softmax"),
]


@pytest.fixture(scope="module", autouse=True)
def _device():
    torch.cuda.init()
    yield
    torch.cuda.synchronize()


@pytest.mark.parametrize("w", SMALL, ids=[w.name for w in SMALL])
def test_small_parity(w):
    inp = W.make_inputs(w, device="cuda")
    cfg = cfg_of(w)
    ws = moe.workspace(cfg)
    sep = host(run_separate(cfg, inp, ws))
    fwd = host(run_forward(cfg, inp, ws))
    assert moe.moe_check_error(ws) == moe.MOE_OK
    rt = O.forward(w, oracle_inputs(inp))
    check_routing(sep, rt, sep=True)
    check_routing(fwd, rt, sep=False)
    check_output(sep["y"], rt["y"], w.dtype)
    # the fused call runs the same kernels: identical bits
    assert np.array_equal(fwd["y"], sep["y"])
    # dropped tokens keep exactly their residual when there is no shared expert
    dropped = ~rt["kept"].any(axis=1)
    if dropped.any() and not w.h_shared:
        assert np.array_equal(sep["y"][dropped], inp["x"].float().cpu().numpy()[dropped])


PAIR = [
    _small("mixtral_prefill", T=300, d=256, h=384),
    _small("switch_top1", T=640, d=256, h=512),
    _small("deepseek_fine", T=200, d=256, N=16, k=4, h=128, h_shared=192),
    _small("mixtral_prefill", T=1100, d=128, h=256, N=2, k=1),
    # hidden sizes that are not a multiple of the 128/256-wide weight blocks
    _small("deepseek_fine", T=333, d=192, N=12, k=3, h=320, h_shared=192),
    _small("switch_top1", T=700, d=320, h=448, N=4),
]


@pytest.mark.parametrize("w", PAIR, ids=[w.name for w in PAIR])
def test_all_tensor_core_ffn_kernels(w):
    """The three tensor-core kernels (weights-as-M CTA pair with token tiles of 32..256,
    row-tile CTA pair with 256-row tiles, row-tile single CTA with 128-row tiles)
    match the oracle on the same inputs."""
    inp = W.make_inputs(w, device="cuda")
    ws = moe.workspace(cfg_of(w))
    rt = O.forward(w, oracle_inputs(inp))
    outs = {}
    for name, flag in (("swap", moe.MOE_DEBUG_FFN_SWAP), ("pair", moe.MOE_DEBUG_FFN_PAIR),
                       ("single", moe.MOE_DEBUG_FFN_SINGLE)):
        outs[name] = host(run_forward(cfg_of(w, debug_flags=flag), inp, ws))
        assert moe.moe_check_error(ws) == moe.MOE_OK, name
        check_routing(outs[name], rt, sep=False)
        check_output(outs[name]["y"], rt["y"], w.dtype)
    assert rel_max_err(outs["pair"]["y"], outs["single"]["y"]) <= 2e-2
    assert rel_max_err(outs["swap"]["y"], outs["single"]["y"]) <= 2e-2


# every product over several rounds of the persistent schedule: 256 and 128 tiles on the
# 74 CTA pairs, 512 and 256 on the 148 single CTAs
ROUNDS = _small("mixtral_prefill", T=2048, d=2048, h=2048, N=8, k=2)


@pytest.mark.parametrize("kernel", ["pair", "single"])
def test_products_over_several_rounds(kernel):
    """Each CTA (pair) of the persistent kernels takes several tiles in turn, with the
    operand ring and both accumulators carried from tile to tile: the layer output and
    the expert outputs of rows from every expert and 256-row block match the oracle."""
    w = ROUNDS
    flags = moe.MOE_DEBUG_FFN_PAIR if kernel == "pair" else moe.MOE_DEBUG_FFN_SINGLE
    inp = W.make_inputs(w, device="cuda")
    cfg = cfg_of(w, debug_flags=flags)
    ws = moe.workspace(cfg)
    sep = host(run_separate(cfg, inp, ws))
    assert moe.moe_check_error(ws) == moe.MOE_OK
    check_expert_rows(w, inp, sep, np.random.default_rng(5))
    rt = O.forward(w, oracle_inputs(inp))
    check_routing(sep, rt, sep=True)
    check_output(sep["y"], rt["y"], w.dtype)


@pytest.mark.parametrize("name", ["mixtral_prefill", "deepseek_fine"])
def test_simt_and_tensor_core_ffn_agree(name):
    w = _small(name, T=160, d=256, h=256, N=8, k=2, h_shared=128 if name == "deepseek_fine" else 0)
    inp = W.make_inputs(w, device="cuda")
    ws = moe.workspace(cfg_of(w))
    tc = host(run_forward(cfg_of(w), inp, ws))
    simt = host(run_forward(cfg_of(w, debug_flags=moe.MOE_DEBUG_FORCE_SIMT_FFN), inp, ws))
    assert np.array_equal(tc["topk_idx"], simt["topk_idx"])
    assert rel_max_err(tc["y"], simt["y"]) <= 2e-2


def test_worked_example_on_gpu():
    """The pages' d=8, four-expert, top-2 router example through moe_router_topk."""
    w = W.Workload("worked", 1, T=1, d=8, N=4, k=2, h=8, dtype="f32")
    x = torch.zeros((1, 8), dtype=torch.float32, device="cuda")
    x[0, 0] = 1.0
    w_r = torch.zeros((8, 4), dtype=torch.float32, device="cuda")
    w_r[0] = torch.tensor([1.0, 0.0, 2.0, -1.0])
    cfg = cfg_of(w)
    ws = moe.workspace(cfg)
    idx = torch.empty((1, 2), dtype=torch.int32, device="cuda")
    gate = torch.empty((1, 2), dtype=torch.float32, device="cuda")
    off = torch.empty(5, dtype=torch.int32, device="cuda")
    sr = torch.empty((1, 2), dtype=torch.int32, device="cuda")
    perm = torch.empty(2, dtype=torch.int32, device="cuda")
    moe.moe_router_topk(cfg, x, w_r, None, idx, gate, None, None, off, sr, perm, None, ws)
    assert idx.cpu().tolist() == [[2, 0]]
    g = gate.cpu().numpy()[0]
    assert abs(g[0] - 1 / (1 + np.exp(-1.0))) < 1e-6 and abs(g[1] - 1 / (1 + np.exp(1.0))) < 1e-6
    assert off.cpu().tolist() == [0, 1, 1, 2, 2]
    assert perm.cpu().tolist() == [0, 0]
    assert sr.cpu().tolist() == [[1, 0]]


def test_three_token_example_on_gpu():
    """The pages' three-token dispatch example: groups E1{1,3}, E2{2}, E3{1,2,3}, E4{}."""
    import math
    scores = np.full((3, 4), -8.0, np.float32)
    scores[0, 0], scores[0, 2] = 0.0, math.log(0.73 / 0.27)
    scores[1, 1], scores[1, 2] = 0.0, 0.25
    scores[2, 0], scores[2, 2] = math.log(0.88 / 0.12), 0.0
    x = torch.zeros((3, 8), dtype=torch.float32, device="cuda")
    w_r = torch.zeros((8, 4), dtype=torch.float32, device="cuda")
    for t in range(3):
        x[t, t] = 1.0
        w_r[t] = torch.from_numpy(scores[t])
    w = W.Workload("three", 1, T=3, d=8, N=4, k=2, h=8, dtype="f32")
    cfg = cfg_of(w)
    ws = moe.workspace(cfg)
    rmax = moe.moe_max_rows(cfg)
    o = {n: torch.empty(s, dtype=torch.int32, device="cuda") for n, s in
         [("idx", (3, 2)), ("off", (5,)), ("sr", (3, 2)), ("perm", (rmax,)), ("cr", (4,)),
          ("ck", (4,))]}
    gate = torch.empty((3, 2), dtype=torch.float32, device="cuda")
    moe.moe_router_topk(cfg, x, w_r, None, o["idx"], gate, o["cr"], o["ck"], o["off"], o["sr"],
                        o["perm"], None, ws)
    assert o["ck"].cpu().tolist() == [2, 1, 3, 0]
    assert o["off"].cpu().tolist() == [0, 2, 3, 6, 6]
    assert o["perm"].cpu().tolist()[:6] == [0, 2, 1, 0, 1, 2]
    g = gate.cpu().numpy()
    i = o["idx"].cpu().numpy()
    assert abs(g[0][list(i[0]).index(0)] - 0.27) < 0.005
    assert abs(g[2][list(i[2]).index(0)] - 0.88) < 0.005


def test_run_to_run_determinism():
    w = _small("deepseek_fine", T=256, d=256, N=32, k=4, h=128, h_shared=128)
    inp = W.make_inputs(w, device="cuda")
    cfg = cfg_of(w)
    ws = moe.workspace(cfg)
    first = host(run_forward(cfg, inp, ws))
    for _ in range(5):
        again = host(run_forward(cfg, inp, ws))
        for k in first:
            assert np.array_equal(first[k], again[k]), k


KEEP = [_small("mixtral_prefill", T=1024, d=256, h=256),
        _small("deepseek_fine", T=200, d=256, N=16, k=4, h=128, h_shared=128),
        _small("switch_top1", T=333, d=128, h=256),
        _small("switch_top1", T=150, d=192, h=128, N=4, k=2, h_shared=192, capacity_factor=None),
        # ReLU experts of ~550 rows on the pair kernel, whose last blocks are tail tiles
        _small("switch_top1", T=1100, d=128, h=256, N=2, capacity_factor=None),
        # the pair kernel with the shared expert's segment (1100 rows: a 76-row tail tile)
        _small("deepseek_fine", T=1100, d=256, N=8, k=2, h=128, h_shared=128)]


@pytest.mark.parametrize("w", KEEP, ids=[w.name for w in KEEP])
def test_forward_keeping_preactivations(w):
    """save_preact only adds stores: the forward's outputs are bit for bit those of the
    plain forward, and the kept pre-activations of every kept row and of the shared
    expert are those of the oracle's experts (x W_gateᵀ, x W_upᵀ / x W1ᵀ)."""
    inp = W.make_inputs(w, device="cuda")
    plain_cfg, keep_cfg = cfg_of(w), cfg_of(w, save_preact=True)
    ws0, ws1 = moe.workspace(plain_cfg), moe.workspace(keep_cfg)
    assert ws1.numel() > ws0.numel()
    a, b = host(run_forward(plain_cfg, inp, ws0)), host(run_forward(keep_cfg, inp, ws1))
    for k in a:
        assert np.array_equal(a[k], b[k]), k
    assert moe.moe_check_error(ws1) == moe.MOE_OK
    # pre-activations of a sample of kept rows against the oracle's products on that token
    oi = oracle_inputs(inp)
    sep = host(run_separate(plain_cfg, inp, moe.workspace(plain_cfg)))
    offs, perm = sep["expert_offsets"], sep["perm_token"]
    gated = w.act == "silu_gated"
    width = 2 * w.h if gated else w.h
    rmax = moe.moe_max_rows(keep_cfg)
    pre = moe.preact_view(keep_cfg, ws1)
    assert tuple(pre.shape) == (rmax, width)
    rng = np.random.default_rng(0)
    for e in range(w.N):
        lo, hi = int(offs[e]), int(offs[e + 1])
        for r in sorted(set(rng.integers(lo, hi, size=min(4, hi - lo)).tolist())) if hi > lo else []:
            xt = oi["x"][int(perm[r])].astype(np.float64)
            want = xt @ oi["w_gate"][e].astype(np.float64).T
            if gated:
                want = np.concatenate([want, xt @ oi["w_up"][e].astype(np.float64).T])
            check_output(pre[r].float().cpu().numpy(), want, "bf16")
    if w.h_shared:
        pre_sh = moe.preact_view(keep_cfg, ws1, shared=True)
        xs = oi["x"].astype(np.float64)
        want = np.concatenate([xs @ oi["shared_w_gate"].astype(np.float64).T,
                               xs @ oi["shared_w_up"].astype(np.float64).T], axis=1)
        check_output(pre_sh.float().cpu().numpy(), want, "bf16")


def test_dispatch_rejects_out_of_range_token():
    """A perm_token entry outside [0, T) is skipped and reported, never followed."""
    w = _small("mixtral_prefill", T=64, d=128, h=128)
    cfg = cfg_of(w)
    ws = moe.workspace(cfg)
    x = torch.randn((64, 128), device="cuda").to(torch.bfloat16)
    rmax = moe.moe_max_rows(cfg)
    perm = torch.arange(rmax, dtype=torch.int32, device="cuda") % 64
    perm[5] = 64
    perm[9] = -3
    off = torch.tensor([0] * 8 + [rmax], dtype=torch.int32, device="cuda")
    x_perm = torch.zeros((rmax + 1, 128), dtype=torch.bfloat16, device="cuda")
    moe.moe_dispatch(cfg, x, perm, off, x_perm, ws)
    assert moe.moe_check_error(ws) == moe.MOE_ERR_DEVICE_FAULT
    assert moe.moe_check_error(ws) == moe.MOE_OK          # the word was cleared
    xp = x_perm.float().cpu()
    xs = x.float().cpu()
    assert torch.equal(xp[0], xs[0]) and torch.equal(xp[6], xs[6])
    assert torch.all(xp[5] == 0) and torch.all(xp[9] == 0) and torch.all(xp[rmax] == 0)


# ------------------------------------------------------------ full-size workloads

FULL = [("switch_top1", None), ("mixtral_decode_16", None), ("mixtral_decode_64", None),
        ("mixtral_decode_128", 24), ("mixtral_prefill", 16), ("deepseek_fine", 8)]


def _expert_block_rows(offsets, rng):
    """Dispatched rows to check: one random row of every 128-row block of every
    expert (the tiles of both tensor-core kernels: 256-row pair tiles and 128-row
    single-CTA tiles) and every expert's last row (its last, partial block)."""
    rows = []
    for e in range(len(offsets) - 1):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        for b0 in range(lo, hi, 128):
            rows.append(int(rng.integers(b0, min(b0 + 128, hi))))
        if hi > lo:
            rows.append(hi - 1)
    return np.array(sorted(set(rows)), dtype=np.int64)


def check_expert_rows(w, inp, sep, rng):
    """Expert outputs y_perm of sampled rows of every expert against the oracle's
    FFN_e of the row's token (the DeepSeekMoE layer equation's FFN_i for every expert
    with a non-zero gate), element by element at the layer tolerance."""
    oi = oracle_inputs(inp)
    off, perm = sep["expert_offsets"], sep["perm_token"]
    rows = _expert_block_rows(off, rng)
    got, ref = [], []
    for e in range(w.N):
        r = rows[(rows >= off[e]) & (rows < off[e + 1])]
        if r.size == 0:
            continue
        xr = oi["x"][perm[r]]
        ref.append(O.expert_ffn(xr, oi["w_gate"][e], None if oi["w_up"] is None else oi["w_up"][e],
                                oi["w_down"][e], w.act))
        got.append(sep["y_perm"][r])
    experts_hit = int(np.count_nonzero(np.diff(off)))
    assert len(ref) == experts_hit
    check_output(np.concatenate(got), np.concatenate(ref), w.dtype)
    return rows.size, experts_hit


@pytest.mark.parametrize("name,sample", FULL, ids=[n for n, _ in FULL])
def test_full_size_parity(name, sample):
    """Full-size layer as the benchmark runs it (moe_forward, one call): routing,
    counts and aux bit-exact / toleranced over all tokens; layer outputs on a token
    sample; expert outputs of every expert on rows drawn from each of its blocks."""
    w = W.WORKLOADS[name]
    inp = W.make_inputs(w, device="cuda")
    cfg = cfg_of(w)
    ws = moe.workspace(cfg)
    fwd = host(run_forward(cfg, inp, ws))
    sep = host(run_separate(cfg, inp, ws))
    assert moe.moe_check_error(ws) == moe.MOE_OK
    rng = np.random.default_rng(1234)
    tokens = None if sample is None else np.sort(rng.choice(w.T, size=sample, replace=False))
    rt = O.forward(w, oracle_inputs(inp), tokens=tokens)
    check_routing(sep, rt, sep=True)
    check_routing(fwd, rt, sep=False)
    ysel = fwd["y"] if tokens is None else fwd["y"][tokens]
    check_output(ysel, rt["y"], w.dtype)
    assert np.array_equal(fwd["y"], sep["y"])
    check_expert_rows(w, inp, sep, rng)


# One expert takes every token, so its row count is T: the pair kernel's last block
# holds T mod 256 rows, handled as a tile with the tokens on the MMA's N side (1, 32,
# 33, 49, 128, 129, 255 rows), or none (T = 768); below 512 rows the experts with a
# short last block move to the single-CTA kernel (T = 300, 304, 305) and the others
# keep the pair kernel's tail tile (T = 400). Gated, ReLU and shared-expert variants.
TAILS = [_small("mixtral_prefill", T=t, d=128, h=256, N=1, k=1) for t in (513, 544, 545, 561, 640, 641, 767, 768,
                                                                          300, 304, 305, 400)]
TAILS += [_small("switch_top1", T=t, d=128, h=384, N=1, k=1, capacity_factor=None) for t in (545, 767)]
TAILS += [_small("deepseek_fine", T=t, d=128, N=1, k=1, h=128, h_shared=128) for t in (545, 767)]
# About 272 rows per expert (most experts just over one 256-row block, as in the
# DeepSeekMoE-shaped layer): both launches of the split, several tiles per CTA pair.
TAILS += [_small("deepseek_fine", T=4352, d=128, N=32, k=2, h=1024, h_shared=0),
          _small("switch_top1", T=2176, d=128, h=2048, N=8, k=1, capacity_factor=None)]


@pytest.mark.parametrize("w", TAILS, ids=[w.name for w in TAILS])
def test_pair_kernel_tail_tiles(w):
    inp = W.make_inputs(w, device="cuda")
    ws = moe.workspace(cfg_of(w))
    rt = O.forward(w, oracle_inputs(inp))
    out = host(run_forward(cfg_of(w, debug_flags=moe.MOE_DEBUG_FFN_PAIR), inp, ws))
    assert moe.moe_check_error(ws) == moe.MOE_OK
    check_routing(out, rt, sep=False)
    check_output(out["y"], rt["y"], w.dtype)


# The largest batch the library accepts (T = 65536) with the most experts and slots
# (N = 256, top-8, a capacity that drops slots) and with the N <= 32 router: routing,
# counts, dispatch order and drop set bit-exact for all tokens, outputs on a sample.
MAXIMAL = [
    _small("deepseek_fine", T=65536, d=128, N=256, k=8, h=128, h_shared=0, capacity_factor=(1, 1)),
    _small("mixtral_prefill", T=65536, d=256, N=32, k=8, h=128),
]


@pytest.mark.parametrize("w", MAXIMAL, ids=[w.name for w in MAXIMAL])
def test_maximum_batch(w):
    inp = W.make_inputs(w, device="cuda")
    cfg = cfg_of(w)
    ws = moe.workspace(cfg)
    fwd = host(run_forward(cfg, inp, ws))
    sep = host(run_separate(cfg, inp, ws))
    assert moe.moe_check_error(ws) == moe.MOE_OK
    tokens = np.sort(np.random.default_rng(99).choice(w.T, size=24, replace=False))
    rt = O.forward(w, oracle_inputs(inp), tokens=tokens)
    check_routing(sep, rt, sep=True)
    check_routing(fwd, rt, sep=False)
    check_output(fwd["y"][tokens], rt["y"], w.dtype)
    if w.capacity_factor:
        assert int(rt["counts_kept"].sum()) < w.T * w.k  # the capacity dropped slots


# The smallest shapes the tensor-core path takes: d = h = 64 (one 64-wide k-block per
# tile, output narrower than one 128- or 256-column tile), with and without a shared
# expert, on the pair kernel (forced) and the single-CTA kernel.
TINY_TC = [
    _small("mixtral_prefill", T=70, d=64, h=64, N=4, k=2),
    _small("deepseek_fine", T=300, d=64, N=4, k=2, h=64, h_shared=64),
    _small("switch_top1", T=600, d=64, h=64, N=2, k=1),
]


@pytest.mark.parametrize("w", TINY_TC, ids=[w.name for w in TINY_TC])
@pytest.mark.parametrize("flags", [0, 2, 4], ids=["auto", "pair", "single"])
def test_smallest_tensor_core_shapes(w, flags):
    inp = W.make_inputs(w, device="cuda")
    ws = moe.workspace(cfg_of(w))
    rt = O.forward(w, oracle_inputs(inp))
    out = host(run_forward(cfg_of(w, debug_flags=flags), inp, ws))
    assert moe.moe_check_error(ws) == moe.MOE_OK
    check_routing(out, rt, sep=False)
    check_output(out["y"], rt["y"], w.dtype)
