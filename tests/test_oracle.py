"""Pins for the CPU oracle: each checks it against something other than itself.

The pins are the pages' worked examples (fixtures under tests/golden/), closed
forms, invariants, textbook/library routines on special cases and brute force on
tiny inputs. The last group plants plausible mistakes in the oracle and checks
that some pin catches each of them.
"""
import math
import os
import random
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch

from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_fixture(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


def _kv(rows):
    out = {}
    for r in rows:
        out.setdefault(r[0], []).append(r[1:])
    return out


# ----------------------------------------------------------------- exact arithmetic

def _round_f32(v: Fraction) -> float:
    """Round a rational to the nearest binary32 value, ties to even (IEEE 754)."""
    if v == 0:
        return 0.0
    s = -1 if v < 0 else 1
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    ulp = Fraction(2) ** (max(e, -126) - 23)
    q = a / ulp
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    return float(np.float32(s * n * ulp))


def _fma_f32(a, b, c):
    return _round_f32(Fraction(float(a)) * Fraction(float(b)) + Fraction(float(c)))


def _logit_exact(xrow, wcol, b=None):
    """The specified fp32 order, evaluated with exact rationals and IEEE
    round-to-nearest-even at every step: 32 partials over 8-feature blocks
    (block b -> partial b mod 32, features in increasing order, one fma each),
    five pairwise rounds p_l <- p_l + p_(l^o) for o = 16, 8, 4, 2, 1, take p_0,
    then add the bias."""
    part = [0.0] * 32
    for i in range(len(xrow)):
        lane = (i // 8) % 32
        part[lane] = _fma_f32(xrow[i], wcol[i], part[lane])
    for o in (16, 8, 4, 2, 1):
        part = [_round_f32(Fraction(part[lane]) + Fraction(part[lane ^ o])) for lane in range(32)]
    acc = part[0]
    if b is not None:
        acc = _round_f32(Fraction(acc) + Fraction(float(b)))
    return np.float32(acc)


def pin_router_logits_exact(O):
    """Each logit equals the specified fp32 summation, re-evaluated exactly: 8-feature
    blocks dealt round-robin to 32 fma partials, a five-round pairwise combine, bias."""
    rng = np.random.default_rng(7)
    T, d, N = 2, 8 * 32 * 2 + 24, 3          # two full passes over the 32 partials + a tail
    x = rng.standard_normal((T, d)).astype(np.float32) * np.float32(3.0)
    w = rng.standard_normal((d, N)).astype(np.float32)
    b = rng.standard_normal(N).astype(np.float32)
    L = O.router_logits(x, w, b)
    for t in range(T):
        for e in range(N):
            want = _logit_exact(x[t], w[:, e], b[e])
            assert L[t, e] == want, (t, e, L[t, e], want)
    # short inputs leave most partials at zero
    x2 = rng.standard_normal((3, 24)).astype(np.float32)
    w2 = rng.standard_normal((24, 4)).astype(np.float32)
    L2 = O.router_logits(x2, w2)
    for t in range(3):
        for e in range(4):
            assert L2[t, e] == _logit_exact(x2[t], w2[:, e])


def pin_router_logits_error_bound(O):
    """|fp32 logit - exact dot| <= gamma_d * sum |x_i w_i| (+ one rounding for b)."""
    rng = np.random.default_rng(11)
    for (T, d, N) in [(5, 64, 4), (3, 768, 8), (2, 1000, 7)]:
        x = rng.standard_normal((T, d)).astype(np.float32)
        w = (rng.standard_normal((d, N)) / math.sqrt(d)).astype(np.float32)
        L = O.router_logits(x, w)
        exact = x.astype(np.float64) @ w.astype(np.float64)
        mag = np.abs(x.astype(np.float64)) @ np.abs(w.astype(np.float64))
        u = 2.0 ** -24
        gamma = d * u / (1 - d * u)
        assert np.all(np.abs(L - exact) <= gamma * mag + 1e-30)


def pin_topk_brute_force(O):
    """Top-k equals a brute-force ordering by (value descending, index ascending),
    including exact ties and signed zeros."""
    rng = random.Random(3)
    for _ in range(200):
        N = rng.randint(1, 12)
        k = rng.randint(1, N)
        vals = [rng.choice([-2.0, -1.0, -0.0, 0.0, 0.5, 1.0, 3.0]) for _ in range(N)]
        L = np.array([vals], dtype=np.float32)
        want = sorted(range(N), key=lambda e: (-vals[e], e))[:k]
        got = O.select_topk(L, k)[0].tolist()
        assert got == want, (vals, k, got, want)


def pin_worked_example(O):
    """Fixture: the pages' d=8, four-expert, top-2 router example."""
    kv = _kv(_read_fixture("router_worked_example.txt"))
    d, N, k = int(kv["d"][0][0]), int(kv["N"][0][0]), int(kv["k"][0][0])
    scores = [float(v) for v in kv["scores"][0]]
    sel = [int(v) - 1 for v in kv["selected"][0]]
    wts = [float(v) for v in kv["weights"][0]]
    tol = float(kv["tolerance"][0][0])
    x = np.zeros((1, d), np.float32)
    x[0, 0] = 1.0                                 # x = e_1, so the scores are W_r row 0
    w_r = np.zeros((d, N), np.float32)
    w_r[0] = scores
    L = O.router_logits(x, w_r)
    assert L[0].tolist() == scores
    idx = O.select_topk(L, k)
    assert idx[0].tolist() == sel
    g = O.gates(L, idx, O.GATING_TOPK_THEN_SOFTMAX)
    assert np.allclose(g[0], wts, atol=tol)
    # closed form: e^2 / (e^1 + e^2) = 1 / (1 + e^-1)
    assert abs(g[0, 0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-12
    assert abs(g[0, 1] - 1.0 / (1.0 + math.exp(1.0))) < 1e-12
    assert abs(g[0].sum() - 1.0) < 1e-12


def _three_token_setup():
    kv = _kv(_read_fixture("dispatch_three_tokens.txt"))
    T, d, N, k = (int(kv[n][0][0]) for n in ("tokens", "d", "N", "k"))
    w = {(int(a), int(b)): float(c) for a, b, c in kv["weight"]}
    # Scores chosen so that each token's top-2 and softmax weights are the page's:
    # a gap ln(w / (1 - w)) between the two selected experts, others far below.
    scores = np.full((T, N), -8.0)
    scores[0, 0], scores[0, 2] = 0.0, math.log(w[(1, 3)] / w[(1, 1)])
    scores[1, 1], scores[1, 2] = 0.0, 0.25
    scores[2, 0], scores[2, 2] = math.log(w[(3, 1)] / (1 - w[(3, 1)])), 0.0
    x = np.zeros((T, d), np.float32)
    w_r = np.zeros((d, N), np.float32)
    for t in range(T):
        x[t, t] = 1.0
        w_r[t] = scores[t].astype(np.float32)
    return kv, T, d, N, k, w, x, w_r


def pin_three_token_dispatch(O):
    """Fixture: the pages' three-token Router -> Dispatch -> Combine example."""
    kv, T, d, N, k, w, x, w_r = _three_token_setup()
    cfg = O.config_from(T=T, d=d, N=N, k=k, h=8)
    rt = O.route(cfg, x, w_r)
    for tok, a, b in kv["select"]:
        assert sorted((rt["topk_idx"][int(tok) - 1] + 1).tolist()) == [int(a), int(b)]
    tol = float(kv["tolerance"][0][0])
    for (tok, e), val in w.items():
        j = rt["topk_idx"][tok - 1].tolist().index(e - 1)
        assert abs(rt["topk_gate"][tok - 1, j] - val) <= tol
    groups = {int(g[0]): [int(v) - 1 for v in g[1:]] for g in kv["group"]}
    counts = [len(groups[e + 1]) for e in range(N)]
    assert rt["counts_kept"].tolist() == counts == [2, 1, 3, 0]
    assert rt["expert_offsets"].tolist() == [0, 2, 3, 6, 6]
    perm = sum((groups[e + 1] for e in range(N)), [])
    assert rt["perm_token"].tolist() == perm == [0, 2, 1, 0, 1, 2]
    # every slot points at a row holding its own token
    for t in range(T):
        for j in range(k):
            assert rt["perm_token"][rt["slot_row"][t, j]] == t


def pin_softmax_library(O):
    """Full softmax equals scipy's softmax; softmax-then-top-k gates are p at the
    selected experts, sum to <= 1, and to 1 when k = N."""
    rng = np.random.default_rng(5)
    L = rng.standard_normal((50, 9)).astype(np.float32) * 4
    p = O.softmax_all(L)
    assert np.allclose(p, scipy.special.softmax(L.astype(np.float64), axis=1), rtol=1e-13, atol=0)
    for k in (1, 3, 9):
        idx = O.select_topk(L, k)
        g = O.gates(L, idx, O.GATING_SOFTMAX_THEN_TOPK)
        assert np.all(g.sum(axis=1) <= 1 + 1e-12)
        assert np.allclose(g, scipy.special.softmax(L.astype(np.float64), axis=1)[
            np.arange(50)[:, None], idx], rtol=1e-13)
        if k == 9:
            assert np.allclose(g.sum(axis=1), 1.0, atol=1e-12)
        g2 = O.gates(L, idx, O.GATING_TOPK_THEN_SOFTMAX)
        assert np.allclose(g2.sum(axis=1), 1.0, atol=1e-12)
        # top-k-then-softmax is the full softmax restricted to k and renormalised
        assert np.allclose(g2, g / g.sum(axis=1, keepdims=True), rtol=1e-12)


def pin_aux_closed_forms(O):
    """Aux loss: W_r = 0 gives form0 = 1, form1 = 0; balanced counts give form0 = 1;
    a two-expert hand case gives 1.5 and 0.0625."""
    T, d, N, k = 12, 8, 4, 2
    cfg = O.config_from(T=T, d=d, N=N, k=k, h=8)
    x = np.random.default_rng(0).standard_normal((T, d)).astype(np.float32)
    rt = O.route(cfg, x, np.zeros((d, N), np.float32))
    assert rt["topk_idx"].tolist() == [[0, 1]] * T      # ties -> lowest indices
    a0, a1 = rt["aux"]
    assert a0 == 1.0 and a1 == 0.0
    # balanced: token t picks expert t mod N (k = 1), one-hot inputs
    T2 = 8
    x2 = np.zeros((T2, d), np.float32)
    w2 = np.zeros((d, N), np.float32)
    for t in range(T2):
        x2[t, t] = 1.0
        w2[t, t % N] = 2.0
    rt2 = O.route(O.config_from(T=T2, d=d, N=N, k=1, h=8), x2, w2)
    assert rt2["counts_routed"].tolist() == [2, 2, 2, 2]
    assert abs(rt2["aux"][0] - 1.0) < 1e-12
    # hand case: 2 tokens, 2 experts, logits [ln 3, 0] for both -> p = [.75, .25]
    x3 = np.ones((2, 1), np.float32)
    w3 = np.array([[math.log(3.0), 0.0]], np.float32)
    rt3 = O.route(O.config_from(T=2, d=1, N=2, k=1, h=8), x3, w3)
    assert np.allclose(rt3["p"][:, 0], 0.75, atol=1e-7)
    assert abs(rt3["aux"][0] - 1.5) < 1e-6
    assert abs(rt3["aux"][1] - 0.0625) < 1e-6


def pin_capacity(O):
    """Capacity: C = ceil(T cf / N); kept_e = min(routed_e, C); kept + dropped = T k;
    all-tied routing keeps tokens 0..C-1; slot-major priority for k = 2."""
    assert O.capacity(4096, 8, (5, 4)) == 640
    assert O.capacity(10, 4, (1, 1)) == 3
    assert O.capacity(10, 4, None) is None
    T, d, N = 10, 4, 4
    x = np.random.default_rng(1).standard_normal((T, d)).astype(np.float32)
    cfg = O.config_from(T=T, d=d, N=N, k=1, h=8, capacity_factor=(1, 1))
    rt = O.route(cfg, x, np.zeros((d, N), np.float32))
    assert rt["capacity"] == 3
    assert rt["kept"][:, 0].tolist() == [True] * 3 + [False] * 7
    assert rt["perm_token"].tolist() == [0, 1, 2]
    assert rt["slot_row"][:, 0].tolist() == [0, 1, 2] + [-1] * 7
    rng = np.random.default_rng(2)
    for _ in range(20):
        T, N, k = 40, 5, 2
        L = rng.standard_normal((T, N)).astype(np.float32)
        L[:, 0] += 2.0                                   # overload expert 0
        idx = O.select_topk(L, k)
        C = O.capacity(T, N, (1, 1))
        kept = O.keep_within_capacity(idx, N, C)
        routed = O.counts_routed(idx, N)
        ck, off, perm, sr = O.group_by_expert(idx, kept, N)
        assert ck.tolist() == np.minimum(routed, C).tolist()
        assert int(ck.sum()) + int((~kept).sum()) == T * k
        # slot-major: a dropped first choice implies the expert was already full
        # with first choices of earlier tokens
        for t in range(T):
            if not kept[t, 0]:
                e = idx[t, 0]
                assert int(np.sum(idx[:t, 0] == e)) >= C
            if kept[t, 1]:
                e = idx[t, 1]
                assert int(np.sum(idx[:, 0] == e)) + int(np.sum(idx[:t, 1] == e)) < C


def _rand_layer(rng, T, d, N, k, h, hs=0, act="silu_gated", gating=O.GATING_TOPK_THEN_SOFTMAX,
                cf=None, bias=False):
    cfg = O.config_from(T=T, d=d, N=N, k=k, h=h, h_shared=hs, gating=gating, act=act,
                        capacity_factor=cf)
    inp = dict(x=rng.standard_normal((T, d)).astype(np.float32),
               w_r=(rng.standard_normal((d, N)) / math.sqrt(d)).astype(np.float32),
               b_r=rng.standard_normal(N).astype(np.float32) if bias else None,
               w_gate=rng.standard_normal((N, h, d)) / math.sqrt(d),
               w_up=(rng.standard_normal((N, h, d)) / math.sqrt(d)) if act == "silu_gated" else None,
               w_down=rng.standard_normal((N, d, h)) / math.sqrt(h))
    if hs:
        inp.update(shared_w_gate=rng.standard_normal((hs, d)) / math.sqrt(d),
                   shared_w_up=rng.standard_normal((hs, d)) / math.sqrt(d),
                   shared_w_down=rng.standard_normal((d, hs)) / math.sqrt(hs))
    return cfg, inp


def _torch_mlp(x, wg, wu, wd):
    F = torch.nn.functional
    xt = torch.as_tensor(np.asarray(x, np.float64))
    return F.linear(F.silu(F.linear(xt, torch.as_tensor(wg))) * F.linear(xt, torch.as_tensor(wu)),
                    torch.as_tensor(wd)).numpy()


def pin_single_expert_is_dense_mlp(O):
    """N = 1, k = 1 (top-k then softmax: gate 1) reduces to x + MLP(x), checked
    against torch's own linear/SiLU; ReLU variant against torch's relu; SiLU(1)."""
    rng = np.random.default_rng(4)
    cfg, inp = _rand_layer(rng, T=7, d=16, N=1, k=1, h=24)
    y = O.forward(cfg, inp)["y"]
    ref = inp["x"].astype(np.float64) + _torch_mlp(inp["x"], inp["w_gate"][0], inp["w_up"][0],
                                                   inp["w_down"][0])
    assert np.allclose(y, ref, rtol=1e-12, atol=1e-12)
    cfg, inp = _rand_layer(rng, T=7, d=16, N=1, k=1, h=24, act="relu")
    y = O.forward(cfg, inp)["y"]
    F = torch.nn.functional
    xt = torch.as_tensor(inp["x"].astype(np.float64))
    ref = xt + F.linear(F.relu(F.linear(xt, torch.as_tensor(inp["w_gate"][0]))),
                        torch.as_tensor(inp["w_down"][0]))
    assert np.allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)
    assert abs(O.silu(np.array([1.0]))[0] - 1.0 / (1.0 + math.exp(-1.0))) < 1e-15
    assert O.silu(np.array([0.0]))[0] == 0.0


def pin_identical_experts(O):
    """With identical experts, y = x + (sum of gates) * FFN(x) whatever the routing."""
    rng = np.random.default_rng(6)
    for gating in (O.GATING_TOPK_THEN_SOFTMAX, O.GATING_SOFTMAX_THEN_TOPK):
        cfg, inp = _rand_layer(rng, T=9, d=8, N=5, k=3, h=12, gating=gating)
        for name in ("w_gate", "w_up", "w_down"):
            inp[name] = np.repeat(inp[name][:1], 5, axis=0)
        rt = O.forward(cfg, inp)
        ffn = _torch_mlp(inp["x"], inp["w_gate"][0], inp["w_up"][0], inp["w_down"][0])
        ref = inp["x"].astype(np.float64) + rt["topk_gate"].sum(axis=1, keepdims=True) * ffn
        assert np.allclose(rt["y"], ref, rtol=1e-12, atol=1e-12)


def pin_dense_brute_force(O):
    """Sparse path (dispatch, grouped experts, combine) equals the dense sum of the
    DeepSeekMoE equation with every expert computed and masked."""
    rng = np.random.default_rng(8)
    cases = [dict(T=11, d=8, N=4, k=2, h=6),
             dict(T=13, d=8, N=5, k=3, h=6, gating=O.GATING_SOFTMAX_THEN_TOPK, hs=5),
             dict(T=16, d=8, N=3, k=1, h=4, act="relu", gating=O.GATING_SOFTMAX_THEN_TOPK,
                  cf=(1, 1), bias=True),
             dict(T=17, d=8, N=4, k=2, h=4, cf=(1, 2))]
    for c in cases:
        cfg, inp = _rand_layer(rng, **c)
        y = O.forward(cfg, inp)["y"]
        yd = O.forward_dense(cfg, inp)
        assert np.allclose(y, yd, rtol=1e-12, atol=1e-12)
        sub = [0, 3, cfg.T - 1]                       # the token-sample path agrees too
        assert np.allclose(O.forward(cfg, inp, tokens=sub)["y"], yd[sub], rtol=1e-12, atol=1e-12)


def pin_dropped_tokens_are_residual(O):
    """A token with every slot dropped leaves the layer as exactly x (no shared
    expert) and as x + S(x) with a shared expert."""
    rng = np.random.default_rng(9)
    cfg, inp = _rand_layer(rng, T=12, d=8, N=4, k=1, h=6, cf=(1, 2))
    inp["w_r"] = np.zeros_like(inp["w_r"])            # everyone ties onto expert 0
    rt = O.forward(cfg, inp)
    dropped = ~rt["kept"].any(axis=1)
    assert dropped.sum() == cfg.T - rt["capacity"]
    assert np.array_equal(rt["y"][dropped], inp["x"][dropped].astype(np.float64))
    cfg, inp = _rand_layer(rng, T=12, d=8, N=4, k=1, h=6, cf=(1, 2), hs=7)
    inp["w_r"] = np.zeros_like(inp["w_r"])
    rt = O.forward(cfg, inp)
    dropped = ~rt["kept"].any(axis=1)
    s = _torch_mlp(inp["x"], inp["shared_w_gate"], inp["shared_w_up"], inp["shared_w_down"])
    assert np.allclose(rt["y"][dropped], inp["x"][dropped] + s[dropped], rtol=1e-12, atol=1e-12)


# ------------------------------------------------- training-time router variants

def pin_noisy_logits_exact(O):
    """H = fl(L + fl(w * n)): two correctly rounded fp32 steps, checked in exact
    rational arithmetic; w = 0 and n = 0 leave the logits unchanged."""
    rng = np.random.default_rng(7)
    L = rng.standard_normal((40, 50)).astype(np.float32) * np.float32(3)
    n = rng.standard_normal((40, 50)).astype(np.float32)
    for w in (0.37, 1.0, 2.5e-3, 13.0):
        H = O.noisy_logits(L, n, w)
        w32 = float(np.float32(w))
        for t in range(L.shape[0]):
            for e in range(L.shape[1]):
                prod = _round_f32(Fraction(w32) * Fraction(float(n[t, e])))
                want = _round_f32(Fraction(float(L[t, e])) + Fraction(prod))
                assert float(H[t, e]) == want
    assert np.array_equal(O.noisy_logits(L, n, 0.0), L)
    assert np.array_equal(O.noisy_logits(L, np.zeros_like(n), 5.0), L)


def pin_noisy_selection(O):
    """With a zero router weight every logit is 0, so the noise alone decides:
    the top-k follow the noise in descending order (brute force), and the gates of
    top-k-then-softmax are the softmax of the selected noise values times w."""
    rng = np.random.default_rng(11)
    T, d, N, k = 9, 8, 6, 3
    cfg = O.config_from(T, d, N, k, h=4)
    x = rng.standard_normal((T, d)).astype(np.float32)
    w_r = np.zeros((d, N), np.float32)
    noise = rng.standard_normal((T, N)).astype(np.float32)
    rt = O.route_train(cfg, x, w_r, None, noise, 0.5)
    for t in range(T):
        order = sorted(range(N), key=lambda e: (-float(noise[t, e]), e))[:k]
        assert list(rt["topk_idx"][t]) == order
        v = np.array([0.5 * float(noise[t, e]) for e in order])
        g = np.exp(v - v.max()) / np.exp(v - v.max()).sum()
        assert np.allclose(rt["topk_gate"][t], g, rtol=1e-6, atol=1e-7)


def pin_route_train_without_noise(O):
    """Without noise route_train selects, gates and counts exactly as route."""
    rng = np.random.default_rng(12)
    cfg = O.config_from(37, 16, 5, 2, h=4, capacity_factor=(1, 1))
    x = rng.standard_normal((37, 16)).astype(np.float32)
    w_r = rng.standard_normal((16, 5)).astype(np.float32)
    a = O.route(cfg, x, w_r)
    b = O.route_train(cfg, x, w_r)
    for key in ("topk_idx", "topk_gate", "kept", "perm_token", "slot_row", "expert_offsets"):
        assert np.array_equal(a[key], b[key]), key


def pin_z_loss_closed_forms(O):
    """z = mean_t (log sum_e exp L)^2: zero logits give (ln N)^2; the two-expert
    case [0, ln 3] gives (ln 4)^2; a per-token shift c gives mean((lse0 + c)^2);
    random logits agree with scipy's logsumexp; noise does not enter z."""
    for N in (1, 2, 7, 256):
        assert math.isclose(O.z_loss(np.zeros((5, N), np.float32)), math.log(N) ** 2,
                            rel_tol=1e-14, abs_tol=1e-15)
    assert math.isclose(O.z_loss(np.array([[0.0, math.log(3.0)]])), math.log(4.0) ** 2, rel_tol=1e-14)
    c = np.array([[-2.0], [0.5], [30.0]])
    L = np.zeros((3, 4)) + c
    assert math.isclose(O.z_loss(L), float(np.mean((math.log(4.0) + c[:, 0]) ** 2)), rel_tol=1e-13)
    rng = np.random.default_rng(13)
    L = rng.standard_normal((50, 9)) * 4
    want = float(np.mean(scipy.special.logsumexp(L, axis=1) ** 2))
    assert math.isclose(O.z_loss(L), want, rel_tol=1e-12)
    cfg = O.config_from(20, 8, 5, 2, h=4)
    x = rng.standard_normal((20, 8)).astype(np.float32)
    w_r = rng.standard_normal((8, 5)).astype(np.float32)
    noise = rng.standard_normal((20, 5)).astype(np.float32)
    plain = O.route_train(cfg, x, w_r)
    noisy = O.route_train(cfg, x, w_r, None, noise, 3.0)
    assert noisy["z_loss"] == plain["z_loss"]
    assert math.isclose(plain["z_loss"], float(np.mean(
        scipy.special.logsumexp(plain["raw_logits"].astype(np.float64), axis=1) ** 2)), rel_tol=1e-12)


# ------------------------------------------------------------- Expert Choice routing

def _c_hex_constants():
    import re
    src = open(os.path.join(os.path.dirname(O.__file__), "expert_choice.c")).read()
    return {m.group(1): float.fromhex(m.group(2))
            for m in re.finditer(r"static const float (\w+) = (0x[0-9a-fp.+-]+)f;", src)}


def pin_ec_exp(O):
    """The scores' exponential: within 1 ulp of e^x on [-87, 0], exactly 1 at 0,
    monotone; its constants are ln 2 split as Cody and Waite prescribe (high part of
    16 significant bits, low part the fp32 remainder), log2(e) and 1/k! in fp32."""
    from decimal import Decimal, getcontext
    getcontext().prec = 50
    ln2 = Decimal(2).ln()
    c = _c_hex_constants()
    hi = c["LN2_HI"]
    m, e = math.frexp(hi)
    assert m * 2 ** 16 == int(m * 2 ** 16)                      # 16 significant bits
    assert abs(Decimal(hi) - ln2) < Decimal(2) ** -16
    assert c["LN2_LO"] == float(np.float32(float(ln2 - Decimal(hi))))
    assert c["LOG2E"] == float(np.float32(float(1 / ln2)))
    for k in range(2, 8):
        assert c[f"C{k}"] == float(np.float32(1.0 / math.factorial(k)))
    x = np.linspace(-87.0, 0.0, 400001).astype(np.float32)
    y = O.ec_exp(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    assert np.max(np.abs(y - ref) / ulp) <= 1.0
    assert float(O.ec_exp(np.zeros(1, np.float32))[0]) == 1.0
    assert np.all(np.diff(y) >= 0)
    assert float(O.ec_exp(np.array([-88.0, -1e30], np.float32)).max()) == 0.0


def pin_ec_scores(O):
    """Scores are the softmax over experts: within 4e-7 of the float64 softmax, sum
    to 1; equal logits give 1/N exactly for N a power of two; logits [0, ln 3] give
    [1/4, 3/4]."""
    rng = np.random.default_rng(21)
    L = (rng.standard_normal((60, 13)) * 3).astype(np.float32)
    S = O.ec_scores(L).astype(np.float64)
    ref = scipy.special.softmax(L.astype(np.float64), axis=1)
    assert np.max(np.abs(S - ref)) <= 4e-7
    assert np.max(np.abs(S.sum(axis=1) - 1.0)) <= 2e-6
    for N in (1, 2, 8, 256):
        assert np.all(O.ec_scores(np.full((3, N), 0.37, np.float32)) == np.float32(1.0 / N))
    S2 = O.ec_scores(np.array([[0.0, math.log(3.0)]], np.float32))[0]
    assert abs(float(S2[0]) - 0.25) <= 1e-7 and abs(float(S2[1]) - 0.75) <= 1e-7


def pin_ec_selection_brute_force(O):
    """Each expert keeps the min(C, T) tokens of largest score, lower index first on
    ties, listed in token order; all-equal scores keep tokens 0 .. C-1."""
    rng = np.random.default_rng(22)
    for T, N, C in ((9, 3, 4), (20, 5, 7), (6, 4, 10), (31, 8, 8)):
        L = rng.integers(-3, 4, size=(T, N)).astype(np.float32)     # many ties
        S = O.ec_scores(L)
        chosen = O.expert_choice_select(S, C)
        for e in range(N):
            want = sorted(sorted(range(T), key=lambda t: (-float(S[t, e]), t))[:min(C, T)])
            assert chosen[e].tolist() == want
    S = O.ec_scores(np.zeros((10, 4), np.float32))
    assert all(O.expert_choice_select(S, 3)[e].tolist() == [0, 1, 2] for e in range(4))


def pin_ec_dispatch_and_balance(O):
    """Every expert owns exactly Ce = min(C, T) rows holding its tokens ascending;
    the per-token row lists cover every row once, in expert order; row gates are the
    chosen scores."""
    rng = np.random.default_rng(23)
    T, d, N = 50, 8, 6
    cfg = O.config_from(T, d, N, 1, h=4, capacity_factor=(2, 1))
    x = rng.standard_normal((T, d)).astype(np.float32)
    w_r = rng.standard_normal((d, N)).astype(np.float32)
    rt = O.route_expert_choice(cfg, x, w_r)
    Ce = min(O.capacity(T, N, (2, 1)), T)
    assert rt["capacity"] == math.ceil(T * 2 / N) and rt["expert_offsets"].tolist() == [e * Ce for e in range(N + 1)]
    rows = []
    for t in range(T):
        rs = rt["token_rows"][rt["token_ptr"][t]:rt["token_ptr"][t + 1]].tolist()
        assert rs == sorted(rs) and all(rt["perm_token"][r] == t for r in rs)
        rows += rs
    assert sorted(rows) == list(range(N * Ce))
    for e in range(N):
        seg = rt["perm_token"][e * Ce:(e + 1) * Ce]
        assert np.all(np.diff(seg) > 0)
        assert np.array_equal(rt["row_gate"][e * Ce:(e + 1) * Ce], rt["scores"][seg, e])


def pin_ec_dense_brute_force(O):
    """y = x + S(x) + sum_e G[t, e] FFN_e(x) with G the dense score matrix masked to
    the chosen (token, expert) pairs, every expert computed on every token; a token
    no expert chose is exactly its residual (no shared expert)."""
    rng = np.random.default_rng(24)
    for hs in (0, 5):
        cfg, inp = _rand_layer(rng, T=14, d=8, N=4, k=1, h=6, hs=hs, cf=(1, 2))
        rt = O.forward_expert_choice(cfg, inp)
        # selection and gates from the float64 softmax of the logits, brute force
        P = scipy.special.softmax(O.router_logits(inp["x"], inp["w_r"]).astype(np.float64), axis=1)
        C = min(O.capacity(cfg.T, cfg.N, (1, 2)), cfg.T)
        G = np.zeros((cfg.T, cfg.N))
        for e in range(cfg.N):
            top = sorted(range(cfg.T), key=lambda t: (-P[t, e], t))[:C]
            G[top, e] = P[top, e]
        x = inp["x"].astype(np.float64)
        y = x.copy()
        for e in range(cfg.N):
            y += G[:, e:e + 1] * _torch_mlp(inp["x"], inp["w_gate"][e], inp["w_up"][e], inp["w_down"][e])
        if hs:
            y += _torch_mlp(inp["x"], inp["shared_w_gate"], inp["shared_w_up"], inp["shared_w_down"])
        assert np.allclose(rt["y"], y, rtol=1e-6, atol=1e-6)
        unchosen = ~np.isin(np.arange(cfg.T), rt["chosen"])
        assert unchosen.any()
        if not hs:
            assert np.array_equal(rt["y"][unchosen], x[unchosen])


# ------------------------------------------------------------------------- backward

def _torch_loss(cfg, inp, rt, dy, aux_coef, z_coef):
    """The layer's loss in torch float64 with the routing of `rt` held fixed; the
    logits take the oracle's fp32 values with the gradient of x W_r + b."""
    T, N, k = cfg.T, cfg.N, cfg.k
    t64 = lambda a: torch.tensor(np.asarray(a, np.float64), requires_grad=True)  # noqa: E731
    x, w_r = t64(inp["x"]), t64(inp["w_r"])
    b = t64(inp["b_r"]) if inp.get("b_r") is not None else None
    lin = x @ w_r + (b if b is not None else 0.0)
    L = torch.tensor(rt["logits"].astype(np.float64)) + (lin - lin.detach())
    p = torch.softmax(L, dim=1)
    idx = torch.tensor(rt["topk_idx"], dtype=torch.long)
    if cfg.gating == O.GATING_TOPK_THEN_SOFTMAX:
        g = torch.softmax(torch.gather(L, 1, idx), dim=1)
    else:
        g = torch.gather(p, 1, idx)
    W = {n: [t64(inp[n][e]) for e in range(N)] if inp.get(n) is not None else None
         for n in ("w_gate", "w_up", "w_down")}
    y = x.clone()
    for t in range(T):
        for j in range(k):
            if rt["kept"][t, j]:
                e = int(idx[t, j])
                a = W["w_gate"][e] @ x[t]
                hdn = torch.nn.functional.silu(a) * (W["w_up"][e] @ x[t]) if cfg.act == "silu_gated" else torch.relu(a)
                y[t] = y[t] + g[t, j] * (W["w_down"][e] @ hdn)
    sh = None
    if cfg.h_shared:
        sh = [t64(inp[n]) for n in ("shared_w_gate", "shared_w_up", "shared_w_down")]
        y = y + (torch.nn.functional.silu(x @ sh[0].T) * (x @ sh[1].T)) @ sh[2].T
    loss = torch.sum(torch.tensor(np.asarray(dy, np.float64)) * y)
    if aux_coef:
        f = torch.tensor(rt["counts_routed"], dtype=torch.float64) / (T * k)
        loss = loss + aux_coef * N * torch.sum(f * p.mean(dim=0))
    if z_coef:
        loss = loss + z_coef * torch.mean(torch.logsumexp(L, dim=1) ** 2)
    loss.backward()
    return x, w_r, b, W, sh


def pin_backward_autograd(O):
    """Every gradient equals torch autograd of the same loss (routing held fixed):
    both gating conventions, SiLU-gated and ReLU experts, a shared expert, router
    bias, capacity drops, the aux and z terms."""
    rng = np.random.default_rng(31)
    for kw in (dict(gating=O.GATING_TOPK_THEN_SOFTMAX, hs=5, bias=False, cf=None),
               dict(gating=O.GATING_SOFTMAX_THEN_TOPK, hs=0, bias=True, cf=(1, 1)),
               dict(gating=O.GATING_SOFTMAX_THEN_TOPK, hs=6, bias=False, cf=None, act="relu")):
        act = kw.pop("act", "silu_gated")
        cfg, inp = _rand_layer(rng, T=11, d=6, N=4, k=2, h=5, act=act, **kw)
        dy = rng.standard_normal((cfg.T, cfg.d))
        gb = O.backward(cfg, inp, dy, aux_coef=0.3, z_coef=0.05)
        x, w_r, b, W, sh = _torch_loss(cfg, inp, gb["route"], dy, 0.3, 0.05)
        close = lambda a, ref: np.allclose(a, ref.grad.numpy(), rtol=1e-9, atol=1e-11)  # noqa: E731
        assert close(gb["dx"], x) and close(gb["dw_r"], w_r)
        if b is not None:
            assert close(gb["db_r"], b)
        for e in range(cfg.N):
            for n, key in (("w_gate", "dw_gate"), ("w_up", "dw_up"), ("w_down", "dw_down")):
                if W[n] is None:
                    continue
                want = W[n][e].grad
                got = gb[key][e]
                if want is None:
                    assert got is None
                else:
                    assert got is not None and np.allclose(got, want.numpy(), rtol=1e-9, atol=1e-11)
        if sh is not None:
            for tsr, key in zip(sh, ("dw_gate", "dw_up", "dw_down")):
                assert np.allclose(gb["shared"][key], tsr.grad.numpy(), rtol=1e-9, atol=1e-11)


def pin_backward_finite_differences(O):
    """Central differences of the loss in float64 along expert and shared-expert
    weight coordinates (the routing does not move with them)."""
    rng = np.random.default_rng(32)
    cfg, inp = _rand_layer(rng, T=9, d=5, N=3, k=2, h=4, hs=3)
    dy = rng.standard_normal((cfg.T, cfg.d))
    gb = O.backward(cfg, inp, dy)

    def loss():
        return float(np.sum(dy * O.forward(cfg, inp)["y"]))
    eps = 1e-6
    for name, key, e in (("w_gate", "dw_gate", 0), ("w_up", "dw_up", 1), ("w_down", "dw_down", 2),
                         ("shared_w_gate", None, None), ("shared_w_down", None, None)):
        for _ in range(3):
            tgt = inp[name][e] if e is not None else inp[name]
            i, j = rng.integers(tgt.shape[0]), rng.integers(tgt.shape[1])
            keep = tgt[i, j]
            tgt[i, j] = keep + eps
            lp = loss()
            tgt[i, j] = keep - eps
            lm = loss()
            tgt[i, j] = keep
            fd = (lp - lm) / (2 * eps)
            an = (gb[key][e] if e is not None else gb["shared"][name.replace("shared_", "d")])[i, j]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an))


def pin_backward_special_cases(O):
    """dy = 0 without aux or z: every gradient is zero. One expert with top-1 and
    top-k-then-softmax: the gate is 1, so the router gets no gradient and dx is
    dy plus the dense MLP's input gradient (torch autograd)."""
    rng = np.random.default_rng(33)
    cfg, inp = _rand_layer(rng, T=7, d=6, N=3, k=2, h=4, hs=2)
    gb = O.backward(cfg, inp, np.zeros((cfg.T, cfg.d)))
    assert not np.any(gb["dx"]) and not np.any(gb["dw_r"])
    assert all(w is None or not np.any(w) for w in gb["dw_gate"] + gb["dw_down"])
    cfg, inp = _rand_layer(rng, T=8, d=6, N=1, k=1, h=5)
    dy = rng.standard_normal((cfg.T, cfg.d))
    gb = O.backward(cfg, inp, dy)
    assert np.allclose(gb["dlogits"], 0.0, atol=1e-15) and np.allclose(gb["dw_r"], 0.0, atol=1e-14)
    x = torch.tensor(inp["x"].astype(np.float64), requires_grad=True)
    wg, wu, wd = (torch.tensor(np.asarray(inp[n][0], np.float64)) for n in ("w_gate", "w_up", "w_down"))
    y = x + (torch.nn.functional.silu(x @ wg.T) * (x @ wu.T)) @ wd.T
    torch.sum(torch.tensor(dy) * y).backward()
    assert np.allclose(gb["dx"], x.grad.numpy(), rtol=1e-10, atol=1e-12)


PINS = [pin_router_logits_exact, pin_router_logits_error_bound, pin_topk_brute_force,
        pin_worked_example, pin_three_token_dispatch, pin_softmax_library, pin_aux_closed_forms,
        pin_capacity, pin_single_expert_is_dense_mlp, pin_identical_experts,
        pin_dense_brute_force, pin_dropped_tokens_are_residual, pin_noisy_logits_exact,
        pin_noisy_selection, pin_route_train_without_noise, pin_z_loss_closed_forms, pin_ec_exp,
        pin_ec_scores, pin_ec_selection_brute_force, pin_ec_dispatch_and_balance,
        pin_ec_dense_brute_force, pin_backward_autograd, pin_backward_finite_differences,
        pin_backward_special_cases]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(O)


# ----------------------------------------------------------- planted mistakes

def _mut_tie_high_index(mp):
    mp.setattr(O, "select_topk", lambda L, k: (L.shape[1] - 1 - np.argsort(
        -L[:, ::-1], axis=1, kind="stable"))[:, :k])


def _mut_swap_gating(mp):
    real = O.gates
    mp.setattr(O, "gates", lambda L, idx, g: real(
        L, idx, O.GATING_SOFTMAX_THEN_TOPK if g == O.GATING_TOPK_THEN_SOFTMAX
        else O.GATING_TOPK_THEN_SOFTMAX))


def _mut_token_major_rows(mp):
    def grp(idx, kept, N):
        ck, off, perm, sr = real(idx, kept, N)
        order = np.argsort(perm, kind="stable")       # rows by token instead of expert
        inv = np.empty_like(order)
        inv[order] = np.arange(len(order))
        sr2 = np.where(sr >= 0, inv[np.maximum(sr, 0)], -1)
        return ck, off, perm[order], sr2
    real = O.group_by_expert
    mp.setattr(O, "group_by_expert", grp)


def _mut_no_residual(mp):
    real = O.layer_output

    def lo(cfg, x, rt, *a, **kw):
        toks = a[6] if len(a) > 6 else kw.get("tokens")
        xs = np.asarray(x, np.float64)
        return real(cfg, x, rt, *a, **kw) - (xs if toks is None else xs[toks])
    mp.setattr(O, "layer_output", lo)


def _mut_sigmoid_act(mp):
    mp.setattr(O, "silu", lambda z: 1.0 / (1.0 + np.exp(-z)))


def _mut_dropped_term(mp):
    real = O.router_logits
    mp.setattr(O, "router_logits", lambda x, w, b=None: real(
        np.ascontiguousarray(np.asarray(x, np.float32)[:, 1:]),
        np.ascontiguousarray(np.asarray(w, np.float32)[1:]), b))


def _mut_mul_then_add(mp):
    def logits(x, w, b=None):
        x = np.asarray(x, np.float32)
        w = np.asarray(w, np.float32)
        acc = np.zeros((x.shape[0], w.shape[1]), np.float32)
        for i in range(x.shape[1]):
            acc = acc + x[:, i:i + 1] * w[i:i + 1]       # two roundings per term
        return acc if b is None else acc + np.asarray(b, np.float32)
    mp.setattr(O, "router_logits", logits)


def _mut_reverse_order(mp):
    real = O.router_logits
    mp.setattr(O, "router_logits", lambda x, w, b=None: real(
        np.ascontiguousarray(np.asarray(x, np.float32)[:, ::-1]),
        np.ascontiguousarray(np.asarray(w, np.float32)[::-1]), b))


def _mut_sequential_order(mp):
    def logits(x, w, b=None):
        x = np.asarray(x, np.float32)
        w = np.asarray(w, np.float32)
        out = np.zeros((x.shape[0], w.shape[1]), np.float32)
        for t in range(x.shape[0]):
            for e in range(w.shape[1]):
                acc = 0.0
                for i in range(x.shape[1]):
                    acc = _fma_f32(x[t, i], w[i, e], acc)
                if b is not None:
                    acc = _round_f32(Fraction(acc) + Fraction(float(b[e])))
                out[t, e] = acc
        return out
    mp.setattr(O, "router_logits", logits)


def _mut_butterfly_ascending(mp):
    def logits(x, w, b=None):
        x = np.asarray(x, np.float32)
        w = np.asarray(w, np.float32)
        out = np.zeros((x.shape[0], w.shape[1]), np.float32)
        for t in range(x.shape[0]):
            for e in range(w.shape[1]):
                part = [0.0] * 32
                for i in range(x.shape[1]):
                    part[(i // 8) % 32] = _fma_f32(x[t, i], w[i, e], part[(i // 8) % 32])
                for o in (1, 2, 4, 8, 16):
                    part = [_round_f32(Fraction(part[q]) + Fraction(part[q ^ o])) for q in range(32)]
                acc = part[0]
                if b is not None:
                    acc = _round_f32(Fraction(acc) + Fraction(float(b[e])))
                out[t, e] = acc
        return out
    mp.setattr(O, "router_logits", logits)


def _mut_capacity_floor(mp):
    mp.setattr(O, "capacity", lambda T, N, cf: None if cf is None else (T * cf[0]) // (N * cf[1]))


def _mut_renormalise_softmax_gates(mp):
    real = O.gates
    def g(L, idx, gating):
        out = real(L, idx, gating)
        return out / out.sum(axis=1, keepdims=True)
    mp.setattr(O, "gates", g)


def _mut_noise_subtracted(mp):
    real = O.noisy_logits
    mp.setattr(O, "noisy_logits", lambda L, n, w: real(L, -np.asarray(n, np.float32), w))


def _mut_noise_one_rounding(mp):
    mp.setattr(O, "noisy_logits", lambda L, n, w: (np.asarray(L, np.float64) + float(np.float32(w))
                                                   * np.asarray(n, np.float64)).astype(np.float32))


def _mut_z_not_squared(mp):
    def z(L):
        L = np.asarray(L, np.float64)
        m = L.max(axis=1, keepdims=True)
        return float(np.mean(m[:, 0] + np.log(np.exp(L - m).sum(axis=1))))
    mp.setattr(O, "z_loss", z)


def _mut_z_on_noisy_logits(mp):
    def rt(cfg, x, w_r, b_r=None, noise=None, noise_weight=0.0):
        L = O.router_logits(x, w_r, b_r)
        H = L if noise is None else O.noisy_logits(L, noise, noise_weight)
        out = O.route_from_logits(cfg, H)
        out["raw_logits"] = L
        out["z_loss"] = O.z_loss(H)
        return out
    mp.setattr(O, "route_train", rt)


def _mut_ec_tie_high_index(mp):
    def sel(S, C):
        T, N = S.shape
        Ce = min(C, T)
        return np.stack([np.sort(np.lexsort((-np.arange(T), -S[:, e].astype(np.float64)))[:Ce])
                         for e in range(N)])
    mp.setattr(O, "expert_choice_select", sel)


def _mut_ec_select_by_logits(mp):
    real = O.route_expert_choice

    def route(cfg, x, w_r, b_r=None):
        L = O.router_logits(x, w_r, b_r)
        mp.setattr(O, "ec_scores", lambda _L: L)       # selection and gates on logits
        return real(cfg, x, w_r, b_r)
    mp.setattr(O, "route_expert_choice", route)


def _mut_ec_rows_by_score(mp):
    def sel(S, C):
        T, N = S.shape
        Ce = min(C, T)
        return np.stack([np.lexsort((np.arange(T), -S[:, e].astype(np.float64)))[:Ce] for e in range(N)])
    mp.setattr(O, "expert_choice_select", sel)


def _mut_ec_exp_short_series(mp):
    mp.setattr(O, "ec_exp", lambda x: (1.0 + np.asarray(x, np.float32) + np.asarray(x, np.float32) ** 2 / 2)
               .astype(np.float32))


def _mut_bwd_sigmoid_for_silu_derivative(mp):
    mp.setattr(O, "_silu_parts", lambda A: (A / (1.0 + np.exp(-A)), 1.0 / (1.0 + np.exp(-A))))


def _mut_bwd_no_residual_gradient(mp):
    real = O.backward

    def bw(cfg, inp, dy, **kw):
        out = real(cfg, inp, dy, **kw)
        out["dx"] = out["dx"] - np.asarray(dy, np.float64)
        return out
    mp.setattr(O, "backward", bw)


def _mut_bwd_down_grad_sign(mp):
    real = O.expert_ffn_backward

    def fb(X, dO, wa, wb, wo, act):
        dX, da, db, do = real(X, dO, wa, wb, wo, act)
        return dX, da, db, -do
    mp.setattr(O, "expert_ffn_backward", fb)


MUTATIONS = [
    (_mut_tie_high_index, pin_topk_brute_force),
    (_mut_swap_gating, pin_worked_example),
    (_mut_token_major_rows, pin_three_token_dispatch),
    (_mut_no_residual, pin_dropped_tokens_are_residual),
    (_mut_sigmoid_act, pin_single_expert_is_dense_mlp),
    (_mut_dropped_term, pin_router_logits_error_bound),
    (_mut_mul_then_add, pin_router_logits_exact),
    (_mut_reverse_order, pin_router_logits_exact),
    (_mut_sequential_order, pin_router_logits_exact),
    (_mut_butterfly_ascending, pin_router_logits_exact),
    (_mut_capacity_floor, pin_capacity),
    (_mut_renormalise_softmax_gates, pin_softmax_library),
    (_mut_noise_subtracted, pin_noisy_selection),
    (_mut_noise_one_rounding, pin_noisy_logits_exact),
    (_mut_z_not_squared, pin_z_loss_closed_forms),
    (_mut_z_on_noisy_logits, pin_z_loss_closed_forms),
    (_mut_ec_tie_high_index, pin_ec_selection_brute_force),
    (_mut_ec_select_by_logits, pin_ec_dense_brute_force),
    (_mut_ec_rows_by_score, pin_ec_dispatch_and_balance),
    (_mut_ec_exp_short_series, pin_ec_exp),
    (_mut_bwd_sigmoid_for_silu_derivative, pin_backward_autograd),
    (_mut_bwd_no_residual_gradient, pin_backward_special_cases),
    (_mut_bwd_down_grad_sign, pin_backward_finite_differences),
]


@pytest.mark.parametrize("mut,pin", MUTATIONS, ids=[m.__name__ for m, _ in MUTATIONS])
def test_planted_mistake_is_caught(mut, pin, monkeypatch):
    with monkeypatch.context() as mp:
        mut(mp)
        with pytest.raises(AssertionError):
            pin(O)
