"""Token-sharded router on the GPU against the oracle run on the whole batch.

The shards of one batch run one after another on one GPU (each with its own
workspace): phase 1 on every shard, the bases of the exchange (sharded.slot_bases,
the rank-order sums), phase 2 on every shard. Together they must reproduce the
oracle's routing of the whole batch: selections, gates, the global capacity
decisions, per-shard dispatch order, and the batch's aux loss."""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import moe_oracle as O

pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import sparse_mixture_experts_64_b300 as moe
    from sparse_mixture_experts_64_b300 import sharded
    from moe_harness import TOL_AUX, TOL_GATE, cfg_of, oracle_inputs


def _w(name, **kw):
    return W.WORKLOADS[name].replace(name=name + "_" + "_".join(f"{a}{b}" for a, b in kw.items()), **kw)


CASES = [
    # Switch top-1 with bias and capacity 1.25
    (_w("switch_top1", T=700, d=128, h=128), 2),
    # GShard-style top-2 with capacity 1, three unequal shards
    (_w("mixtral_prefill", T=333, d=192, h=128, N=8, k=2, capacity_factor=(1, 1)), 3),
    # fine-grained: N > 32 router path, top-8, capacity 1
    (_w("deepseek_fine", T=260, d=256, N=64, k=8, h=128, h_shared=0, capacity_factor=(1, 1)), 2),
    # no capacity limit, fp32
    (_w("tiny_fp32", T=150, N=4, k=2), 2),
]


def _shards(T, R):
    cuts = np.linspace(0, T, R + 1).astype(int)
    cuts[1:-1] += 7                                  # unequal shards
    return list(zip(cuts[:-1], cuts[1:]))


def _run_sharded(w, inp, R):
    dev = "cuda"
    i32 = dict(dtype=torch.int32, device=dev)
    shards = []
    for a, b in _shards(w.T, R):
        ws_ = w.replace(T=int(b - a), capacity_factor=None)
        cfg = cfg_of(ws_)
        s = dict(a=int(a), b=int(b), cfg=cfg, ws=moe.workspace(cfg),
                 topk_idx=torch.empty((b - a, w.k), **i32), topk_gate=torch.empty((b - a, w.k), device=dev),
                 slot_counts=torch.empty((w.N, w.k), **i32), prob_sums=torch.empty(w.N, device=dev))
        moe.moe_router_shard_stats(cfg, inp["x"][a:b], inp["w_r"], inp["b_r"], s["topk_idx"], s["topk_gate"],
                                   s["slot_counts"], s["prob_sums"], s["ws"])
        shards.append(s)
    counts = np.stack([s["slot_counts"].cpu().numpy() for s in shards])
    bases = sharded.slot_bases(counts)
    g_routed = torch.as_tensor(counts.sum(axis=(0, 2)), dtype=torch.int32, device=dev)
    g_psum = np.zeros(w.N, np.float32)
    for s in shards:
        g_psum = (g_psum + s["prob_sums"].cpu().numpy()).astype(np.float32)
    g_psum = torch.as_tensor(g_psum, device=dev)
    C = sharded.global_capacity(w.T, w.N, w.capacity_factor)
    for r, s in enumerate(shards):
        n = s["b"] - s["a"]
        s.update(counts_kept=torch.full((w.N,), -7, **i32), expert_offsets=torch.full((w.N + 1,), -7, **i32),
                 slot_row=torch.full((n, w.k), -7, **i32),
                 perm_token=torch.full((moe.moe_max_rows(s["cfg"]),), -7, **i32), aux=torch.zeros(2, device=dev))
        base = torch.as_tensor(bases[r], dtype=torch.int32, device=dev)
        moe.moe_router_shard_assign(s["cfg"], s["topk_idx"], base, C, g_routed, g_psum, w.T, s["counts_kept"],
                                    s["expert_offsets"], s["slot_row"], s["perm_token"], s["aux"], s["ws"])
        assert moe.moe_check_error(s["ws"]) == moe.MOE_OK
    return shards, C


@pytest.mark.parametrize("w,R", CASES, ids=[c[0].name for c in CASES])
def test_sharded_router_matches_whole_batch(w, R):
    inp = W.make_inputs(w, device="cuda", router_only=True)
    oi = oracle_inputs(inp)
    rt = O.route(w, oi["x"], oi["w_r"], oi["b_r"])
    shards, C = _run_sharded(w, inp, R)
    assert C == (rt["capacity"] or 0)
    for s in shards:
        a, b = s["a"], s["b"]
        idx = s["topk_idx"].cpu().numpy()
        assert np.array_equal(idx, rt["topk_idx"][a:b])
        assert np.max(np.abs(s["topk_gate"].cpu().numpy() - rt["topk_gate"][a:b])) <= TOL_GATE
        kept = rt["kept"][a:b]
        ck, off, perm, sr = O.group_by_expert(rt["topk_idx"][a:b], kept, w.N)
        assert np.array_equal(s["counts_kept"].cpu().numpy(), ck)
        assert np.array_equal(s["expert_offsets"].cpu().numpy(), off)
        R_ = int(off[-1])
        assert np.array_equal(s["perm_token"].cpu().numpy()[:R_], perm)
        assert np.array_equal(s["slot_row"].cpu().numpy(), sr)
        for i in range(2):
            ref = rt["aux"][i]
            assert abs(float(s["aux"][i]) - ref) <= TOL_AUX * max(abs(ref), 1e-6)
    # the decisions really are global: some shard's local capacity would differ
    assert sum(int((s["slot_row"] < 0).sum()) for s in shards) == int((~rt["kept"]).sum())


def test_one_shard_is_the_unsharded_router():
    """R = 1 with the batch's own capacity: the same bits as moe_router_topk."""
    w = _w("mixtral_prefill", T=301, d=128, h=128, N=8, k=2, capacity_factor=(1, 1))
    inp = W.make_inputs(w, device="cuda", router_only=True)
    (s,), C = _run_sharded(w, inp, 1)
    cfg = cfg_of(w)
    ws = moe.workspace(cfg)
    i32 = dict(dtype=torch.int32, device="cuda")
    o = dict(topk_idx=torch.empty((w.T, w.k), **i32), topk_gate=torch.empty((w.T, w.k), device="cuda"),
             counts_routed=torch.empty(w.N, **i32), counts_kept=torch.empty(w.N, **i32),
             expert_offsets=torch.empty(w.N + 1, **i32), slot_row=torch.empty((w.T, w.k), **i32),
             perm_token=torch.full((moe.moe_max_rows(cfg),), -7, **i32), aux=torch.empty(2, device="cuda"))
    moe.moe_router_topk(cfg, inp["x"], inp["w_r"], inp["b_r"], *o.values(), ws)
    for key in ("topk_idx", "topk_gate", "counts_kept", "expert_offsets", "slot_row"):
        assert torch.equal(s[key], o[key]), key
    R_ = int(o["expert_offsets"][-1])
    assert torch.equal(s["perm_token"][:R_], o["perm_token"][:R_])
    assert torch.allclose(s["aux"], o["aux"], rtol=1e-6)


def test_full_size_switch_two_shards():
    w = W.WORKLOADS["switch_top1"]
    inp = W.make_inputs(w, device="cuda", router_only=True)
    oi = oracle_inputs(inp)
    rt = O.route(w, oi["x"], oi["w_r"], oi["b_r"])
    shards, C = _run_sharded(w, inp, 2)
    assert C == rt["capacity"] == 640
    for s in shards:
        a, b = s["a"], s["b"]
        assert np.array_equal(s["slot_row"].cpu().numpy() >= 0, rt["kept"][a:b])
