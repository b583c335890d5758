"""Token-sharded routing on CPU ranks: the exchange between the router's two phases.

A batch routed by the oracle as a whole fixes the global capacity decisions. Each
gloo rank takes its shard of that batch (its selections are the global selections
of its tokens, since routing is per token), exchanges its per-(expert, slot) counts
and softmax sums through sharded.exchange, places its selections at the returned
global priorities and must reproduce the global decisions for its tokens.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from oracle import moe_oracle as O
from sparse_mixture_experts_64_b300 import sharded


def _local_stats(idx, p, N):
    k = idx.shape[1]
    counts = np.zeros((N, k), np.int32)
    for j in range(k):
        np.add.at(counts[:, j], idx[:, j], 1)
    return counts, p.sum(axis=0).astype(np.float32)


def _keep_from_bases(idx, base, C):
    """The capacity rule at global priorities: slot j of a token keeps its expert
    if base[e][j] + (earlier selections of (e, j) on this rank) < C."""
    T, k = idx.shape
    seen = np.zeros_like(base)
    kept = np.ones((T, k), bool)
    for j in range(k):
        for t in range(T):
            e = idx[t, j]
            kept[t, j] = C == 0 or base[e, j] + seen[e, j] < C
            seen[e, j] += 1
    return kept


def _batch(seed, T, N, k, skew=2.0):
    rng = np.random.default_rng(seed)
    L = rng.standard_normal((T, N)).astype(np.float32)
    L[:, 0] += skew                         # overload expert 0 so that drops happen
    idx = O.select_topk(L, k)
    return L, idx, O.softmax_all(L)


def test_slot_bases_brute_force():
    """Base of (rank r, e, j) = number of selections of e that come earlier in the
    global slot-major order, counted one by one."""
    rng = np.random.default_rng(3)
    for R, N, k in ((1, 4, 2), (3, 5, 2), (4, 8, 3), (2, 16, 8)):
        counts = rng.integers(0, 6, size=(R, N, k))
        got = sharded.slot_bases(counts)
        for r in range(R):
            for e in range(N):
                for j in range(k):
                    want = sum(int(counts[rr, e, jj]) for jj in range(j) for rr in range(R))
                    want += sum(int(counts[rr, e, j]) for rr in range(r))
                    assert got[r, e, j] == want


def test_global_capacity():
    assert sharded.global_capacity(4096, 8, (5, 4)) == O.capacity(4096, 8, (5, 4)) == 640
    assert sharded.global_capacity(10, 4, (1, 1)) == 3
    assert sharded.global_capacity(10, 4, None) == 0


@pytest.mark.parametrize("R,N,k", [(1, 4, 2), (2, 8, 1), (3, 8, 2), (4, 16, 4)])
def test_bases_reproduce_global_capacity(R, N, k):
    """Without processes: shards of unequal size, bases from slot_bases, decisions
    equal to the oracle's decisions on the whole batch."""
    T = 97
    L, idx, p = _batch(R * 10 + k, T, N, k)
    C = O.capacity(T, N, (1, 1))
    want = O.keep_within_capacity(idx, N, C)
    cuts = np.linspace(0, T, R + 1).astype(int)
    cuts[1:-1] += np.arange(1, R) * 3          # unequal shards
    stats = [_local_stats(idx[a:b], p[a:b], N) for a, b in zip(cuts[:-1], cuts[1:])]
    bases = sharded.slot_bases(np.stack([c for c, _ in stats]))
    for r, (a, b) in enumerate(zip(cuts[:-1], cuts[1:])):
        assert np.array_equal(_keep_from_bases(idx[a:b], bases[r], C), want[a:b])


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, T, N, k, seed, q):
    try:
        os.environ["MASTER_ADDR"] = "127.0.0.1"
        os.environ["MASTER_PORT"] = str(port)
        dist.init_process_group("gloo", rank=rank, world_size=world)
        L, idx, p = _batch(seed, T, N, k)
        cuts = [0, T // 3 + 5, T] if world == 2 else np.linspace(0, T, world + 1).astype(int)
        a, b = int(cuts[rank]), int(cuts[rank + 1])
        counts, psum = _local_stats(idx[a:b], p[a:b], N)
        base, g_routed, g_psum, T_global = sharded.exchange(
            torch.from_numpy(counts), torch.from_numpy(psum), b - a)
        C = sharded.global_capacity(T_global, N, (1, 1))
        kept = _keep_from_bases(idx[a:b], base.numpy().astype(np.int64), C)
        want = O.keep_within_capacity(idx, N, O.capacity(T, N, (1, 1)))
        ok = (T_global == T and np.array_equal(kept, want[a:b])
              and np.array_equal(g_routed.numpy(), O.counts_routed(idx, N))
              and np.allclose(g_psum.numpy(), p.sum(axis=0), rtol=1e-5))
        # the aux loss from the exchanged sums is the batch's aux loss
        f = g_routed.numpy() / (T_global * k)
        Pm = g_psum.numpy().astype(np.float64) / T_global
        ok = ok and abs(N * float(np.sum(f * Pm)) - O.aux_losses(p, O.counts_routed(idx, N), k)[0]) < 1e-5
        q.put((rank, bool(ok)))
    except Exception as ex:  # reported to the parent, which fails the test
        q.put((rank, repr(ex)))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


@pytest.mark.parametrize("world,N,k", [(2, 8, 2), (2, 8, 1), (3, 16, 4)])
def test_gloo_ranks_exchange(world, N, k):
    """world gloo ranks on CPU: exchange + global priorities = global decisions."""
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, 120, N, k, 40 + world + k, q))
             for r in range(world)]
    for pr in procs:
        pr.start()
    res = dict(q.get(timeout=120) for _ in range(world))
    for pr in procs:
        pr.join(timeout=60)
    assert all(v is True for v in res.values()), res
