"""bench.py's multi-rank plumbing on CPU gloo ranks (world size 2): the process group
from the launcher's environment, the barrier around the timed region, and the
max-over-ranks time that the whole-job value divides the ranks' tokens by."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    try:
        # the environment torchrun gives each rank
        os.environ.update(WORLD_SIZE=str(world), RANK=str(rank), LOCAL_RANK=str(rank),
                          MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        import bench
        w, r, local = bench._dist()
        bench._barrier(w)
        ms = 2.0 + 3.0 * r  # this rank's step time
        ms_max = bench._max_over_ranks(ms, w)
        tokens_per_rank = 4096
        value = w * tokens_per_rank / (ms_max / 1e3)
        q.put((rank, (w, r, local, dist.get_backend(), ms_max, value)))
    except Exception as ex:  # reported to the parent, which fails the test
        q.put((rank, repr(ex)))
    finally:
        if dist.is_initialized():
            dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for pr in procs:
        pr.start()
    res = dict(q.get(timeout=180) for _ in range(world))
    for pr in procs:
        pr.join(timeout=60)
    for r in range(world):
        assert not isinstance(res[r], str), res[r]
        w, rr, local, backend, ms_max, value = res[r]
        assert (w, rr, local, backend) == (world, r, r, "gloo")
        # every rank sees the slowest rank's time: 5 ms, so 2 x 4096 tokens / 5 ms
        assert ms_max == pytest.approx(5.0)
        assert value == pytest.approx(2 * 4096 / 5e-3)
