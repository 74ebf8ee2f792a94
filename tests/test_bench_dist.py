"""Multi-rank host logic of bench.py, on CPU with gloo and two ranks: every
rank serves its own requests of the workload's request stream (weak scaling,
no data-path collective), and the reported step time is the max over ranks."""
import multiprocessing as mp
import os
import socket

import numpy as np

import bench
import workload as wl


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    r, wsz, local = bench.dist_env()
    bench.init_dist(wsz, "gloo")
    w = wl.LONG_CONTEXT
    first = bench.first_request(r, w)
    lens = wl.ctx_lens(w, first).tolist()
    t = bench.max_over_ranks(1.0 + r, wsz)
    bench.barrier(wsz)
    q.put((r, local, first, lens, t))
    dist.destroy_process_group()


def test_two_ranks_shard_requests_and_take_the_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, l0, f0, lens0, t0), (r1, l1, f1, lens1, t1) = out
    w = wl.LONG_CONTEXT
    assert (r0, r1) == (0, 1) and (l0, l1) == (0, 1)
    assert (f0, f1) == (0, w.B)                 # disjoint request ranges
    assert t0 == t1 == 2.0                      # max over ranks on every rank
    # the ranks' requests are the first 2B requests of one stream
    both = wl.ctx_lens(wl.scaled(w, B=2 * w.B))
    assert lens0 + lens1 == both.tolist()
