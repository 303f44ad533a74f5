"""Host-side logic of the multi-GPU bench path on CPU ranks (gloo, world 2):
each rank runs its own replica (a different seed, so a different batch), the
timed region ends at the slowest rank (max over ranks) and the work is the sum
over ranks; no collective touches the data path."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import bench
    from workloads import PagedDecodeWorkload, get
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = bench.max_over_ranks(dist, 1.0 + rank)
        n = bench.sum_over_ranks(dist, 10.0 * (rank + 1))
        cfg = get("tiny_f32")
        w = PagedDecodeWorkload(cfg, bench.SEED_BASE + 1000 * rank)
        lens = w.next_step().context_lens.tolist()
        q.put((rank, t, n, lens))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_bench():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, t0, n0, l0), (r1, t1, n1, l1) = res
    assert t0 == t1 == 2.0            # max over ranks
    assert n0 == n1 == 30.0           # sum over ranks
    assert l0 != l1                   # each rank works on its own batch
