"""bench.py's multi-rank logic on CPU: two gloo ranks agree on the max time and draw distinct
token batches (replicas with weak scaling, no collective on the data path)."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    import synth
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    mx = bench.reduce_max(10.0 + rank, w)
    seed = bench.rank_seed(0, r)
    x = synth.workload("tiny", seed=seed).x()
    dist.barrier()
    dist.destroy_process_group()
    q.put((r, w, lr, mx, seed, x[:2].copy()))


def test_two_gloo_ranks_share_max_time_and_draw_distinct_batches():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted([q.get(timeout=120) for _ in procs], key=lambda t: t[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, w0, l0, m0, s0, x0), (r1, w1, l1, m1, s1, x1) = res
    assert (r0, r1) == (0, 1) and w0 == w1 == 2 and (l0, l1) == (0, 1)
    assert m0 == m1 == 11.0
    assert s0 != s1 and not (x0 == x1).all()


def test_single_rank_reduce_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5, 1) == 3.5
    assert bench.rank_seed(0, 0) == 0
