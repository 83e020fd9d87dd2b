"""The data-parallel bookkeeping of bench.py with two gloo ranks on CPU: every rank runs its own
batch (no collective on the data path); only timing (max) and token counts (sum) are reduced."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    import torch.distributed as dist

    r, w, local = bench.dist_setup(backend="gloo")
    spec = bench.make_spec(2, r)
    slowest = bench.reduce_over_ranks(1.5 + r, "max", w)
    tokens = bench.reduce_over_ranks(float(spec.num_tokens), "sum", w)
    bench.barrier(w)
    out.put((r, w, slowest, tokens, spec.num_computed.tolist()))
    dist.destroy_process_group()


def test_two_rank_weak_scaling_bookkeeping():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, w0, m0, t0, c0), (r1, w1, m1, t1, c1) = res
    assert (r0, r1, w0, w1) == (0, 1, 2, 2)
    assert m0 == m1 == 2.5            # max over ranks
    assert t0 == t1 == 2 * 2518.0     # whole-job tokens
    assert c0 != c1                   # each rank owns a different batch
