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
    _, steps = bench.stream_steps(r, 3)      # this rank's own chunked-prefill request stream
    slowest = bench.reduce_over_ranks(1.5 + r, "max", w)
    tokens = bench.reduce_over_ranks(float(spec.num_tokens), "sum", w)
    stream_tokens = bench.reduce_over_ranks(float(sum(x.num_tokens for x in steps)), "sum", w)
    bench.barrier(w)
    out.put((r, w, slowest, tokens, spec.num_computed.tolist(),
             [sorted(x.scheduled) for x in steps], stream_tokens,
             sum(x.num_tokens for x in steps)))
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
    (r0, w0, m0, t0, c0, s0, st0, own0), (r1, w1, m1, t1, c1, s1, st1, own1) = res
    assert (r0, r1, w0, w1) == (0, 1, 2, 2)
    assert m0 == m1 == 2.5            # max over ranks
    assert t0 == t1 == 2 * 2518.0     # whole-job tokens
    assert c0 != c1                   # each rank owns a different batch
    assert st0 == st1 == own0 + own1  # the streams' tokens add up over ranks
    assert own0 != own1               # each rank draws its own request stream
