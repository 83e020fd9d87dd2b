"""rb_step (one memset and two launches) against the four separate calls: every output bit for
bit — metadata, phase flags, both caches, attention output, gathered rows, error word — and,
on a few cases, directly against the oracle; rb_step_host (host buffers in and out) against
rb_step."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_cases import (check_kv_write, compare_attention, config4_specs, oracle_attention,
                       oracle_meta, sample_rows)

pytestmark = pytest.mark.gpu


def _buffers(rb, spec):
    tens = wl.make_tensors(spec, device="cuda")
    tables = wl.device_tables(spec, "cuda")
    buf = rb.StepBuffers.allocate(rb.Dims.of(spec.dims), spec.num_reqs, spec.num_reqs_padded,
                                  spec.num_tokens, spec.num_tokens_padded, tables, tens.q,
                                  tens.k, tens.v, tens.hidden, tens.k_cache, tens.v_cache)
    return buf, tens


def _twins(rb, spec):
    """Two StepBuffers over the same inputs, each with its own copy of the paged cache."""
    a, tens = _buffers(rb, spec)
    b, _ = _buffers(rb, spec)
    b.k_cache.copy_(a.k_cache)
    b.v_cache.copy_(a.v_cache)
    return a, b, tens


def _same(a, b):
    for k in a.meta:
        assert torch.equal(a.meta[k], b.meta[k]), k
    assert torch.equal(a.k_cache, b.k_cache)
    assert torch.equal(a.v_cache, b.v_cache)
    assert torch.equal(a.attn_out, b.attn_out)
    assert torch.equal(a.rows_out, b.rows_out)


CASES = {
    "cfg1": lambda: wl.config1(),
    "cfg1_pad24": lambda: wl.config1(num_tokens_padded=24),
    "cfg2": lambda: wl.config2(),
    "cfg2_r2": lambda: wl.config2(manager_ratio=2),
    "cfg3": lambda: wl.config3(),
    "cfg3_pad": lambda: wl.config3(num_real=250),
    "cfg5": lambda: wl.config5(),
    "mix_step57": lambda: config4_specs()[57],
    "many_decodes": lambda: wl.batch_from_lists([int(x) for x in np.arange(3000) % 300 + 1],
                                                [1] * 3000, num_q_heads=8, num_kv_heads=2,
                                                head_dim=128, seed=3),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_fused_step_equals_four_calls(rb, name):
    spec = CASES[name]()
    a, b, _ = _twins(rb, spec)
    rb.run_step(a)
    rb.run_step_fused(b)
    torch.cuda.synchronize()
    assert int(a.meta["scalars"][3].item()) == 0
    _same(a, b)


@pytest.mark.parametrize("seed", range(16))
def test_fused_step_fuzz(rb, seed):
    """Head groups that are powers of two and not, head_dim 64 and 128, padding, manager
    blocks."""
    nh, nkv = [(32, 8), (6, 2), (8, 1), (4, 4), (28, 4), (12, 1)][seed % 6]
    spec = wl.random_batch(seed, num_q_heads=nh, num_kv_heads=nkv, head_dim=[64, 128][seed % 2],
                           max_reqs=9, max_q=150, max_c=300, pad_tokens=seed % 5,
                           pad_reqs=seed % 3, manager_ratio=[1, 2, 4, 1][seed % 4])
    a, b, _ = _twins(rb, spec)
    rb.run_step(a)
    rb.run_step_fused(b)
    torch.cuda.synchronize()
    _same(a, b)


ORACLE_CASES = {
    "cfg1_pad24": (lambda: wl.config1(num_tokens_padded=24), None),
    "fuzz": (lambda: wl.random_batch(9, num_q_heads=8, num_kv_heads=2, head_dim=128,
                                     pad_tokens=3), None),
    "cfg2": (lambda: wl.config2(), None),
    "cfg3_pad": (lambda: wl.config3(num_real=250), None),
    "cfg5": (lambda: wl.config5(), 96),   # every decode row + a sample of the chunk's rows
}


@pytest.mark.parametrize("name", sorted(ORACLE_CASES))
def test_fused_step_vs_oracle(rb, name):
    """rb_step (the entry point bench.py times) against the oracle directly: metadata, phase
    flags and scalars bit for bit, the KV write (changed rows = the oracle's real slots plus
    the null page, each real slot holding its token's K and V), attention element-wise, the
    gathered rows bit for bit."""
    make, n_random = ORACLE_CASES[name]
    spec = make()
    buf, tens = _buffers(rb, spec)
    kc0, vc0 = tens.k_cache.clone(), tens.v_cache.clone()
    rb.run_step_fused(buf)
    torch.cuda.synchronize()
    assert int(buf.meta["scalars"][3].item()) == 0
    want = oracle_meta(spec)
    for k in ("input_ids", "positions", "query_start_loc", "seq_lens", "slot_mapping",
              "logits_indices"):
        assert np.array_equal(buf.meta[k].cpu().numpy(), want[k]), k
    assert buf.meta["scalars"][:3].tolist() == [want["max_query_len"], want["max_seq_len"],
                                                want["num_actual_tokens"]]
    check_kv_write(spec, kc0, vc0, tens, want["slot_mapping"])
    rows = None if n_random is None else sample_rows(spec, n_random=n_random, seed=5)
    ref = oracle_attention(spec, tens, want, rows=rows)
    compare_attention(buf.attn_out, ref, spec.num_tokens, rows=rows)
    li = torch.as_tensor(want["logits_indices"], device="cuda")
    assert torch.equal(buf.rows_out, tens.hidden[li])


def test_fused_step_error_bits(rb):
    """A page id outside the pool: the same bits, the same null-page routing."""
    spec = wl.batch_from_lists([3, 0, 9], [2, 4, 1], block_size=16, seed=1,
                               num_q_heads=4, num_kv_heads=2, head_dim=64)
    spec.block_table[1, 0] = spec.dims.num_blocks + 5
    a, b, _ = _twins(rb, spec)
    rb.run_step(a)
    rb.run_step_fused(b)
    torch.cuda.synchronize()
    assert int(a.meta["scalars"][3].item()) & 0x010
    _same(a, b)


@pytest.mark.parametrize("name", ["cfg1_pad24", "cfg2", "mix_step57"])
def test_step_host_equals_device_step(rb, name):
    """rb_step_host (inputs copied in from pinned host memory, results copied back) against
    rb_step on inputs already on the device: the same outputs, bit for bit."""
    spec = CASES[name]()
    a, b, _ = _twins(rb, spec)
    rb.run_step_fused(a)
    host_in = []
    for t in (b.token_table, b.block_table, b.num_computed, b.num_scheduled, b.q, b.k, b.v,
              b.hidden):
        h = t.cpu().pin_memory()
        t.zero_()  # the copies must bring the inputs
        host_in.append((t, h))
    got = {k: torch.empty(t.shape, dtype=t.dtype).pin_memory()
           for k, t in (("attn", b.attn_out), ("rows", b.rows_out), ("scalars", b.meta["scalars"]))}
    host_out = [(got["attn"], b.attn_out), (got["rows"], b.rows_out),
                (got["scalars"], b.meta["scalars"])]
    rb.run_step_host(b, host_in, host_out)
    torch.cuda.synchronize()
    assert int(got["scalars"][3]) == 0
    assert torch.equal(got["attn"], a.attn_out.cpu())
    assert torch.equal(got["rows"], a.rows_out.cpu())
    assert torch.equal(got["scalars"], a.meta["scalars"].cpu())
    _same(a, b)


def test_step_host_async_pipeline_equals_device_steps(rb):
    """rb_step_host_async over a pipelined run of chunked-prefill stream steps (copies on their
    own streams, two buffer sets used by alternate steps, each step's copies overlapping its
    neighbours' compute) gives, step by step, what rb_step gives on inputs already on the
    device: the same attention output, gathered rows and scalars, bit for bit."""
    import dataclasses

    import workloads as wl

    stream = wl.MixedChunkStream(seed=4321)
    steps = [stream.next_step() for _ in range(6)]
    d = stream.dims
    dims = rb.Dims.of(d)
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(7)
    nmax, rmax = stream.BUDGET, d.max_num_reqs
    rnd = lambda *sh: torch.randn(*sh, generator=g, device=dev).to(torch.bfloat16)
    q, k, v = rnd(nmax, d.num_q_heads, d.head_dim), rnd(nmax, d.num_kv_heads, d.head_dim), \
        rnd(nmax, d.num_kv_heads, d.head_dim)
    hidden = rnd(nmax, 256)
    kc0, vc0 = rnd(d.num_slots, d.num_kv_heads, d.head_dim), rnd(d.num_slots, d.num_kv_heads,
                                                                 d.head_dim)
    twins = []
    for t in range(2):  # the same stream applied to two batches with their own KV caches
        batch = rb.PersistentBatch(d.max_num_reqs, d.max_model_len, d.max_blocks_per_req,
                                   device=dev)
        tables = dict(token_table=batch.token_table, block_table=batch.block_table,
                      num_computed=batch.num_computed, num_scheduled=batch.num_scheduled,
                      num_prompt=batch.num_prompt)
        kc, vc = (kc0, vc0) if t == 0 else (kc0.clone(), vc0.clone())
        twins.append((batch, tables, kc, vc))
    # reference: rb_step on the device inputs, one step at a time
    batch, tables, kc, vc = twins[0]
    ref = rb.StepBuffers.allocate(dims, rmax, rmax, nmax, nmax, tables, q, k, v, hidden, kc, vc)
    want = []
    for st in steps:
        batch.apply(st)
        R, N = batch.num_reqs, batch.num_tokens_scheduled
        b = dataclasses.replace(ref, num_reqs=R, num_reqs_padded=R, num_tokens=N,
                                num_tokens_padded=N, q=q[:N], k=k[:N], v=v[:N], hidden=hidden[:N],
                                attn_out=ref.attn_out[:N], rows_out=ref.rows_out[:R],
                                _step_args=None)
        rb.run_step_fused(b)
        torch.cuda.synchronize()
        want.append((b.attn_out.cpu(), b.rows_out.cpu(), b.meta["scalars"].cpu()))
    # pipelined: inputs from pinned host memory, two sets, three streams
    batch, tables, kc, vc = twins[1]
    hq, hk, hv, hh = (t.cpu().pin_memory() for t in (q, k, v, hidden))
    sets = []
    for _ in range(2):
        sb = rb.StepBuffers.allocate(dims, rmax, rmax, nmax, nmax, tables, torch.zeros_like(q),
                                     torch.zeros_like(k), torch.zeros_like(v),
                                     torch.zeros_like(hidden), kc, vc)
        ho = (torch.empty(tuple(sb.attn_out.shape), dtype=sb.attn_out.dtype).pin_memory(),
              torch.empty(tuple(sb.rows_out.shape), dtype=sb.rows_out.dtype).pin_memory(),
              torch.empty(4, dtype=torch.int32).pin_memory())
        sets.append((sb, ho))
    s_comp, s_in, s_out = torch.cuda.current_stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def ev():
        e = torch.cuda.Event()
        e.record(s_comp)
        return e

    in_done, step_done, out_done = ([ev(), ev()] for _ in range(3))
    pending = [None, None]
    seen = {}

    def collect(x):
        if pending[x] is not None:
            out_done[x].synchronize()
            i, N, R = pending[x]
            o_attn, o_rows, o_sc = sets[x][1]
            seen[i] = (o_attn[:N].clone(), o_rows[:R].clone(), o_sc.clone())
            pending[x] = None

    for i, st in enumerate(steps):
        x = i % 2
        sb, (o_attn, o_rows, o_sc) = sets[x]
        collect(x)
        s_in.wait_event(step_done[x])
        s_comp.wait_event(out_done[x])
        batch.apply(st, stream=s_comp)
        R, N = batch.num_reqs, batch.num_tokens_scheduled
        b = dataclasses.replace(sb, num_reqs=R, num_reqs_padded=R, num_tokens=N,
                                num_tokens_padded=N, q=sb.q[:N], k=sb.k[:N], v=sb.v[:N],
                                hidden=sb.hidden[:N], attn_out=sb.attn_out[:N],
                                rows_out=sb.rows_out[:R], _step_args=None)
        ins = [(b.q, hq[:N]), (b.k, hk[:N]), (b.v, hv[:N]), (b.hidden, hh[:N])]
        outs = [(o_attn[:N], b.attn_out), (o_rows[:R], b.rows_out), (o_sc, b.meta["scalars"])]
        rb.run_step_host_async(b, ins, outs, s_comp, s_in, s_out, in_done[x], step_done[x])
        out_done[x].record(s_out)
        pending[x] = (i, N, R)
    collect(0), collect(1)
    torch.cuda.synchronize()
    assert int(batch.error_word.item()) == 0
    for i, (a_attn, a_rows, a_sc) in enumerate(want):
        g_attn, g_rows, g_sc = seen[i]
        assert int(g_sc[3]) == 0, f"step {i}"
        assert torch.equal(g_attn, a_attn), f"step {i}"
        assert torch.equal(g_rows, a_rows), f"step {i}"
        assert torch.equal(g_sc, a_sc), f"step {i}"
