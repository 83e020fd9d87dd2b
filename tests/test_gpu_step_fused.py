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
