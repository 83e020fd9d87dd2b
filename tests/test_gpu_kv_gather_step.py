"""rb_kv_write and rb_gather_rows bit-exact vs the oracle; the whole step (as bench.py times
it) on the padding-example workload and friends."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_cases import (compare_attention, dims_of, i32, oracle_attention, oracle_meta)

pytestmark = pytest.mark.gpu


def _u16(t):
    return t.contiguous().view(torch.int16).cpu().numpy()


def _check_cache(spec, before, after, expected):
    """Every page but the null page must match the oracle byte for byte."""
    B, nb = spec.dims.block_size, spec.dims.null_block
    keep = np.ones(after.shape[0], bool)
    keep[nb * B:(nb + 1) * B] = False
    assert np.array_equal(after[keep], expected[keep])


@pytest.mark.parametrize("name,make", [
    ("cfg1", lambda: wl.config1(num_tokens_padded=24)),
    ("cfg2", lambda: wl.config2()),
    ("cfg3_pad", lambda: wl.config3(num_real=250)),
    ("fuzz", lambda: wl.random_batch(5, num_q_heads=8, num_kv_heads=2, head_dim=128,
                                     pad_tokens=7)),
])
def test_kv_write_bit_exact(rb, name, make):
    spec = make()
    tens = wl.make_tensors(spec, device="cuda")
    meta = oracle_meta(spec)
    kc0, vc0 = _u16(tens.k_cache), _u16(tens.v_cache)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rb.kv_write(dims_of(spec), tens.k, tens.v, i32(meta["slot_mapping"]), tens.k_cache,
                tens.v_cache, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    ek, ev = oracle.kv_write(kc0, vc0, meta["slot_mapping"], _u16(tens.k), _u16(tens.v))
    _check_cache(spec, kc0, _u16(tens.k_cache), ek)
    _check_cache(spec, vc0, _u16(tens.v_cache), ev)


def test_kv_write_skips_negative_and_flags_out_of_range(rb):
    spec = wl.config1()
    tens = wl.make_tensors(spec, device="cuda")
    n = spec.num_tokens
    slots = np.arange(n, dtype=np.int32) + 16
    slots[3] = -1
    slots[5] = spec.dims.num_slots          # outside the pool
    kc0, vc0 = _u16(tens.k_cache), _u16(tens.v_cache)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    rb.kv_write(dims_of(spec), tens.k, tens.v, i32(slots), tens.k_cache, tens.v_cache,
                error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 0x020
    ok = np.array([s >= 0 and s < spec.dims.num_slots for s in slots])
    ek, _ = oracle.kv_write(kc0, vc0, np.where(ok, slots, -1), _u16(tens.k), _u16(tens.v))
    assert np.array_equal(_u16(tens.k_cache), ek)


@pytest.mark.parametrize("H", [128, 4096, 8192])
def test_gather_rows_bit_exact(rb, H):
    g = torch.Generator(device="cuda")
    g.manual_seed(H)
    hidden = torch.randn(300, H, generator=g, device="cuda").to(torch.bfloat16)
    idx = np.random.default_rng(H).integers(0, 300, size=37).astype(np.int32)
    out = rb.gather_rows(hidden, i32(idx))
    torch.cuda.synchronize()
    assert np.array_equal(_u16(out), oracle.gather_rows(_u16(hidden), idx))
    bad = idx.copy()
    bad[4] = 300
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = rb.gather_rows(hidden, i32(bad), error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 0x040
    assert torch.count_nonzero(out[4]) == 0


@pytest.mark.parametrize("name,make", [
    ("cfg2", lambda: wl.config2()),
    ("cfg1_pad24", lambda: wl.config1(num_tokens_padded=24)),
    ("cfg3_pad", lambda: wl.config3(num_real=250)),
])
def test_whole_step(rb, name, make):
    """One pass of the hot path through run_step (the launch sequence bench.py times)."""
    from ragged_mixed_paged_gb300 import StepBuffers, run_step

    spec = make()
    tens = wl.make_tensors(spec, device="cuda")
    kc0, vc0 = _u16(tens.k_cache), _u16(tens.v_cache)
    tables = wl.device_tables(spec, "cuda")
    buf = StepBuffers.allocate(dims_of(spec), spec.num_reqs, spec.num_reqs_padded,
                               spec.num_tokens, spec.num_tokens_padded, tables, tens.q, tens.k,
                               tens.v, tens.hidden, tens.k_cache, tens.v_cache)
    run_step(buf)
    torch.cuda.synchronize()
    meta = oracle_meta(spec)
    m = {k: v.cpu().numpy() for k, v in buf.meta.items()}
    for k in ("input_ids", "positions", "query_start_loc", "seq_lens", "slot_mapping",
              "logits_indices"):
        assert np.array_equal(m[k], meta[k]), k
    assert m["scalars"].tolist() == [meta["max_query_len"], meta["max_seq_len"],
                                     meta["num_actual_tokens"], 0]
    ek, ev = oracle.kv_write(kc0, vc0, meta["slot_mapping"], _u16(tens.k), _u16(tens.v))
    _check_cache(spec, kc0, _u16(tens.k_cache), ek)
    _check_cache(spec, vc0, _u16(tens.v_cache), ev)
    ref = oracle_attention(spec, tens, meta)
    compare_attention(buf.attn_out, ref, spec.num_tokens)
    assert np.array_equal(_u16(buf.rows_out),
                          oracle.gather_rows(_u16(tens.hidden), meta["logits_indices"]))
    # a second step on the same buffers gives the same answer (fixed addresses, no state), also
    # through the profiled attention entry point that records events between its launches
    first = buf.attn_out.clone()
    marks = [torch.cuda.Event(enable_timing=True) for _ in range(5)]
    attn_marks = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for e in attn_marks:
        e.record()
    run_step(buf, marks=marks, attn_marks=attn_marks)
    torch.cuda.synchronize()
    assert torch.equal(buf.attn_out, first)
    times = [marks[2].elapsed_time(attn_marks[0]), attn_marks[0].elapsed_time(attn_marks[1]),
             attn_marks[1].elapsed_time(attn_marks[2]), attn_marks[2].elapsed_time(marks[3])]
    assert all(t >= 0 for t in times)
