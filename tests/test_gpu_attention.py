"""rb_paged_attention vs the float64 oracle (max-abs 2e-2, mean-abs 2e-3), plus invariants:
mixed step == each request alone, page-id permutation invariance, padding rows zero."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_cases import (compare_attention, config4_specs, dims_of, i32, jump_tensors,
                       oracle_attention, oracle_meta, run_attention, sample_rows)

pytestmark = pytest.mark.gpu


def _case(rb, spec, rows=None):
    tens = wl.make_tensors(spec, device="cuda")
    meta = oracle_meta(spec)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_attention(rb, spec, tens, meta, error_word=err)
    assert int(err.item()) == 0
    ref = oracle_attention(spec, tens, meta, rows=rows)
    return compare_attention(got, ref, spec.num_tokens, rows=rows), got, tens, meta


@pytest.mark.parametrize("name,make", [
    ("cfg1", lambda: wl.config1()),
    ("cfg1_pad24", lambda: wl.config1(num_tokens_padded=24)),
    ("cfg2", lambda: wl.config2()),
    ("cfg3", lambda: wl.config3()),
    ("cfg3_pad", lambda: wl.config3(num_real=250)),
])
def test_workloads_full(rb, name, make):
    _case(rb, make())


@pytest.mark.parametrize("step", [0, 57])
def test_chunked_prefill_mix_sampled(rb, step):
    spec = config4_specs()[step]
    _case(rb, spec, rows=sample_rows(spec, n_random=48, seed=step))


def test_long_context_sampled(rb):
    spec = wl.config5()
    _case(rb, spec, rows=sample_rows(spec, n_random=96, seed=5))


@pytest.mark.parametrize("seed", range(48))
def test_fuzzed_mixes(rb, seed):
    """Head groups 1-16, powers of two and not (a 128-row tile then holds 128 // group whole
    tokens and masks its last rows)."""
    nh, nkv = [(4, 4), (4, 2), (8, 2), (16, 2), (32, 8), (16, 1), (6, 2), (12, 2), (28, 4),
               (10, 1), (14, 2), (15, 1)][seed % 12]
    hd = 64 if seed % 2 else 128
    spec = wl.random_batch(seed, num_q_heads=nh, num_kv_heads=nkv, head_dim=hd, max_reqs=7,
                           max_q=150, max_c=400, pad_tokens=seed % 4, decode_frac=0.5)
    _case(rb, spec)


@pytest.mark.parametrize("q,c", [(1, 0), (1, 1), (1, 15), (1, 16), (1, 17), (2, 30), (8, 0),
                                 (9, 40), (63, 1), (64, 0), (65, 64), (200, 0), (1, 1000)])
def test_edge_lengths(rb, q, c):
    """Page and tile edges: sequence lengths at and around multiples of 16 and 64."""
    for nh, nkv in ((8, 1), (4, 2), (8, 8), (6, 2), (7, 1)):
        spec = wl.batch_from_lists([c, 3], [q, 1], num_q_heads=nh, num_kv_heads=nkv,
                                   head_dim=128, seed=q * 1000 + c)
        _case(rb, spec)


def test_mixed_step_equals_each_request_alone(rb):
    """'验证：一次混合前向': one mixed step gives every request what it gets alone."""
    spec = wl.config1()
    (_, _), mixed, tens, meta = _case(rb, spec)
    dims = dims_of(spec)
    qsl, sl = meta["query_start_loc"], meta["seq_lens"]
    for i in range(spec.num_reqs):
        s, e = int(qsl[i]), int(qsl[i + 1])
        bt = np.full((1, spec.dims.max_blocks_per_req), -1, np.int32)
        bt[0] = spec.block_table[i]
        alone = rb.paged_attention(dims, 1, e - s, tens.q[s:e].contiguous(), tens.k_cache,
                                   tens.v_cache, i32(bt), i32([0, e - s]), i32([sl[i]]))
        torch.cuda.synchronize()
        assert torch.equal(alone, mixed[s:e])


def test_page_permutation_invariance(rb):
    """Moving pages to other physical ids (and the page table with them) changes nothing."""
    spec = wl.random_batch(11, num_q_heads=8, num_kv_heads=2, head_dim=128, max_reqs=6,
                           max_q=90, max_c=300)
    (_, _), got, tens, meta = _case(rb, spec)
    d = spec.dims
    rng = np.random.default_rng(0)
    perm = np.concatenate([[0], 1 + rng.permutation(d.num_blocks - 1)])  # keep the null page
    bt2 = np.where(spec.block_table >= 0, perm[np.maximum(spec.block_table, 0)], -1)
    B = d.block_size
    pages = lambda c: c.view(d.num_blocks, B, d.num_kv_heads, d.head_dim)
    k2 = torch.empty_like(tens.k_cache)
    v2 = torch.empty_like(tens.v_cache)
    idx = torch.as_tensor(perm, device="cuda")
    pages(k2)[idx] = pages(tens.k_cache)
    pages(v2)[idx] = pages(tens.v_cache)
    R, N = spec.num_reqs, spec.num_tokens
    out2 = rb.paged_attention(dims_of(spec), R, N, tens.q, k2, v2, i32(bt2),
                              i32(meta["query_start_loc"][:R + 1]), i32(meta["seq_lens"][:R]))
    torch.cuda.synchronize()
    assert torch.equal(out2, got)


def test_metadata_errors_are_flagged(rb):
    spec = wl.batch_from_lists([5, 0], [1, 20], num_q_heads=4, num_kv_heads=2, head_dim=64)
    tens = wl.make_tensors(spec, device="cuda")
    meta = oracle_meta(spec)
    dims = dims_of(spec)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad_sl = meta["seq_lens"][:2].copy()
    bad_sl[1] = 3                                   # shorter than its query
    rb.paged_attention(dims, 2, 21, tens.q, tens.k_cache, tens.v_cache, i32(spec.block_table),
                       i32(meta["query_start_loc"][:3]), i32(bad_sl), error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 0x080
    err.zero_()
    bt = spec.block_table.copy()
    bt[1, 0] = spec.dims.num_blocks + 5             # page id outside the pool
    rb.paged_attention(dims, 2, 21, tens.q, tens.k_cache, tens.v_cache, i32(bt),
                       i32(meta["query_start_loc"][:3]), i32(meta["seq_lens"][:2]),
                       error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) & 0x010


@pytest.mark.parametrize("nh,nkv,hd", [(32, 8, 128), (8, 1, 128), (12, 2, 64)])
def test_score_jumps_across_key_tiles(rb, nh, nkv, hd):
    """A row's maximum rising by far more than 2^20 between key tiles (once, then again): the
    prefill softmax takes its exponents against the reference of an earlier tile, so these
    rows make it re-reference the tile (O and the sum rescaled) — exact either way."""
    spec = wl.batch_from_lists([600, 0, 700], [300, 400, 1], num_q_heads=nh, num_kv_heads=nkv,
                               head_dim=hd, seed=nh * 100 + hd)
    scale = 128 / hd  # the same jumps in log2 units at head_dim 64
    tens = jump_tensors(spec, {(300, 340): 2.0 * scale, (560, 570): 4.0 * scale})
    meta = oracle_meta(spec)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = run_attention(rb, spec, tens, meta, error_word=err)
    assert int(err.item()) == 0
    ref = oracle_attention(spec, tens, meta)
    compare_attention(got, ref, spec.num_tokens)
