"""rb_paged_attention_cascade vs the one-pass float64 oracle ("8.3.2.5 Cascade Attention"):
shared-prefix batches of decodes and chunks, head groups 1-10 (powers of two and not),
manager blocks, the prefix
length the rule allows and shorter ones; P = 0 is the plain call bit for bit; a broken
contract sets ATTN_META."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_cases import (compare_attention, dims_of, i32, jump_tensors, oracle_attention,
                       oracle_meta, sample_rows)

pytestmark = pytest.mark.gpu


def _run(rb, spec, tens, meta, P, err=None):
    d = dims_of(spec)
    R, N = spec.num_reqs, spec.num_tokens
    rb.kv_write(d, tens.k, tens.v, i32(meta["slot_mapping"]), tens.k_cache, tens.v_cache,
                error_word=err)
    out = rb.paged_attention_cascade(d, R, N, P, tens.q, tens.k_cache, tens.v_cache,
                                     i32(spec.block_table), i32(meta["query_start_loc"][:R + 1]),
                                     i32(meta["seq_lens"][:R]), error_word=err)
    torch.cuda.synchronize()
    return out


def _check(rb, spec, P=None, rows=None):
    tens = wl.make_tensors(spec, device="cuda")
    meta = oracle_meta(spec)
    d = spec.dims
    if P is None:
        P = rb.cascade_prefix_len(spec.shared_prefix_tokens, spec.num_computed.tolist(),
                                  d.block_size * d.kernel_blocks_per_manager_block)
        assert P == oracle.cascade_prefix_len(spec.shared_prefix_tokens, spec.num_computed,
                                              d.block_size * d.kernel_blocks_per_manager_block)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _run(rb, spec, tens, meta, P, err)
    assert int(err.item()) == 0
    ref = oracle_attention(spec, tens, meta, rows=rows)
    compare_attention(got, ref, spec.num_tokens, rows=rows)
    return P


@pytest.mark.parametrize("seed", range(16))
def test_shared_prefix_mixes(rb, seed):
    nh, nkv = [(32, 8), (8, 1), (4, 4), (16, 2), (6, 2), (12, 2), (28, 4), (10, 1)][seed % 8]
    spec = wl.shared_prefix_batch(seed, num_decodes=3 + seed, prefix_tokens=[64, 160, 512][seed % 3],
                                  suffix_range=(0, 200), num_chunks=seed % 3, chunk_q=[7, 130][seed % 2],
                                  num_q_heads=nh, num_kv_heads=nkv,
                                  head_dim=128 if seed % 2 else 64, hidden_size=64,
                                  manager_ratio=[1, 2][seed % 2])
    assert _check(rb, spec) > 0


def test_shorter_prefix_and_suffix_free_requests(rb):
    """A prefix shorter than allowed, and decodes whose whole cache is the prefix (c = P)."""
    spec = wl.shared_prefix_batch(3, num_decodes=6, prefix_tokens=256, suffix_range=(0, 3),
                                  num_chunks=1, chunk_q=40, hidden_size=64)
    _check(rb, spec, P=128)
    assert _check(rb, spec) == 256


def test_system_prompt_decodes_sampled(rb):
    """256 decodes after a 4096-token shared prompt plus two 512-token chunks."""
    spec = wl.shared_prefix_batch(11, num_decodes=256, prefix_tokens=4096, suffix_range=(16, 1024),
                                  num_chunks=2, chunk_q=512)
    _check(rb, spec, rows=sample_rows(spec, n_random=32, seed=11))


def test_zero_prefix_is_the_plain_call(rb):
    spec = wl.shared_prefix_batch(5, num_decodes=9, prefix_tokens=64, num_chunks=2, chunk_q=70,
                                  hidden_size=64)
    tens = wl.make_tensors(spec, device="cuda")
    meta = oracle_meta(spec)
    got = _run(rb, spec, tens, meta, 0)
    R, N = spec.num_reqs, spec.num_tokens
    plain = rb.paged_attention(dims_of(spec), R, N, tens.q, tens.k_cache, tens.v_cache,
                               i32(spec.block_table), i32(meta["query_start_loc"][:R + 1]),
                               i32(meta["seq_lens"][:R]))
    torch.cuda.synchronize()
    assert torch.equal(got, plain)


def test_broken_contract_sets_attn_meta(rb):
    """A request whose first page differs from row 0's, or a prefix past a cached length."""
    spec = wl.shared_prefix_batch(6, num_decodes=4, prefix_tokens=64, suffix_range=(0, 40),
                                  hidden_size=64)
    tens = wl.make_tensors(spec, device="cuda")
    meta = oracle_meta(spec)
    for P, mutate in ((64, True), (int(spec.num_computed.min()) // 16 * 16 + 16, False)):
        s = spec
        if mutate:
            s = wl.shared_prefix_batch(6, num_decodes=4, prefix_tokens=64, suffix_range=(0, 40),
                                       hidden_size=64)
            s.block_table[2, 1] = s.block_table[2, 5] if s.block_table[2, 5] >= 0 else 1
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        _run(rb, s, tens, meta, P, err)
        assert int(err.item()) & 0x080, (P, mutate)


def test_shared_prefix_score_jumps(rb):
    """Scores rising by ~2^29 and then ~2^58 inside the shared prefix: the prefix pass (no
    causal mask) re-references its key tiles, and the epilogues merge its log-sum-exp with the
    suffix pass's rows across those magnitudes."""
    spec = wl.shared_prefix_batch(5, num_decodes=6, prefix_tokens=704, suffix_range=(0, 200),
                                  num_chunks=2, chunk_q=130, num_q_heads=32, num_kv_heads=8,
                                  head_dim=128, hidden_size=64)
    tens = jump_tensors(spec, {(300, 340): 2.0, (560, 570): 4.0})
    meta = oracle_meta(spec)
    d = spec.dims
    P = rb.cascade_prefix_len(spec.shared_prefix_tokens, spec.num_computed.tolist(),
                              d.block_size * d.kernel_blocks_per_manager_block)
    assert P >= 576  # both jumps lie inside the shared prefix
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = _run(rb, spec, tens, meta, P, err)
    assert int(err.item()) == 0
    ref = oracle_attention(spec, tens, meta)
    compare_attention(got, ref, spec.num_tokens)
