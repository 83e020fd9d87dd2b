"""Pins of the cascade oracle: the prefix-length rule as printed, and the two-pass attention
against the one-pass definition (softmax over the union of two key sets is the log-sum-exp
merge of the softmaxes over each)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl


def test_prefix_len_rule_page_example():
    """"8.3.2.5": request 1 has 3 cached tokens, request 2 has 4, the shared prefix is 5
    tokens; the printed code caps at the smallest num_computed and aligns to the block."""
    assert oracle.cascade_prefix_len(5, [3, 4], 1) == 3
    assert oracle.cascade_prefix_len(5, [3, 4], 2) == 2
    assert oracle.cascade_prefix_len(100, [40, 70], 16) == 32
    assert oracle.cascade_prefix_len(100, [], 16) == 0
    assert oracle.cascade_prefix_len(0, [40, 70], 16) == 0


def _spec_and_tensors(seed, **kw):
    spec = wl.shared_prefix_batch(seed, num_q_heads=4, num_kv_heads=2, head_dim=64,
                                  hidden_size=64, **kw)
    return spec, wl.make_tensors(spec, with_pool=False)


def _meta(spec):
    d = spec.dims
    return oracle.prepare_inputs(block_size=d.block_size, null_block=d.null_block,
                                 token_table=spec.token_table, block_table=spec.block_table,
                                 num_computed=spec.num_computed, num_scheduled=spec.num_scheduled)


@pytest.mark.parametrize("seed", range(4))
def test_two_passes_equal_one_pass(seed):
    spec, t = _spec_and_tensors(seed, num_decodes=3, prefix_tokens=48, suffix_range=(1, 30),
                                num_chunks=2, chunk_q=9)
    m = _meta(spec)
    f = lambda x: x.float().numpy().astype(np.float64)
    args = (f(t.q), [f(h) for h in t.hist_k], [f(h) for h in t.hist_v], f(t.k), f(t.v),
            m["query_start_loc"], m["seq_lens"], spec.num_reqs)
    plain = oracle.paged_attention(*args)
    P_max = oracle.cascade_prefix_len(48, spec.num_computed, 16)
    assert P_max == 48
    for P in (0, 16, P_max):
        casc = oracle.cascade_attention(*args, prefix_len=P)
        assert np.abs(casc - plain).max() < 1e-12


def test_prefix_past_a_cached_length_is_refused():
    """The prefix pass has no mask, so P may not exceed any request's cached keys."""
    spec, t = _spec_and_tensors(0, num_decodes=2, prefix_tokens=32, suffix_range=(0, 0))
    m = _meta(spec)
    f = lambda x: x.float().numpy().astype(np.float64)
    with pytest.raises(ValueError):
        oracle.cascade_attention(f(t.q), [f(h) for h in t.hist_k], [f(h) for h in t.hist_v],
                                 f(t.k), f(t.v), m["query_start_loc"], m["seq_lens"],
                                 spec.num_reqs, prefix_len=48)
