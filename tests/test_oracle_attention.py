"""Pins of the attention oracle: library special cases, closed forms and the pages' visibility example."""
import math

import numpy as np
import pytest
import torch

import oracle


def _meta(num_computed, num_scheduled):
    out = oracle.prepare_inputs(block_size=1, null_block=0,
                                token_table=np.zeros((len(num_scheduled), 1 + max(
                                    c + q for c, q in zip(num_computed, num_scheduled))), np.int64),
                                block_table=np.tile(np.arange(1, 1 + max(
                                    c + q for c, q in zip(num_computed, num_scheduled))),
                                    (len(num_scheduled), 1)),
                                num_computed=num_computed, num_scheduled=num_scheduled)
    return out["query_start_loc"], out["seq_lens"]


def _rand_batch(rng, num_computed, num_scheduled, nh, nkv, hd, pad=0):
    N = sum(num_scheduled)
    q = rng.standard_normal((N + pad, nh, hd))
    k = rng.standard_normal((N + pad, nkv, hd))
    v = rng.standard_normal((N + pad, nkv, hd))
    hk = [rng.standard_normal((c, nkv, hd)) for c in num_computed]
    hv = [rng.standard_normal((c, nkv, hd)) for c in num_computed]
    return q, k, v, hk, hv


def _sdpa(q, k, v, mask=None, causal=False, gqa=1):
    """torch SDPA in float64: q [L, nh, hd], k/v [S, nkv, hd] -> [L, nh, hd]."""
    Q = torch.from_numpy(q).permute(1, 0, 2)[None]
    K = torch.from_numpy(k).permute(1, 0, 2)[None].repeat_interleave(gqa, dim=1)
    V = torch.from_numpy(v).permute(1, 0, 2)[None].repeat_interleave(gqa, dim=1)
    m = None if mask is None else torch.from_numpy(mask)
    o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=m, is_causal=causal)
    return o[0].permute(1, 0, 2).numpy()


def test_fresh_prefill_equals_causal_sdpa():
    """c = 0, g = 1, one request: plain causal multi-head attention."""
    rng = np.random.default_rng(0)
    q, k, v, hk, hv = _rand_batch(rng, [0], [37], 3, 3, 32)
    qsl, sl = _meta([0], [37])
    got = oracle.paged_attention(q, hk, hv, k, v, qsl, sl, 1)
    ref = _sdpa(q, k, v, causal=True)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_single_query_equals_unmasked_sdpa():
    """A decode (q = 1) reads every cached key plus its own: softmax over all of them."""
    rng = np.random.default_rng(1)
    q, k, v, hk, hv = _rand_batch(rng, [50], [1], 4, 4, 16)
    qsl, sl = _meta([50], [1])
    got = oracle.paged_attention(q, hk, hv, k, v, qsl, sl, 1)
    K = np.concatenate([hk[0], k]); V = np.concatenate([hv[0], v])
    ref = _sdpa(q, K, V)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


@pytest.mark.parametrize("nh,nkv", [(4, 2), (8, 2), (8, 1), (6, 3)])
def test_chunk_with_history_gqa_equals_masked_sdpa(nh, nkv):
    """A chunk on top of cached context with grouped heads: SDPA with a bottom-right causal mask
    and each kv head repeated for its group of query heads."""
    rng = np.random.default_rng(nh * 10 + nkv)
    c, n = 23, 11
    q, k, v, hk, hv = _rand_batch(rng, [c], [n], nh, nkv, 16)
    qsl, sl = _meta([c], [n])
    got = oracle.paged_attention(q, hk, hv, k, v, qsl, sl, 1)
    K = np.concatenate([hk[0], k]); V = np.concatenate([hv[0], v])
    mask = np.tril(np.ones((n, c + n), bool), k=c)
    ref = _sdpa(q, K, V, mask=mask, gqa=nh // nkv)
    np.testing.assert_allclose(got, ref, rtol=0, atol=1e-12)


def test_visible_lengths_of_the_runner_example():
    """Zero queries make every visible key weigh the same, so with V[k] = k the output is the
    mean key index (L - 1) / 2; the pages print L = 6, 1, 2, 3, 9, 10 for A, B, C."""
    c, qn = [5, 0, 8], [1, 3, 2]
    qsl, sl = _meta(c, qn)
    N = sum(qn)
    q = np.zeros((N, 2, 4))
    k = np.random.default_rng(2).standard_normal((N, 1, 4))
    hk = [np.random.default_rng(3 + i).standard_normal((ci, 1, 4)) for i, ci in enumerate(c)]
    hv = [np.broadcast_to(np.arange(ci, dtype=float)[:, None, None], (ci, 1, 4)).copy() for ci in c]
    v = np.concatenate([np.broadcast_to((ci + np.arange(n, dtype=float))[:, None, None], (n, 1, 4))
                        for ci, n in zip(c, qn)])
    out = oracle.paged_attention(q, hk, hv, k, v, qsl, sl, 3)
    visible = np.round(out[:, :, 0] * 2 + 1).astype(int)
    assert visible[:, 0].tolist() == [6, 1, 2, 3, 9, 10]
    assert visible[:, 1].tolist() == [6, 1, 2, 3, 9, 10]


def test_softmax_scale_closed_form():
    """Two keys, scores 0 and a*b: the weight of key 1 is 1 / (1 + exp(-a*b/sqrt(hd)))."""
    hd = 64
    a, b = 3.0, 2.5
    q = np.zeros((1, 1, hd)); q[0, 0, 0] = a
    hk = [np.zeros((1, 1, hd))]
    k = np.zeros((1, 1, hd)); k[0, 0, 0] = b
    hv = [np.zeros((1, 1, hd))]
    v = np.ones((1, 1, hd))
    qsl, sl = _meta([1], [1])
    out = oracle.paged_attention(q, hk, hv, k, v, qsl, sl, 1)
    w = 1.0 / (1.0 + math.exp(-a * b / math.sqrt(hd)))
    np.testing.assert_allclose(out[0, 0], w, rtol=1e-14)


def test_mixed_step_equals_each_request_alone_and_padding_is_zero():
    """'验证：一次混合前向': one mixed step gives each request what it gets alone."""
    rng = np.random.default_rng(4)
    c, qn = [0, 5, 10], [7, 1, 12]
    q, k, v, hk, hv = _rand_batch(rng, c, qn, 4, 2, 8, pad=4)
    qsl, sl = _meta(c, qn)
    mixed = oracle.paged_attention(q, hk, hv, k, v, qsl, sl, 3)
    assert np.all(mixed[20:] == 0)
    for i in range(3):
        s, e = qsl[i], qsl[i + 1]
        qs1, sl1 = _meta([c[i]], [qn[i]])
        alone = oracle.paged_attention(q[s:e], [hk[i]], [hv[i]], k[s:e], v[s:e], qs1, sl1, 1)
        np.testing.assert_array_equal(mixed[s:e], alone)


def test_row_subset_matches_full():
    rng = np.random.default_rng(5)
    c, qn = [3, 0, 9], [4, 6, 1]
    q, k, v, hk, hv = _rand_batch(rng, c, qn, 4, 2, 8)
    qsl, sl = _meta(c, qn)
    full = oracle.paged_attention(q, hk, hv, k, v, qsl, sl, 3)
    part = oracle.paged_attention(q, hk, hv, k, v, qsl, sl, 3, rows=[0, 5, 10])
    for r in (0, 5, 10):
        np.testing.assert_array_equal(part[r], full[r])
    assert np.isnan(part[1]).all()


def test_threaded_evaluation_equals_one_call():
    """oracle.threads evaluates each request on its own rows in a thread pool: the same rows as
    one call over the whole batch (up to BLAS summation order), NaN elsewhere, padding zero."""
    from oracle.threads import oracle_attention_threads

    rng = np.random.default_rng(6)
    c, qn = [30, 0, 12, 7], [1, 9, 5, 1]
    q, k, v, hk, hv = _rand_batch(rng, c, qn, 8, 2, 16, pad=2)
    qsl, sl = _meta(c, qn)
    rows = [0, 1, 4, 9, 10, 12, 15]
    full = oracle.paged_attention(q, hk, hv, k, v, qsl, sl, 4)
    got = oracle_attention_threads(q, hk, hv, k, v, qsl, sl, 4, rows, workers=3)
    np.testing.assert_allclose(got[rows], full[rows], rtol=0, atol=1e-13)
    others = [r for r in range(16) if r not in rows]
    assert np.isnan(got[others]).all() and np.all(got[16:] == 0)


def test_threaded_evaluation_cuts_long_requests():
    """A request holding most of the rows x keys is cut into several calls on parts of its rows
    (so that it does not keep one thread busy while the others wait): the rows come out as one
    call over the whole batch gives them."""
    from oracle.threads import oracle_attention_threads

    rng = np.random.default_rng(7)
    c, qn = [300, 2, 0], [48, 1, 3]
    q, k, v, hk, hv = _rand_batch(rng, c, qn, 8, 2, 16, pad=1)
    qsl, sl = _meta(c, qn)
    rows = list(range(0, 52, 1))
    full = oracle.paged_attention(q, hk, hv, k, v, qsl, sl, 3)
    got = oracle_attention_threads(q, hk, hv, k, v, qsl, sl, 3, rows, workers=4)
    np.testing.assert_allclose(got[rows], full[rows], rtol=0, atol=1e-13)
    assert np.all(got[52:] == 0)
