"""Cascade (shared-prefix) attention — float64, one row at a time (oracle; test infrastructure).

Source: "第8章 ModelRunner：从 SchedulerOutput 到 GPU Kernel", "8.3.2.5 Cascade Attention 的
"最小 num_computed_tokens - 1" 规则":

* when many requests share a long common prefix (a system prompt, few-shot examples), the
  shared keys and values are attended once for all requests: a first pass over the shared
  prefix and a second pass over each request's own suffix, whose results are combined;
* the usable prefix length is capped by the smallest num_computed of the batch and then
  rounded down to a multiple of the block size (the printed code), because a prefix pass runs
  without a mask: every query must be allowed to see every prefix key.

The section's prose and example disagree with its code (the prose speaks of
``min(num_computed) - 1``; the example calls a 4-token prefix correct where the smallest
num_computed is 3).  This oracle takes the printed code, which never lets the prefix reach a
key some query must not see; the two-pass combination below is exact for any prefix length
no larger than every request's cached length.

``cascade_attention`` merges the two passes by log-sum-exp: with s1, o1 the prefix pass's
log-sum-exp and softmax-weighted values, and s2, o2 the suffix pass's, the row is
``(e^s1 o1 + e^s2 o2) / (e^s1 + e^s2)`` — softmax over the union of the two key sets.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np


def cascade_prefix_len(shared_prefix_tokens: int, num_computed: Sequence[int],
                       block_size: int) -> int:
    """min(shared prefix, smallest num_computed), rounded down to a multiple of block_size."""
    p = int(shared_prefix_tokens)
    for c in num_computed:
        p = min(p, int(c))
    if not len(num_computed):
        return 0
    return p // int(block_size) * int(block_size)


def _softmax_pass(scores: np.ndarray, values: np.ndarray):
    """log-sum-exp and softmax-weighted values of one row over one key set."""
    if scores.size == 0:
        return -math.inf, np.zeros(values.shape[1], np.float64)
    m = scores.max()
    w = np.exp(scores - m)
    return m + math.log(w.sum()), (w / w.sum()) @ values


def cascade_attention(q: np.ndarray, hist_k: Sequence[np.ndarray], hist_v: Sequence[np.ndarray],
                      k_new: np.ndarray, v_new: np.ndarray, query_start_loc: Sequence[int],
                      seq_lens: Sequence[int], num_reqs: int, prefix_len: int, *,
                      scale: Optional[float] = None, rows=None) -> np.ndarray:
    """Attention output ``[N_pad, nh, hd]`` computed as a prefix pass over keys [0, P) of each
    request (the shared ones) and a causal suffix pass over keys [P, c_i + j], merged by
    log-sum-exp.  Arguments as ``oracle.attention.paged_attention``; P must not exceed any
    request's cached length (the prefix pass has no mask)."""
    q = np.asarray(q, np.float64)
    k_new = np.asarray(k_new, np.float64)
    v_new = np.asarray(v_new, np.float64)
    N_pad, nh, hd = q.shape
    group = nh // k_new.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(hd)
    P = int(prefix_len)
    out = np.zeros((N_pad, nh, hd), np.float64)
    wanted = None if rows is None else set(int(r) for r in rows)
    if wanted is not None:
        out[: int(query_start_loc[num_reqs])] = np.nan
    for i in range(num_reqs):
        s, e = int(query_start_loc[i]), int(query_start_loc[i + 1])
        c = int(seq_lens[i]) - (e - s)
        if P > c:
            raise ValueError("the prefix reaches past a request's cached keys")
        K = np.concatenate([np.asarray(hist_k[i], np.float64), k_new[s:e]], axis=0)
        V = np.concatenate([np.asarray(hist_v[i], np.float64), v_new[s:e]], axis=0)
        for j in range(e - s):
            if wanted is not None and (s + j) not in wanted:
                continue
            for h in range(nh):
                kv = h // group
                qv = q[s + j, h, :]
                # pass 1: the shared prefix, every key visible
                s1, o1 = _softmax_pass(K[:P, kv, :] @ qv * scale, V[:P, kv, :])
                # pass 2: the request's own keys P .. c + j
                s2, o2 = _softmax_pass(K[P:c + j + 1, kv, :] @ qv * scale, V[P:c + j + 1, kv, :])
                mx = max(s1, s2)
                w1 = 0.0 if s1 == -math.inf else math.exp(s1 - mx)
                w2 = 0.0 if s2 == -math.inf else math.exp(s2 - mx)
                out[s + j, h, :] = (w1 * o1 + w2 * o2) / (w1 + w2)
    return out
