"""Varlen causal GQA attention of a mixed batch — dense float64, one request at a time
(oracle; test infrastructure).

Sources (page title, then section):

* "vLLM 源码完全拆解（五）…", "4. 注意力读取边界": a query only reads its own request;
  query j of request i sees the c_i cached keys plus the new keys up to and including its
  own position, c_i + j + 1 keys in all (A sees 6; B sees 1, 2, 3; C sees 9, 10);
  "为什么不显式构造巨大 Attention Mask": the bound comes from query_start_loc, seq_lens and
  causal=True rather than from a stored mask.
* "变长批处理与一次混合前向", runner.py: scale = 1 / sqrt(head_dim); the step writes the new
  K/V first and then reads the whole context ("先写入，再读出整段上下文").

Here the keys and values of request i are NOT read through the page table: they are the
request's contiguous cached history (the copy the harness placed into the pool) followed by
this step's new rows, so a paging error on the device side cannot hide in the oracle.

Readings where the pages are silent: query head h reads kv head ``h // (nh / nkv)``
(contiguous groups); no soft-cap, window or bias; padded rows (t >= N) are zero.
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Sequence

import numpy as np


def paged_attention(q: np.ndarray, hist_k: Sequence[np.ndarray], hist_v: Sequence[np.ndarray],
                    k_new: np.ndarray, v_new: np.ndarray, query_start_loc: Sequence[int],
                    seq_lens: Sequence[int], num_reqs: int, *, scale: Optional[float] = None,
                    rows: Optional[Iterable[int]] = None) -> np.ndarray:
    """Attention output ``[N_pad, nh, hd]`` in float64.

    ``q [N_pad, nh, hd]``, ``k_new/v_new [N_pad, nkv, hd]``: this step's rows (flat order).
    ``hist_k[i]/hist_v[i] [c_i, nkv, hd]``: request i's cached keys/values, contiguous.
    ``rows``: if given, only these flat token indices are computed; the other real rows are NaN.
    """
    q = np.asarray(q, np.float64)
    k_new = np.asarray(k_new, np.float64)
    v_new = np.asarray(v_new, np.float64)
    N_pad, nh, hd = q.shape
    nkv = k_new.shape[1]
    assert nh % nkv == 0
    group = nh // nkv
    if scale is None:
        scale = 1.0 / math.sqrt(hd)
    out = np.zeros((N_pad, nh, hd), np.float64)
    wanted = None if rows is None else set(int(r) for r in rows)
    if wanted is not None:
        out[: int(query_start_loc[num_reqs])] = np.nan

    for i in range(num_reqs):
        s, e = int(query_start_loc[i]), int(query_start_loc[i + 1])
        n_new = e - s
        c = int(seq_lens[i]) - n_new
        assert c == hist_k[i].shape[0], "seq_len - query_len must equal the cached length"
        js = [j for j in range(n_new) if wanted is None or (s + j) in wanted]
        if not js:
            continue
        K = np.concatenate([np.asarray(hist_k[i], np.float64), k_new[s:e]], axis=0)  # [L, nkv, hd]
        V = np.concatenate([np.asarray(hist_v[i], np.float64), v_new[s:e]], axis=0)
        for h in range(nh):
            kv = h // group
            for j in js:
                visible = c + j + 1                       # keys 0 .. c + j
                scores = K[:visible, kv, :] @ q[s + j, h, :] * scale
                scores = scores - scores.max()
                p = np.exp(scores)
                p = p / p.sum()
                out[s + j, h, :] = p @ V[:visible, kv, :]
    return out
