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

    For request i and kv head kv the selected queries of the head group are stacked: the scores
    of query j against every key of the request are one matrix product, the keys past its
    visible length ``c_i + j + 1`` get weight exp(-inf) = 0, each row is normalised by its own
    maximum and sum, and the output is the weights times V.  Every query row is computed on its
    own (stacking rows only batches independent products), so the result of a row does not
    depend on which other rows are asked for.
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
        js = np.array([j for j in range(n_new) if wanted is None or (s + j) in wanted], np.int64)
        if js.size == 0:
            continue
        L = c + n_new
        key = np.arange(L)
        # rows per product: bounds the [rows, group, L] score array (~32M values)
        step = max(1, (1 << 25) // (group * L))
        for kv in range(nkv):
            # keys and values of this kv head: the cached history, then this step's rows
            Kh = np.empty((L, hd), np.float64)
            Vh = np.empty((L, hd), np.float64)
            Kh[:c] = hist_k[i][:, kv, :]
            Vh[:c] = hist_v[i][:, kv, :]
            Kh[c:] = k_new[s:e, kv, :]
            Vh[c:] = v_new[s:e, kv, :]
            heads = slice(kv * group, (kv + 1) * group)      # query heads reading this kv head
            for b in range(0, js.size, step):
                jb = js[b:b + step]
                Qb = q[s + jb, heads, :]                       # [J, group, hd]
                scores = np.matmul(Qb, Kh.T) * scale           # [J, group, L]
                visible = c + jb + 1                           # keys 0 .. c + j
                hidden = key[None, :] >= visible[:, None]      # [J, L]
                scores = np.where(hidden[:, None, :], -np.inf, scores)
                scores = scores - scores.max(axis=-1, keepdims=True)
                p = np.exp(scores)
                p = p / p.sum(axis=-1, keepdims=True)
                out[s + jb, heads, :] = np.matmul(p, Vh)
    return out
