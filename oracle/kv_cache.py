"""Paged K/V write by slot_mapping — plain loop (oracle; test infrastructure).

Sources: "vLLM 源码完全拆解（五）…", "3. 物理 KV 槽位" (the t-th new K/V goes to
slot_mapping[t]; the write needs no request id); "变长批处理与一次混合前向", runner.py
(``kv.write(i, slot_mapping, k, v)`` before attention reads the context); the nano-vLLM notes
("Nano-VLLM全代码解析笔记(4)-model_runner") where a slot of -1 marks a token to skip.

Works on any dtype (bytes are copied as they are); the caches are returned as new arrays.
"""
from __future__ import annotations

import numpy as np


def kv_write(k_cache: np.ndarray, v_cache: np.ndarray, slot_mapping, k: np.ndarray,
             v: np.ndarray):
    """Return copies of the caches with row ``slot_mapping[t]`` set to ``k[t]`` / ``v[t]``.

    Rows are written in flat-token order; a negative slot is skipped.
    """
    k_out = k_cache.copy()
    v_out = v_cache.copy()
    for t, s in enumerate(slot_mapping):
        s = int(s)
        if s < 0:
            continue
        k_out[s] = k[t]
        v_out[s] = v[t]
    return k_out, v_out
