"""Selection of the hidden rows that feed the LM head (oracle; test infrastructure).

Sources: "vLLM 源码完全拆解（五）…", "第四步：只在必要位置计算 logits" (only the selected
hidden states go through the vocabulary projection); "04 · 模型执行与 CUDA Graph", step ⑤
(``hidden_states[logits_indices]``); "变长批处理与一次混合前向", runner.py
(``x[b.logits_indices]``).
"""
from __future__ import annotations

import numpy as np


def gather_rows(hidden: np.ndarray, indices) -> np.ndarray:
    """``out[i] = hidden[indices[i]]`` row by row."""
    out = np.empty((len(indices),) + hidden.shape[1:], dtype=hidden.dtype)
    for i, r in enumerate(indices):
        out[i] = hidden[int(r)]
    return out
