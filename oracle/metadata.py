"""Step metadata of a flattened, unpadded mixed batch — plain loops (oracle; test infrastructure).

Sources (page title, then section):

* "vLLM 源码完全拆解（五）：GPUModelRunner 如何把动态请求拼成一次 GPU 前向"
  - "第一步：从每请求 token 数得到边界": query_start_loc is the length-(R+1) prefix sum of
    the scheduled counts, request i owns the half-open interval [s_i, s_{i+1});
  - "第二步：相对位置加已计算长度得到模型位置": position = num_computed[i] + offset j,
    seq_lens = num_computed + num_scheduled;
  - "第三步：从二维 token 历史抽取本轮切片": token (i, j) is row i, column c_i + j of the
    [max_num_reqs, max_model_len] token table;
  - "第四步：只在必要位置计算 logits": logits index of request i = query_start_loc[i+1] - 1;
  - "Block table 是逐请求的页表": logical block = p // B, offset = p % B,
    slot = block_table[i, p // B] * B + p % B;
  - "固定地址与动态有效长度如何共存": padding to a captured size Q' >= Q keeps the real count
    in num_actual_tokens, repeats the total in the query_start_loc tail (empty intervals) and
    points padded slots at a reserved place.
* "第8章 ModelRunner：从 SchedulerOutput 到 GPU Kernel"
  - "8.3.1.6 np.repeat + cumsum 的向量化 req_indices 构造" (req_indices, in-request offsets),
  - "8.3.2 slot_mapping：新 token 写到哪个 KV 槽" (per-token slot loop),
  - "8.5.0.5 pad_for_cudagraph 的实现" (smallest captured size >= the token count).
* "04 · 模型执行与 CUDA Graph", "5. 关键细节与坑": padding tokens use the null block (block 0),
  which never holds real cache.
* same GPUModelRunner page, "混合 KV Cache：一条请求不止一张页表": when the manager's block is
  larger than the kernel's, each manager block id expands into several kernel block ids
  (32-token manager blocks over 16-token kernel pages: [0, 1, 2] -> [0, 1, 2, 3, 4, 5]), and
  the slot map works on the expanded ids.
* "变长批处理与一次混合前向", "布局与元数据" and "为什么不填充".

Readings where the pages are silent: padded requests get seq_len 0 and the empty interval at
the end; a padded token t (t >= N) gets input id 0, position 0 and slot
``null_block * B + (t - N) % B``; a padded request's logits index is ``max(N - 1, 0)``.
"""
from __future__ import annotations

import bisect
from typing import Dict, Sequence

import numpy as np


def req_indices_and_query_pos(num_scheduled: Sequence[int]):
    """Owner request and in-request offset of every flat token (8.3.1.6; "第一步")."""
    req_indices, query_pos = [], []
    for i, q in enumerate(num_scheduled):
        for j in range(int(q)):
            req_indices.append(i)
            query_pos.append(j)
    return np.array(req_indices, np.int64), np.array(query_pos, np.int64)


def map_to_kernel_blocks(manager_ids: Sequence[int], kernel_blocks_per_manager_block: int):
    """Kernel block ids of a row of manager block ids ("混合 KV Cache：一条请求不止一张页表"):
    manager block m of r kernel blocks becomes kernel blocks r*m, r*m + 1, ..., r*m + r - 1,
    in order, so [0, 1, 2] with r = 2 is [0, 1, 2, 3, 4, 5] as the page prints."""
    r = int(kernel_blocks_per_manager_block)
    out = []
    for m in manager_ids:
        for j in range(r):
            out.append(int(m) * r + j)
    return out


def prepare_inputs(*, block_size: int, null_block: int, token_table: np.ndarray,
                   block_table: np.ndarray, num_computed: Sequence[int],
                   num_scheduled: Sequence[int], num_reqs_padded: int | None = None,
                   num_tokens_padded: int | None = None,
                   num_prompt: Sequence[int] | None = None,
                   kernel_blocks_per_manager_block: int = 1) -> Dict[str, np.ndarray]:
    """Flat step inputs and attention metadata of one batch, as plain loops.

    Returns int64 arrays ``query_start_loc [R_pad+1]``, ``seq_lens [R_pad]``,
    ``positions [N_pad]``, ``input_ids [N_pad]``, ``slot_mapping [N_pad]``,
    ``logits_indices [R_pad]``, ``visible_keys [N]`` (keys each query may read, "4. 注意力读取边界")
    and ints ``max_query_len``, ``max_seq_len``, ``num_actual_tokens``.  With ``num_prompt``
    also ``is_prefilling [R_pad]`` and ``discard_request_mask [R_pad]`` (see request_flags).
    With ``kernel_blocks_per_manager_block`` r > 1 the rows of ``block_table`` hold manager
    block ids, expanded to kernel block ids (``map_to_kernel_blocks``) before the slot map;
    ``block_size`` and ``null_block`` are then the kernel's.
    """
    B = int(block_size)
    R = len(num_scheduled)
    R_pad = R if num_reqs_padded is None else int(num_reqs_padded)
    assert R_pad >= R

    # 第一步: boundaries from per-request counts
    qsl = [0]
    for i in range(R):
        qsl.append(qsl[-1] + int(num_scheduled[i]))
    N = qsl[-1]
    N_pad = N if num_tokens_padded is None else int(num_tokens_padded)
    assert N_pad >= N
    for _ in range(R, R_pad):  # padded requests: empty intervals at the end
        qsl.append(N)

    # 第二步: sequence lengths after this step
    seq_lens = [int(num_computed[i]) + int(num_scheduled[i]) for i in range(R)] + [0] * (R_pad - R)

    positions, input_ids, slots, visible = [], [], [], []
    for i in range(R):
        kernel_row = (block_table[i] if kernel_blocks_per_manager_block == 1 else
                      map_to_kernel_blocks(block_table[i], kernel_blocks_per_manager_block))
        c = int(num_computed[i])
        for j in range(int(num_scheduled[i])):
            p = c + j                                     # 第二步
            positions.append(p)
            input_ids.append(int(token_table[i, p]))      # 第三步
            logical_block, offset = p // B, p % B         # Block table 是逐请求的页表
            slots.append(int(kernel_row[logical_block]) * B + offset)
            visible.append(c + j + 1)                     # 4. 注意力读取边界
    for t in range(N, N_pad):                              # padding tokens -> the null block
        positions.append(0)
        input_ids.append(0)
        slots.append(null_block * B + (t - N) % B)

    # 第四步: last flat token of every request
    logits = [qsl[i + 1] - 1 for i in range(R)] + [max(N - 1, 0)] * (R_pad - R)

    flags = {} if num_prompt is None else request_flags(num_computed, num_scheduled, num_prompt,
                                                        R_pad)
    return dict(
        **flags,
        query_start_loc=np.array(qsl, np.int64),
        seq_lens=np.array(seq_lens, np.int64),
        positions=np.array(positions, np.int64),
        input_ids=np.array(input_ids, np.int64),
        slot_mapping=np.array(slots, np.int64),
        logits_indices=np.array(logits, np.int64),
        visible_keys=np.array(visible, np.int64),
        max_query_len=max([int(x) for x in num_scheduled] + [0]),
        max_seq_len=max(seq_lens[:R] + [0]),
        num_actual_tokens=N,
    )


def request_flags(num_computed: Sequence[int], num_scheduled: Sequence[int],
                  num_prompt: Sequence[int], num_reqs_padded: int | None = None):
    """Phase flags of each request ("Chunked Prefill：query 很长，但仍只是一段区间" and
    "第四步：只在必要位置计算 logits" on the GPUModelRunner page).

    is_prefilling[i]: the request has not yet computed its whole prompt before this step
    (num_computed < num_prompt) — the page's rule, not "query length 1 means decode".
    discard_request_mask[i]: this step's chunk still stops inside the prompt
    (num_computed + num_scheduled < num_prompt), so the token sampled from its last position is
    not an output.  Reading: a padded request is not prefilling and its logits are discarded.
    """
    R = len(num_scheduled)
    R_pad = R if num_reqs_padded is None else int(num_reqs_padded)
    prefilling, discard = [], []
    for i in range(R):
        c, q, p = int(num_computed[i]), int(num_scheduled[i]), int(num_prompt[i])
        prefilling.append(1 if c < p else 0)
        discard.append(1 if c + q < p else 0)
    prefilling += [0] * (R_pad - R)
    discard += [1] * (R_pad - R)
    return dict(is_prefilling=np.array(prefilling, np.int64),
                discard_request_mask=np.array(discard, np.int64))


def pad_for_graph(capture_sizes: Sequence[int], num_tokens: int) -> int:
    """Smallest captured size >= num_tokens; num_tokens itself above the largest (eager).

    "8.5.0.5 pad_for_cudagraph 的实现：二分查找最接近的上界" (bisect_left over the sorted
    sizes) and "8.5 pad_for_cudagraph" (beyond the largest size the runner stays eager).
    """
    sizes = sorted(int(s) for s in capture_sizes)
    if not sizes or num_tokens > sizes[-1]:
        return int(num_tokens)
    return sizes[bisect.bisect_left(sizes, num_tokens)]


def padded_layout_tokens(query_lens: Sequence[int]) -> int:
    """Tokens a rectangular [batch, max_len] layout computes ("为什么不填充")."""
    return len(query_lens) * max(query_lens)
