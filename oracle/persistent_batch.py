"""Row operations of the persistent batch, as plain Python lists (oracle; test infrastructure).

The runner keeps one row per resident request in column arrays (token history, counters, page
table) and merges each step's scheduler deltas into them before it flattens the step.  This
module restates that merge with one Python dict per row; nothing is vectorised.

Sources (page title, then section):

* "vLLM 源码完全拆解（五）：GPUModelRunner 如何把动态请求拼成一次 GPU 前向"
  - "行号是一种短生命周期地址": a row is only an address in the current layout; a finished
    request's row may be reused by a new request; condense() moves tail rows into the holes,
    and a move carries every column of the row (example: rows A B C D, B finishes, D moves
    to row 1, giving A D C);
  - "为什么删除后还要压紧": after the update the live rows are the prefix [0, num_reqs);
  - "先删除完成和本轮未调度的请求": finished requests and requests not scheduled this step
    leave the batch;
  - "新请求建立完整状态": a new request brings its full prompt history, its initial page ids
    and its num_computed (prefix hits included);
  - "驻留请求只合并差量": a resident request only sets num_computed and appends its new page
    ids to its row; a request resumed from preemption replaces its page row instead;
  - "最后压紧并刷新派生 metadata": condense runs after every removal and addition, and the
    step is flattened only from the settled layout.
* "第8章 ModelRunner：从 SchedulerOutput 到 GPU Kernel"
  - "8.2.2 三种变更操作": new requests take a free row; a continuing request appends its new
    tokens to its row; a finished request's row is marked free and its data is not cleared;
  - "8.2.2.5 _update_states 的真实四段执行": removals come first, then new requests fill
    the rows the removals freed;
  - "8.2.2.6 \"aborted 后相同 ID resubmit\" 的边界处理": an id that is both finished and
    newly scheduled names two distinct requests: the old state is dropped and the new
    request is installed from scratch.
* "04 · 模型执行与 CUDA Graph", "4.2 块表：BlockTable": append_row adds the scheduler's new
  page ids to the used part of a request's page-table row.

Readings where the pages are silent (each is also a test in tests/test_oracle_batch.py):

* the rows a step keeps are those whose request is scheduled this step and is not announced
  again as new (the abort-and-resubmit case drops the old row);
* new requests, in the order given, take the freed rows in ascending order, then the rows
  after the old end of the batch;
* condense pairs the lowest remaining hole with the highest live row, the next lowest with the
  next highest, and stops when no live row lies above a hole;
* a continuing request's new tokens are appended after its current history length; a request
  resumed from preemption with its row still resident replaces its page row (a request that
  left the batch comes back as a new request with its full history);
* contents past a row's history length or page count, and of rows past the batch end, are
  unspecified: only the valid prefixes are state;
* request ids are non-negative integer handles (the pages use strings; -1 marks a free row).
"""
from __future__ import annotations

from typing import Dict, List, Optional

import numpy as np


class InputBatch:
    """Rows of resident requests; ``rows[r]`` is a dict of that row's columns or None (a hole)."""

    def __init__(self, max_num_reqs: int, max_model_len: int, max_blocks_per_req: int):
        self.max_num_reqs = int(max_num_reqs)
        self.max_model_len = int(max_model_len)
        self.max_blocks_per_req = int(max_blocks_per_req)
        self.rows: List[Optional[dict]] = []
        self.moves = 0

    # -- the four stages of one update -------------------------------------------------------
    def apply(self, step) -> List[int]:
        """Merge one step's deltas; returns the row of every scheduled request, in the order of
        ``step.scheduled``.  Raises ValueError for an inconsistent step, leaving the batch as
        it was.

        ``step`` carries ``scheduled`` (dict req_id -> tokens this step), ``new`` (items with
        ``req_id, num_computed, num_prompt, tokens, blocks``: the whole state of a request
        entering the batch) and ``cached`` (items with ``req_id, num_computed, new_tokens,
        new_blocks, replace_blocks``: what a resident request adds).
        """
        rows = [None if r is None else dict(r) for r in self.rows]
        new_ids = [n.req_id for n in step.new]
        if any(int(i) < 0 for i in step.scheduled):
            raise ValueError("request ids are non-negative handles")
        if len(set(new_ids)) != len(new_ids):
            raise ValueError("a request is announced as new twice")
        for n in step.new:
            if n.req_id not in step.scheduled:
                raise ValueError("a new request is not scheduled")

        # 1. removals: finished or unscheduled requests, and the old state of an id that is
        #    announced again as new (abort and resubmit)
        holes = []
        for r, row in enumerate(rows):
            if row is None or row["req_id"] not in step.scheduled or row["req_id"] in new_ids:
                rows[r] = None
                holes.append(r)

        # 2. merge the deltas of resident requests
        index = {row["req_id"]: r for r, row in enumerate(rows) if row is not None}
        seen = set()
        for d in step.cached:
            if d.req_id not in index or d.req_id in seen:
                raise ValueError("a delta names a request that is not resident (or twice)")
            seen.add(d.req_id)
            row = rows[index[d.req_id]]
            row["num_computed"] = int(d.num_computed)
            row["tokens"] = list(row["tokens"]) + [int(t) for t in d.new_tokens]
            if d.replace_blocks:
                row["blocks"] = [int(b) for b in d.new_blocks]
            else:
                row["blocks"] = list(row["blocks"]) + [int(b) for b in d.new_blocks]

        # 3. new requests fill the freed rows, lowest first, then extend the batch
        for k, n in enumerate(step.new):
            state = dict(req_id=int(n.req_id), num_computed=int(n.num_computed),
                         num_prompt=int(n.num_prompt), tokens=[int(t) for t in n.tokens],
                         blocks=[int(b) for b in n.blocks])
            if k < len(holes):
                rows[holes[k]] = state
            else:
                rows.append(state)
        holes = holes[len(step.new):]

        # 4. condense: the highest live row moves into the lowest remaining hole
        moves = 0
        while holes:
            while rows and rows[-1] is None:
                rows.pop()
            holes = [h for h in holes if h < len(rows)]
            if not holes:
                break
            h = holes.pop(0)
            rows[h] = rows.pop()
            moves += 1

        for row in rows:
            if row is None:
                raise AssertionError("condense left a hole")
            if len(row["tokens"]) > self.max_model_len:
                raise ValueError("token history longer than max_model_len")
            if len(row["blocks"]) > self.max_blocks_per_req:
                raise ValueError("page row longer than max_blocks_per_req")
        if len(rows) > self.max_num_reqs:
            raise ValueError("more resident requests than rows")
        index = {row["req_id"]: r for r, row in enumerate(rows)}
        if set(index) != set(step.scheduled):
            raise ValueError("a scheduled request is neither resident nor new")
        self.rows = rows
        self.moves += moves
        return [index[i] for i in step.scheduled]

    # -- column views ------------------------------------------------------------------------
    @property
    def num_reqs(self) -> int:
        return len(self.rows)

    def columns(self, num_scheduled: Optional[Dict[int, int]] = None) -> Dict[str, np.ndarray]:
        """Row-order arrays of the live rows: ``req_id``, ``num_tokens``, ``num_prompt``,
        ``num_computed``, ``num_blocks`` and, given this step's schedule, ``num_scheduled``;
        the token and page rows as lists (their valid prefixes only)."""
        out = dict(
            req_id=np.array([r["req_id"] for r in self.rows], np.int64),
            num_tokens=np.array([len(r["tokens"]) for r in self.rows], np.int64),
            num_prompt=np.array([r["num_prompt"] for r in self.rows], np.int64),
            num_computed=np.array([r["num_computed"] for r in self.rows], np.int64),
            num_blocks=np.array([len(r["blocks"]) for r in self.rows], np.int64),
            tokens=[list(r["tokens"]) for r in self.rows],
            blocks=[list(r["blocks"]) for r in self.rows],
        )
        if num_scheduled is not None:
            out["num_scheduled"] = np.array([num_scheduled[r["req_id"]] for r in self.rows],
                                            np.int64)
        return out

    def tables(self, pad_token: int = 0, pad_block: int = -1):
        """Dense [max_num_reqs, max_model_len] token table and page table of the live rows,
        padded with ``pad_token`` / ``pad_block`` (the padding is not state)."""
        tok = np.full((self.max_num_reqs, self.max_model_len), pad_token, np.int32)
        blk = np.full((self.max_num_reqs, self.max_blocks_per_req), pad_block, np.int32)
        for r, row in enumerate(self.rows):
            tok[r, :len(row["tokens"])] = row["tokens"]
            blk[r, :len(row["blocks"])] = row["blocks"]
        return tok, blk
