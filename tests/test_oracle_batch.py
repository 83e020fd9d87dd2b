"""Pins of the persistent-batch oracle (oracle.persistent_batch.InputBatch).

Each test fixes the row rule to something outside the oracle's own code: the pages' printed
example, their stated reuse and ordering rules, or a request-keyed dictionary model in which
rows do not exist at all (so a wrong move, a dropped column or a stale row shows as a
difference in some request's state).
"""
import numpy as np
import pytest

import workloads as wl
from oracle.persistent_batch import InputBatch

A, B, C, D, E = 10, 11, 12, 13, 14


def new(i, tokens=(1, 2, 3), blocks=(5,), computed=0, prompt=None):
    return wl.NewRequest(i, computed, len(tokens) if prompt is None else prompt,
                         np.array(tokens, np.int32), np.array(blocks, np.int32))


def delta(i, computed, tokens=(), blocks=(), replace=False):
    return wl.CachedDelta(i, computed, np.array(tokens, np.int32), np.array(blocks, np.int32),
                          replace_blocks=replace)


def step(sched, new_=(), cached=()):
    return wl.SchedulerStep(scheduled=dict(sched), new=list(new_), cached=list(cached))


def ids(batch):
    return [r["req_id"] for r in batch.rows]


def abcd():
    b = InputBatch(8, 64, 8)
    b.apply(step({A: 3, B: 3, C: 3, D: 3},
                 [new(A, (1,)), new(B, (2, 2)), new(C, (3, 3, 3)), new(D, (4, 4, 4, 4))]))
    return b


def test_page_example_condense_moves_d_into_bs_row():
    """"行号是一种短生命周期地址": rows A B C D; B finishes; condense moves D to row 1."""
    b = abcd()
    assert ids(b) == [A, B, C, D]
    rows = b.apply(step({A: 1, C: 1, D: 1}))
    assert ids(b) == [A, D, C]
    assert rows == [0, 2, 1]
    assert b.moves == 1
    # the move carried D's whole state, not only its id
    assert b.rows[1]["tokens"] == [4, 4, 4, 4]


def test_new_request_reuses_the_freed_row():
    """"该行可能被新请求复用" and "8.2.2.5": the new request fills B's row; nothing moves."""
    b = abcd()
    b.apply(step({A: 1, C: 1, D: 1, E: 5}, [new(E, (9, 9))]))
    assert ids(b) == [A, E, C, D]
    assert b.moves == 0
    assert b.rows[1]["tokens"] == [9, 9]


def test_new_requests_take_lowest_holes_then_the_tail():
    b = abcd()
    b.apply(step({B: 1, E: 1, 20: 1, 21: 1, 22: 1},
                 [new(E), new(20), new(21), new(22)]))  # A, C, D leave
    assert ids(b) == [E, B, 20, 21, 22]


def test_unscheduled_request_leaves_the_batch():
    """"先删除完成和本轮未调度的请求": a request the scheduler skipped is removed too."""
    b = abcd()
    b.apply(step({A: 1, B: 1, D: 1}))  # C neither finished nor scheduled
    assert ids(b) == [A, B, D]


def test_abort_and_resubmit_is_a_new_request():
    """"8.2.2.6": an id scheduled as new while resident names a new request."""
    b = abcd()
    b.apply(step({A: 1, B: 1, C: 1, D: 1}, [new(B, (7,), (40, 41), prompt=1)]))
    row = b.rows[ids(b).index(B)]
    assert row["tokens"] == [7] and row["blocks"] == [40, 41] and row["num_prompt"] == 1


def test_delta_sets_computed_and_appends():
    """"驻留请求只合并差量" and "4.2 块表" (append_row)."""
    b = abcd()
    b.apply(step({A: 1, B: 1, C: 1, D: 1}, cached=[delta(C, 3, (8,), (6, 7))]))
    row = b.rows[2]
    assert row["num_computed"] == 3
    assert row["tokens"] == [3, 3, 3, 8]
    assert row["blocks"] == [5, 6, 7]


def test_resumed_request_replaces_its_page_row():
    """"驻留请求只合并差量": a request resumed from preemption must not append to stale ids."""
    b = abcd()
    b.apply(step({A: 1, B: 1, C: 1, D: 1}, cached=[delta(C, 3, (), (30, 31), replace=True)]))
    assert b.rows[2]["blocks"] == [30, 31]


def test_condense_pairs_lowest_hole_with_highest_row():
    b = InputBatch(16, 8, 2)
    b.apply(step({i: 1 for i in range(10)}, [new(i, (i,)) for i in range(10)]))
    b.apply(step({i: 1 for i in (0, 3, 5, 8, 9)}))  # holes 1 2 4 6 7: 9 -> 1, 8 -> 2, 5 -> 4
    assert ids(b) == [0, 9, 8, 3, 5]
    assert b.moves == 3


def test_inconsistent_steps_raise_and_leave_the_batch():
    b = abcd()
    before = [dict(r) for r in b.rows]
    bad = [
        step({A: 1, 99: 1}),                                  # scheduled, neither resident nor new
        step({A: 1}, cached=[delta(B, 1)]),                   # delta for a request that leaves
        step({A: 1}, [new(E)]),                               # new but not scheduled
        step({A: 1, E: 1}, [new(E), new(E)]),                 # new twice
        step({A: 1}, cached=[delta(A, 1, tokens=[0] * 70)]),  # history past max_model_len
        step({A: 1}, cached=[delta(A, 1, blocks=[1] * 8)]),   # page row past max_blocks_per_req
    ]
    for s in bad:
        with pytest.raises(ValueError):
            b.apply(s)
        assert b.rows == before


class DictModel:
    """The same deltas applied to a dict keyed by request id (no rows anywhere)."""

    def __init__(self):
        self.state = {}

    def apply(self, s):
        new_ids = {n.req_id for n in s.new}
        self.state = {i: v for i, v in self.state.items() if i in s.scheduled and i not in new_ids}
        for d in s.cached:
            v = self.state[d.req_id]
            v["num_computed"] = int(d.num_computed)
            v["tokens"] = v["tokens"] + [int(t) for t in d.new_tokens]
            v["blocks"] = ([int(x) for x in d.new_blocks] if d.replace_blocks
                           else v["blocks"] + [int(x) for x in d.new_blocks])
        for n in s.new:
            self.state[n.req_id] = dict(num_computed=int(n.num_computed),
                                        num_prompt=int(n.num_prompt),
                                        tokens=[int(t) for t in n.tokens],
                                        blocks=[int(x) for x in n.blocks])


@pytest.mark.parametrize("seed", range(12))
def test_rows_are_a_compact_permutation_of_the_request_state(seed):
    """Brute force over random request streams: the batch, read by request id, equals the
    row-free model; rows [0, S) are exactly the scheduled requests; a live row below the new
    end never moves; the number of moves is the number of live rows at or past the new end."""
    stream = wl.RandomRequestStream(seed, max_live=12, max_model_len=64, max_blocks=8)
    b, model = InputBatch(stream.max_rows, 64, 8), DictModel()
    for _ in range(40):
        s = stream.next_step()
        prev_ids, moves0 = ids(b), b.moves
        rows = b.apply(s)
        model.apply(s)
        assert sorted(ids(b)) == sorted(s.scheduled) and len(ids(b)) == len(s.scheduled)
        assert rows == [ids(b).index(i) for i in s.scheduled]
        for r in b.rows:
            v = model.state[r["req_id"]]
            assert (r["num_computed"], r["num_prompt"], r["tokens"], r["blocks"]) == \
                (v["num_computed"], v["num_prompt"], v["tokens"], v["blocks"])
        F = len(s.scheduled)
        new_ids = {n.req_id for n in s.new}
        kept = {i: r for r, i in enumerate(prev_ids) if i in s.scheduled and i not in new_ids}
        for i, r in kept.items():
            if r < F:
                assert ids(b)[r] == i
        assert b.moves - moves0 == sum(1 for r in kept.values() if r >= F)


def test_chunked_prefill_stream_exercises_every_path():
    """The 8192-token mix reaches holes, tail appends, condense moves, replaced page rows and
    requests that come back after preemption."""
    st = wl.MixedChunkStream()
    b = InputBatch(160, 65536, 4096)
    seen_replace = seen_resumed = 0
    left = set()
    for _ in range(60):
        s = st.next_step()
        seen_replace += sum(1 for d in s.cached if d.replace_blocks)
        seen_resumed += sum(1 for n in s.new if n.req_id in left)
        left |= {i for i in ids(b) if i not in s.scheduled}
        b.apply(s)
        assert s.num_tokens <= st.BUDGET
    assert b.moves > 0 and seen_replace > 0 and seen_resumed > 0
