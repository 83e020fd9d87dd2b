"""Pins of the metadata oracle against the pages' worked examples, invariants and brute force."""
import itertools

import numpy as np
import pytest

import oracle
import workloads as wl
from conftest import load_golden


def _tables(num_computed, num_scheduled, block_size, block_rows=None, token_rows=None,
            max_len=None):
    """Token table and page table for a batch; pages default to distinct ids 1, 2, 3, ..."""
    R = len(num_scheduled)
    lens = [c + q for c, q in zip(num_computed, num_scheduled)]
    M = max_len or (max(lens) + block_size)
    MB = -(-M // block_size)
    tok = np.zeros((R, M), np.int64)
    for i in range(R):
        tok[i, :] = 1000 * (i + 1) + np.arange(M)
    if token_rows is not None:
        for i, (base, n) in enumerate(token_rows):
            tok[i, :n] = base + np.arange(n)
    bt = np.full((R, MB), -1, np.int64)
    if block_rows is not None:
        for i, row in enumerate(block_rows):
            bt[i, :len(row)] = row
    else:
        nxt = 1
        for i in range(R):
            n = -(-lens[i] // block_size)
            bt[i, :n] = np.arange(nxt, nxt + n)
            nxt += n
    return tok, bt


def _run(num_computed, num_scheduled, block_size=16, **kw):
    tok, bt = _tables(num_computed, num_scheduled, block_size, kw.pop("block_rows", None),
                      kw.pop("token_rows", None))
    return oracle.prepare_inputs(block_size=block_size, null_block=0, token_table=tok,
                                 block_table=bt, num_computed=num_computed,
                                 num_scheduled=num_scheduled, **kw)


def test_runner_flatten_example():
    g = load_golden("runner_flatten_example.json")
    i, e = g["inputs"], g["expected"]
    out = _run(i["num_computed"], i["num_scheduled"], i["block_size"], block_rows=i["block_table"],
               token_rows=i["token_rows"])
    for key in ("query_start_loc", "input_ids", "positions", "seq_lens", "slot_mapping",
                "visible_keys", "logits_indices"):
        assert out[key].tolist() == e[key], key
    ri, qp = oracle.req_indices_and_query_pos(i["num_scheduled"])
    assert ri.tolist() == e["req_indices"] and qp.tolist() == e["query_pos"]


def test_runner_cumsum_example():
    g = load_golden("runner_cumsum_example.json")
    q = g["inputs"]["num_scheduled"]
    out = _run([0] * len(q), q)
    ri, qp = oracle.req_indices_and_query_pos(q)
    assert out["query_start_loc"].tolist() == g["expected"]["query_start_loc"]
    assert out["logits_indices"].tolist() == g["expected"]["logits_indices"]
    assert ri.tolist() == g["expected"]["req_indices"]
    assert qp.tolist() == g["expected"]["query_pos"]


def test_book_logits_example():
    g = load_golden("book_logits_example.json")
    q = g["inputs"]["num_scheduled"]
    out = _run([3] * len(q), q)
    assert out["query_start_loc"].tolist() == g["expected"]["query_start_loc"]
    assert out["logits_indices"].tolist() == g["expected"]["logits_indices"]


@pytest.mark.parametrize("name", ["batch_layout_abc.json", "batch_layout_step2.json",
                                  "runner_debug_example.json", "batch_layout_exercise.json"])
def test_layout_examples(name):
    g = load_golden(name)
    i, e = g["inputs"], g["expected"]
    out = _run(i["num_computed"], i["num_scheduled"])
    assert out["query_start_loc"].tolist() == e["query_start_loc"]
    assert out["seq_lens"].tolist() == e["seq_lens"]
    assert out["positions"].tolist() == e["positions"]
    if "logits_indices" in e:
        assert out["logits_indices"].tolist() == e["logits_indices"]
    if "num_tokens" in e:
        assert out["num_actual_tokens"] == e["num_tokens"]
    if "logits_indices_needed" in e:
        # the exercise's answer keeps only requests whose prompt is complete after this step
        done = [c + q >= p for c, q, p in zip(i["num_computed"], i["num_scheduled"], i["num_prompt"])]
        kept = [int(x) for x, d in zip(out["logits_indices"], done) if d]
        assert kept == e["logits_indices_needed"]


def test_nano_slot_ranges():
    g = load_golden("nano_slot_ranges.json")
    i, e = g["inputs"], g["expected"]
    start, end, B = i["start"], i["end"], i["block_size"]
    out = _run([start], [end - start], B, block_rows=[i["block_table"]])
    slots = out["slot_mapping"].tolist()
    assert slots == e["slot_mapping"] and len(slots) == e["num_slots"]
    # the page's per-page ranges: runs of slots that share a physical page
    ranges = []
    for s in slots:
        if ranges and s // B == (ranges[-1][1] - 1) // B and s == ranges[-1][1]:
            ranges[-1][1] = s + 1
        else:
            ranges.append([s, s + 1])
    assert ranges == e["ranges"]


def test_padding_waste():
    g = load_golden("padding_waste.json")
    i, e = g["inputs"], g["expected"]
    ql = i["query_lens"]
    assert oracle.padded_layout_tokens(ql) == e["padded_tokens"]
    assert sum(ql) == e["real_tokens"]
    assert round(100 * (1 - sum(ql) / e["padded_tokens"])) == e["waste_percent"]
    for n, padded, waste in e["graph_padding"]:
        got = oracle.pad_for_graph(i["capture_sizes"], n)
        assert got == padded
        assert round(100 * (got - n) / got) == waste
    # beyond the largest captured size the runner stays eager (no padding)
    assert oracle.pad_for_graph(i["capture_sizes"], 257) == 257
    assert oracle.pad_for_graph(i["capture_sizes"], 256) == 256


def _check_invariants(num_computed, num_scheduled, B, out, bt, R_pad=None, N_pad=None,
                      null_block=0):
    """Invariants 3-7 of '八条必须成立的不变量' plus the null-page routing of padding."""
    R = len(num_scheduled)
    N = sum(num_scheduled)
    qsl = out["query_start_loc"]
    assert qsl[0] == 0 and np.all(np.diff(qsl) >= 0) and qsl[R] == N          # 3, 4
    assert out["num_actual_tokens"] == N
    for i in range(R):
        c, q = num_computed[i], num_scheduled[i]
        s = qsl[i]
        pos = out["positions"][s:s + q]
        assert pos.tolist() == list(range(c, c + q))                            # 5
        L = out["seq_lens"][i]
        pages = [int(x) for x in bt[i] if x >= 0]
        assert pos[-1] + 1 <= L <= len(pages) * B                               # 6
        sl = out["slot_mapping"][s:s + q]
        assert all(int(x) // B in pages for x in sl)                             # 7
        assert len(set(sl.tolist())) == q
        assert all(int(x) % B == int(p) % B for x, p in zip(sl, pos))
        if q == 1:
            # nano-vLLM prepare_decode: last page * B + tokens in the last page - 1
            n_pages = -(-int(L) // B)
            last_block_tokens = int(L) - (n_pages - 1) * B
            assert sl[0] == bt[i, n_pages - 1] * B + last_block_tokens - 1
        # nano-vLLM prepare_prefill: per-page slot ranges from start to end
        start, end = c, c + q
        ref = []
        for blk in range(start // B, (end + B - 1) // B):
            lo = bt[i, blk] * B + (start % B if blk == start // B else 0)
            hi = bt[i, blk] * B + (B if blk != (end + B - 1) // B - 1 else end - blk * B)
            ref.extend(range(int(lo), int(hi)))
        assert sl.tolist() == ref
    if N_pad is not None:
        pad = out["slot_mapping"][N:N_pad]
        assert all(int(x) // B == null_block for x in pad)
        assert out["positions"][N:N_pad].tolist() == [0] * (N_pad - N)
    if R_pad is not None:
        assert qsl[R:].tolist() == [N] * (R_pad - R + 1)
        assert out["seq_lens"][R:].tolist() == [0] * (R_pad - R)


@pytest.mark.parametrize("B", [1, 2, 4, 16])
def test_brute_force_small_batches(B):
    """Every batch with R <= 2, q in 1..4, c in 0..7 (plus padding) keeps the invariants."""
    qs, cs = range(1, 5), range(0, 8)
    for R in (1, 2):
        for q in itertools.product(qs, repeat=R):
            for c in itertools.product(cs, repeat=R):
                tok, bt = _tables(list(c), list(q), B)
                out = oracle.prepare_inputs(block_size=B, null_block=0, token_table=tok,
                                            block_table=bt, num_computed=list(c),
                                            num_scheduled=list(q), num_reqs_padded=R + 1,
                                            num_tokens_padded=sum(q) + 3)
                _check_invariants(list(c), list(q), B, out, bt, R_pad=R + 1, N_pad=sum(q) + 3)
                ri, qp = oracle.req_indices_and_query_pos(q)
                # the vectorised form on '8.3.1.6': repeat(arange(R), q), arange - repeat(cu - q, q)
                cu = np.cumsum(q)
                assert ri.tolist() == np.repeat(np.arange(R), q).tolist()
                assert qp.tolist() == (np.arange(cu[-1]) - np.repeat(cu - np.array(q), q)).tolist()
                assert out["input_ids"][:sum(q)].tolist() == [
                    1000 * (i + 1) + c[i] + j for i in range(R) for j in range(q[i])]


def test_random_three_request_batches():
    rng = np.random.default_rng(7)
    for _ in range(400):
        R = 3
        q = [int(x) for x in rng.integers(1, 20, R)]
        c = [int(x) for x in rng.integers(0, 60, R)]
        B = int(rng.choice([2, 4, 8, 16]))
        tok, bt = _tables(c, q, B)
        perm = rng.permutation(np.arange(1, bt.max() + 1))
        bt = np.where(bt >= 0, perm[np.maximum(bt, 1) - 1], -1)   # random physical ids
        out = oracle.prepare_inputs(block_size=B, null_block=0, token_table=tok, block_table=bt,
                                    num_computed=c, num_scheduled=q)
        _check_invariants(c, q, B, out, bt)


def test_request_flags_debug_example():
    """'最小可复现实验': the page prints discard=[False, True] for A (decode) and B (chunk)."""
    g = load_golden("runner_debug_example.json")
    i, e = g["inputs"], g["expected"]
    out = _run(i["num_computed"], i["num_scheduled"], num_prompt=i["num_prompt"])
    assert out["discard_request_mask"].astype(bool).tolist() == e["discard_request_mask"]
    assert out["is_prefilling"].astype(bool).tolist() == e["is_prefilling"]


def test_request_flags_exercise_answer():
    """'练习' 1: request 3 stops at 20 of its 40 prompt tokens, so its logits are not sampled; the
    answer keeps logits only where the discard mask is clear."""
    g = load_golden("batch_layout_exercise.json")
    i, e = g["inputs"], g["expected"]
    out = _run(i["num_computed"], i["num_scheduled"], num_prompt=i["num_prompt"])
    assert out["discard_request_mask"].astype(bool).tolist() == e["discard_request_mask"]
    kept = [int(x) for x, d in zip(out["logits_indices"], out["discard_request_mask"]) if not d]
    assert kept == e["logits_indices_needed"]


def test_one_token_query_can_still_be_prefilling():
    """'Chunked Prefill' section: a short query does not mean decode; the phase comes from
    num_computed against num_prompt."""
    flags = oracle.request_flags([5, 9, 12, 0], [1, 1, 1, 4], [9, 9, 12, 2], num_reqs_padded=6)
    assert flags["is_prefilling"].tolist() == [1, 0, 0, 1, 0, 0]
    assert flags["discard_request_mask"].tolist() == [1, 0, 0, 0, 1, 1]


def test_manager_to_kernel_blocks_page_example():
    """"混合 KV Cache：一条请求不止一张页表": 32-token manager blocks over 16-token kernel pages,
    manager ids [0, 1, 2] become kernel ids [0, 1, 2, 3, 4, 5]."""
    assert oracle.map_to_kernel_blocks([0, 1, 2], 2) == [0, 1, 2, 3, 4, 5]
    assert oracle.map_to_kernel_blocks([7, 3], 1) == [7, 3]
    assert oracle.map_to_kernel_blocks([], 4) == []


@pytest.mark.parametrize("ratio", [2, 4])
@pytest.mark.parametrize("seed", range(6))
def test_manager_table_slots_equal_one_big_page(ratio, seed):
    """Closed form: manager block m is r consecutive kernel pages, i.e. r*B consecutive slots,
    so the slot of position p is m * (r*B) + p % (r*B) with m = table[i, p // (r*B)]."""
    spec = wl.random_batch(seed, block_size=8, manager_ratio=ratio, max_q=50, max_c=120)
    d = spec.dims
    got = oracle.prepare_inputs(block_size=d.block_size, null_block=d.null_block,
                                token_table=spec.token_table, block_table=spec.block_table,
                                num_computed=spec.num_computed, num_scheduled=spec.num_scheduled,
                                kernel_blocks_per_manager_block=ratio)
    big = ratio * d.block_size
    want = []
    for i, (c, q) in enumerate(zip(spec.num_computed, spec.num_scheduled)):
        for j in range(int(q)):
            p = int(c) + j
            want.append(int(spec.block_table[i, p // big]) * big + p % big)
    assert got["slot_mapping"].tolist() == want
    # every real slot lies in a manager block the request owns, never in the null one
    for s in want:
        assert s // big != d.null_block // ratio


def test_batch_maxima_on_worked_examples():
    """max_query_len / max_seq_len (the scalars the attention metadata carries, nano-vLLM's
    max_seqlen_q / max_seqlen_k) on the printed examples: A/B/C of '布局与元数据' has query
    lengths 7, 1, 12 and sequence lengths 7, 6, 22, so 12 and 22 (both from C); the runner's
    example of '2. 模型位置与完整序列长度' has query lengths 1, 3, 2 and sequence lengths 6, 3, 10,
    so 3 (from B) and 10 (from C) -- a maximum over num_computed would give 8 there."""
    g = load_golden("batch_layout_abc.json")
    out = _run(g["inputs"]["num_computed"], g["inputs"]["num_scheduled"], num_reqs_padded=5,
               num_tokens_padded=24)
    assert (out["max_query_len"], out["max_seq_len"]) == (12, 22)
    g = load_golden("runner_flatten_example.json")
    i = g["inputs"]
    out = _run(i["num_computed"], i["num_scheduled"], i["block_size"],
               block_rows=i["block_table"], token_rows=i["token_rows"], num_reqs_padded=4)
    assert (out["max_query_len"], out["max_seq_len"]) == (3, 10)
    # nano-vLLM's flattening example (question 8): Seq_0 4 tokens, Seq_1 6 tokens -> max q 6;
    # scheduled again with 4 cached and 4 new -> seqlen_k 8
    out = _run([0, 0], [4, 6])
    assert (out["max_query_len"], out["max_seq_len"]) == (6, 6)
    out = _run([4], [4])
    assert (out["max_query_len"], out["max_seq_len"]) == (4, 8)
    # padded requests (q = 0, seq_len 0) never raise either maximum
    out = _run([100, 3], [1, 2], num_reqs_padded=8, num_tokens_padded=16)
    assert (out["max_query_len"], out["max_seq_len"]) == (2, 101)
