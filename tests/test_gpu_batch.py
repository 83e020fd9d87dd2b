"""rb_batch_apply_update vs the oracle's persistent batch: bit-exact row state every step."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_cases import config4_layouts, dims_of, oracle_meta, spec_of_layout
from oracle.persistent_batch import InputBatch

pytestmark = pytest.mark.gpu


def assert_same(dev, ref: InputBatch, step=None, check_tokens=True):
    snap = dev.snapshot()
    cols = ref.columns(None if step is None else step.scheduled)
    R = ref.num_reqs
    assert snap["num_rows"] == R
    for k in ("req_id", "num_tokens", "num_prompt", "num_computed", "num_blocks"):
        assert np.array_equal(snap[k].astype(np.int64), cols[k]), k
    if step is not None:
        assert np.array_equal(snap["num_scheduled"][:R], cols["num_scheduled"])
        assert not snap["num_scheduled"][R:].any()
        rows = dev.row_of_sched[:R].cpu().numpy()
        want = [int(np.nonzero(cols["req_id"] == i)[0][0]) for i in step.scheduled]
        assert rows.tolist() == want
    for r in range(R):
        assert snap["blocks"][r].tolist() == cols["blocks"][r], f"page row {r}"
        if check_tokens:
            assert snap["tokens"][r].tolist() == cols["tokens"][r], f"token row {r}"


def make(max_rows, M, MB):
    import ragged_mixed_paged_gb300 as rb

    return rb.PersistentBatch(max_rows, M, MB), InputBatch(max_rows, M, MB)


def apply_both(dev, ref, step):
    dev.apply(step)
    ref.apply(step)
    torch.cuda.synchronize()
    assert int(dev.error_word.item()) == 0


def test_page_example_on_device():
    """A B C D; B finishes; D moves into row 1 with all of its columns."""
    dev, ref = make(8, 64, 8)
    s0 = wl.SchedulerStep({10: 1, 11: 1, 12: 1, 13: 1}, [
        wl.NewRequest(10 + i, i, 4, np.full(i + 1, i, np.int32), np.array([i + 1], np.int32))
        for i in range(4)])
    apply_both(dev, ref, s0)
    s1 = wl.SchedulerStep({10: 1, 12: 1, 13: 1})
    apply_both(dev, ref, s1)
    assert dev.req_id[:3].tolist() == [10, 13, 12]
    assert_same(dev, ref, s1)


@pytest.mark.parametrize("seed", range(16))
def test_random_streams_bit_exact(seed):
    stream = wl.RandomRequestStream(seed, max_live=12 + seed, max_model_len=64, max_blocks=8)
    dev, ref = make(stream.max_rows, 64, 8)
    for _ in range(40):
        s = stream.next_step()
        apply_both(dev, ref, s)
        assert_same(dev, ref, s)


def test_chunked_prefill_stream_bit_exact():
    """60 steps of the 8192-token mix (132 rows, histories up to 64K tokens)."""
    import ragged_mixed_paged_gb300 as rb

    d = wl.MixedChunkStream().dims
    dev = rb.PersistentBatch(d.max_num_reqs, d.max_model_len, d.max_blocks_per_req)
    for s, step, ref in config4_layouts(60):
        dev.apply(step)
        torch.cuda.synchronize()
        assert int(dev.error_word.item()) == 0
        assert_same(dev, ref, step, check_tokens=(s % 5 == 0 or s < 3))


def test_device_layout_feeds_prepare_inputs():
    """The device batch after each update is a valid rb_prepare_inputs input: metadata equals
    the oracle's, computed on the oracle's own layout, bit for bit (phase flags included)."""
    import ragged_mixed_paged_gb300 as rb

    d = wl.MixedChunkStream().dims
    dev = rb.PersistentBatch(d.max_num_reqs, d.max_model_len, d.max_blocks_per_req)
    for s, step, ref in config4_layouts(25):
        dev.apply(step)
        spec = spec_of_layout("mix", d, step, ref, 0)
        t = dev.tables()
        got = rb.prepare_inputs(dims_of(spec), dev.num_reqs, dev.num_reqs, dev.num_tokens_scheduled,
                                dev.num_tokens_scheduled, t["token_table"], t["num_computed"],
                                t["num_scheduled"], t["block_table"], num_prompt=t["num_prompt"])
        torch.cuda.synchronize()
        want = oracle_meta(spec)
        for k in ("input_ids", "positions", "query_start_loc", "seq_lens", "slot_mapping",
                  "logits_indices", "is_prefilling", "discard_request_mask"):
            assert np.array_equal(got[k].cpu().numpy(), want[k]), (s, k)
        assert int(got["scalars"][3].item()) == 0


def test_large_batch_multi_tile_scans():
    """4096 rows (every scan spans four 1024-thread tiles), then every other request leaves and
    2048 rows condense; then the tail refills."""
    dev, ref = make(4096, 32, 4)
    rng = np.random.default_rng(7)
    new = [wl.NewRequest(i, 0, 3, rng.integers(0, 100, size=1 + i % 30).astype(np.int32),
                         rng.integers(1, 99, size=i % 5).astype(np.int32)) for i in range(4096)]
    apply_both(dev, ref, wl.SchedulerStep({i: 1 for i in range(4096)}, new))
    assert_same(dev, ref)
    keep = {i: 1 for i in range(4096) if i % 2 == 0 or i < 100}
    apply_both(dev, ref, wl.SchedulerStep(keep))
    assert_same(dev, ref, wl.SchedulerStep(keep))
    refill = dict(keep)
    more = [wl.NewRequest(10000 + i, 1, 2, np.array([i], np.int32), np.array([i + 1], np.int32))
            for i in range(4096 - len(keep))]
    refill.update({n.req_id: 2 for n in more})
    s = wl.SchedulerStep(refill, more)
    apply_both(dev, ref, s)
    assert_same(dev, ref, s)


def test_empty_and_all_leave():
    dev, ref = make(4, 16, 2)
    apply_both(dev, ref, wl.SchedulerStep({}))
    assert dev.num_rows.item() == 0
    s = wl.SchedulerStep({1: 1, 2: 1}, [wl.NewRequest(i, 0, 1, np.array([i], np.int32),
                                                       np.array([], np.int32)) for i in (1, 2)])
    apply_both(dev, ref, s)
    assert_same(dev, ref, s)
    apply_both(dev, ref, wl.SchedulerStep({}))
    assert dev.num_rows.item() == 0
    assert dev.req_id.tolist()[:2] == [-1, -1]


def _bad_steps():
    def new(i, n=1, nb=1):
        return wl.NewRequest(i, 0, n, np.zeros(n, np.int32), np.ones(nb, np.int32))

    def delta(i, toks=0, blocks=0, replace=False):
        return wl.CachedDelta(i, 1, np.zeros(toks, np.int32), np.ones(blocks, np.int32), replace)

    ID, SIZE = 0x200, 0x400
    return [
        ("unknown scheduled", wl.SchedulerStep({0: 1, 99: 1}), ID),
        ("delta of a leaving request", wl.SchedulerStep({0: 1}, cached=[delta(1)]), ID),
        ("delta of a request not in the batch", wl.SchedulerStep({0: 1, 5: 1}, [new(5)],
                                                                 [delta(6)]), ID),
        ("new not scheduled", wl.SchedulerStep({0: 1}, [new(7)]), ID),
        ("new twice", wl.SchedulerStep({0: 1, 7: 1}, [new(7), new(7)]), ID),
        ("negative id", wl.SchedulerStep({0: 1, -3: 1}, [new(-3)]), ID),
        ("delta twice", wl.SchedulerStep({0: 1, 1: 1}, cached=[delta(0), delta(0)]), ID),
        ("history too long", wl.SchedulerStep({0: 1}, cached=[delta(0, toks=16)]), SIZE),
        ("page row too long", wl.SchedulerStep({0: 1}, cached=[delta(0, blocks=4)]), SIZE),
        ("new history too long", wl.SchedulerStep({0: 1, 8: 1}, [new(8, n=17)]), SIZE),
    ]


@pytest.mark.parametrize("case", range(10))
def test_device_errors_leave_the_batch_unchanged(case):
    name, bad, bit = _bad_steps()[case]
    dev, ref = make(4, 16, 4)
    s = wl.SchedulerStep({0: 1, 1: 1}, [wl.NewRequest(i, 0, 2, np.array([i, i], np.int32),
                                                       np.array([i + 1], np.int32)) for i in (0, 1)])
    apply_both(dev, ref, s)
    before = dev.snapshot()
    dev.apply(bad)
    torch.cuda.synchronize()
    assert int(dev.error_word.item()) & bit, name
    after = dev.snapshot()
    for k in ("num_rows", "req_id", "num_tokens", "num_prompt", "num_computed", "num_blocks"):
        assert np.array_equal(np.asarray(after[k]), np.asarray(before[k])), (name, k)
    for r in range(before["num_rows"]):
        assert after["tokens"][r].tolist() == before["tokens"][r].tolist()
        assert after["blocks"][r].tolist() == before["blocks"][r].tolist()
    with pytest.raises(ValueError):
        ref.apply(bad)
