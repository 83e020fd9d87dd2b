"""rb_prepare_inputs vs the oracle: bit-exact on every workload, fuzzed mixes and edge cases."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_cases import config4_specs, dims_of, i32, oracle_meta

pytestmark = pytest.mark.gpu

KEYS = ("input_ids", "positions", "query_start_loc", "seq_lens", "slot_mapping", "logits_indices")


def _run(rb, spec, num_tokens=None):
    t = wl.device_tables(spec, "cuda")
    out = rb.prepare_inputs(dims_of(spec), spec.num_reqs, spec.num_reqs_padded,
                            spec.num_tokens if num_tokens is None else num_tokens,
                            spec.num_tokens_padded, t["token_table"], t["num_computed"],
                            t["num_scheduled"], t["block_table"], num_prompt=t.get("num_prompt"))
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def _assert_exact(got, spec):
    ref = oracle_meta(spec)
    for k in KEYS:
        assert np.array_equal(got[k], ref[k]), k
    if spec.num_prompt is not None:
        for k in ("is_prefilling", "discard_request_mask"):
            assert np.array_equal(got[k], ref[k]), k
    assert got["scalars"].tolist() == [ref["max_query_len"], ref["max_seq_len"],
                                       ref["num_actual_tokens"], 0]


CASES = {
    "cfg1": lambda: wl.config1(),
    "cfg1_pad24": lambda: wl.config1(num_tokens_padded=24),
    "cfg2": lambda: wl.config2(),
    "cfg3": lambda: wl.config3(),
    "cfg3_pad": lambda: wl.config3(num_real=250),
    "cfg5": lambda: wl.config5(),
    "runner_example_B4": lambda: wl.batch_from_lists([5, 0, 8], [1, 3, 2], block_size=4),
    "nano_example_B8": lambda: wl.batch_from_lists([1], [37], block_size=8),
    "many_decodes": lambda: wl.batch_from_lists([int(x) for x in np.arange(5000) % 300 + 1],
                                                [1] * 5000, block_size=16, seed=3),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_workloads_bit_exact(rb, name):
    spec = CASES[name]()
    _assert_exact(_run(rb, spec), spec)


@pytest.mark.parametrize("step", [0, 1, 57, 99])
def test_chunked_prefill_mix_steps_bit_exact(rb, step):
    spec = config4_specs()[step]
    _assert_exact(_run(rb, spec), spec)


@pytest.mark.parametrize("seed", range(60))
def test_fuzzed_mixes_bit_exact(rb, seed):
    B = [1, 2, 4, 8, 16, 32][seed % 6]
    spec = wl.random_batch(seed, block_size=B, max_reqs=12, max_q=70, max_c=200,
                           pad_tokens=seed % 5, pad_reqs=seed % 3)
    _assert_exact(_run(rb, spec), spec)


def test_phase_flags_page_examples(rb):
    """The debug example prints discard=[False, True]; the exercise drops request 3's logits."""
    from conftest import load_golden

    for name in ("runner_debug_example.json", "batch_layout_exercise.json"):
        g = load_golden(name)
        spec = wl.batch_from_lists(g["inputs"]["num_computed"], g["inputs"]["num_scheduled"])
        spec.num_prompt = np.array(g["inputs"]["num_prompt"], np.int32)
        got = _run(rb, spec)
        assert got["discard_request_mask"].astype(bool).tolist() == \
            g["expected"]["discard_request_mask"]
        _assert_exact(got, spec)


def test_empty_batch(rb):
    spec = wl.batch_from_lists([], [])
    got = _run(rb, spec)
    assert got["query_start_loc"].tolist() == [0]
    assert got["scalars"].tolist() == [0, 0, 0, 0]


def test_all_padding_batch(rb):
    spec = wl.with_padding(wl.batch_from_lists([], [], num_reqs_padded=3), 3, 5)
    got = _run(rb, spec)
    _assert_exact(got, spec)
    assert set((got["slot_mapping"] // 16).tolist()) == {0}


def test_error_bits(rb):
    base = wl.batch_from_lists([3, 0, 9], [2, 4, 1], block_size=4, seed=1)
    # a real request with nothing scheduled
    s = wl.batch_from_lists([3, 0, 9], [2, 0, 1], block_size=4, seed=1)
    assert _run(rb, s)["scalars"][3] & 0x001
    # token count disagrees with the sum of scheduled tokens
    assert _run(rb, wl.with_padding(base, 3, 9), num_tokens=8)["scalars"][3] & 0x008
    # sequence longer than the token table
    s = wl.batch_from_lists([3, 0, 9], [2, 4, 1], block_size=4, seed=1)
    s.num_computed[2] = s.dims.max_model_len
    assert _run(rb, s)["scalars"][3] & 0x004
    # page id outside the pool / the null page in a real row: slot routed to the null page
    for bad in (-1, 0, s.dims.num_blocks):
        s = wl.batch_from_lists([3, 0, 9], [2, 4, 1], block_size=4, seed=1)
        s.block_table[1, 0] = bad
        got = _run(rb, s)
        assert got["scalars"][3] & 0x010
        assert np.all(got["slot_mapping"][2:6] // 4 == 0)
