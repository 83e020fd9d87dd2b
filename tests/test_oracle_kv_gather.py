"""Pins of the KV-write and row-gather oracles."""
import numpy as np

import oracle
from conftest import load_golden


def test_kv_write_runner_example():
    """'3. 物理 KV 槽位': the six new rows land in slots 9, 20, 21, 22, 16, 17 and nothing else moves."""
    slots = load_golden("runner_flatten_example.json")["expected"]["slot_mapping"]
    rng = np.random.default_rng(0)
    kc = rng.integers(0, 2**16, (6 * 4, 2, 8), dtype=np.uint16)   # 6 pages of 4 slots
    vc = rng.integers(0, 2**16, (6 * 4, 2, 8), dtype=np.uint16)
    k = rng.integers(0, 2**16, (6, 2, 8), dtype=np.uint16)
    v = rng.integers(0, 2**16, (6, 2, 8), dtype=np.uint16)
    k2, v2 = oracle.kv_write(kc, vc, slots, k, v)
    for t, s in enumerate(slots):
        assert np.array_equal(k2[s], k[t]) and np.array_equal(v2[s], v[t])
    untouched = [s for s in range(24) if s not in slots]
    assert np.array_equal(k2[untouched], kc[untouched])
    assert np.array_equal(v2[untouched], vc[untouched])
    assert np.array_equal(kc, kc.copy())  # inputs not modified


def test_kv_write_skips_negative_slots():
    """nano-vLLM marks graph-padding slots with -1 and the store skips them."""
    kc = np.zeros((8, 1, 2)); vc = np.zeros((8, 1, 2))
    k = np.ones((3, 1, 2)); v = 2 * np.ones((3, 1, 2))
    k2, v2 = oracle.kv_write(kc, vc, [3, -1, 5], k, v)
    assert k2[3].sum() == 2 and k2[5].sum() == 2 and k2.sum() == 4
    assert v2.sum() == 8


def test_gather_rows_picks_last_tokens():
    """'5. logits 选择与丢弃': rows 0, 3, 5 of the six-token example."""
    idx = load_golden("runner_flatten_example.json")["expected"]["logits_indices"]
    hidden = np.arange(6 * 3, dtype=np.float64).reshape(6, 3)
    out = oracle.gather_rows(hidden, idx)
    assert out[:, 0].tolist() == [0.0, 9.0, 15.0]
