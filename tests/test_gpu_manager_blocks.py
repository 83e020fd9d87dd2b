"""Page tables of manager blocks ("混合 KV Cache：一条请求不止一张页表"): the slot map and the
attention page walk expand each manager block id into its kernel pages on the fly.  Bit-exact
metadata and oracle-tolerance attention against the oracle, which expands the table first."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_cases import dims_of, i32, oracle_meta
from test_gpu_attention import _case

pytestmark = pytest.mark.gpu

KEYS = ("input_ids", "positions", "query_start_loc", "seq_lens", "slot_mapping", "logits_indices")


def _meta(rb, spec):
    t = wl.device_tables(spec, "cuda")
    out = rb.prepare_inputs(dims_of(spec), spec.num_reqs, spec.num_reqs_padded, spec.num_tokens,
                            spec.num_tokens_padded, t["token_table"], t["num_computed"],
                            t["num_scheduled"], t["block_table"])
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


@pytest.mark.parametrize("ratio", [2, 4])
@pytest.mark.parametrize("seed", range(12))
def test_metadata_bit_exact(rb, ratio, seed):
    spec = wl.random_batch(seed, block_size=16, manager_ratio=ratio, max_reqs=10, max_q=80,
                           max_c=300, pad_tokens=seed % 3, pad_reqs=seed % 2)
    got, want = _meta(rb, spec), oracle_meta(spec)
    for k in KEYS:
        assert np.array_equal(got[k], want[k]), k
    assert got["scalars"][3] == 0


@pytest.mark.parametrize("name,make", [
    ("padding_example_r2", lambda: wl.config2(manager_ratio=2)),
    ("pure_decode_r2", lambda: wl.config3(manager_ratio=2)),
    ("pure_decode_pad_r4", lambda: wl.config3(num_real=250, manager_ratio=4)),
])
def test_workloads_attention(rb, name, make):
    spec = make()
    got, want = _meta(rb, spec), oracle_meta(spec)
    for k in KEYS:
        assert np.array_equal(got[k], want[k]), k
    _case(rb, spec)


@pytest.mark.parametrize("seed", range(16))
def test_fuzzed_attention(rb, seed):
    """Manager blocks of 2 and 4 kernel pages under head groups that are powers of two and
    not (decode units and tcgen05 prefill units both walk the expanded pages)."""
    nh, nkv = [(32, 8), (8, 1), (6, 2), (4, 4), (12, 2), (7, 1)][seed % 6]
    spec = wl.random_batch(seed, num_q_heads=nh, num_kv_heads=nkv, head_dim=128 if seed % 2 else 64,
                           manager_ratio=[2, 4][seed % 2], max_reqs=6, max_q=140, max_c=500,
                           decode_frac=0.5)
    _case(rb, spec)


def test_null_and_out_of_pool_manager_blocks(rb):
    """A manager id naming the null page's manager block, or past the pool, sets BLOCK_ID and
    its tokens write to the null page; the attention flags it too."""
    for bad in (0, -1, 10_000):
        spec = wl.batch_from_lists([20, 3], [5, 1], manager_ratio=2, seed=4)
        spec.block_table[0, 0] = bad
        got = _meta(rb, spec)
        assert got["scalars"][3] & 0x010
        B = spec.dims.block_size
        assert np.all(got["slot_mapping"][:5] // B != -1)
        d = dims_of(spec)
        tens = wl.make_tensors(spec, device="cuda", with_history=False)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        rb.paged_attention(d, spec.num_reqs, spec.num_tokens, tens.q, tens.k_cache, tens.v_cache,
                           i32(spec.block_table), i32(got["query_start_loc"][:3]),
                           i32(got["seq_lens"][:2]), error_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) & 0x010
