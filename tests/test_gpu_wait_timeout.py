"""The fused attention launch's bounded waits, made to run out without faulting anything: with
the test hook rb_debug_attention_wait_limit the producer of CTA 0 withholds its first prefill
unit before any copy or MMA of it is issued, so that CTA's MMA issuer and softmax warps wait for
a unit that never arrives.  After a few milliseconds they give up: the call must flag
RB_EBIT_TIMEOUT, the CTA must drain and return (the stream synchronises, no fault), and the next
ordinary call on the same context must be right."""
import pytest
import torch

import workloads as wl
from gpu_cases import compare_attention, oracle_attention, oracle_meta, run_attention

pytestmark = pytest.mark.gpu


def _set(rb, limit_ns, withhold):
    assert rb.lib.rb_debug_attention_wait_limit(limit_ns, withhold) == 0


def test_withheld_unit_times_out_cleanly_and_the_next_call_is_right(rb):
    # prefills only (every CTA starts on prefill units and takes at least one): 4 x 2048 tokens
    spec = wl.batch_from_lists([0, 100, 0, 37], [2048, 2048, 2048, 2048], num_q_heads=32,
                               num_kv_heads=8, head_dim=128, seed=21)
    tens = wl.make_tensors(spec, device="cuda")
    meta = oracle_meta(spec)
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    try:
        _set(rb, 5_000_000, 1)                       # 5 ms waits, CTA 0 withholds a unit
        run_attention(rb, spec, tens, meta, error_word=err)
        torch.cuda.synchronize()
        assert int(err.item()) & rb.EBIT_TIMEOUT, "the withheld unit's waits must run out"
    finally:
        _set(rb, 0, 0)                               # defaults: 1 s, nothing withheld
    err.zero_()
    out = run_attention(rb, spec, tens, meta, error_word=err)
    assert int(err.item()) == 0
    compare_attention(out, oracle_attention(spec, tens, meta), spec.num_tokens)

