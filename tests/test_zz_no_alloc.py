"""rb_paged_attention_static_ws: the attention entry point for callers that cannot allocate
device memory (its scratch is an array inside the library).  Through the C ABI it must give
what rb_paged_attention gives with a caller-allocated workspace, bit for bit, on calls in a row
over different batches, and reject batches whose scratch would not fit.  This file is
collected last on purpose."""
import ctypes
import math

import pytest
import torch

import workloads as wl
from gpu_cases import dims_of, i32, oracle_meta

pytestmark = pytest.mark.gpu


def _static_ws_fn(rb):
    lib = ctypes.CDLL(rb.LIB_PATH)
    fn = lib.rb_paged_attention_static_ws
    P, I32 = ctypes.c_void_p, ctypes.c_int32
    fn.restype = I32
    fn.argtypes = [ctypes.POINTER(rb._binding.rb_dims), I32, I32, I32, P, P, P, P, P, P,
                   ctypes.c_float, P, P, P]
    return fn


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _case(rb, spec):
    """Inputs of one attention call (this step's K/V already written) and the allocating entry
    point's output for them."""
    tens = wl.make_tensors(spec, device="cuda")
    meta = oracle_meta(spec)
    dims = dims_of(spec)
    R, N = spec.num_reqs, spec.num_tokens
    rb.kv_write(dims, tens.k, tens.v, i32(meta["slot_mapping"]), tens.k_cache, tens.v_cache)
    qsl, sl, bt = i32(meta["query_start_loc"][:R + 1]), i32(meta["seq_lens"][:R]), \
        i32(spec.block_table)
    ref = rb.paged_attention(dims, R, N, tens.q, tens.k_cache, tens.v_cache, bt, qsl, sl)
    torch.cuda.synchronize()
    return dict(spec=spec, tens=tens, dims=dims, qsl=qsl, sl=sl, bt=bt, ref=ref)


def _call(fn, c):
    spec, tens = c["spec"], c["tens"]
    d = c["dims"].c()
    scale = 1.0 / math.sqrt(spec.dims.head_dim)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    out = torch.full_like(tens.q, float("nan"))
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    st = fn(ctypes.byref(d), spec.num_reqs, spec.num_tokens, tens.q.shape[0], _ptr(tens.q),
            _ptr(tens.k_cache), _ptr(tens.v_cache), _ptr(c["bt"]), _ptr(c["qsl"]), _ptr(c["sl"]),
            ctypes.c_float(scale), _ptr(out), _ptr(err), stream)
    assert st == 0
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out


def test_static_workspace_matches_allocating_entry_point(rb):
    """Two calls in a row on the shared array: first a batch with many requests and split-KV
    partials (256 decodes, padded to 256 rows), then the padding example, whose planner header,
    unit offsets and split counters must not inherit anything from the first call.  Both
    entry points run the same kernels on the same plan, so the outputs agree bit for bit."""
    fn = _static_ws_fn(rb)
    big = _case(rb, wl.config3(num_real=250))
    small = _case(rb, wl.config2())
    for c in (big, small, small):
        out = _call(fn, c)
        assert torch.equal(out, c["ref"])


def test_static_workspace_rejects_batches_beyond_its_capacity(rb):
    fn = _static_ws_fn(rb)
    spec = wl.config2()
    d = dims_of(spec).c()
    d.max_num_reqs = 4096
    fake = ctypes.c_void_p(0x100000)  # never used: the size check fails first
    st = fn(ctypes.byref(d), 4000, 4000, 4000, fake, fake, fake, fake, fake, fake,
            ctypes.c_float(0.1), fake, None, None)
    assert st == 2  # RB_ERR_CAPACITY
