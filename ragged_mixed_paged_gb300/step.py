"""One pass of the hot path over a batch: prepare_inputs -> kv_write -> paged_attention ->
gather_rows, on one stream, with no host synchronisation inside.

``StepBuffers`` holds fixed-address device buffers sized once (as a CUDA-graph runner keeps
them); ``run_step`` enqueues the four library calls, ``run_step_fused`` the single ``rb_step``
call that does the same work in one memset and two launches (same results, bit for bit), and
``run_step_host`` the ``rb_step_host`` call that also copies the inputs in from host memory
and the results back.  The
step's error word is the fourth scalar written by ``prepare_inputs``; the KV write and the
attention OR their bits into it.
"""
from __future__ import annotations

import ctypes
import math

from dataclasses import dataclass
from typing import Optional

from . import _binding as rb


@dataclass
class StepBuffers:
    dims: rb.Dims
    num_reqs: int
    num_reqs_padded: int
    num_tokens: int
    num_tokens_padded: int
    token_table: object
    block_table: object
    num_computed: object
    num_scheduled: object
    q: object
    k: object
    v: object
    hidden: object
    k_cache: object
    v_cache: object
    meta: dict
    attn_out: object
    workspace: object
    rows_out: object
    num_prompt: object = None  # int32 prompt lengths: enables is_prefilling / discard mask
    _step_args: object = None  # rb_step_args built on first use (the buffers never move)

    @classmethod
    def allocate(cls, dims: rb.Dims, num_reqs: int, num_reqs_padded: int, num_tokens: int,
                 num_tokens_padded: int, tables: dict, q, k, v, hidden, k_cache, v_cache):
        import torch

        dev = q.device
        i32 = torch.int32
        meta = dict(
            input_ids=torch.empty(num_tokens_padded, dtype=i32, device=dev),
            positions=torch.empty(num_tokens_padded, dtype=i32, device=dev),
            query_start_loc=torch.empty(num_reqs_padded + 1, dtype=i32, device=dev),
            seq_lens=torch.empty(num_reqs_padded, dtype=i32, device=dev),
            slot_mapping=torch.empty(num_tokens_padded, dtype=i32, device=dev),
            logits_indices=torch.empty(num_reqs_padded, dtype=i32, device=dev),
            scalars=torch.zeros(4, dtype=i32, device=dev))
        if tables.get("num_prompt") is not None:
            meta["is_prefilling"] = torch.empty(num_reqs_padded, dtype=i32, device=dev)
            meta["discard_request_mask"] = torch.empty(num_reqs_padded, dtype=i32, device=dev)
        ws = torch.empty(rb.workspace_size(dims, max(num_reqs, 1), max(num_tokens, 1)),
                         dtype=torch.uint8, device=dev)
        return cls(dims=dims, num_reqs=num_reqs, num_reqs_padded=num_reqs_padded,
                   num_tokens=num_tokens, num_tokens_padded=num_tokens_padded,
                   token_table=tables["token_table"], block_table=tables["block_table"],
                   num_computed=tables["num_computed"], num_scheduled=tables["num_scheduled"],
                   q=q, k=k, v=v, hidden=hidden, k_cache=k_cache, v_cache=v_cache, meta=meta,
                   attn_out=torch.empty_like(q), workspace=ws,
                   rows_out=torch.empty((num_reqs_padded, hidden.shape[1]), dtype=hidden.dtype,
                                        device=dev),
                   num_prompt=tables.get("num_prompt"))

    @property
    def error_word(self):
        return self.meta["scalars"][3:4]


def run_step(b: StepBuffers, stream=None, softmax_scale: Optional[float] = None,
             marks=None, attn_marks=None) -> None:
    """Enqueue one whole step (all four library calls) on ``stream``.

    ``marks``: optional five CUDA events, recorded on the same stream before the first call
    and after each of the four calls (for per-call timing).  ``attn_marks``: optional three
    recorded-once events the attention call re-records after its planner, decode and prefill
    launches (per-kernel timing).
    """
    def mark(i):
        if marks is not None:
            marks[i].record(stream)

    m = b.meta
    mark(0)
    rb.prepare_inputs(b.dims, b.num_reqs, b.num_reqs_padded, b.num_tokens, b.num_tokens_padded,
                      b.token_table, b.num_computed, b.num_scheduled, b.block_table, out=m,
                      stream=stream, num_prompt=b.num_prompt)
    mark(1)
    rb.kv_write(b.dims, b.k, b.v, m["slot_mapping"], b.k_cache, b.v_cache,
                error_word=b.error_word, num_tokens_padded=b.num_tokens_padded, stream=stream)
    mark(2)
    rb.paged_attention(b.dims, b.num_reqs, b.num_tokens, b.q, b.k_cache, b.v_cache,
                       b.block_table, m["query_start_loc"], m["seq_lens"], out=b.attn_out,
                       workspace=b.workspace, softmax_scale=softmax_scale,
                       error_word=b.error_word, stream=stream, events=attn_marks)
    mark(3)
    rb.gather_rows(b.hidden, m["logits_indices"], num_rows=b.num_reqs_padded, out=b.rows_out,
                   error_word=b.error_word, stream=stream)
    mark(4)


def _step_args(b: StepBuffers, softmax_scale: Optional[float]):
    import torch

    i32, bf = torch.int32, torch.bfloat16
    m = b.meta
    p = lambda t, dt=None: rb._ptr(t, dt).value
    flags = b.num_prompt is not None
    b._dims_c = b.dims.c()  # kept alive with the struct that points at it
    scale = 1.0 / math.sqrt(b.dims.head_dim) if softmax_scale is None else softmax_scale
    return rb.rb_step_args(
        ctypes.pointer(b._dims_c), b.num_reqs, b.num_reqs_padded, b.num_tokens,
        b.num_tokens_padded, b.hidden.shape[1], b.hidden.shape[0], scale,
        p(b.token_table, i32), p(b.num_computed, i32), p(b.num_scheduled, i32),
        p(b.block_table, i32), p(b.num_prompt, i32) if flags and b.num_prompt.numel() else None,
        p(b.q, bf), p(b.k, bf), p(b.v, bf), p(b.hidden, bf), p(b.k_cache, bf), p(b.v_cache, bf),
        p(m["input_ids"], i32), p(m["positions"], i32), p(m["query_start_loc"], i32),
        p(m["seq_lens"], i32), p(m["slot_mapping"], i32), p(m["logits_indices"], i32),
        p(m["scalars"], i32), p(m["is_prefilling"], i32) if flags else None,
        p(m["discard_request_mask"], i32) if flags else None, p(b.attn_out, bf),
        p(b.rows_out, bf), p(b.workspace, torch.uint8), b.workspace.numel())


def run_step_fused(b: StepBuffers, stream=None, softmax_scale: Optional[float] = None,
                   events=None) -> None:
    """Enqueue the whole step as one ``rb_step`` call (one memset and two launches).

    ``events``: optional recorded-once torch.cuda.Event objects that the library re-records
    after its preparation launch and after its attention launch (``rb_step_profiled``)."""
    if b._step_args is None or softmax_scale is not None:
        b._step_args = _step_args(b, softmax_scale)
    if events is None:
        rb._check("rb_step", rb.lib.rb_step(ctypes.byref(b._step_args), rb._stream(stream)))
        return
    handles = [e.cuda_event for e in events]
    if not all(handles):
        raise ValueError("record each event once before passing it (torch creates them lazily)")
    arr = (ctypes.c_void_p * len(handles))(*handles)
    rb._check("rb_step_profiled", rb.lib.rb_step_profiled(ctypes.byref(b._step_args), arr,
                                                          len(handles), rb._stream(stream)))


def _copies(pairs):
    arr = (rb.rb_host_copy * max(len(pairs), 1))()
    for i, (dst, src) in enumerate(pairs):
        n = src.numel() * src.element_size()
        if dst.numel() * dst.element_size() != n:
            raise ValueError("a host copy's source and destination differ in size")
        arr[i] = rb.rb_host_copy(dst.data_ptr(), src.data_ptr(), n)
    return arr


def run_step_host_async(b: StepBuffers, host_in, host_out, stream, in_stream, out_stream,
                        in_done, step_done, softmax_scale: Optional[float] = None) -> None:
    """Enqueue one ``rb_step_host_async`` call: the ``host_in`` copies on ``in_stream`` (then
    ``in_done`` recorded there), the step on ``stream`` after ``in_done`` (then ``step_done``),
    the ``host_out`` copies on ``out_stream`` after ``step_done``.  The events are
    torch.cuda.Event objects already recorded once (torch creates them lazily); the caller
    keeps the buffers of steps in flight apart and orders their reuse."""
    if b._step_args is None or softmax_scale is not None:
        b._step_args = _step_args(b, softmax_scale)
    if not (in_done.cuda_event and step_done.cuda_event):
        raise ValueError("record each event once before passing it (torch creates them lazily)")
    ins, outs = _copies(host_in), _copies(host_out)
    rb._check("rb_step_host_async",
              rb.lib.rb_step_host_async(ctypes.byref(b._step_args), ins, len(host_in), outs,
                                        len(host_out), rb._stream(stream), rb._stream(in_stream),
                                        rb._stream(out_stream), in_done.cuda_event,
                                        step_done.cuda_event))


def run_step_host(b: StepBuffers, host_in, host_out, stream=None,
                  softmax_scale: Optional[float] = None) -> None:
    """Enqueue one ``rb_step_host`` call: the ``host_in`` copies (``(device_dst, host_src)``
    tensor pairs, contiguous), the step, then the ``host_out`` copies (``(host_dst,
    device_src)``).  Page-locked host tensors keep the copies asynchronous."""
    if b._step_args is None or softmax_scale is not None:
        b._step_args = _step_args(b, softmax_scale)
    ins, outs = _copies(host_in), _copies(host_out)
    rb._check("rb_step_host", rb.lib.rb_step_host(ctypes.byref(b._step_args), ins, len(host_in),
                                                  outs, len(host_out), rb._stream(stream)))
