"""ctypes binding of librb.so: argument marshalling only.

Every step of the path runs in the library's CUDA kernels; this module checks tensor
devices, dtypes and contiguity, passes raw pointers and sizes, and turns status codes into
exceptions.  There is no fallback: if the library is missing or fails to load, importing the
package raises.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "librb.so")

RB_OK = 0
STATUS_NAMES = {0: "RB_OK", 1: "RB_ERR_INVALID_ARG", 2: "RB_ERR_CAPACITY", 4: "RB_ERR_CUDA",
                5: "RB_ERR_UNSUPPORTED"}

# device error-word bits (rb.h)
EBIT_NUM_SCHEDULED = 0x001
EBIT_NUM_COMPUTED = 0x002
EBIT_SEQ_LEN = 0x004
EBIT_TOKEN_SUM = 0x008
EBIT_BLOCK_ID = 0x010
EBIT_SLOT = 0x020
EBIT_ROW_INDEX = 0x040
EBIT_ATTN_META = 0x080
EBIT_TIMEOUT = 0x100
EBIT_BATCH_ID = 0x200
EBIT_BATCH_SIZE = 0x400


class RbError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {STATUS_NAMES.get(status, status)}")
        self.status = status


class rb_dims(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in (
        "block_size", "num_q_heads", "num_kv_heads", "head_dim", "max_num_reqs", "max_model_len",
        "max_blocks_per_req", "num_blocks", "null_block", "kernel_blocks_per_manager_block")]


class rb_batch(ctypes.Structure):
    _fields_ = [("max_num_reqs", ctypes.c_int32), ("max_model_len", ctypes.c_int32),
                ("max_blocks_per_req", ctypes.c_int32), ("reserved", ctypes.c_int32)] + [
        (n, ctypes.c_void_p) for n in (
            "d_req_id", "d_token_table", "d_num_tokens", "d_num_prompt", "d_num_computed",
            "d_block_table", "d_num_blocks", "d_num_rows")]


class rb_batch_update(ctypes.Structure):
    _fields_ = [("num_scheduled", ctypes.c_int32), ("num_new", ctypes.c_int32),
                ("num_cached", ctypes.c_int32), ("reserved", ctypes.c_int32)] + [
        (n, ctypes.c_void_p) for n in (
            "d_sched_req_id", "d_sched_num_tokens", "d_new_req_id", "d_new_num_computed",
            "d_new_num_prompt", "d_new_token_start", "d_new_tokens", "d_new_block_start",
            "d_new_blocks", "d_cached_req_id", "d_cached_num_computed", "d_cached_replace",
            "d_cached_token_start", "d_cached_tokens", "d_cached_block_start",
            "d_cached_blocks")]


class rb_host_copy(ctypes.Structure):
    _fields_ = [("dst", ctypes.c_void_p), ("src", ctypes.c_void_p), ("bytes", ctypes.c_size_t)]


class rb_step_args(ctypes.Structure):
    _fields_ = ([("dims", ctypes.POINTER(rb_dims))] +
                [(n, ctypes.c_int32) for n in ("num_reqs", "num_reqs_padded", "num_tokens",
                                               "num_tokens_padded", "hidden_size",
                                               "num_hidden_rows")] +
                [("softmax_scale", ctypes.c_float)] +
                [(n, ctypes.c_void_p) for n in (
                    "d_token_table", "d_num_computed", "d_num_scheduled", "d_block_table",
                    "d_num_prompt", "d_q", "d_k", "d_v", "d_hidden", "d_k_cache", "d_v_cache",
                    "d_input_ids", "d_positions", "d_query_start_loc", "d_seq_lens",
                    "d_slot_mapping", "d_logits_indices", "d_scalars", "d_is_prefilling",
                    "d_discard_request_mask", "d_attn_out", "d_rows_out", "d_workspace")] +
                [("workspace_bytes", ctypes.c_size_t)])


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is missing: build it with `python ragged_mixed_paged_gb300/build.py` "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    I32 = ctypes.c_int32
    PD = ctypes.POINTER(rb_dims)
    sig = {
        "rb_status_string": (ctypes.c_char_p, [I32]),
        "rb_kernel_launch_count": (ctypes.c_uint64, []),
        "rb_debug_attention_wait_limit": (I32, [ctypes.c_uint64, I32]),
        "rb_pad_for_graph": (I32, [P, I32, I32]),
        "rb_prepare_inputs": (I32, [PD, I32, I32, I32, I32, P, P, P, P, P, P, P, P, P, P, P, P,
                                    P, P, P]),
        "rb_kv_write": (I32, [PD, I32, P, P, P, P, P, P, P]),
        "rb_paged_attention_workspace_size": (ctypes.c_size_t, [PD, I32, I32]),
        "rb_paged_attention": (I32, [PD, I32, I32, I32, P, P, P, P, P, P, ctypes.c_float, P, P,
                                     ctypes.c_size_t, P, P]),
        "rb_paged_attention_profiled": (I32, [PD, I32, I32, I32, P, P, P, P, P, P,
                                              ctypes.c_float, P, P, ctypes.c_size_t, P, P,
                                              ctypes.POINTER(ctypes.c_void_p), I32]),
        "rb_gather_rows": (I32, [I32, I32, I32, P, P, P, P, P]),
        "rb_batch_update_workspace_size": (I32, [I32, ctypes.POINTER(ctypes.c_size_t)]),
        "rb_cascade_prefix_len": (I32, [I32, P, I32, I32]),
        "rb_step": (I32, [ctypes.POINTER(rb_step_args), P]),
        "rb_step_profiled": (I32, [ctypes.POINTER(rb_step_args), ctypes.POINTER(ctypes.c_void_p),
                                   I32, P]),
        "rb_step_host": (I32, [ctypes.POINTER(rb_step_args), ctypes.POINTER(rb_host_copy), I32,
                               ctypes.POINTER(rb_host_copy), I32, P]),
        "rb_step_host_async": (I32, [ctypes.POINTER(rb_step_args), ctypes.POINTER(rb_host_copy),
                                     I32, ctypes.POINTER(rb_host_copy), I32, P, P, P, P, P]),
        "rb_paged_attention_cascade_workspace_size": (ctypes.c_size_t, [PD, I32, I32]),
        "rb_paged_attention_cascade": (I32, [PD, I32, I32, I32, I32, P, P, P, P, P, P,
                                             ctypes.c_float, P, P, ctypes.c_size_t, P, P]),
        "rb_batch_apply_update": (I32, [ctypes.POINTER(rb_batch), ctypes.POINTER(rb_batch_update),
                                        P, P, P, ctypes.c_size_t, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


lib = _load()


@dataclass(frozen=True)
class Dims:
    block_size: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    max_num_reqs: int
    max_model_len: int
    max_blocks_per_req: int
    num_blocks: int
    null_block: int = 0
    kernel_blocks_per_manager_block: int = 1  # kernel pages per page-table entry

    def c(self) -> rb_dims:
        return rb_dims(self.block_size, self.num_q_heads, self.num_kv_heads, self.head_dim,
                       self.max_num_reqs, self.max_model_len, self.max_blocks_per_req,
                       self.num_blocks, self.null_block, self.kernel_blocks_per_manager_block)

    @classmethod
    def of(cls, d) -> "Dims":
        return cls(d.block_size, d.num_q_heads, d.num_kv_heads, d.head_dim, d.max_num_reqs,
                   d.max_model_len, d.max_blocks_per_req, d.num_blocks, d.null_block,
                   getattr(d, "kernel_blocks_per_manager_block", 1))


def _check(fn: str, status: int) -> None:
    if status != RB_OK:
        raise RbError(fn, status)


def _ptr(t, dtype=None, name="tensor"):
    """Device pointer of a contiguous CUDA tensor (or None)."""
    if t is None:
        return None
    import torch

    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def launch_count() -> int:
    return int(lib.rb_kernel_launch_count())


def status_string(status: int) -> str:
    return lib.rb_status_string(status).decode()


def pad_for_graph(capture_sizes: Sequence[int], num_tokens: int) -> int:
    arr = (ctypes.c_int32 * len(capture_sizes))(*capture_sizes)
    return int(lib.rb_pad_for_graph(ctypes.cast(arr, ctypes.c_void_p), len(capture_sizes),
                                    num_tokens))


def workspace_size(dims: Dims, max_num_reqs: int, max_num_tokens: int) -> int:
    d = dims.c()
    return int(lib.rb_paged_attention_workspace_size(ctypes.byref(d), max_num_reqs,
                                                     max_num_tokens))


def prepare_inputs(dims: Dims, num_reqs: int, num_reqs_padded: int, num_tokens: int,
                   num_tokens_padded: int, token_table, num_computed, num_scheduled, block_table,
                   out: Optional[dict] = None, stream=None, num_prompt=None) -> dict:
    """Flat step inputs + metadata; returns the output tensors (allocated unless given).

    With ``num_prompt`` (int32 prompt lengths) the output also holds ``is_prefilling`` and
    ``discard_request_mask`` ([num_reqs_padded] int32)."""
    import torch

    i32 = torch.int32
    dev = block_table.device
    if out is None:
        out = dict(
            input_ids=torch.empty(num_tokens_padded, dtype=i32, device=dev),
            positions=torch.empty(num_tokens_padded, dtype=i32, device=dev),
            query_start_loc=torch.empty(num_reqs_padded + 1, dtype=i32, device=dev),
            seq_lens=torch.empty(num_reqs_padded, dtype=i32, device=dev),
            slot_mapping=torch.empty(num_tokens_padded, dtype=i32, device=dev),
            logits_indices=torch.empty(num_reqs_padded, dtype=i32, device=dev),
            scalars=torch.empty(4, dtype=i32, device=dev))
    if num_prompt is not None and "is_prefilling" not in out:
        out["is_prefilling"] = torch.empty(num_reqs_padded, dtype=i32, device=dev)
        out["discard_request_mask"] = torch.empty(num_reqs_padded, dtype=i32, device=dev)
    with_flags = num_prompt is not None
    d = dims.c()
    st = lib.rb_prepare_inputs(
        ctypes.byref(d), num_reqs, num_reqs_padded, num_tokens, num_tokens_padded,
        _ptr(token_table, i32, "token_table"), _ptr(num_computed, i32, "num_computed"),
        _ptr(num_scheduled, i32, "num_scheduled"), _ptr(block_table, i32, "block_table"),
        _ptr(out["input_ids"], i32), _ptr(out["positions"], i32),
        _ptr(out["query_start_loc"], i32), _ptr(out["seq_lens"], i32),
        _ptr(out["slot_mapping"], i32), _ptr(out["logits_indices"], i32),
        _ptr(out["scalars"], i32),
        _ptr(num_prompt, i32, "num_prompt") if with_flags and num_prompt.numel() else None,
        _ptr(out["is_prefilling"], i32) if with_flags else None,
        _ptr(out["discard_request_mask"], i32) if with_flags else None, _stream(stream))
    _check("rb_prepare_inputs", st)
    return out


def kv_write(dims: Dims, k, v, slot_mapping, k_cache, v_cache, error_word=None,
             num_tokens_padded: Optional[int] = None, stream=None) -> None:
    import torch

    bf = torch.bfloat16
    n = k.shape[0] if num_tokens_padded is None else num_tokens_padded
    d = dims.c()
    st = lib.rb_kv_write(ctypes.byref(d), n, _ptr(k, bf, "k"), _ptr(v, bf, "v"),
                         _ptr(slot_mapping, torch.int32, "slot_mapping"),
                         _ptr(k_cache, bf, "k_cache"), _ptr(v_cache, bf, "v_cache"),
                         _ptr(error_word, torch.int32, "error_word"), _stream(stream))
    _check("rb_kv_write", st)


def paged_attention(dims: Dims, num_reqs: int, num_tokens: int, q, k_cache, v_cache,
                    block_table, query_start_loc, seq_lens, out=None, workspace=None,
                    softmax_scale: Optional[float] = None, error_word=None, stream=None,
                    events=None):
    """``events``: optional up to three recorded-once torch.cuda.Event objects that the library
    re-records after its planner, decode and prefill launches (per-kernel timing)."""
    import torch

    bf = torch.bfloat16
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = torch.empty(workspace_size(dims, num_reqs, num_tokens), dtype=torch.uint8,
                                device=q.device)
    scale = 1.0 / math.sqrt(dims.head_dim) if softmax_scale is None else softmax_scale
    d = dims.c()
    args = (ctypes.byref(d), num_reqs, num_tokens, q.shape[0], _ptr(q, bf, "q"),
            _ptr(k_cache, bf, "k_cache"), _ptr(v_cache, bf, "v_cache"),
            _ptr(block_table, torch.int32, "block_table"),
            _ptr(query_start_loc, torch.int32, "query_start_loc"),
            _ptr(seq_lens, torch.int32, "seq_lens"), ctypes.c_float(scale), _ptr(out, bf, "out"),
            _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
            _ptr(error_word, torch.int32, "error_word"), _stream(stream))
    if events is None:
        _check("rb_paged_attention", lib.rb_paged_attention(*args))
    else:
        handles = [e.cuda_event for e in events]
        if not all(handles):
            raise ValueError("record each event once before passing it (torch creates them lazily)")
        arr = (ctypes.c_void_p * len(handles))(*handles)
        _check("rb_paged_attention_profiled",
               lib.rb_paged_attention_profiled(*args, arr, len(handles)))
    return out


def cascade_prefix_len(shared_prefix_tokens: int, num_computed: Sequence[int],
                       block_size: int) -> int:
    """Shared-prefix length a cascade call may use (host rule; -1 for invalid input)."""
    arr = (ctypes.c_int32 * len(num_computed))(*[int(x) for x in num_computed])
    return int(lib.rb_cascade_prefix_len(shared_prefix_tokens, ctypes.cast(arr, ctypes.c_void_p),
                                         len(num_computed), block_size))


def cascade_workspace_size(dims: Dims, max_num_reqs: int, max_num_tokens: int) -> int:
    d = dims.c()
    return int(lib.rb_paged_attention_cascade_workspace_size(ctypes.byref(d), max_num_reqs,
                                                             max_num_tokens))


def paged_attention_cascade(dims: Dims, num_reqs: int, num_tokens: int, common_prefix_len: int,
                            q, k_cache, v_cache, block_table, query_start_loc, seq_lens,
                            out=None, workspace=None, softmax_scale: Optional[float] = None,
                            error_word=None, stream=None):
    """Attention of a batch whose requests share their first ``common_prefix_len`` tokens."""
    import torch

    bf = torch.bfloat16
    if out is None:
        out = torch.empty_like(q)
    if workspace is None:
        workspace = torch.empty(cascade_workspace_size(dims, num_reqs, num_tokens),
                                dtype=torch.uint8, device=q.device)
    scale = 1.0 / math.sqrt(dims.head_dim) if softmax_scale is None else softmax_scale
    d = dims.c()
    st = lib.rb_paged_attention_cascade(
        ctypes.byref(d), num_reqs, num_tokens, q.shape[0], common_prefix_len, _ptr(q, bf, "q"),
        _ptr(k_cache, bf, "k_cache"), _ptr(v_cache, bf, "v_cache"),
        _ptr(block_table, torch.int32, "block_table"),
        _ptr(query_start_loc, torch.int32, "query_start_loc"),
        _ptr(seq_lens, torch.int32, "seq_lens"), ctypes.c_float(scale), _ptr(out, bf, "out"),
        _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
        _ptr(error_word, torch.int32, "error_word"), _stream(stream))
    _check("rb_paged_attention_cascade", st)
    return out


def gather_rows(hidden, indices, num_rows: Optional[int] = None, out=None, error_word=None,
                stream=None):
    import torch

    n = indices.shape[0] if num_rows is None else num_rows
    if out is None:
        out = torch.empty((n, hidden.shape[1]), dtype=hidden.dtype, device=hidden.device)
    st = lib.rb_gather_rows(n, hidden.shape[1], hidden.shape[0],
                            _ptr(hidden, torch.bfloat16, "hidden"),
                            _ptr(indices, torch.int32, "indices"), _ptr(out, torch.bfloat16),
                            _ptr(error_word, torch.int32, "error_word"), _stream(stream))
    _check("rb_gather_rows", st)
    return out
