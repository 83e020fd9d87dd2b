"""CPU oracle for one flattened mixed-batch step — TEST INFRASTRUCTURE ONLY.

Plain, slow, obviously correct restatements of what the step computes, written
from the pages' prose and worked examples:

* ``metadata``  — query_start_loc, seq_lens, positions, input_ids, slot_mapping,
  logits_indices, phase flags, the manager-to-kernel page expansion and the padding of a step
  to a captured graph size;
* ``persistent_batch`` — the runner's per-step merge of scheduler deltas into the rows of
  the persistent batch (remove, append, install, condense);
* ``kv_cache``  — the paged K/V write by slot_mapping;
* ``attention`` — per-request dense causal GQA attention in float64 over an
  unpaged, contiguous copy of each request's keys and values;
* ``cascade``   — the shared-prefix length rule and the two-pass (prefix, suffix) attention
  merged by log-sum-exp;
* ``gather``    — selection of the last-token hidden rows.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.  The library under
``ragged_mixed_paged_gb300/`` never imports it, and this package imports
nothing from the library: the two share no code.  Integers are exact; floating
point is float64 over bf16 inputs widened exactly.

Every function is pinned by ``tests/test_oracle_*.py`` against values the pages
print, closed forms, special cases that reduce to library routines, and brute
force over tiny inputs.
"""
from .metadata import (prepare_inputs, pad_for_graph, padded_layout_tokens,
                       req_indices_and_query_pos, request_flags, map_to_kernel_blocks)
from .persistent_batch import InputBatch
from .kv_cache import kv_write
from .attention import paged_attention
from .cascade import cascade_attention, cascade_prefix_len
from .gather import gather_rows

__all__ = ["cascade_attention", "cascade_prefix_len", "prepare_inputs", "request_flags", "map_to_kernel_blocks", "InputBatch", "pad_for_graph", "padded_layout_tokens", "req_indices_and_query_pos",
           "kv_write", "paged_attention", "gather_rows"]
