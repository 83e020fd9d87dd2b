"""Ragged mixed-batch step for GB300: Python face of the librb C ABI (include/rb.h).

    prepare_inputs   persistent batch -> input_ids, positions, query_start_loc, seq_lens,
                     slot_mapping, logits_indices (+ max_query_len, max_seq_len, error word)
    kv_write         new K/V rows -> paged cache by slot_mapping
    paged_attention  varlen causal GQA attention through the page table
    paged_attention_cascade  the same when all requests share a prefix (read once), with
                     cascade_prefix_len giving the usable prefix length
    gather_rows      hidden rows at logits_indices
    PersistentBatch  device-resident rows of the resident requests; ``apply`` merges one
                     step's scheduler output (remove, append, install, condense) on the GPU
    pad_for_graph    smallest captured graph size >= the token count

All compute runs in the library's sm_103a kernels; tensors are caller-owned CUDA tensors.
"""
from ._binding import (Dims, RbError, EBIT_ATTN_META, EBIT_BLOCK_ID, EBIT_NUM_COMPUTED,
                       EBIT_NUM_SCHEDULED, EBIT_ROW_INDEX, EBIT_SEQ_LEN, EBIT_SLOT, EBIT_TIMEOUT,
                       EBIT_TOKEN_SUM, LIB_PATH, gather_rows, kv_write, launch_count, lib,
                       pad_for_graph, paged_attention, prepare_inputs, status_string,
                       workspace_size, cascade_prefix_len, cascade_workspace_size,
                       paged_attention_cascade)
from ._binding import EBIT_BATCH_ID, EBIT_BATCH_SIZE
from .persistent_batch import PersistentBatch, batch_workspace_size
from .step import StepBuffers, run_step, run_step_fused, run_step_host, run_step_host_async

__all__ = ["Dims", "RbError", "gather_rows", "kv_write", "launch_count", "lib", "pad_for_graph",
           "paged_attention", "prepare_inputs", "status_string", "workspace_size", "StepBuffers",
           "run_step", "run_step_fused", "run_step_host", "run_step_host_async", "LIB_PATH", "PersistentBatch", "batch_workspace_size",
           "cascade_prefix_len", "cascade_workspace_size", "paged_attention_cascade"]
