"""Device-resident persistent batch and the per-step merge of scheduler deltas into it.

``PersistentBatch`` owns the row columns (request id, token history, counters, page row) on
the GPU.  ``apply`` packs one step's scheduler output (request-id keyed: the schedule, the
requests entering the batch with their whole state, the deltas of resident requests) into one
pinned host buffer, copies it to the device in one transfer, and calls
``rb_batch_apply_update``, which removes, merges, installs and condenses rows in the library's
kernels.  Afterwards ``num_scheduled`` holds this step's per-row token counts and the batch's
columns are the inputs of ``rb_prepare_inputs`` for ``num_reqs`` rows.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import numpy as np

from . import _binding as rb

_ALIGN = 4  # int32 elements: every packed section starts on a 16-byte boundary


def batch_workspace_size(max_num_reqs: int) -> int:
    n = ctypes.c_size_t(0)
    rb._check("rb_batch_update_workspace_size",
              rb.lib.rb_batch_update_workspace_size(max_num_reqs, ctypes.byref(n)))
    return int(n.value)


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32).reshape(-1))


def _starts(lengths) -> np.ndarray:
    out = np.zeros(len(lengths) + 1, np.int32)
    if len(lengths):
        out[1:] = np.cumsum(np.asarray(lengths, np.int64))
    return out


class _Staging:
    """Two pinned host buffers and their device twins, used in turn so that packing the next
    step never overwrites a buffer whose copy may still be in flight."""

    def __init__(self, device):
        self.device = device
        self.slots = [None, None]
        self.turn = 0

    def get(self, n_int32: int):
        import torch

        i = self.turn
        self.turn ^= 1
        slot = self.slots[i]
        if slot is None or slot[0].numel() < n_int32:
            size = max(n_int32, 1 << 16, 0 if slot is None else 2 * slot[0].numel())
            host = torch.empty(size, dtype=torch.int32).pin_memory()
            dev = torch.empty(size, dtype=torch.int32, device=self.device)
            slot = [host, dev, None]
            self.slots[i] = slot
        elif slot[2] is not None:
            slot[2].synchronize()  # the copy that last read this host buffer has finished
        return slot


class StagedStep:
    """One step's packed scheduler output, already in device memory."""

    def __init__(self, packet, offsets, num_scheduled, num_new, num_cached, num_tokens, nbytes):
        self.packet = packet
        self.offsets = offsets
        self.num_scheduled = num_scheduled
        self.num_new = num_new
        self.num_cached = num_cached
        self.num_tokens = num_tokens
        self.nbytes = nbytes


class PersistentBatch:
    """One row per resident request; the live rows are always [0, num_reqs)."""

    def __init__(self, max_num_reqs: int, max_model_len: int, max_blocks_per_req: int,
                 device="cuda"):
        import torch

        self.max_num_reqs = int(max_num_reqs)
        self.max_model_len = int(max_model_len)
        self.max_blocks_per_req = int(max_blocks_per_req)
        i32 = torch.int32
        NR = self.max_num_reqs
        self.req_id = torch.full((NR,), -1, dtype=torch.int64, device=device)
        self.token_table = torch.zeros((NR, self.max_model_len), dtype=i32, device=device)
        self.num_tokens = torch.zeros(NR, dtype=i32, device=device)
        self.num_prompt = torch.zeros(NR, dtype=i32, device=device)
        self.num_computed = torch.zeros(NR, dtype=i32, device=device)
        self.block_table = torch.full((NR, self.max_blocks_per_req), -1, dtype=i32, device=device)
        self.num_blocks = torch.zeros(NR, dtype=i32, device=device)
        self.num_rows = torch.zeros(1, dtype=i32, device=device)
        self.num_scheduled = torch.zeros(NR, dtype=i32, device=device)
        self.row_of_sched = torch.zeros(NR, dtype=i32, device=device)
        self.error_word = torch.zeros(1, dtype=i32, device=device)
        self.workspace = torch.empty(batch_workspace_size(NR), dtype=torch.uint8, device=device)
        self.num_reqs = 0
        self.num_tokens_scheduled = 0
        self.last_h2d_bytes = 0
        self._staging = _Staging(device)
        self._c = rb.rb_batch(NR, self.max_model_len, self.max_blocks_per_req, 0,
                              *(t.data_ptr() for t in (
                                  self.req_id, self.token_table, self.num_tokens,
                                  self.num_prompt, self.num_computed, self.block_table,
                                  self.num_blocks, self.num_rows)))

    # ------------------------------------------------------------------------------ packing
    @staticmethod
    def pack(step):
        """Sections of one step's packet, as (name, int32 array) in upload order."""
        sched_ids = np.fromiter(step.scheduled.keys(), dtype=np.int64, count=len(step.scheduled))
        sched_q = np.fromiter(step.scheduled.values(), dtype=np.int32, count=len(step.scheduled))
        new, cached = list(step.new), list(step.cached)
        ids64 = lambda xs: np.array([x.req_id for x in xs], np.int64).view(np.int32)
        cat = lambda arrs: (np.concatenate([_i32(a) for a in arrs]) if arrs
                            else np.zeros(0, np.int32))
        return [
            ("sched_req_id", sched_ids.view(np.int32)),
            ("new_req_id", ids64(new)),
            ("cached_req_id", ids64(cached)),
            ("sched_num_tokens", sched_q),
            ("new_num_computed", _i32([n.num_computed for n in new])),
            ("new_num_prompt", _i32([n.num_prompt for n in new])),
            ("new_token_start", _starts([len(n.tokens) for n in new])),
            ("new_block_start", _starts([len(n.blocks) for n in new])),
            ("cached_num_computed", _i32([c.num_computed for c in cached])),
            ("cached_replace", _i32([1 if c.replace_blocks else 0 for c in cached])),
            ("cached_token_start", _starts([len(c.new_tokens) for c in cached])),
            ("cached_block_start", _starts([len(c.new_blocks) for c in cached])),
            ("new_tokens", cat([n.tokens for n in new])),
            ("new_blocks", cat([n.blocks for n in new])),
            ("cached_tokens", cat([c.new_tokens for c in cached])),
            ("cached_blocks", cat([c.new_blocks for c in cached])),
        ], len(sched_ids), len(new), len(cached)

    @classmethod
    def _layout(cls, step):
        sections, S, NN, NC = cls.pack(step)
        offsets, n = {}, 0
        for name, arr in sections:
            offsets[name] = n
            n += -(-arr.size // _ALIGN) * _ALIGN
        return sections, offsets, n, S, NN, NC

    def _launch(self, base: int, offsets: dict, S: int, NN: int, NC: int, stream) -> None:
        import torch

        ptr = {name: base + 4 * off for name, off in offsets.items()}
        u = rb.rb_batch_update(S, NN, NC, 0, *(ptr[f[0][2:]] for f in rb.rb_batch_update._fields_[4:]))
        st = rb.lib.rb_batch_apply_update(
            ctypes.byref(self._c), ctypes.byref(u), rb._ptr(self.num_scheduled, torch.int32),
            rb._ptr(self.row_of_sched, torch.int32), rb._ptr(self.workspace),
            self.workspace.numel(), rb._ptr(self.error_word, torch.int32), rb._stream(stream))
        rb._check("rb_batch_apply_update", st)
        self.num_reqs = S

    def apply(self, step, stream=None, copied_event=None) -> int:
        """Merge one step's scheduler output into the batch (enqueued on ``stream``); returns
        the bytes copied host -> device.  Sets ``num_reqs`` / ``num_tokens_scheduled``.
        ``copied_event``, if given, is recorded between the packet copy and the kernels."""
        import torch

        sections, offsets, n, S, NN, NC = self._layout(step)
        host, dev, _ = slot = self._staging.get(n)
        view = host.numpy()
        for name, arr in sections:
            view[offsets[name]:offsets[name] + arr.size] = arr
        s = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            dev[:n].copy_(host[:n], non_blocking=True)
            ev = torch.cuda.Event()
            ev.record(s)
        slot[2] = ev
        if copied_event is not None:
            copied_event.record(s)
        self._launch(dev.data_ptr(), offsets, S, NN, NC, s)
        self.num_tokens_scheduled = int(sum(step.scheduled.values()))
        self.last_h2d_bytes = 4 * n
        return self.last_h2d_bytes

    def stage(self, step, device=None) -> "StagedStep":
        """Pack one step's scheduler output and copy it into a device buffer of its own, ahead
        of time (a caller that has the step before it runs, e.g. a benchmark); the copy is
        complete when this returns.  ``apply_staged`` then merges it with no host work."""
        import torch

        sections, offsets, n, S, NN, NC = self._layout(step)
        host = np.zeros(max(n, 1), np.int32)
        for name, arr in sections:
            host[offsets[name]:offsets[name] + arr.size] = arr
        dev = torch.from_numpy(host).to(device or self.req_id.device)
        return StagedStep(dev, offsets, S, NN, NC, int(sum(step.scheduled.values())), 4 * n)

    def apply_staged(self, staged: "StagedStep", stream=None) -> None:
        """``apply`` for a packet already on the device (``stage``): only the update's
        launches are enqueued on ``stream``."""
        import torch

        s = stream if stream is not None else torch.cuda.current_stream()
        self._launch(staged.packet.data_ptr(), staged.offsets, staged.num_scheduled,
                     staged.num_new, staged.num_cached, s)
        self.num_tokens_scheduled = staged.num_tokens
        self.last_h2d_bytes = 0

    # ------------------------------------------------------------------------------ views
    def tables(self) -> dict:
        """The inputs ``rb_prepare_inputs`` reads, as views of the batch's columns."""
        return {"token_table": self.token_table, "block_table": self.block_table,
                "num_computed": self.num_computed, "num_scheduled": self.num_scheduled,
                "num_prompt": self.num_prompt}

    def snapshot(self) -> dict:
        """Host copies of the live rows' state (valid prefixes only)."""
        R = int(self.num_rows.item())
        nt = self.num_tokens[:R].cpu().numpy()
        nb = self.num_blocks[:R].cpu().numpy()
        tok = self.token_table[:R].cpu().numpy()
        blk = self.block_table[:R].cpu().numpy()
        return dict(num_rows=R, req_id=self.req_id[:R].cpu().numpy(), num_tokens=nt,
                    num_prompt=self.num_prompt[:R].cpu().numpy(),
                    num_computed=self.num_computed[:R].cpu().numpy(), num_blocks=nb,
                    num_scheduled=self.num_scheduled.cpu().numpy(),
                    tokens=[tok[r, :nt[r]].copy() for r in range(R)],
                    blocks=[blk[r, :nb[r]].copy() for r in range(R)])
