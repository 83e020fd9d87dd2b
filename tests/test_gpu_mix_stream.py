"""The chunked-prefill mix as a stream of 100 seeded steps, through the product's own entry
points: every step merges the scheduler's deltas into the device-resident batch
(``rb_batch_apply_update``) and runs the whole step in one ``rb_step`` call.  The KV cache
carries over from step to step, so each step's attention reads what earlier steps wrote.

At every step, against the oracle (its ``InputBatch`` for the rows, ``prepare_inputs`` for the
metadata, its attention over each request's contiguous history):

* metadata, phase flags and the three scalars bit for bit;
* the KV cache: the rows this step changed are exactly the oracle's slots, and each holds the
  token's new K and V ("先写入，再读出": the write that precedes attention);
* attention on every decode row and on a seeded sample of each chunk's rows (first, last,
  page edges, 32 random), element-wise within max-abs 2e-2 / mean-abs 2e-3;
* the gathered hidden rows bit for bit.

Each request's cached history is drawn when it first enters the batch and placed into its
pages by the test (a preempted request brings its history back the same way, as does a
request whose page row is replaced); after that only the library writes the cache.
"""
import dataclasses

import numpy as np
import pytest
import torch

import workloads as wl
from gpu_cases import (compare_attention, oracle_attention_threads, oracle_meta, sample_rows,
                       spec_of_layout, to64, _Lazy)
from oracle.persistent_batch import InputBatch

pytestmark = pytest.mark.gpu

STEPS = 100
SEED = 4000          # the chunked-prefill stream's seed (rank 0 of bench.py --config 4)


class _History:
    """One request's cached K and V rows in host memory (bf16), grown by appends."""

    def __init__(self, k, v):
        self.n = k.shape[0]
        cap = max(64, int(self.n * 1.25) + 64)
        self.k = torch.empty((cap,) + tuple(k.shape[1:]), dtype=k.dtype)
        self.v = torch.empty_like(self.k)
        self.k[:self.n] = k
        self.v[:self.n] = v

    def append(self, k, v):
        m = self.n + k.shape[0]
        if m > self.k.shape[0]:
            cap = int(m * 1.5) + 64
            for name in ("k", "v"):
                old = getattr(self, name)
                new = torch.empty((cap,) + tuple(old.shape[1:]), dtype=old.dtype)
                new[:self.n] = old[:self.n]
                setattr(self, name, new)
        self.k[self.n:m] = k
        self.v[self.n:m] = v
        self.n = m


def _place(cache, block_size, pages, rows):
    """Write a request's contiguous history rows into its pages (page-table order)."""
    n = rows.shape[0]
    if n == 0:
        return
    view = cache.view(-1, block_size, *cache.shape[1:])
    full = n // block_size
    dev_rows = rows.to(cache.device)
    if full:
        idx = torch.as_tensor(np.asarray(pages[:full], np.int64), device=cache.device)
        view[idx] = dev_rows[:full * block_size].view(full, block_size, *cache.shape[1:])
    rem = n - full * block_size
    if rem:
        view[int(pages[full]), :rem] = dev_rows[full * block_size:]


def test_chunked_prefill_stream_every_step(rb):
    stream = wl.MixedChunkStream(seed=SEED)
    d = stream.dims
    dims = rb.Dims.of(d)
    B, nh, nkv, hd = d.block_size, d.num_q_heads, d.num_kv_heads, d.head_dim
    bf = torch.bfloat16
    g = torch.Generator(device="cuda").manual_seed(SEED * 1000 + 17)

    def randn(*shape):
        return torch.randn(*shape, generator=g, device="cuda", dtype=torch.float32).to(bf)

    k_cache = torch.empty((d.num_slots, nkv, hd), dtype=bf, device="cuda").normal_(generator=g)
    v_cache = torch.empty_like(k_cache).normal_(generator=g)
    dev = rb.PersistentBatch(d.max_num_reqs, d.max_model_len, d.max_blocks_per_req)
    ref = InputBatch(d.max_num_reqs, d.max_model_len, d.max_blocks_per_req)
    nmax, rmax, H = stream.BUDGET, d.max_num_reqs, 4096
    buf = rb.StepBuffers.allocate(dims, rmax, rmax, nmax, nmax, dev.tables(),
                                  randn(nmax, nh, hd), randn(nmax, nkv, hd),
                                  randn(nmax, nkv, hd), randn(nmax, H), k_cache, v_cache)
    hist, last_seen = {}, {}
    checked_rows = decode_rows = 0
    for s in range(STEPS):
        step = stream.next_step()
        dev.apply(step)
        ref.apply(step)
        torch.cuda.synchronize()
        assert int(dev.error_word.item()) == 0, f"step {s}: batch update error bits"
        R, N = ref.num_reqs, step.num_tokens
        assert (dev.num_reqs, dev.num_tokens_scheduled) == (R, N)
        cols = ref.columns(step.scheduled)

        # requests entering with a cached history, or whose page row was replaced: their
        # history goes into their (new) pages
        entering = {n.req_id for n in step.new} | {c.req_id for c in step.cached
                                                    if c.replace_blocks}
        for r in range(R):
            uid, c = int(cols["req_id"][r]), int(cols["num_computed"][r])
            last_seen[uid] = s
            if uid not in entering:
                continue
            if uid not in hist:
                hk, hv = randn(c, nkv, hd), randn(c, nkv, hd)
                hist[uid] = _History(hk.cpu(), hv.cpu())
            h = hist[uid]
            assert h.n == c, f"step {s}: request {uid} re-enters with {c} tokens, history {h.n}"
            _place(k_cache, B, cols["blocks"][r], h.k[:c])
            _place(v_cache, B, cols["blocks"][r], h.v[:c])

        q, k, v, hidden = randn(N, nh, hd), randn(N, nkv, hd), randn(N, nkv, hd), randn(N, H)
        b = dataclasses.replace(buf, num_reqs=R, num_reqs_padded=R, num_tokens=N,
                                num_tokens_padded=N, q=q, k=k, v=v, hidden=hidden,
                                attn_out=buf.attn_out[:N], rows_out=buf.rows_out[:R])
        kc0, vc0 = k_cache.clone(), v_cache.clone()
        rb.run_step_fused(b)
        torch.cuda.synchronize()

        spec = spec_of_layout(f"stream step {s}", d, step, ref, SEED * 1000 + s)
        want = oracle_meta(spec)
        m = buf.meta
        assert int(m["scalars"][3].item()) == 0, f"step {s}: device error word"
        for key, n in (("input_ids", N), ("positions", N), ("slot_mapping", N),
                       ("query_start_loc", R + 1), ("seq_lens", R), ("logits_indices", R),
                       ("is_prefilling", R), ("discard_request_mask", R)):
            assert np.array_equal(m[key][:n].cpu().numpy(), want[key][:n]), f"step {s}: {key}"
        assert m["scalars"][:3].tolist() == [want["max_query_len"], want["max_seq_len"],
                                             want["num_actual_tokens"]], f"step {s}: scalars"

        # KV write: the changed rows are the oracle's slots, holding this step's K and V
        slots = torch.as_tensor(want["slot_mapping"], device="cuda")
        changed = ((k_cache != kc0).flatten(1).any(1) | (v_cache != vc0).flatten(1).any(1))
        changed = torch.nonzero(changed).flatten()
        del kc0, vc0
        assert bool(torch.isin(changed, slots).all()), f"step {s}: a row outside the slots changed"
        assert torch.equal(k_cache[slots], k) and torch.equal(v_cache[slots], v), f"step {s}: KV"

        # gathered hidden rows
        li = torch.as_tensor(want["logits_indices"], device="cuda")
        assert torch.equal(b.rows_out, hidden[li]), f"step {s}: gathered rows"

        # attention: every decode row plus a seeded sample of each chunk's rows
        rows = sample_rows(spec, n_random=32, seed=s)
        hk = [_Lazy(hist[int(u)].k[:int(c)]) for u, c in zip(cols["req_id"], cols["num_computed"])]
        hv = [_Lazy(hist[int(u)].v[:int(c)]) for u, c in zip(cols["req_id"], cols["num_computed"])]
        ref_out = oracle_attention_threads(to64(q), hk, hv, to64(k), to64(v),
                                           want["query_start_loc"], want["seq_lens"], R, rows)
        compare_attention(b.attn_out, ref_out, N, rows=rows)
        checked_rows += len(rows)
        decode_rows += int((spec.num_scheduled == 1).sum())

        # this step's K and V join each request's history; requests gone for two steps leave
        kh, vh = k.cpu(), v.cpu()
        qsl = want["query_start_loc"]
        for r in range(R):
            hist[int(cols["req_id"][r])].append(kh[qsl[r]:qsl[r + 1]], vh[qsl[r]:qsl[r + 1]])
        for uid in [u for u, t in last_seen.items() if t < s - 1]:
            hist.pop(uid, None)
            last_seen.pop(uid)
    assert decode_rows >= 100 * 100 and checked_rows > decode_rows
