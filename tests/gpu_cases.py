"""Shared helpers of the GPU parity tests: seeded cases, oracle evaluation, comparisons."""
import functools

import numpy as np
import torch

import oracle
import workloads as wl
from oracle.threads import oracle_attention_threads

ATTN_MAX_ABS = 2e-2   # bf16 output vs the float64 oracle
ATTN_MEAN_ABS = 2e-3


def dims_of(spec):
    from ragged_mixed_paged_gb300 import Dims

    return Dims.of(spec.dims)


def oracle_meta(spec):
    d = spec.dims
    return oracle.prepare_inputs(block_size=d.block_size, null_block=d.null_block,
                                 token_table=spec.token_table, block_table=spec.block_table,
                                 num_computed=spec.num_computed, num_scheduled=spec.num_scheduled,
                                 num_reqs_padded=spec.num_reqs_padded,
                                 num_tokens_padded=spec.num_tokens_padded,
                                 num_prompt=spec.num_prompt,
                                 kernel_blocks_per_manager_block=d.kernel_blocks_per_manager_block)


def i32(a, device="cuda"):
    return torch.as_tensor(np.ascontiguousarray(a, dtype=np.int32), device=device)


def to64(t):
    return t.detach().cpu().to(torch.float64).numpy()


class _Lazy:
    """A bf16 history tensor widened only when the oracle reads it (whole, or one kv head's
    slice as float32, which widens to float64 exactly on assignment)."""

    def __init__(self, t):
        self.t = t
        self.shape = tuple(t.shape)

    def __array__(self, dtype=None, copy=None):
        a = to64(self.t)
        return a if dtype is None else a.astype(dtype)

    def __getitem__(self, idx):
        return self.t[idx].float().cpu().numpy()


def config4_layouts(num_steps):
    """The chunked-prefill stream laid out by the oracle's persistent batch, step by step:
    yields (step index, scheduler step, oracle InputBatch after the update)."""
    from oracle.persistent_batch import InputBatch

    stream = wl.MixedChunkStream()
    d = stream.dims
    batch = InputBatch(d.max_num_reqs, d.max_model_len, d.max_blocks_per_req)
    for s in range(num_steps):
        step = stream.next_step()
        batch.apply(step)
        yield s, step, batch


def spec_of_layout(name, dims, step, batch, seed):
    cols = batch.columns(step.scheduled)
    tok, blk = batch.tables()
    return wl.spec_from_columns(name, dims, cols["num_computed"], cols["num_scheduled"],
                                cols["num_prompt"], tok, blk, seed)


@functools.lru_cache(maxsize=1)
def config4_specs(steps=(0, 1, 57, 99)):
    out = {}
    dims = wl.MixedChunkStream().dims
    for s, step, batch in config4_layouts(max(steps) + 1):
        if s in steps:
            out[s] = spec_of_layout(f"chunked-prefill mix step {s}", dims, step, batch,
                                    4000 * 1000 + s)
    return out


def sample_rows(spec, n_random=64, seed=0):
    """Every decode row, plus the first/last rows, page-boundary rows and random rows of longer
    queries."""
    rng = np.random.default_rng(seed)
    rows, s = [], 0
    for c, q in zip(spec.num_computed, spec.num_scheduled):
        c, q = int(c), int(q)
        if q <= 8:
            rows.extend(range(s, s + q))
        else:
            cand = {s, s + q - 1}
            edges = [s + j for j in range(q) if (c + j) % 16 in (0, 15)]
            cand.update(edges[:: max(1, len(edges) // 32)])
            cand.update(int(x) for x in rng.integers(s, s + q, size=n_random))
            rows.extend(sorted(cand))
        s += q
    return sorted(set(rows))


def run_attention(rb, spec, tens, meta, error_word=None):
    """KV write of this step's rows (oracle slots), then the library's attention."""
    dims = dims_of(spec)
    R, N = spec.num_reqs, spec.num_tokens
    rb.kv_write(dims, tens.k, tens.v, i32(meta["slot_mapping"]), tens.k_cache, tens.v_cache,
                error_word=error_word)
    out = rb.paged_attention(dims, R, N, tens.q, tens.k_cache, tens.v_cache,
                             i32(spec.block_table), i32(meta["query_start_loc"][:R + 1]),
                             i32(meta["seq_lens"][:R]), error_word=error_word)
    torch.cuda.synchronize()
    return out


def oracle_attention(spec, tens, meta, rows=None):
    """The oracle's attention of a step (rows not asked for are NaN, padding rows 0)."""
    R = spec.num_reqs
    rows = range(spec.num_tokens) if rows is None else rows
    return oracle_attention_threads(to64(tens.q), [_Lazy(h) for h in tens.hist_k],
                                    [_Lazy(h) for h in tens.hist_v], to64(tens.k), to64(tens.v),
                                    meta["query_start_loc"][:R + 1], meta["seq_lens"][:R], R,
                                    rows)


def compare_attention(got, ref, N, rows=None):
    g = got.float().cpu().numpy().astype(np.float64)
    sel = np.arange(N) if rows is None else np.asarray(rows)
    diff = np.abs(g[sel] - ref[sel])
    assert np.isfinite(g[sel]).all()
    max_abs, mean_abs = float(diff.max(initial=0.0)), float(diff.mean()) if diff.size else 0.0
    assert max_abs <= ATTN_MAX_ABS, f"max abs {max_abs}"
    assert mean_abs <= ATTN_MEAN_ABS, f"mean abs {mean_abs}"
    assert np.all(g[N:] == 0.0), "padding rows must be zero"
    return max_abs, mean_abs


def check_kv_write(spec, k_before, v_before, tens, slot_mapping):
    """The paged KV write of one step, checked on the device: ``cache[slot[t]] = kv[t]`` for
    every real token t and nothing else changes, except padding tokens' writes, which land in
    the null page (any winner: its contents are not state)."""
    d = spec.dims
    N = spec.num_tokens
    slots = torch.as_tensor(np.asarray(slot_mapping[:N], np.int64), device=tens.k_cache.device)
    changed = ((tens.k_cache != k_before).flatten(1).any(1) |
               (tens.v_cache != v_before).flatten(1).any(1))
    changed = torch.nonzero(changed).flatten()
    null_rows = (changed // d.block_size) == d.null_block
    assert bool(torch.isin(changed[~null_rows], slots).all()), "a row outside the slots changed"
    assert not bool(((slots // d.block_size) == d.null_block).any()), "a real token in the null page"
    assert torch.equal(tens.k_cache[slots], tens.k[:N])
    assert torch.equal(tens.v_cache[slots], tens.v[:N])


def jump_tensors(spec, hot, device="cuda"):
    """Inputs whose scores jump across key tiles: every query is a common direction u plus small
    noise and the keys at the positions of `hot` ({(start, end): beta}) are beta * u, so a row's
    scores rise by ~16 beta (log2 units, head_dim 128) where it reaches those keys."""
    tens = wl.make_tensors(spec, device=device)
    d = spec.dims
    g = torch.Generator(device=device).manual_seed(spec.seed + 17)
    u = torch.randn(d.head_dim, generator=g, device=device)
    q = u + 0.1 * torch.randn(tens.q.shape, generator=g, device=device)
    tens.q.copy_(q.to(torch.bfloat16))
    qsl = np.concatenate([[0], np.cumsum(spec.num_scheduled)])
    for i in range(spec.num_reqs):
        c = int(spec.num_computed[i])
        for (s, e), beta in hot.items():
            key = (beta * u).to(torch.bfloat16)
            hs, he = min(s, c), min(e, c)          # hot keys in the history
            tens.hist_k[i][hs:he] = key
            ns, ne = max(s, c) - c, max(min(e, c + int(spec.num_scheduled[i])), c) - c
            tens.k[int(qsl[i]) + ns:int(qsl[i]) + ne] = key   # hot keys among the new tokens
    wl.place_history(spec, tens.hist_k, tens.k_cache)
    return tens
