"""Seeded synthetic workloads for one flattened mixed-batch step.

This module only builds inputs: the request structure (cached and scheduled
token counts), the persistent token table, a page table whose physical page ids
are a seeded random permutation, and random bf16 activations standing in for the
Q/K/V projections and the hidden states.  None of the step's own arithmetic is
here: no prefix sums, positions, slots, attention or gathers.  Both the CPU
oracle (``oracle/``) and the CUDA library consume what this module returns, and
neither is imported from here.

Recipe (all synthetic; the pages name no dataset):

* host structure: ``numpy.random.Generator(PCG64(seed))`` with
  ``seed = 1000 * config + step``;
* token ids uniform in [0, 32000);
* physical page ids: a seeded permutation of every page but the reserved null
  page (id 0 unless stated); unused page-table entries hold -1;
* Q/K/V/hidden: bf16 draws of N(0, 1) from a seeded ``torch.Generator``;
* cached history K/V: one contiguous bf16 tensor per request, placed page by
  page into the pool (the pool starts filled with N(0, 1) noise so stale or
  misplaced data is visible).
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import Iterator, List, Optional

import numpy as np

VOCAB = 32000

# Capture sizes quoted for vLLM's piecewise CUDA graphs (vLLM book, ch. 8,
# "8.4.3 实际效果" and "8.5 pad_for_cudagraph").
GRAPH_CAPTURE_SIZES = (1, 2, 4, 8, 16, 24, 32, 48, 64, 96, 128, 192, 256)


@dataclass(frozen=True)
class Dims:
    """Static sizes of the persistent batch and the paged KV pool (one layer)."""

    block_size: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    max_num_reqs: int
    max_model_len: int
    max_blocks_per_req: int
    num_blocks: int
    null_block: int = 0
    # page-table entries are manager blocks of this many kernel pages (block_size tokens each);
    # a manager block is kernel-page aligned and spans that many consecutive pages of the pool
    kernel_blocks_per_manager_block: int = 1

    @property
    def num_slots(self) -> int:
        return self.num_blocks * self.block_size


@dataclass
class BatchSpec:
    """Host-side description of one scheduled step (what the scheduler hands the runner)."""

    name: str
    dims: Dims
    num_computed: np.ndarray  # int32 [R]   tokens already in the KV cache
    num_scheduled: np.ndarray  # int32 [R]  tokens scheduled this step
    num_reqs_padded: int
    num_tokens_padded: int
    token_table: np.ndarray  # int32 [max_num_reqs, max_model_len]
    block_table: np.ndarray  # int32 [max_num_reqs, max_blocks_per_req], -1 = unused
    hidden_size: int
    seed: int
    num_prompt: Optional[np.ndarray] = None  # int32 [R] prompt lengths, where known
    shared_prefix_tokens: int = 0  # every request's first tokens, pages and history are shared

    @property
    def num_reqs(self) -> int:
        return int(self.num_scheduled.shape[0])

    @property
    def num_tokens(self) -> int:
        # the scheduler's own total (total_num_scheduled_tokens)
        return int(self.num_scheduled.sum(dtype=np.int64))


# --------------------------------------------------------------------------- #
# page allocation (a seeded free list; the KV-cache manager's job, not the step's)
# --------------------------------------------------------------------------- #
class PagePool:
    """Free list of physical pages in seeded random order; the null page is never handed out."""

    def __init__(self, num_blocks: int, null_block: int, rng: np.random.Generator):
        ids = np.array([b for b in range(num_blocks) if b != null_block], dtype=np.int64)
        self.free: List[int] = [int(x) for x in rng.permutation(ids)]
        self.in_use = 0
        self.peak = 0

    def take(self, n: int) -> List[int]:
        if n > len(self.free):
            raise RuntimeError(f"page pool exhausted: need {n}, have {len(self.free)}")
        out, self.free = self.free[:n], self.free[n:]
        self.in_use += n
        self.peak = max(self.peak, self.in_use)
        return out

    def give_back(self, pages: List[int]) -> None:
        self.free.extend(pages)
        self.in_use -= len(pages)


def pages_for(num_tokens: int, block_size: int) -> int:
    """Pages a request must own to hold ``num_tokens`` tokens (allocator rule)."""
    return -(-int(num_tokens) // block_size)


def _build_spec(name, dims, computed, scheduled, rng, hidden_size, seed,
                num_reqs_padded=None, num_tokens_padded=None, num_prompt=None,
                shared_prefix=0) -> BatchSpec:
    computed = np.asarray(computed, dtype=np.int32)
    scheduled = np.asarray(scheduled, dtype=np.int32)
    R = computed.shape[0]
    assert R <= dims.max_num_reqs
    token_table = np.zeros((dims.max_num_reqs, dims.max_model_len), dtype=np.int32)
    block_table = np.full((dims.max_num_reqs, dims.max_blocks_per_req), -1, dtype=np.int32)
    r = dims.kernel_blocks_per_manager_block
    pool = PagePool(dims.num_blocks // r, dims.null_block // r, rng)  # manager block ids
    n_shared = shared_prefix // (dims.block_size * r)
    assert n_shared * dims.block_size * r == shared_prefix, "shared prefix in whole entries"
    shared_pages = pool.take(n_shared) if n_shared else []
    shared_tokens = rng.integers(0, VOCAB, size=shared_prefix, dtype=np.int32)
    for i in range(R):
        total = int(computed[i]) + int(scheduled[i])
        token_table[i, :total] = rng.integers(0, VOCAB, size=total, dtype=np.int32)
        token_table[i, :shared_prefix] = shared_tokens
        n = pages_for(total, dims.block_size * r)
        block_table[i, :n_shared] = shared_pages
        block_table[i, n_shared:n] = pool.take(n - n_shared)
    n_tok = int(scheduled.sum(dtype=np.int64))
    if num_prompt is None:  # decodes: prompt already computed; longer queries finish their prompt
        num_prompt = [int(c) if int(q) == 1 else int(c) + int(q) for c, q in zip(computed, scheduled)]
    return BatchSpec(name=name, dims=dims, num_computed=computed, num_scheduled=scheduled,
                     num_reqs_padded=R if num_reqs_padded is None else num_reqs_padded,
                     num_tokens_padded=n_tok if num_tokens_padded is None else num_tokens_padded,
                     token_table=token_table, block_table=block_table, hidden_size=hidden_size,
                     seed=seed, num_prompt=None if num_prompt is None else np.asarray(num_prompt, np.int32),
                     shared_prefix_tokens=int(shared_prefix))


def _pool_blocks_for(computed, scheduled, block_size, slack=1.25, ratio=1) -> int:
    """Kernel pages of a pool with room for the batch (in whole manager blocks of ``ratio``
    pages, the null manager block included)."""
    need = sum(pages_for(int(c) + int(q), block_size * ratio) for c, q in zip(computed, scheduled))
    return (int(np.ceil(need * slack)) + 1) * ratio


def _round_up(x: int, m: int) -> int:
    return -(-x // m) * m


# --------------------------------------------------------------------------- #
# the five workloads
# --------------------------------------------------------------------------- #
def config1(step: int = 0, num_tokens_padded: Optional[int] = None) -> BatchSpec:
    """Pages' worked example: A prefill 7, B decode with 5 cached, C chunk 10 cached + 12 new.

    block_size 16, 64 physical pages, 4 q heads / 2 kv heads, head_dim 64.
    """
    seed = 1000 * 1 + step
    rng = np.random.default_rng(seed)
    dims = Dims(block_size=16, num_q_heads=4, num_kv_heads=2, head_dim=64, max_num_reqs=4,
                max_model_len=64, max_blocks_per_req=4, num_blocks=64, null_block=0)
    return _build_spec("worked example A/B/C", dims, [0, 5, 10], [7, 1, 12], rng, 256, seed,
                       num_tokens_padded=num_tokens_padded)


def config2(step: int = 0, manager_ratio: int = 1) -> BatchSpec:
    """Padding example: query_lens [2000, 512, 1 x 6]; decodes have 1000..4000 cached tokens.

    32 q heads / 8 kv heads, head_dim 128, block_size 16, hidden 4096.
    """
    seed = 1000 * 2 + step
    rng = np.random.default_rng(seed)
    scheduled = [2000, 512] + [1] * 6
    computed = [0, 0] + [int(x) for x in rng.integers(1000, 4000, size=6, endpoint=True)]
    M = _round_up(max(c + q for c, q in zip(computed, scheduled)), 16) + 16
    dims = Dims(block_size=16, num_q_heads=32, num_kv_heads=8, head_dim=128, max_num_reqs=8,
                max_model_len=M, max_blocks_per_req=-(-M // (16 * manager_ratio)),
                num_blocks=_pool_blocks_for(computed, scheduled, 16, ratio=manager_ratio),
                kernel_blocks_per_manager_block=manager_ratio)
    return _build_spec("padding example (2 prefills + 6 decodes)", dims, computed, scheduled, rng,
                       4096, seed)


def config3(step: int = 0, num_real: int = 256, manager_ratio: int = 1,
            context_scale: float = 1.0) -> BatchSpec:
    """Pure decode: ``num_real`` requests x 1 token, cached context U[512, 8192], padded to 256.

    ``num_real=256`` is the workload as stated (no padding tokens); ``num_real=250`` exercises the
    null-page route for 6 padding tokens and 6 padding requests.  ``context_scale`` < 1 shrinks
    every cached length by that factor (a smaller case of the same shape, e.g. for a profiler).
    """
    seed = 1000 * 3 + step + (0 if num_real == 256 else 500)
    rng = np.random.default_rng(seed)
    computed = [max(1, int(int(x) * context_scale))
                for x in rng.integers(512, 8192, size=num_real, endpoint=True)]
    scheduled = [1] * num_real
    M = _round_up(8192 + 1, 16)
    dims = Dims(block_size=16, num_q_heads=32, num_kv_heads=8, head_dim=128, max_num_reqs=256,
                max_model_len=M, max_blocks_per_req=-(-M // (16 * manager_ratio)),
                num_blocks=_pool_blocks_for(computed, scheduled, 16, ratio=manager_ratio),
                kernel_blocks_per_manager_block=manager_ratio)
    return _build_spec(f"pure decode ({num_real} real, padded to 256)", dims, computed, scheduled, rng,
                       4096, seed, num_reqs_padded=256, num_tokens_padded=256)


def config5(step: int = 0, pool_gb: float = 0.0, context_scale: float = 1.0) -> BatchSpec:
    """Long context: 8 decodes at 131072 cached + one 4096-token chunk with 65536 cached.

    64 q heads / 8 kv heads, head_dim 128, block_size 16.  One layer of the KV cache is
    materialised; ``pool_gb`` > 0 spreads the pages over a larger pool of that many GB (K+V).
    ``context_scale`` < 1 shrinks every cached length by that factor (a smaller case of the
    same shape, e.g. for a profiler).
    """
    seed = 1000 * 5 + step
    rng = np.random.default_rng(seed)
    computed = [int(131072 * context_scale)] * 8 + [int(65536 * context_scale)]
    scheduled = [1] * 8 + [4096]
    M = _round_up(max(c + q for c, q in zip(computed, scheduled)), 16) + 16
    nb = _pool_blocks_for(computed, scheduled, 16)
    if pool_gb > 0:
        page_bytes = 2 * 16 * 8 * 128 * 2
        nb = max(nb, int(pool_gb * 1e9 // page_bytes))
    dims = Dims(block_size=16, num_q_heads=64, num_kv_heads=8, head_dim=128, max_num_reqs=9,
                max_model_len=M, max_blocks_per_req=M // 16, num_blocks=nb)
    return _build_spec("long context (8 x 131072 decodes + 4096 chunk at 65536)", dims, computed,
                       scheduled, rng, 8192, seed)


def random_batch(seed: int, *, max_reqs: int = 6, max_q: int = 40, max_c: int = 90,
                 block_size: int = 16, num_q_heads: int = 4, num_kv_heads: int = 2,
                 head_dim: int = 64, pad_tokens: int = 0, pad_reqs: int = 0,
                 decode_frac: float = 0.4, hidden_size: int = 128,
                 manager_ratio: int = 1) -> BatchSpec:
    """A small ragged mix for fuzzing: a seeded blend of decodes, fresh prefills and chunks."""
    rng = np.random.default_rng(seed)
    R = int(rng.integers(1, max_reqs + 1))
    computed, scheduled = [], []
    for _ in range(R):
        u = rng.random()
        if u < decode_frac:
            computed.append(int(rng.integers(1, max_c + 1)))
            scheduled.append(1)
        elif u < decode_frac + 0.3:
            computed.append(0)
            scheduled.append(int(rng.integers(1, max_q + 1)))
        else:
            computed.append(int(rng.integers(1, max_c + 1)))
            scheduled.append(int(rng.integers(1, max_q + 1)))
    M = _round_up(max_c + max_q + 1, block_size) + block_size
    r = manager_ratio
    dims = Dims(block_size=block_size, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                head_dim=head_dim, max_num_reqs=R + pad_reqs + 1, max_model_len=M,
                max_blocks_per_req=-(-M // (block_size * r)),
                num_blocks=_pool_blocks_for(computed, scheduled, block_size, ratio=r) + 3 * r,
                kernel_blocks_per_manager_block=r)
    n = sum(scheduled)
    spec = _build_spec(f"random mix seed={seed}", dims, computed, scheduled, rng, hidden_size,
                       seed, num_reqs_padded=R + pad_reqs, num_tokens_padded=n + pad_tokens)
    # some chunks stop inside their prompt (drawn last so the other draws do not move)
    extra = rng.integers(0, 2, size=R) * rng.integers(1, max_q + 1, size=R)
    spec.num_prompt = np.where(spec.num_scheduled > 1, spec.num_prompt + extra,
                               spec.num_prompt).astype(np.int32)
    return spec


def batch_from_lists(num_computed, num_scheduled, *, block_size=16, num_q_heads=4, num_kv_heads=2,
                     head_dim=64, seed=0, num_reqs_padded=None, num_tokens_padded=None,
                     hidden_size=128, extra_blocks=3, max_model_len=None,
                     manager_ratio=1) -> BatchSpec:
    """A batch with the given per-request counts (and seeded pages/tokens)."""
    rng = np.random.default_rng(seed)
    mx = max([c + q for c, q in zip(num_computed, num_scheduled)] + [1])
    M = max_model_len or (_round_up(mx, block_size) + block_size)
    R = len(num_scheduled)
    r = manager_ratio
    dims = Dims(block_size=block_size, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                head_dim=head_dim, max_num_reqs=max(R, num_reqs_padded or 0, 1), max_model_len=M,
                max_blocks_per_req=-(-M // (block_size * r)),
                num_blocks=(_pool_blocks_for(num_computed, num_scheduled, block_size, ratio=r)
                            + extra_blocks * r),
                kernel_blocks_per_manager_block=r)
    return _build_spec("explicit", dims, num_computed, num_scheduled, rng, hidden_size, seed,
                       num_reqs_padded=num_reqs_padded, num_tokens_padded=num_tokens_padded)


def shared_prefix_batch(seed: int, *, num_decodes: int, prefix_tokens: int,
                        suffix_range=(16, 1024), num_chunks: int = 0, chunk_q: int = 512,
                        num_q_heads: int = 32, num_kv_heads: int = 8, head_dim: int = 128,
                        block_size: int = 16, manager_ratio: int = 1,
                        hidden_size: int = 4096) -> BatchSpec:
    """Requests that all start with the same ``prefix_tokens`` (a shared system prompt: same
    token ids, same pages, same cached K/V): ``num_decodes`` decodes with U[suffix_range] own
    cached tokens after the prefix, and ``num_chunks`` prefill chunks of ``chunk_q`` new tokens
    on top of U[0, 256] own cached tokens."""
    rng = np.random.default_rng(seed)
    lo, hi = suffix_range
    computed = [prefix_tokens + int(x) for x in rng.integers(lo, hi, size=num_decodes, endpoint=True)]
    scheduled = [1] * num_decodes
    for _ in range(num_chunks):
        computed.append(prefix_tokens + int(rng.integers(0, 256, endpoint=True)))
        scheduled.append(chunk_q)
    M = _round_up(max(c + q for c, q in zip(computed, scheduled)), block_size * manager_ratio) + \
        block_size * manager_ratio
    r = manager_ratio
    dims = Dims(block_size=block_size, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                head_dim=head_dim, max_num_reqs=len(computed), max_model_len=M,
                max_blocks_per_req=-(-M // (block_size * r)),
                num_blocks=_pool_blocks_for(computed, scheduled, block_size, ratio=r) + 2 * r,
                kernel_blocks_per_manager_block=r)
    return _build_spec(f"shared prefix {prefix_tokens} x {len(computed)} requests", dims,
                       computed, scheduled, rng, hidden_size, seed, shared_prefix=prefix_tokens)


# --------------------------------------------------------------------------- #
# chunked-prefill mixed workload: a request stream, one scheduler output per step
# --------------------------------------------------------------------------- #
@dataclass
class NewRequest:
    """A request entering the persistent batch with its whole state."""

    req_id: int
    num_computed: int
    num_prompt: int
    tokens: np.ndarray   # int32 history known so far (prompt, then any outputs)
    blocks: np.ndarray   # int32 page ids of the request's first len(blocks) pages


@dataclass
class CachedDelta:
    """What a resident request adds this step."""

    req_id: int
    num_computed: int
    new_tokens: np.ndarray            # int32, appended to the request's history
    new_blocks: np.ndarray            # int32, appended to its page row (or the whole row)
    replace_blocks: bool = False      # resumed from preemption: the page row is replaced


@dataclass
class SchedulerStep:
    """One step's scheduler output, keyed by request id (no batch rows in it)."""

    scheduled: "dict"                 # req_id -> tokens scheduled this step (insertion order)
    new: List[NewRequest] = field(default_factory=list)
    cached: List[CachedDelta] = field(default_factory=list)

    @property
    def num_tokens(self) -> int:
        return int(sum(self.scheduled.values()))


@dataclass
class _Req:
    uid: int
    kind: str  # "chunk" or "decode"
    computed: int
    prompt_len: int
    tokens: np.ndarray      # every token this request will ever show (drawn at arrival)
    sent: int = 0           # history tokens already handed to the batch
    pages: List[int] = field(default_factory=list)


class MixedChunkStream:
    """Request stream of the 8192-token-budget chunked-prefill workload.

    It starts with 4 chunked-prefill requests (chunks of U[1024, 2048] tokens on top of
    U[0, 16384] prior context, prompts U[4096, 24576] tokens longer) and 128 decodes (context
    U[256, 32768]).  A chunked prefill leaves when its prompt is done; every request leaves
    with probability 5% per step (or near the model length); a fresh request of the same kind
    arrives one step later.  A running decode is preempted with probability 1% per step: it
    sits out one step and then comes back as a new request carrying its history; with another
    1% its page row is replaced by fresh pages.  Chunk lengths are drawn first and then shrunk
    in proportion until the step fits the token budget.

    Each step is emitted as a ``SchedulerStep`` keyed by request id; which batch row holds a
    request is the runner's business, not the stream's.
    """

    BUDGET = 8192
    N_CHUNK = 4
    N_DECODE = 128
    FINISH_P = 0.05
    PREEMPT_P = 0.01
    REPLACE_P = 0.01

    def __init__(self, seed: int = 4000, num_blocks: int = 180_001, max_model_len: int = 65536,
                 max_num_reqs: int = 160):
        self.rng = np.random.default_rng(seed)
        self.seed = seed
        self.dims = Dims(block_size=16, num_q_heads=32, num_kv_heads=8, head_dim=128,
                         max_num_reqs=max_num_reqs, max_model_len=max_model_len,
                         max_blocks_per_req=max_model_len // 16, num_blocks=num_blocks)
        self.pool = PagePool(num_blocks, 0, self.rng)
        self.running: List[_Req] = []
        self.arrivals: List[str] = []
        self.resuming: List[_Req] = []
        self.next_uid = 0
        self.step_index = 0
        self.fresh: List[_Req] = []
        for kind in ["chunk"] * self.N_CHUNK + ["decode"] * self.N_DECODE:
            self.running.append(self._draw(kind))
        self.fresh = list(self.running)

    def _draw(self, kind: str) -> _Req:
        M = self.dims.max_model_len
        if kind == "chunk":
            c = int(self.rng.integers(0, 16384, endpoint=True))
            prompt = min(M - 1, c + int(self.rng.integers(4096, 24576, endpoint=True)))
        else:
            c = int(self.rng.integers(256, 32768, endpoint=True))
            prompt = c
        toks = self.rng.integers(0, VOCAB, size=M, dtype=np.int32)
        r = _Req(uid=self.next_uid, kind=kind, computed=c, prompt_len=prompt, tokens=toks)
        self.next_uid += 1
        return r

    def _retire(self) -> None:
        """Requests that finished or were preempted after the previous step leave."""
        M = self.dims.max_model_len
        keep, finished, preempted = [], [], []
        for r in self.running:
            done = (r.kind == "chunk" and r.computed >= r.prompt_len) or \
                r.computed + 2048 >= M or self.rng.random() < self.FINISH_P
            if done:
                self.pool.give_back(r.pages)
                finished.append(r.kind)
            elif r.kind == "decode" and self.rng.random() < self.PREEMPT_P:
                self.pool.give_back(r.pages)
                r.pages, r.sent = [], 0
                preempted.append(r)
            else:
                keep.append(r)
        self.fresh = [self._draw(kind) for kind in self.arrivals] + self.resuming
        self.running = keep + self.fresh
        self.arrivals, self.resuming = finished, preempted

    def next_step(self) -> SchedulerStep:
        if self.step_index > 0:
            self._retire()
        fresh = {r.uid for r in self.fresh}
        replace = {r.uid for r in self.running
                   if r.uid not in fresh and r.kind == "decode" and self.rng.random() < self.REPLACE_P}
        q = []
        for r in self.running:
            if r.kind == "chunk":
                q.append(int(self.rng.integers(1024, 2048, endpoint=True)))
            else:
                q.append(1)
        chunk_idx = [i for i, r in enumerate(self.running) if r.kind == "chunk"]
        total = sum(q)
        if total > self.BUDGET and chunk_idx:
            room = self.BUDGET - (total - sum(q[i] for i in chunk_idx))
            scale = room / sum(q[i] for i in chunk_idx)
            for i in chunk_idx:
                q[i] = max(1, int(q[i] * scale))
        for i, r in enumerate(self.running):  # the last chunk of a prompt stops at its end
            if r.kind == "chunk" and r.computed < r.prompt_len:
                q[i] = min(q[i], r.prompt_len - r.computed)

        step = SchedulerStep(scheduled={})
        B = self.dims.block_size
        for i, r in enumerate(self.running):
            step.scheduled[r.uid] = q[i]
            need_tokens = max(r.computed + q[i], r.prompt_len if r.uid in fresh else 0)
            if r.uid in fresh:
                r.pages = self.pool.take(pages_for(r.computed + q[i], B))
                r.sent = need_tokens
                step.new.append(NewRequest(r.uid, r.computed, r.prompt_len,
                                           r.tokens[:r.sent].copy(),
                                           np.array(r.pages, np.int32)))
                continue
            if r.uid in replace:
                self.pool.give_back(r.pages)
                r.pages = []
            add = self.pool.take(pages_for(r.computed + q[i], B) - len(r.pages))
            new_tokens = r.tokens[r.sent:need_tokens].copy() if need_tokens > r.sent else \
                np.zeros(0, np.int32)
            r.sent = max(r.sent, need_tokens)
            r.pages = r.pages + add
            step.cached.append(CachedDelta(
                r.uid, r.computed, new_tokens,
                np.array(r.pages if r.uid in replace else add, np.int32),
                replace_blocks=r.uid in replace))
        for i, r in enumerate(self.running):
            r.computed += q[i]
        self.step_index += 1
        return step


def config4_stream(num_steps: int = 100, seed: int = 4000) -> Iterator[SchedulerStep]:
    stream = MixedChunkStream(seed=seed)
    for _ in range(num_steps):
        yield stream.next_step()


def spec_from_columns(name: str, dims: Dims, num_computed, num_scheduled, num_prompt,
                      token_table: np.ndarray, block_table: np.ndarray, seed: int,
                      hidden_size: int = 4096) -> BatchSpec:
    """A step description from a persistent batch's row-order columns (no padding)."""
    num_scheduled = np.asarray(num_scheduled, np.int32)
    return BatchSpec(name=name, dims=dims, num_computed=np.asarray(num_computed, np.int32),
                     num_scheduled=num_scheduled, num_reqs_padded=int(num_scheduled.shape[0]),
                     num_tokens_padded=int(num_scheduled.sum(dtype=np.int64)),
                     token_table=token_table, block_table=block_table, hidden_size=hidden_size,
                     seed=seed, num_prompt=np.asarray(num_prompt, np.int32))

# --------------------------------------------------------------------------- #
# activations and the paged pool (torch; CPU or CUDA)
# --------------------------------------------------------------------------- #
@dataclass
class Tensors:
    """bf16 tensors of one step: new Q/K/V rows, hidden rows, per-request history, the pool."""

    q: "object"  # [N_pad, nh, hd]
    k: "object"  # [N_pad, nkv, hd]
    v: "object"  # [N_pad, nkv, hd]
    hidden: "object"  # [N_pad, H]
    hist_k: list  # per request [c_i, nkv, hd]
    hist_v: list
    k_cache: "object"  # [num_blocks * B, nkv, hd]
    v_cache: "object"


def make_tensors(spec: BatchSpec, device="cpu", with_pool: bool = True, with_history: bool = True):
    """Seeded bf16 activations; the history of request i is placed page by page into the pool."""
    import torch

    d = spec.dims
    g = torch.Generator(device=device)
    g.manual_seed(spec.seed)
    Np = spec.num_tokens_padded
    bf = torch.bfloat16

    def randn(*shape):
        return torch.randn(*shape, generator=g, device=device, dtype=torch.float32).to(bf)

    q = randn(Np, d.num_q_heads, d.head_dim)
    k = randn(Np, d.num_kv_heads, d.head_dim)
    v = randn(Np, d.num_kv_heads, d.head_dim)
    hidden = randn(Np, spec.hidden_size)
    hist_k, hist_v = [], []
    if with_history:
        P = spec.shared_prefix_tokens
        if P:  # one history for the shared prefix, then each request's own
            pk, pv = randn(P, d.num_kv_heads, d.head_dim), randn(P, d.num_kv_heads, d.head_dim)
        for i in range(spec.num_reqs):
            c = int(spec.num_computed[i])
            if P:
                hist_k.append(torch.cat([pk, randn(c - P, d.num_kv_heads, d.head_dim)]))
                hist_v.append(torch.cat([pv, randn(c - P, d.num_kv_heads, d.head_dim)]))
            else:
                hist_k.append(randn(c, d.num_kv_heads, d.head_dim))
                hist_v.append(randn(c, d.num_kv_heads, d.head_dim))
    k_cache = v_cache = None
    if with_pool:
        k_cache = randn(d.num_slots, d.num_kv_heads, d.head_dim)
        v_cache = randn(d.num_slots, d.num_kv_heads, d.head_dim)
        if with_history:
            place_history(spec, hist_k, k_cache)
            place_history(spec, hist_v, v_cache)
    return Tensors(q=q, k=k, v=v, hidden=hidden, hist_k=hist_k, hist_v=hist_v,
                   k_cache=k_cache, v_cache=v_cache)


def place_history(spec: BatchSpec, hist: list, cache) -> None:
    """Copy each request's contiguous history into its pages, one whole page-table entry (a
    manager block of consecutive kernel pages) at a time."""
    import torch

    d = spec.dims
    r = d.kernel_blocks_per_manager_block
    B = d.block_size * r  # tokens per page-table entry: one manager block of r kernel pages
    pages = cache.view(d.num_blocks // r, B, d.num_kv_heads, d.head_dim)
    for i, h in enumerate(hist):
        c = h.shape[0]
        full = c // B
        row = torch.as_tensor(spec.block_table[i], device=cache.device, dtype=torch.long)
        if full:
            pages[row[:full]] = h[: full * B].view(full, B, d.num_kv_heads, d.head_dim)
        rem = c - full * B
        if rem:
            pages[int(spec.block_table[i, full]), :rem] = h[full * B:]


def device_tables(spec: BatchSpec, device):
    """The persistent arrays as int32 device tensors (token table, page table, counters)."""
    import torch

    def t(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(device)

    out = dict(token_table=t(spec.token_table), block_table=t(spec.block_table),
               num_computed=t(spec.num_computed), num_scheduled=t(spec.num_scheduled))
    if spec.num_prompt is not None:
        out["num_prompt"] = t(spec.num_prompt)
    return out


def with_padding(spec: BatchSpec, num_reqs_padded: int, num_tokens_padded: int) -> BatchSpec:
    return dataclasses.replace(spec, num_reqs_padded=num_reqs_padded,
                               num_tokens_padded=num_tokens_padded)


class RandomRequestStream:
    """Small seeded request streams for fuzzing the batch update: arrivals, finishes, requests
    the scheduler skips for a step (they come back later as new requests with their history),
    ids resubmitted while still resident, deltas with appended tokens and page ids, and
    replaced page rows.  Request-level only: it never decides which row holds what."""

    def __init__(self, seed: int, max_live: int = 12, max_model_len: int = 64,
                 max_blocks: int = 8, p_finish: float = 0.2, p_skip: float = 0.1,
                 p_resubmit: float = 0.05, p_replace: float = 0.1):
        self.rng = np.random.default_rng(seed)
        self.max_live, self.M, self.MB = max_live, max_model_len, max_blocks
        self.max_rows = max_live
        self.p = dict(finish=p_finish, skip=p_skip, resubmit=p_resubmit, replace=p_replace)
        self.live: dict = {}     # id -> [computed, prompt, tokens list, blocks list]
        self.parked: dict = {}   # skipped last step: id -> state, back as new next time
        self.next_id = 0

    def _fresh_state(self):
        n = int(self.rng.integers(1, self.M // 2))
        toks = [int(x) for x in self.rng.integers(0, VOCAB, size=n)]
        blocks = [int(x) for x in self.rng.integers(1, 10_000, size=int(self.rng.integers(0, self.MB // 2 + 1)))]
        return [int(self.rng.integers(0, n + 1)), n, toks, blocks]

    def next_step(self) -> SchedulerStep:
        rng, p = self.rng, self.p
        step = SchedulerStep(scheduled={})
        back, self.parked = self.parked, {}
        for i, st in list(self.live.items()):
            u = rng.random()
            if u < p["finish"] or len(st[2]) >= self.M - 4 or len(st[3]) >= self.MB - 2:
                del self.live[i]
            elif u < p["finish"] + p["skip"]:
                self.parked[i] = self.live.pop(i)
        for i, st in back.items():  # skipped last step: the batch dropped it, resend it whole
            self.live[i] = st
        arrivals = int(rng.integers(0, 4))
        for _ in range(arrivals):
            if len(self.live) + len(self.parked) >= self.max_live:
                break
            self.live[self.next_id] = self._fresh_state()
            self.next_id += 1
        fresh = set(back) | set(range(self.next_id - arrivals, self.next_id))
        for i, st in self.live.items():
            step.scheduled[i] = int(rng.integers(1, 6))
            if i not in fresh and rng.random() < p["resubmit"]:
                st[:] = self._fresh_state()
                fresh.add(i)
            if i in fresh:
                step.new.append(NewRequest(i, st[0], st[1], np.array(st[2], np.int32),
                                           np.array(st[3], np.int32)))
                continue
            if rng.random() < 0.3:
                continue  # resident and unchanged: no delta this step
            toks = [int(x) for x in rng.integers(0, VOCAB, size=int(rng.integers(0, 4)))]
            replace = rng.random() < p["replace"]
            nb = int(rng.integers(1, self.MB // 2 + 1)) if replace else int(rng.integers(0, 3))
            blocks = [int(x) for x in rng.integers(1, 10_000, size=nb)]
            st[0] = min(len(st[2]) + len(toks), st[0] + int(rng.integers(0, 4)))
            st[2] = st[2] + toks
            st[3] = blocks if replace else st[3] + blocks
            step.cached.append(CachedDelta(i, st[0], np.array(toks, np.int32),
                                           np.array(blocks, np.int32), replace_blocks=replace))
        return step
