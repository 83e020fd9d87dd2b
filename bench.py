#!/usr/bin/env python
"""Throughput of the flattened mixed-batch step on GB300, one attention layer, synthetic data.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config C]

Prints ONE JSON line on rank 0.

Headline workload (``--config 4``, the default): the chunked-prefill mix as a seeded request
stream with an 8192-token budget -- 4 chunked prefills of U[1024, 2048] tokens on U[0, 16384]
cached tokens and 128 decodes on U[256, 32768] cached tokens, 32 q / 8 kv heads, head_dim 128,
pages of 16 tokens, requests finishing, arriving, being preempted and having their page rows
replaced -- over max(100, W + K) scheduler steps.  One step is the whole hot path on the
device: ``rb_batch_apply_update`` (the scheduler's deltas merged into the device-resident
persistent batch, its packet staged in device memory before the timed region) and one
``rb_step`` (metadata, KV write, paged attention, last-token row gather).  Steps 0..W-1 warm
up; steps W..W+K-1 are timed; the rest of the stream runs after the timed region and is
reported as ``stream_all``.  ``value`` = real tokens of the timed steps / their device time.

In the same line, ``configs`` carries the other single-GPU workloads, each timed as a captured
``rb_step`` graph replayed with a cold L2 (median of its steps): ``2`` the pages' padding
example, ``3`` pure decode (256 x U[512, 8192]), ``5`` long context (8 decodes at 131072 plus a
4096-token chunk on 65536, 64 q heads); each with the roofline of its dominant kernel.
``--config 2|3|5`` makes one of them the headline instead.

Timing: CUDA events on the launching stream around each step, a 512 MiB write between steps
(outside the events) so every step starts with a cold L2, barrier + synchronize around the
whole region, max over ranks.  Under torchrun every rank runs its own independent stream
(data parallel: no collective on the data path).  ``e2e``: the same steps through the public
API with host buffers (the scheduler packet and q / k / v / hidden copied in from pinned host
memory, the attention output, gathered rows and scalars copied back, every step synchronised),
wall clock.  ``cpu_baseline``: the CPU oracle (float64) on a bounded row sample of the same
workload, on all host cores (each request's rows in pieces of about equal cost, one per thread).  ``--impl reference`` times that oracle
alone on the headline workload.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import math
import os
import platform
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "mixed-step tokens/s; decode-attn HBM GB/s & prefill TFLOPS vs peak"
UNIT = "tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
STREAM_STEPS = 100
HIDDEN = 4096
FLUSH_BYTES = 512 << 20

# DRAM bytes (read + write) per launch of the fused attention kernel measured by ncu
# (dram__bytes_read.sum + dram__bytes_write.sum), keyed by (workload, hash of the kernel's and
# its planner's code, comments left out): a figure is reported only while the code is the code
# it was measured on.
KNOWN_TRAFFIC = {
    (2, "9a8026878da7e19f"): 78976256 + 3943680,
    (3, "9a8026878da7e19f"): 4545474816 + 26148352,
    # the stream: mean over the launches of stream steps 5..99 (the default timed steps)
    (4, "9a8026878da7e19f"): 9567950312 + 80911815,
    (5, "9a8026878da7e19f"): 8588893440 + 115581440,
}

WORKLOAD_NAMES = {1: "pages' worked example A/B/C", 2: "pages' padding example",
                  3: "pure decode x256", 4: "chunked-prefill mix stream (8192-token budget)",
                  5: "long-context 70B-like step"}


# ----------------------------------------------------------------------------- workloads
def make_spec(config: int, rank: int = 0, manager_ratio: int = 1, context_scale: float = 1.0):
    import workloads as wl

    if config == 1:
        return wl.config1(step=rank)
    if config == 2:
        return wl.config2(step=rank, manager_ratio=manager_ratio)
    if config == 3:
        return wl.config3(step=rank, manager_ratio=manager_ratio, context_scale=context_scale)
    if config == 5:
        return wl.config5(step=rank, context_scale=context_scale)
    raise SystemExit(f"config {config} is not a single fixed batch")


def stream_seed(rank: int) -> int:
    return 4000 + 7919 * rank


def stream_steps(rank: int, n: int):
    """The first n scheduler outputs of this rank's chunked-prefill request stream."""
    import workloads as wl

    stream = wl.MixedChunkStream(seed=stream_seed(rank))
    return stream, [stream.next_step() for _ in range(n)]


def step_cq(step):
    """(cached, scheduled) token counts of every request of a scheduler step, in schedule
    order (the counts the scheduler hands the runner)."""
    computed = {n.req_id: int(n.num_computed) for n in step.new}
    computed.update({c.req_id: int(c.num_computed) for c in step.cached})
    return [(computed[i], int(q)) for i, q in step.scheduled.items()]


def work_of(cq, nh, nkv, hd, block_size, N, Np, R, Rp, hidden):
    """Algorithmic work of a step (what the pages define, not what the kernels do)."""
    g = nh // nkv
    dec_bytes = pre_flops = dec_flops = 0
    for c, q in cq:
        visible = q * c + q * (q + 1) // 2                 # sum over j of (c + j + 1)
        flops = 4 * nh * hd * visible
        if q * g <= 8:  # decode-like: bound by reading the request's K/V once per kv head
            L = c + q
            dec_bytes += L * 2 * nkv * hd * 2 + 2 * q * nh * hd * 2 + -(-L // block_size) * 4
            dec_flops += flops
        else:
            pre_flops += flops
    row = nkv * hd * 2
    return dict(prefill_flops=pre_flops, decode_flops=dec_flops, decode_bytes=dec_bytes,
                kv_write_bytes=2 * 2 * Np * row,
                meta_bytes=Np * (4 + 4 + 3 * 4) + R * (2 * 4 + 3 * 4),
                gather_bytes=2 * Rp * hidden * 2)


def spec_work(spec):
    d = spec.dims
    cq = list(zip(spec.num_computed.tolist(), spec.num_scheduled.tolist()))
    return work_of(cq, d.num_q_heads, d.num_kv_heads, d.head_dim, d.block_size, spec.num_tokens,
                   spec.num_tokens_padded, spec.num_reqs, spec.num_reqs_padded, spec.hidden_size)


def fixed_config_desc(spec, config):
    d = spec.dims
    return {
        "workload": WORKLOAD_NAMES[config],
        "query_lens": (spec.num_scheduled.tolist() if spec.num_reqs <= 9
                       else f"{spec.num_reqs} requests"),
        "num_reqs": spec.num_reqs, "num_tokens": spec.num_tokens,
        "num_tokens_padded": spec.num_tokens_padded, "q_heads": d.num_q_heads,
        "kv_heads": d.num_kv_heads, "head_dim": d.head_dim, "block_size": d.block_size,
        "hidden": spec.hidden_size, "kv_pages": d.num_blocks,
        "kernel_pages_per_table_entry": d.kernel_blocks_per_manager_block,
        "l2": "flushed before every timed step (512 MiB write, outside the events)",
    }


def stream_config_desc(dims, warmup, steps, total):
    return {
        "workload": WORKLOAD_NAMES[4],
        "stream": f"{total} seeded scheduler steps (seed {stream_seed(0)} + 7919 x rank); "
                  f"steps {warmup}..{warmup + steps - 1} timed",
        "mix": "4 chunks U[1024, 2048] on U[0, 16384] cached + 128 decodes on U[256, 32768] "
               "cached, budget 8192 tokens; 5% finish / 1% preempt / 1% page-row replace "
               "per step",
        "q_heads": dims.num_q_heads, "kv_heads": dims.num_kv_heads, "head_dim": dims.head_dim,
        "block_size": dims.block_size, "hidden": HIDDEN, "kv_pages": dims.num_blocks,
        "max_num_reqs": dims.max_num_reqs, "max_model_len": dims.max_model_len,
        "step": "rb_batch_apply_update (packet pre-staged in HBM) + rb_step, eager",
        "l2": "flushed before every timed step (512 MiB write, outside the events)",
    }


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


FUSED_SOURCES = ("attn_prefill_tc.cu", "attn_decode_warp.cuh", "tc_ptx.cuh", "attn_common.cuh",
                 "rb_internal.cuh", "attn_plan.cuh")


def _code_only(text: str) -> str:
    """Source text without comments, blank lines and runs of spaces (an edit of comments or
    layout keeps the hash)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    lines = (" ".join(re.sub(r"//.*", "", ln).split()) for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_sources_hash():
    """Hash of the code the fused attention kernel and its planner are built from."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ragged_mixed_paged_gb300", "csrc")
    for f in FUSED_SOURCES:
        with open(os.path.join(csrc, f), encoding="utf-8") as fh:
            h.update(f.encode() + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def roofline(work, launch_s, config, launches=1):
    """Roofline of the fused attention launch: the dominant resource's algorithmic work (prefill
    FLOPs or decode bytes, whichever takes longer at peak) over the measured launch time."""
    pk, pk_kind = peaks()
    t_tensor = work["prefill_flops"] / (pk["bf16_tflops"] * 1e12)
    t_hbm = work["decode_bytes"] / (pk["hbm_gbs"] * 1e9)
    tensor_bound = t_tensor >= t_hbm
    tflops = work["prefill_flops"] / launch_s / 1e12
    gbs = work["decode_bytes"] / launch_s / 1e9
    achieved = tflops if tensor_bound else gbs
    peak = pk["bf16_tflops"] if tensor_bound else pk["hbm_gbs"]
    traffic = KNOWN_TRAFFIC.get((config, kernel_sources_hash()))
    return {"bound": "tensor" if tensor_bound else "hbm", "achieved": achieved, "peak": peak,
            "unit": "TFLOP/s" if tensor_bound else "GB/s", "frac": achieved / peak,
            "traffic": traffic,
            "kernel": "attn_prefill_tc_kernel (fused launch: split-KV decode units + tcgen05 "
                      "prefill units)",
            "launch_ms": launch_s * 1000.0 / launches,
            "tensor_frac": tflops / pk["bf16_tflops"],
            "tensor_frac_sustained": tflops / pk["bf16_tflops_sustained"],
            "hbm_frac": gbs / pk["hbm_gbs"],
            "overlap_frac": max(t_tensor, t_hbm) / launch_s,
            "peak_kind": f"{'bf16 dense burst' if tensor_bound else 'HBM copy'}, {pk_kind}",
            "work_per_launch": {"prefill_gflop": work["prefill_flops"] / 1e9 / launches,
                                "decode_kv_gb": work["decode_bytes"] / 1e9 / launches}}


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        try:
            import torch

            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.ident = uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"
        except Exception:
            self.ident = str(device_index)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.ident, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        sm, mx, reasons = [], [], set()
        for line in out.strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, val in zip(self.NAMES, parts[3:7]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- ranks
def dist_setup(backend=None):
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0
    import torch
    import torch.distributed as dist

    local = int(os.environ.get("LOCAL_RANK", "0"))
    if backend is None:
        backend = "nccl" if torch.cuda.is_available() else "gloo"
    if backend == "nccl":
        torch.cuda.set_device(local)
    dist.init_process_group(backend)
    return dist.get_rank(), dist.get_world_size(), local


def reduce_over_ranks(value: float, op: str, world: int, device=None) -> float:
    """max / sum of a float over all ranks (timing bookkeeping only, never step data)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ----------------------------------------------------------------------------- oracle (CPU)
def host_cpu():
    """CPU model and the cores this process may use."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if model is None:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith(("model name", "cpu part")):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return {"model": model or platform.processor() or platform.machine(),
            "arch": platform.machine(), "host_cores": len(os.sched_getaffinity(0))}


class OracleStream:
    """The oracle's side of the chunked-prefill stream on the host: its persistent batch, one
    layer's K/V pool (bf16 bit patterns, lazily zero), and random float32 activations and
    histories (a request's history is a prefix of one shared random array: the oracle reads
    histories, never the pool, and any values will do)."""

    def __init__(self, rank):
        import numpy as np

        from oracle.persistent_batch import InputBatch

        self.stream, _ = stream_steps(rank, 0)
        d = self.dims = self.stream.dims
        self.batch = InputBatch(d.max_num_reqs, d.max_model_len, d.max_blocks_per_req)
        self.k_pool = np.zeros((d.num_slots, d.num_kv_heads, d.head_dim), np.int16)
        self.v_pool = np.zeros_like(self.k_pool)
        rng = np.random.default_rng(stream_seed(rank) + 99)
        shape = (d.max_model_len, d.num_kv_heads, d.head_dim)
        self.hist_k = rng.standard_normal(shape, np.float32)
        self.hist_v = rng.standard_normal(shape, np.float32)
        n = self.stream.BUDGET
        self.q = rng.standard_normal((n, d.num_q_heads, d.head_dim)).astype(np.float64)
        self.k = rng.standard_normal((n, d.num_kv_heads, d.head_dim)).astype(np.float64)
        self.v = rng.standard_normal((n, d.num_kv_heads, d.head_dim)).astype(np.float64)
        bits = lambda a: (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        self.k16, self.v16 = bits(self.k).view(np.int16), bits(self.v).view(np.int16)
        self.hidden = np.zeros((n, HIDDEN), np.int16)

    def advance(self):
        """The next scheduler step (not yet merged into the oracle's batch)."""
        return self.stream.next_step()

    def timed_step(self, step, row_stride, offset):
        """The oracle's whole step: the batch merge, metadata for every token, the KV write,
        attention for every ``row_stride``-th query row (all heads), the row gather.  Returns
        (seconds, rows evaluated, process CPU seconds)."""
        import numpy as np

        import oracle
        from oracle.threads import oracle_attention_threads

        d = self.dims
        N = step.num_tokens
        rows = list(range(offset % row_stride, N, row_stride))
        c0, w0 = time.process_time(), time.perf_counter()
        self.batch.apply(step)
        cols = self.batch.columns(step.scheduled)
        tok, blk = self.batch.tables()
        meta = oracle.prepare_inputs(block_size=d.block_size, null_block=d.null_block,
                                     token_table=tok, block_table=blk,
                                     num_computed=cols["num_computed"],
                                     num_scheduled=cols["num_scheduled"],
                                     num_prompt=cols["num_prompt"])
        oracle.kv_write(self.k_pool, self.v_pool, meta["slot_mapping"], self.k16[:N],
                        self.v16[:N])
        c = cols["num_computed"].tolist()
        a0, ca0 = time.perf_counter(), time.process_time()
        oracle_attention_threads(self.q[:N], [self.hist_k[:x] for x in c],
                                 [self.hist_v[:x] for x in c], self.k[:N], self.v[:N],
                                 meta["query_start_loc"], meta["seq_lens"], len(c), rows)
        attn, attn_cpu = time.perf_counter() - a0, time.process_time() - ca0
        oracle.gather_rows(self.hidden[:N], meta["logits_indices"])
        wall = time.perf_counter() - w0
        return {"wall": wall, "attn": attn, "attn_cpu": attn_cpu, "rows": len(rows),
                "cpu": time.process_time() - c0}


def oracle_stream_run(rank, warmup, steps, budget_s):
    """The oracle over the stream: W warm-up steps (the last one a full step with a small row
    sample, the others only merged into the batch), then K timed steps whose row sample is
    sized so they take about ``budget_s`` together (the probe step's attention time per row
    and its time outside attention)."""
    os_ = OracleStream(rank)
    probe = None
    for w in range(warmup):
        step = os_.advance()
        if w < warmup - 1:
            os_.batch.apply(step)
            continue
        probe = os_.timed_step(step, 64, w)
    per_row = probe["attn"] / max(probe["rows"], 1) if probe else 0.1
    fixed = probe["wall"] - probe["attn"] if probe else 5.0
    rows_budget = max(1.0, (budget_s / max(steps, 1) - fixed) / max(per_row, 1e-6))
    stride = max(1, math.ceil(6000 / rows_budget))
    times, rows, cpu, attn, attn_cpu = [], 0, 0.0, 0.0, 0.0
    for k in range(steps):
        step = os_.advance()
        r = os_.timed_step(step, stride, k)
        times.append(r["wall"])
        rows += r["rows"]
        cpu += r["cpu"]
        attn += r["attn"]
        attn_cpu += r["attn_cpu"]
    total = sum(times)
    # the attention rows spread over the host's cores; the rest of the oracle's step (batch
    # merge, metadata, the KV write's copy of the whole pool, gather) runs on one
    return {"value": rows / total, "wall_s": total, "rows": rows, "stride": stride,
            "cores": round(cpu / max(total, 1e-9), 1),
            "cores_attention": round(attn_cpu / max(attn, 1e-9), 1),
            "attention_s": attn, "times": times}


def fixed_oracle_run(spec, target_s):
    """The oracle on one fixed batch: full metadata, KV write and gather, attention for a row
    sample sized to about ``target_s``.  Returns (rows/s, rows, stride, cores, seconds)."""
    import numpy as np
    import torch

    import oracle
    import workloads as wl
    from oracle.threads import oracle_attention_threads

    tens = wl.make_tensors(spec, device="cpu")
    d = spec.dims
    f64 = lambda t: t.to(torch.float64).numpy()
    u16 = lambda t: t.view(torch.int16).numpy()
    q64, k64, v64 = f64(tens.q), f64(tens.k), f64(tens.v)
    hk = [f64(h) for h in tens.hist_k]
    hv = [f64(h) for h in tens.hist_v]

    def run(rows):
        c0, w0 = time.process_time(), time.perf_counter()
        meta = oracle.prepare_inputs(block_size=d.block_size, null_block=d.null_block,
                                     token_table=spec.token_table, block_table=spec.block_table,
                                     num_computed=spec.num_computed,
                                     num_scheduled=spec.num_scheduled,
                                     num_reqs_padded=spec.num_reqs_padded,
                                     num_tokens_padded=spec.num_tokens_padded)
        oracle.kv_write(u16(tens.k_cache), u16(tens.v_cache), meta["slot_mapping"], u16(tens.k),
                        u16(tens.v))
        R = spec.num_reqs
        oracle_attention_threads(q64, hk, hv, k64, v64, meta["query_start_loc"][:R + 1],
                                 meta["seq_lens"][:R], R, rows)
        oracle.gather_rows(u16(tens.hidden), meta["logits_indices"])
        return time.perf_counter() - w0, time.process_time() - c0

    N = spec.num_tokens
    probe = list(range(0, N, max(1, N // 48)))
    t, _ = run(probe)
    stride = max(1, math.ceil(N * t / len(probe) / target_s))
    rows = list(range(0, N, stride))
    t, c = run(rows)
    return len(rows) / t, len(rows), stride, round(c / max(t, 1e-9), 1), t


def run_reference(args, rank, world):
    """--impl reference: the CPU oracle (float64) on the headline workload, on this host's
    cores; rank 0 only."""
    if rank != 0:
        return
    cpu = host_cpu()
    budget = 150.0
    if args.config == 4:
        r = oracle_stream_run(rank, args.warmup, args.steps, budget)
        import workloads as wl

        value, total = r["value"], r["wall_s"]
        config = stream_config_desc(wl.MixedChunkStream().dims, args.warmup, args.steps,
                                    args.warmup + args.steps)
        sample = (f"each step: the oracle's batch merge, metadata for every token, KV write and "
                  f"row gather in full, attention (all heads) for 1 in {r['stride']} query "
                  f"rows, over all host threads; {r['rows']} rows over {args.steps} steps")
        cores = r["cores"]
        cpu = {**cpu, "cores_attention": r["cores_attention"]}
    else:
        spec = make_spec(args.config)
        per = budget / max(1, args.steps + args.warmup)
        value, nrows, stride, cores, t = fixed_oracle_run(spec, per)
        total = t * args.steps
        config = fixed_config_desc(spec, args.config)
        sample = f"1 in {stride} of {spec.num_tokens} query rows per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000 * total / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config,
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample, **cpu},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def cpu_baseline(config, rank):
    """The oracle on this host's cores, on a bounded sample of the headline workload."""
    cpu = host_cpu()
    if config == 4:
        r = oracle_stream_run(rank, 1, 1, 20.0)
        return {"value": r["value"], "unit": UNIT, "cores": r["cores"],
                "cores_attention": r["cores_attention"], "kind": "oracle",
                "sample": (f"stream step 1 (after a probe of step 0): the oracle's batch "
                           f"merge, metadata, KV write (a copy of the whole pool) and gather in "
                           f"full, attention for 1 in {r['stride']} query rows (all heads) over "
                           f"all host threads; {r['rows']} rows in "
                           f"{r['wall_s']:.1f} s, of which {r['attention_s']:.1f} s attention "
                           f"on {r['cores_attention']} cores and the rest on one"), **cpu}
    spec = make_spec(config, rank)
    value, nrows, stride, cores, t = fixed_oracle_run(spec, 12.0)
    return {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"1 in {stride} of {spec.num_tokens} query rows with the full "
                      f"metadata, KV write and gather; {t:.1f} s", **cpu}


# ----------------------------------------------------------------------------- our arm
def _events(n):
    import torch

    return [torch.cuda.Event(enable_timing=True) for _ in range(n)]


def _recorded_events(n):
    """Events the library re-records (rb_step_profiled): torch creates the handle lazily."""
    import torch

    ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(n)]
    for e in ev:
        e.record()
    return ev


def measure_stream(args, rank, world, local):
    """The headline: the chunked-prefill stream, each step rb_batch_apply_update + rb_step."""
    import torch

    import ragged_mixed_paged_gb300 as rb

    dev = torch.device("cuda", local)
    total = max(STREAM_STEPS, args.warmup + args.steps)
    stream, steps = stream_steps(rank, total)
    d = stream.dims
    dims = rb.Dims.of(d)
    nmax, rmax = stream.BUDGET, d.max_num_reqs
    g = torch.Generator(device=dev).manual_seed(stream_seed(rank))
    bf = torch.bfloat16

    def rnd(*shape):
        return torch.randn(*shape, generator=g, device=dev, dtype=torch.float32).to(bf)

    q, k, v = rnd(nmax, d.num_q_heads, d.head_dim), rnd(nmax, d.num_kv_heads, d.head_dim), \
        rnd(nmax, d.num_kv_heads, d.head_dim)
    hidden = rnd(nmax, HIDDEN)
    k_cache = torch.empty((d.num_slots, d.num_kv_heads, d.head_dim), dtype=bf,
                          device=dev).normal_(generator=g)
    v_cache = torch.empty_like(k_cache).normal_(generator=g)
    batch = rb.PersistentBatch(d.max_num_reqs, d.max_model_len, d.max_blocks_per_req, device=dev)
    staged = [batch.stage(s) for s in steps]             # every step's packet in HBM
    buf = rb.StepBuffers.allocate(dims, rmax, rmax, nmax, nmax, batch.tables(), q, k, v, hidden,
                                  k_cache, v_cache)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    cq = [step_cq(s) for s in steps]
    works = [work_of(x, d.num_q_heads, d.num_kv_heads, d.head_dim, d.block_size,
                     sum(qq for _, qq in x), sum(qq for _, qq in x), len(x), len(x), HIDDEN)
             for x in cq]
    tokens = [s.num_tokens for s in steps]
    # per step: start | after the update | after the preparation launch | after attention
    marks = [(_events(2), _recorded_events(2)) for _ in steps]

    def run(i):
        st = staged[i]
        R, N = st.num_scheduled, st.num_tokens
        b = dataclasses.replace(buf, num_reqs=R, num_reqs_padded=R, num_tokens=N,
                                num_tokens_padded=N, q=q[:N], k=k[:N], v=v[:N],
                                hidden=hidden[:N], attn_out=buf.attn_out[:N],
                                rows_out=buf.rows_out[:R])
        (a, u), inner = marks[i]
        flush.zero_()
        a.record()
        batch.apply_staged(st)
        u.record()
        rb.run_step_fused(b, events=inner)

    torch.cuda.synchronize()
    for i in range(args.warmup):
        run(i)
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    launches0 = rb.launch_count()
    w0 = time.perf_counter()
    timed = range(args.warmup, args.warmup + args.steps)
    for i in timed:
        run(i)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - w0
    launches = rb.launch_count() - launches0
    clocks = sampler.stop()
    for i in range(args.warmup + args.steps, total):  # the rest of the stream
        run(i)
    torch.cuda.synchronize()
    err = int(buf.meta["scalars"][3].item()) | int(batch.error_word.item())
    if err:
        raise SystemExit(f"device error word {err:#x}")

    def spans(i):
        (a, u), (p, z) = marks[i]
        return a.elapsed_time(u), u.elapsed_time(p), p.elapsed_time(z), a.elapsed_time(z)

    sp = [spans(i) for i in range(total)]
    step_ms = [x[3] for x in sp]
    t_timed = sum(step_ms[i] for i in timed)
    tok_timed = sum(tokens[i] for i in timed)
    t_max = reduce_over_ranks(t_timed, "max", world, dev)
    tok_sum = reduce_over_ranks(float(tok_timed), "sum", world, dev)
    value = tok_sum / (t_max / 1000.0)

    def agg(idx):
        w = {k2: sum(works[i][k2] for i in idx) for k2 in works[0]}
        launch_s = sum(sp[i][2] for i in idx) / 1000.0
        return w, launch_s

    w, launch_s = agg(timed)
    roof = roofline(w, launch_s, 4, launches=len(timed))
    all_idx = range(total)
    w_all, launch_all = agg(all_idx)
    roof_all = roofline(w_all, launch_all, 4, launches=total)
    comp = {"batch_update": statistics.mean(sp[i][0] for i in timed),
            "prep_launch": statistics.mean(sp[i][1] for i in timed),
            "attention_launch": statistics.mean(sp[i][2] for i in timed)}
    result = {
        "value": value, "ms_per_step": t_max / len(timed), "tokens_timed": tok_timed,
        "median_step_tokens_per_s": statistics.median(tokens[i] / (step_ms[i] / 1000.0)
                                                      for i in timed),
        "config": stream_config_desc(d, args.warmup, args.steps, total),
        "roofline": roof, "components_ms": comp, "gpu_launches": launches,
        "clocks": clocks, "wall_s": wall,
        "stream_all": {"steps": total, "tokens": sum(tokens),
                       "value": sum(tokens) / (sum(step_ms) / 1000.0),
                       "ms_per_step": sum(step_ms) / total,
                       "hbm_frac": roof_all["hbm_frac"], "tensor_frac": roof_all["tensor_frac"],
                       "attention_launch_ms": roof_all["launch_ms"]},
    }
    e2e = stream_e2e_pipelined(args, rank, world, dev, steps, buf, q, k, v, hidden, k_cache,
                               v_cache)
    e2e["synchronised"] = stream_e2e(args, rank, world, dev, steps, buf, q, k, v, hidden,
                                     k_cache, v_cache, flush)
    del batch, staged, buf, k_cache, v_cache, flush
    torch.cuda.empty_cache()
    return result, e2e


def stream_e2e_pipelined(args, rank, world, dev, steps, buf, q, k, v, hidden, k_cache, v_cache):
    """The stream end to end through the public API as a serving loop runs it: per step
    PersistentBatch.apply (host packing, the packet copy, the update) and rb_step_host_async
    (q / k / v / hidden in from pinned host memory on a copy stream, the step on the compute
    stream once they landed, attention output, gathered rows and scalars back on a third
    stream), two sets of device and pinned buffers used by alternate steps, so that each step's
    copies overlap its neighbours' compute; the host checks each step's error word two steps
    later.  Wall clock over the timed steps, from their first enqueue to the last result on the
    host.  No L2 flush: every step reads ~8 GB of KV pages, far more than L2."""
    import torch

    import ragged_mixed_paged_gb300 as rb

    d = buf.dims
    batch = rb.PersistentBatch(d.max_num_reqs, d.max_model_len, d.max_blocks_per_req, device=dev)
    tables = dict(token_table=batch.token_table, block_table=batch.block_table,
                  num_computed=batch.num_computed, num_scheduled=batch.num_scheduled,
                  num_prompt=batch.num_prompt)
    nmax, rmax = q.shape[0], buf.rows_out.shape[0]
    pin = lambda t: t.cpu().pin_memory()
    hq, hk, hv, hh = pin(q), pin(k), pin(v), pin(hidden)
    sets = []
    for x in range(2):  # device inputs / outputs and pinned outputs of alternate steps
        dq, dk, dv, dh = ((t if x == 0 else torch.empty_like(t)) for t in (q, k, v, hidden))
        sb = rb.StepBuffers.allocate(d, rmax, rmax, nmax, nmax, tables, dq, dk, dv, dh, k_cache,
                                     v_cache)
        ho = (torch.empty(tuple(sb.attn_out.shape), dtype=sb.attn_out.dtype).pin_memory(),
              torch.empty(tuple(sb.rows_out.shape), dtype=sb.rows_out.dtype).pin_memory(),
              torch.empty(4, dtype=torch.int32).pin_memory())
        sets.append((sb, ho))
    s_comp, s_in, s_out = torch.cuda.current_stream(), torch.cuda.Stream(), torch.cuda.Stream()

    def event():
        e = torch.cuda.Event()
        e.record(s_comp)  # torch creates events lazily: record once so the handle exists
        return e

    in_done, step_done, out_done = ([event(), event()] for _ in range(3))
    pending = [None, None]  # (step index) whose outputs sit in each pinned set
    h2d = d2h = tok = 0

    def check(x):
        if pending[x] is None:
            return
        out_done[x].synchronize()
        if int(sets[x][1][2][3]) != 0:
            raise SystemExit(f"e2e step {pending[x]}: device error word "
                             f"{int(sets[x][1][2][3]):#x}")
        pending[x] = None

    def run(i):
        nonlocal h2d, d2h, tok
        x = i % 2
        sb, (o_attn, o_rows, o_sc) = sets[x]
        check(x)                                   # step i - 2's results, read on the host
        s_in.wait_event(step_done[x])              # step i - 2 has read this input set
        s_comp.wait_event(out_done[x])             # ... and its outputs have left this set
        nbytes = batch.apply(steps[i], stream=s_comp)
        R, N = batch.num_reqs, batch.num_tokens_scheduled
        b = dataclasses.replace(sb, num_reqs=R, num_reqs_padded=R, num_tokens=N,
                                num_tokens_padded=N, q=sb.q[:N], k=sb.k[:N], v=sb.v[:N],
                                hidden=sb.hidden[:N], attn_out=sb.attn_out[:N],
                                rows_out=sb.rows_out[:R], _step_args=None)
        ins = [(b.q, hq[:N]), (b.k, hk[:N]), (b.v, hv[:N]), (b.hidden, hh[:N])]
        outs = [(o_attn[:N], b.attn_out), (o_rows[:R], b.rows_out), (o_sc, b.meta["scalars"])]
        rb.run_step_host_async(b, ins, outs, s_comp, s_in, s_out, in_done[x], step_done[x])
        out_done[x].record(s_out)
        pending[x] = i
        if i >= args.warmup:
            tok += N
            h2d += nbytes + sum(t.numel() * t.element_size() for _, t in ins)
            d2h += sum(t.numel() * t.element_size() for t, _ in outs)

    for i in range(args.warmup):
        run(i)
    check(0), check(1)
    torch.cuda.synchronize()
    barrier(world)
    t0 = time.perf_counter()
    for i in range(args.warmup, args.warmup + args.steps):
        run(i)
    check(0), check(1)
    total = time.perf_counter() - t0
    if int(batch.error_word.item()) != 0:
        raise SystemExit(f"e2e: batch error word {int(batch.error_word.item()):#x}")
    K = max(1, args.steps)
    total = reduce_over_ranks(total, "max", world, dev)
    toks = reduce_over_ranks(float(tok), "sum", world, dev)
    del batch, sets
    return {"value": toks / total, "unit": UNIT, "ms_per_step": 1000.0 * total / K,
            "h2d_bytes_per_step": h2d / K, "d2h_bytes_per_step": d2h / K,
            "entry": "PersistentBatch.apply (packet copy + rb_batch_apply_update) + "
                     "rb_step_host_async (C ABI, host buffers; copies on their own streams "
                     "overlapping the neighbouring steps' compute, two buffer sets), wall "
                     "clock from the first timed enqueue to the last result on the host",
            "l2": "not flushed: every step reads ~8 GB of KV pages (L2 is 129 MB)",
            "timed_steps": f"{args.warmup}..{args.warmup + args.steps - 1}"}


def stream_e2e(args, rank, world, dev, steps, buf, q, k, v, hidden, k_cache, v_cache, flush):
    """The stream end to end through the public API: per step PersistentBatch.apply (host
    packing, one packet copy from pinned memory, the update) and rb_step_host (q / k / v /
    hidden in from pinned host memory, the step, attention output, gathered rows and scalars
    back), synchronised; wall clock per step, L2 flushed outside it."""
    import torch

    import ragged_mixed_paged_gb300 as rb

    d = buf.dims
    batch = rb.PersistentBatch(d.max_num_reqs, d.max_model_len, d.max_blocks_per_req, device=dev)
    b0 = dataclasses.replace(buf, token_table=batch.token_table, block_table=batch.block_table,
                             num_computed=batch.num_computed, num_scheduled=batch.num_scheduled,
                             num_prompt=batch.num_prompt, _step_args=None)
    nmax = q.shape[0]
    pin = lambda t: t.cpu().pin_memory()
    hq, hk, hv, hh = pin(q), pin(k), pin(v), pin(hidden)
    out_attn = torch.empty(tuple(buf.attn_out.shape), dtype=buf.attn_out.dtype).pin_memory()
    out_rows = torch.empty(tuple(buf.rows_out.shape), dtype=buf.rows_out.dtype).pin_memory()
    out_sc = torch.empty(4, dtype=torch.int32).pin_memory()
    times, h2d, d2h, tok = [], 0, 0, 0
    for i in range(args.warmup + args.steps):
        step = steps[i]
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        nbytes = batch.apply(step)
        R, N = batch.num_reqs, batch.num_tokens_scheduled
        b = dataclasses.replace(b0, num_reqs=R, num_reqs_padded=R, num_tokens=N,
                                num_tokens_padded=N, q=q[:N], k=k[:N], v=v[:N],
                                hidden=hidden[:N], attn_out=buf.attn_out[:N],
                                rows_out=buf.rows_out[:R], _step_args=None)
        ins = [(b.q, hq[:N]), (b.k, hk[:N]), (b.v, hv[:N]), (b.hidden, hh[:N])]
        outs = [(out_attn[:N], b.attn_out), (out_rows[:R], b.rows_out), (out_sc, b.meta["scalars"])]
        rb.run_step_host(b, ins, outs)
        torch.cuda.synchronize()
        t1 = time.perf_counter()
        if int(out_sc[3]) != 0:
            raise SystemExit(f"e2e step {i}: device error word {int(out_sc[3]):#x}")
        if i >= args.warmup:
            times.append(t1 - t0)
            tok += N
            h2d += nbytes + sum(t.numel() * t.element_size() for _, t in ins)
            d2h += sum(t.numel() * t.element_size() for t, _ in outs)
    K = max(1, args.steps)
    total = reduce_over_ranks(sum(times), "max", world, dev)
    toks = reduce_over_ranks(float(tok), "sum", world, dev)
    del batch
    return {"value": toks / total, "unit": UNIT, "ms_per_step": 1000.0 * total / K,
            "h2d_bytes_per_step": h2d / K, "d2h_bytes_per_step": d2h / K,
            "entry": "PersistentBatch.apply (packet copy + rb_batch_apply_update) + rb_step_host "
                     "(C ABI, host buffers), wall clock, synchronised every step",
            "timed_steps": f"{args.warmup}..{args.warmup + args.steps - 1}"}


def measure_fixed(config, rank, world, local, steps, warmup, manager_ratio=1, want_e2e=False,
                  context_scale=1.0):
    """One fixed batch: rb_step captured once as a CUDA graph and replayed with a cold L2; the
    fused launch timed in a second graph of rb_step_profiled (event nodes between launches)."""
    import torch

    import workloads as wl
    import ragged_mixed_paged_gb300 as rb

    dev = torch.device("cuda", local)
    spec = make_spec(config, rank, manager_ratio, context_scale)
    d = spec.dims
    tens = wl.make_tensors(spec, device=dev)
    tables = wl.device_tables(spec, dev)
    buf = rb.StepBuffers.allocate(rb.Dims.of(d), spec.num_reqs, spec.num_reqs_padded,
                                  spec.num_tokens, spec.num_tokens_padded, tables, tens.q,
                                  tens.k, tens.v, tens.hidden, tens.k_cache, tens.v_cache)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(warmup):
        flush.zero_()
        rb.run_step_fused(buf)
    torch.cuda.synchronize()
    if int(buf.meta["scalars"][3].item()) != 0:
        raise SystemExit(f"device error word {int(buf.meta['scalars'][3].item()):#x}")
    inner = _recorded_events(2)
    torch.cuda.synchronize()
    launches0 = rb.launch_count()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        rb.run_step_fused(buf)
    per_step = rb.launch_count() - launches0
    marked = torch.cuda.CUDAGraph()
    with torch.cuda.graph(marked):
        rb.run_step_fused(buf, events=inner)
    graph.replay()
    marked.replay()
    torch.cuda.synchronize()
    ev = [_events(2) for _ in range(steps)]
    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    w0 = time.perf_counter()
    for a, b in ev:
        flush.zero_()
        a.record()
        graph.replay()
        b.record()
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - w0
    clocks = sampler.stop()
    step_times = [a.elapsed_time(b) for a, b in ev]
    # breakdown pass: the same step with the library's events between its two launches
    pre, att = [], []
    for _ in range(steps):
        flush.zero_()
        a = _events(1)[0]
        a.record()
        marked.replay()
        torch.cuda.synchronize()
        pre.append(a.elapsed_time(inner[0]))
        att.append(inner[0].elapsed_time(inner[1]))
    med = statistics.median(step_times)
    med_max = reduce_over_ranks(med, "max", world, dev)
    toks = reduce_over_ranks(float(spec.num_tokens), "sum", world, dev)
    launch_s = statistics.median(att) / 1000.0
    out = {"value": toks / (med_max / 1000.0), "ms_per_step": med_max,
           "ms_per_step_mean": statistics.mean(step_times), "steps": steps, "warmup": warmup,
           "config": fixed_config_desc(spec, config),
           # measured traffic belongs to the workload as named: none for a scaled or
           # manager-block variant
           "roofline": roofline(spec_work(spec), launch_s,
                                config if context_scale == 1.0 and manager_ratio == 1 else None),
           "components_ms": {"prep_launch": statistics.median(pre),
                             "attention_launch": statistics.median(att)},
           "gpu_launches": per_step * steps, "launch": "cuda_graph_replay", "wall_s": wall,
           "clocks": clocks}
    e2e = fixed_e2e(spec, buf, flush, steps, warmup, world, dev) if want_e2e else None
    del buf, tens, tables, flush, graph, marked
    torch.cuda.empty_cache()
    return out, e2e


def fixed_e2e(spec, buf, flush, steps, warmup, world, dev):
    """A fixed batch through rb_step_host with host buffers (inputs in from pinned memory,
    results back), every step synchronised; wall clock."""
    import torch

    import ragged_mixed_paged_gb300 as rb

    host_in = [(t, t.cpu().pin_memory()) for t in (
        buf.token_table, buf.block_table, buf.num_computed, buf.num_scheduled, buf.q, buf.k,
        buf.v, buf.hidden)]
    host_out = [(torch.empty_like(t, device="cpu").pin_memory(), t) for t in (
        buf.attn_out, buf.rows_out, buf.meta["scalars"])]
    h2d = sum(t.numel() * t.element_size() for _, t in host_in)
    d2h = sum(t.numel() * t.element_size() for t, _ in host_out)
    times = []
    for i in range(warmup + steps):
        flush.zero_()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        rb.run_step_host(buf, host_in, host_out)
        torch.cuda.synchronize()
        if i >= warmup:
            times.append(time.perf_counter() - t0)
    ms = reduce_over_ranks(1000.0 * statistics.median(times), "max", world, dev)
    return {"value": world * spec.num_tokens / (ms / 1000.0), "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "entry": "rb_step_host (C ABI, host buffers), wall clock, median"}


def run_ours(args, rank, world, local):
    import torch

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device for --impl ours")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    side_steps = max(3, min(args.steps, 10))
    if args.config == 4:
        head, e2e = measure_stream(args, rank, world, local)
    else:
        head, e2e = measure_fixed(args.config, rank, world, local, args.steps, args.warmup,
                                  args.manager_ratio, want_e2e=True,
                                  context_scale=args.context_scale)
    line = {"metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": head["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 Q/K/V/hidden and KV pool, seeded request "
                    "stream and page ids; no weights)",
            "config": head["config"], "roofline": head["roofline"],
            "gpu_launches": head["gpu_launches"], "clocks": head["clocks"], "e2e": e2e,
            "components_ms": head["components_ms"],
            "kernel_source_hash": kernel_sources_hash()}
    for key in ("stream_all", "median_step_tokens_per_s", "tokens_timed", "launch", "wall_s"):
        if key in head:
            line[key] = head[key]
    if not args.no_side_configs:
        side = {}
        for c in (2, 3, 5):
            if c == args.config:
                continue
            out, _ = measure_fixed(c, rank, world, local, side_steps, 3)
            side[str(c)] = {k2: out[k2] for k2 in ("value", "ms_per_step", "roofline",
                                                    "components_ms", "config", "clocks")}
            side[str(c)]["unit"] = UNIT
            side[str(c)]["timing"] = (f"median of {side_steps} graph replays of rb_step after "
                                      "3 warm-ups, L2 flushed before each")
        line["configs"] = side
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(args.config, rank)
    if rank == 0:
        print(json.dumps(line), flush=True)


def run_cascade_compare(args, rank, world, local):
    """Shared system prompt (256 decodes after a common 4096-token prefix, own suffixes
    U[16, 1024], plus two 512-token chunks): one attention call through the plain path and
    through the cascade path, each timed alone with a cold L2."""
    import numpy as np
    import torch

    import workloads as wl
    import ragged_mixed_paged_gb300 as rb

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    spec = wl.shared_prefix_batch(11 + rank, num_decodes=256, prefix_tokens=4096,
                                  suffix_range=(16, 1024), num_chunks=2, chunk_q=512)
    d = spec.dims
    dims = rb.Dims.of(d)
    tens = wl.make_tensors(spec, device=dev)
    tables = wl.device_tables(spec, dev)
    R, N = spec.num_reqs, spec.num_tokens
    meta = rb.prepare_inputs(dims, R, R, N, N, tables["token_table"], tables["num_computed"],
                             tables["num_scheduled"], tables["block_table"])
    rb.kv_write(dims, tens.k, tens.v, meta["slot_mapping"], tens.k_cache, tens.v_cache)
    P = rb.cascade_prefix_len(spec.shared_prefix_tokens, spec.num_computed.tolist(), d.block_size)
    ws = torch.empty(rb.cascade_workspace_size(dims, R, N), dtype=torch.uint8, device=dev)
    out = torch.empty_like(tens.q)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    bt, qsl, sl = tables["block_table"], meta["query_start_loc"], meta["seq_lens"]
    calls = {
        "plain": lambda: rb.paged_attention(dims, R, N, tens.q, tens.k_cache, tens.v_cache, bt,
                                            qsl, sl, out=out, workspace=ws, error_word=err),
        "cascade": lambda: rb.paged_attention_cascade(dims, R, N, P, tens.q, tens.k_cache,
                                                      tens.v_cache, bt, qsl, sl, out=out,
                                                      workspace=ws, error_word=err),
    }
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    res = {}
    sampler = ClockSampler(local)
    sampler.start()
    for name, fn in calls.items():
        g = torch.cuda.CUDAGraph()
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        with torch.cuda.graph(g):
            fn()
        times = []
        for _ in range(args.steps):
            flush.zero_()
            a, b = _events(2)
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        res[name] = statistics.median(times)
    clocks = sampler.stop()
    if int(err.item()) != 0:
        raise SystemExit(f"device error word {int(err.item()):#x}")
    kv_token = 2 * d.num_kv_heads * d.head_dim * 2  # K and V bytes of one token, all kv heads
    L = spec.num_computed.astype(np.int64) + spec.num_scheduled
    plain_bytes = int(L.sum()) * kv_token
    casc_bytes = (P + int((L - P).sum())) * kv_token
    pk, pk_kind = peaks()
    if rank == 0:
        print(json.dumps({
            "metric": "attention call time with a shared prefix (plain vs cascade)",
            "workload": spec.name, "num_reqs": R, "num_tokens": N, "prefix_len": P,
            "steps": args.steps, "warmup": args.warmup, "launch": "cuda_graph_replay",
            "l2": "512 MiB flush before every call",
            "plain_ms": res["plain"], "cascade_ms": res["cascade"],
            "speedup": res["plain"] / res["cascade"],
            "plain_kv_bytes": plain_bytes, "cascade_kv_bytes": casc_bytes,
            "plain_hbm_frac": plain_bytes / (res["plain"] / 1e3) / 1e9 / pk["hbm_gbs"],
            "cascade_kv_gbs": casc_bytes / (res["cascade"] / 1e3) / 1e9,
            "peak_kind": pk_kind, "clocks": clocks}), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=95)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=4, choices=[2, 3, 4, 5])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-side-configs", action="store_true",
                    help="skip the configs 2/3/5 entries of the line")
    ap.add_argument("--manager-ratio", type=int, default=1,
                    help="--config 2/3: page tables of manager blocks of this many kernel pages")
    ap.add_argument("--context-scale", type=float, default=1.0,
                    help="--config 3 or 5: cached lengths times this factor (a smaller case, e.g. "
                         "for a profiler; not a headline)")
    ap.add_argument("--cascade", action="store_true",
                    help="time one attention call on a shared-prefix batch, plain vs cascade")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    if args.steps < 1:
        raise SystemExit("--steps must be >= 1")
    rank, world, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.cascade:
        run_cascade_compare(args, rank, world, local)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
