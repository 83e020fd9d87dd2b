#!/usr/bin/env python
"""Throughput of one flattened mixed-batch step on GB300 (prepare_inputs -> kv_write ->
paged_attention -> gather_rows, one attention layer, synthetic bf16 activations).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config C]

Prints ONE JSON line on rank 0.  The headline workload is the pages' padding example
(query lens [2000, 512, 1 x 6]; 32 q / 8 kv heads, head_dim 128, block 16, hidden 4096).
``--config`` selects another workload for local study (1 worked example, 3 pure decode,
4 chunked-prefill mix step 0, 5 long context); those lines are not the headline.

Timing: W untimed warm-up steps, then K steps, each bracketed by CUDA events on the launching
stream with a 512 MiB write between steps (outside the events) so every step starts with a
cold L2; barrier + synchronize around the whole region; max over ranks.  Under torchrun every
rank runs its own independent batch (data parallel, no collective on the data path).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
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

# DRAM bytes (read + write) per launch measured by ncu (dram__bytes_read.sum +
# dram__bytes_write.sum), keyed by (kernel, workload, hash of the kernel's sources): a figure is
# reported only while the kernel's sources are the ones it was measured on (profiles/).
KNOWN_TRAFFIC = {
    ("fused", 2, "3b1b6221124298e8"): 79013632 + 4368640,
    ("fused", 3, "3b1b6221124298e8"): 4546843904 + 26761472,
    ("fused", 4, "3b1b6221124298e8"): 10085929472 + 99310336,
}


# ----------------------------------------------------------------------------- workloads
def chunked_mix_step0(rank: int, oracle_layout: bool = False):
    """Step 0 of the chunked-prefill request stream, laid out into batch rows by the library's
    own device-side batch update (the oracle's InputBatch on the reference leg)."""
    import workloads as wl

    stream = wl.MixedChunkStream(seed=4000 + 7919 * rank)
    step, d = stream.next_step(), stream.dims
    if oracle_layout:
        from oracle.persistent_batch import InputBatch

        batch = InputBatch(d.max_num_reqs, d.max_model_len, d.max_blocks_per_req)
        batch.apply(step)
        cols = batch.columns(step.scheduled)
        tok, blk = batch.tables()
        computed, sched, prompt = cols["num_computed"], cols["num_scheduled"], cols["num_prompt"]
    else:
        import torch

        import ragged_mixed_paged_gb300 as rb

        batch = rb.PersistentBatch(d.max_num_reqs, d.max_model_len, d.max_blocks_per_req)
        batch.apply(step)
        torch.cuda.synchronize()
        if int(batch.error_word.item()) != 0:
            raise SystemExit(f"batch update error word {int(batch.error_word.item()):#x}")
        R = batch.num_reqs
        computed = batch.num_computed[:R].cpu().numpy()
        sched = batch.num_scheduled[:R].cpu().numpy()
        prompt = batch.num_prompt[:R].cpu().numpy()
        tok, blk = batch.token_table.cpu().numpy(), batch.block_table.cpu().numpy()
        del batch
    return wl.spec_from_columns("chunked-prefill mix step 0", d, computed, sched, prompt, tok, blk,
                                seed=(4000 + 7919 * rank) * 1000)


def make_spec(config: int, rank: int = 0, oracle_layout: bool = False, manager_ratio: int = 1):
    import workloads as wl

    if config == 1:
        return wl.config1(step=rank)
    if config == 2:
        return wl.config2(step=rank, manager_ratio=manager_ratio)
    if config == 3:
        return wl.config3(step=rank, manager_ratio=manager_ratio)
    if config == 4:
        return chunked_mix_step0(rank, oracle_layout)
    if config == 5:
        return wl.config5(step=rank)
    raise SystemExit(f"unknown config {config}")


def workload_name(spec, config):
    d = spec.dims
    return {
        "workload": {1: "pages' worked example A/B/C", 2: "pages' padding example",
                     3: "pure decode x256", 4: "chunked-prefill mix (step 0)",
                     5: "long-context 70B-like"}[config],
        "query_lens": (spec.num_scheduled.tolist() if spec.num_reqs <= 8
                       else f"{spec.num_reqs} requests"),
        "num_reqs": spec.num_reqs, "num_tokens": spec.num_tokens,
        "num_tokens_padded": spec.num_tokens_padded, "q_heads": d.num_q_heads,
        "kv_heads": d.num_kv_heads, "head_dim": d.head_dim, "block_size": d.block_size,
        "hidden": spec.hidden_size, "kv_pages": d.num_blocks,
        "kernel_pages_per_table_entry": d.kernel_blocks_per_manager_block,
        "l2": "flushed before every timed step (512 MiB write, outside the events)",
    }


def work_counts(spec):
    """Algorithmic work of the step (what the pages define, not what the kernels do)."""
    d = spec.dims
    g = d.num_q_heads // d.num_kv_heads
    dec_bytes = pre_flops = dec_flops = 0
    for c, q in zip(spec.num_computed.tolist(), spec.num_scheduled.tolist()):
        visible = q * c + q * (q + 1) // 2                 # sum over j of (c + j + 1)
        flops = 4 * d.num_q_heads * d.head_dim * visible
        if q * g <= 8:  # decode-like: bound by reading the request's K/V once per kv head
            L = c + q
            dec_bytes += L * 2 * d.num_kv_heads * d.head_dim * 2 \
                + 2 * q * d.num_q_heads * d.head_dim * 2 + -(-L // d.block_size) * 4
            dec_flops += flops
        else:
            pre_flops += flops
    N, Np, R = spec.num_tokens, spec.num_tokens_padded, spec.num_reqs
    row = d.num_kv_heads * d.head_dim * 2
    return dict(
        attn_flops=pre_flops + dec_flops, prefill_flops=pre_flops, decode_flops=dec_flops,
        decode_bytes=dec_bytes,
        kv_write_bytes=2 * 2 * Np * row,                       # K and V, read + write
        meta_bytes=Np * (4 + 4 + 3 * 4) + R * (2 * 4 + 3 * 4),
        gather_bytes=2 * spec.num_reqs_padded * spec.hidden_size * 2)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return FALLBACK_PEAKS, "fallback"


KERNEL_SOURCES = {
    "fused": ("attn_prefill_tc.cu", "attn_decode_warp.cuh", "tc_ptx.cuh", "attn_common.cuh",
              "rb_internal.cuh"),
    "prefill": ("attn_prefill.cu", "attn_common.cuh", "rb_internal.cuh"),
    "decode": ("attn_decode.cu", "attn_decode_warp.cuh", "attn_common.cuh", "rb_internal.cuh"),
}


def kernel_sources_hash(kind):
    """Hash of the sources a kernel is built from (traffic figures are valid for one hash)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "ragged_mixed_paged_gb300", "csrc")
    for f in KERNEL_SOURCES[kind]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


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


# ----------------------------------------------------------------------------- oracle arm
def oracle_step_sample(spec, tens, rows):
    """The CPU oracle on a row sample of the step: metadata, KV write, attention for `rows`,
    gather.  Returns seconds."""
    import numpy as np
    import torch

    import oracle

    d = spec.dims
    f64 = lambda t: t.float().numpy().astype(np.float64)
    u16 = lambda t: t.view(torch.int16).numpy()
    t0 = time.perf_counter()
    meta = oracle.prepare_inputs(block_size=d.block_size, null_block=d.null_block,
                                 token_table=spec.token_table, block_table=spec.block_table,
                                 num_computed=spec.num_computed,
                                 num_scheduled=spec.num_scheduled,
                                 num_reqs_padded=spec.num_reqs_padded,
                                 num_tokens_padded=spec.num_tokens_padded)
    oracle.kv_write(u16(tens.k_cache), u16(tens.v_cache), meta["slot_mapping"], u16(tens.k),
                    u16(tens.v))
    oracle.paged_attention(f64(tens.q), [f64(h) for h in tens.hist_k],
                           [f64(h) for h in tens.hist_v], f64(tens.k), f64(tens.v),
                           meta["query_start_loc"], meta["seq_lens"], spec.num_reqs, rows=rows)
    oracle.gather_rows(u16(tens.hidden), meta["logits_indices"])
    return time.perf_counter() - t0


def row_sample(spec, stride, offset=0):
    return list(range(offset % stride, spec.num_tokens, stride))


def cpu_baseline(spec, target_s=12.0):
    """Oracle timed on this host's cores on a bounded row sample of the same workload."""
    import workloads as wl

    tens = wl.make_tensors(spec, device="cpu")
    probe = max(1, spec.num_tokens // 40)
    t = oracle_step_sample(spec, tens, row_sample(spec, probe))
    per_row = t / len(row_sample(spec, probe))
    stride = max(1, math.ceil(spec.num_tokens * per_row / target_s))
    rows = row_sample(spec, stride)
    c0, w0 = time.process_time(), time.perf_counter()
    t = oracle_step_sample(spec, tens, rows)
    cores = (time.process_time() - c0) / max(time.perf_counter() - w0, 1e-9)
    return {"value": len(rows) / t, "unit": UNIT, "cores": round(cores, 1),
            "host_cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"every {stride}th of {spec.num_tokens} query rows (all heads) with the "
                      f"full metadata, KV write and gather; {t:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    spec = make_spec(args.config, oracle_layout=True)
    import workloads as wl

    tens = wl.make_tensors(spec, device="cpu")
    budget = 150.0 / max(1, args.steps + args.warmup)      # seconds per step
    probe = max(1, spec.num_tokens // 40)
    t = oracle_step_sample(spec, tens, row_sample(spec, probe))
    per_row = t / len(row_sample(spec, probe))
    stride = max(1, math.ceil(spec.num_tokens * per_row / budget))
    for w in range(max(0, args.warmup - 1)):
        oracle_step_sample(spec, tens, row_sample(spec, stride, w))
    times, nrows = [], 0
    c0, w0 = time.process_time(), time.perf_counter()
    for k in range(args.steps):
        rows = row_sample(spec, stride, k)
        times.append(oracle_step_sample(spec, tens, rows))
        nrows += len(rows)
    cores = (time.process_time() - c0) / max(time.perf_counter() - w0, 1e-9)
    total = sum(times)
    value = nrows / total
    sample = (f"each step: the oracle's metadata, KV write and gather in full plus attention "
              f"for every {stride}th query row (all heads), rotating the offset per step")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000 * total / max(1, args.steps), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_name(spec, args.config),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": round(cores, 1),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ----------------------------------------------------------------------------- our arm
def run_ours(args, rank, world, local):
    import torch

    import workloads as wl
    import ragged_mixed_paged_gb300 as rb

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device for --impl ours")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = torch.cuda.current_stream()
    spec = make_spec(args.config, rank, manager_ratio=args.manager_ratio)
    d = spec.dims
    tens = wl.make_tensors(spec, device=dev)
    tables = wl.device_tables(spec, dev)
    buf = rb.StepBuffers.allocate(rb.Dims.of(d), spec.num_reqs, spec.num_reqs_padded,
                                  spec.num_tokens, spec.num_tokens_padded, tables, tens.q,
                                  tens.k, tens.v, tens.hidden, tens.k_cache, tens.v_cache)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    E = lambda: torch.cuda.Event(enable_timing=True)

    # the product's step is one rb_step call (one memset, two launches); --four-calls times the
    # four separate entry points instead
    step_fn = rb.run_step if args.four_calls else rb.run_step_fused
    for _ in range(args.warmup):
        flush.zero_()
        step_fn(buf)
        rb.run_step(buf)
    torch.cuda.synchronize()
    if int(buf.meta["scalars"][3].item()) != 0:
        raise SystemExit(f"device error word {int(buf.meta['scalars'][3].item()):#x}")

    # events recorded inside the step: 5 around the four calls, 3 inside the attention call
    EX = lambda: torch.cuda.Event(enable_timing=True, external=True)
    marks, attn_marks = [EX() for _ in range(5)], [EX() for _ in range(3)]
    for ev in marks + attn_marks:
        ev.record()  # torch creates the handle lazily; the library re-records it in the step
    torch.cuda.synchronize()
    graph = graph_marked = None
    launches_per_step = None
    if not args.eager:
        # the step has only scalar host inputs and fixed-address buffers: capture it once and
        # replay it, as a serving loop would, so host launch latency does not enter the step.
        # The timed graph holds the library's launches only: an event-record node inside a
        # graph costs ~3.5 us, so the per-call and per-kernel events live in a second graph of
        # the same step, replayed after the timed region
        launches0 = rb.launch_count()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step_fn(buf)
        launches_per_step = rb.launch_count() - launches0
        graph_marked = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_marked):
            rb.run_step(buf, marks=marks, attn_marks=attn_marks)
        graph.replay()
        graph_marked.replay()
        torch.cuda.synchronize()
    E = lambda: torch.cuda.Event(enable_timing=True)
    step_events = [(E(), E()) for _ in range(args.steps)]
    samples = []  # per step of the breakdown pass: the 8 event timestamps
    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    launches0 = rb.launch_count()
    w0 = time.perf_counter()
    for k in range(args.steps):
        flush.zero_()
        a, b = step_events[k]
        a.record()
        if graph is not None:
            graph.replay()
        elif args.four_calls:
            rb.run_step(buf, marks=marks, attn_marks=attn_marks)
        else:
            step_fn(buf)
        b.record()
        torch.cuda.synchronize()
        if graph is None and args.four_calls:
            pts = [marks[0], marks[1], marks[2], attn_marks[0], attn_marks[1], attn_marks[2],
                   marks[3], marks[4]]
            samples.append([pts[0].elapsed_time(p) for p in pts])
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - w0
    launches = (launches_per_step * args.steps if graph is not None
                else rb.launch_count() - launches0)
    step_times = [a.elapsed_time(b) for a, b in step_events]
    if not samples:  # breakdown pass: the same steps, four calls with events between launches
        for k in range(args.steps):
            flush.zero_()
            if graph_marked is not None:
                graph_marked.replay()
            else:
                rb.run_step(buf, marks=marks, attn_marks=attn_marks)
            torch.cuda.synchronize()
            pts = [marks[0], marks[1], marks[2], attn_marks[0], attn_marks[1], attn_marks[2],
                   marks[3], marks[4]]
            samples.append([pts[0].elapsed_time(p) for p in pts])
    clocks = sampler.stop()

    # timestamps: 0 start | 1 after prepare | 2 after kv_write | 3 after plan | 4 after decode |
    # 5 after prefill | 6 after attention | 7 after gather
    def span(a, b):
        idx = {0: 0, 1: 1, 2: 2, 3: 6, 4: 7}
        return [s[idx[b]] - s[idx[a]] for s in samples]

    def kspan(a, b):  # inside the attention call: planner | decode kernel | prefill kernel
        return [s[2 + b] - s[2 + a] for s in samples]

    step_ms = statistics.mean(step_times)
    marked_step_ms = statistics.mean(span(0, 4))
    parts = {"prepare_inputs": span(0, 1), "kv_write": span(1, 2),
             "paged_attention": span(2, 3), "gather_rows": span(3, 4)}
    parts_ms = {k: statistics.mean(v) for k, v in parts.items()}
    kernels_ms = {"attn_plan": statistics.mean(kspan(0, 1)),
                  "attn_decode": statistics.mean(kspan(1, 2)),
                  "attn_prefill": statistics.mean(kspan(2, 3))}
    step_ms_max = reduce_over_ranks(step_ms, "max", world, dev)
    total_tokens = reduce_over_ranks(float(spec.num_tokens), "sum", world, dev)
    value = total_tokens / (step_ms_max / 1000.0)

    w = work_counts(spec)
    pk, pk_kind = peaks()
    attn_s = parts_ms["paged_attention"] / 1000.0
    dec_s = kernels_ms["attn_decode"] / 1000.0
    pre_s = kernels_ms["attn_prefill"] / 1000.0
    # decode and prefill units share one launch (timed as the prefill span) when the head group
    # is a power of two and head_dim is 64 or 128 (the tcgen05 path)
    fused = (d.num_q_heads // d.num_kv_heads) in (1, 2, 4, 8, 16) and d.head_dim in (64, 128)
    t_tensor = w["prefill_flops"] / (pk["bf16_tflops"] * 1e12)
    t_hbm = w["decode_bytes"] / (pk["hbm_gbs"] * 1e9)
    if fused:
        kernels_ms = {"attn_plan": kernels_ms["attn_plan"],
                      "attn_fused": kernels_ms["attn_prefill"]}
        tensor_bound = t_tensor >= t_hbm
        achieved = (w["prefill_flops"] / pre_s / 1e12 if tensor_bound
                    else w["decode_bytes"] / pre_s / 1e9)
        peak = pk["bf16_tflops"] if tensor_bound else pk["hbm_gbs"]
        roof = {"bound": "tensor" if tensor_bound else "hbm", "achieved": achieved,
                "peak": peak, "unit": "TFLOP/s" if tensor_bound else "GB/s",
                "frac": achieved / peak,
                "traffic": KNOWN_TRAFFIC.get(("fused", args.config, kernel_sources_hash("fused"))),
                "kernel": "attn_fused (split-KV decode + tcgen05 prefill units, one launch)",
                "launch_ms": pre_s * 1000.0,
                "overlap_frac": max(t_tensor, t_hbm) / pre_s,
                "tensor_frac": w["prefill_flops"] / pre_s / 1e12 / pk["bf16_tflops"],
                "hbm_frac": w["decode_bytes"] / pre_s / 1e9 / pk["hbm_gbs"],
                "peak_kind": f"{'bf16 dense burst' if tensor_bound else 'HBM copy'}, {pk_kind}"}
    # otherwise the dominant kernel: the one with the larger measured share of the step
    elif pre_s >= dec_s:
        achieved = w["prefill_flops"] / pre_s / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"],
                "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
                "traffic": KNOWN_TRAFFIC.get(("prefill", args.config, kernel_sources_hash("prefill"))),
                "kernel": "attn_prefill (tcgen05 tiles)", "launch_ms": kernels_ms["attn_prefill"],
                "peak_kind": f"bf16 dense burst, {pk_kind}"}
    else:
        achieved = w["decode_bytes"] / dec_s / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / pk["hbm_gbs"],
                "traffic": KNOWN_TRAFFIC.get(("decode", args.config, kernel_sources_hash("decode"))),
                "kernel": "attn_decode (split-KV)", "launch_ms": kernels_ms["attn_decode"],
                "peak_kind": f"HBM copy, {pk_kind}"}

    e2e = measure_e2e(spec, tens, buf, dev, args, flush, world)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms_max,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic (seeded N(0,1) bf16 Q/K/V/hidden, random page ids; no weights)",
            "config": workload_name(spec, args.config), "roofline": roof,
            "components_ms": parts_ms, "attention_kernels_ms": kernels_ms,
            "step_entry": "four calls" if args.four_calls else "rb_step (one memset, two launches)",
            "breakdown": ("per-call and per-kernel spans from a second pass of the same steps "
                          "through the four separate calls with events recorded between the "
                          f"launches (step {marked_step_ms:.4f} ms there; an event node in a "
                          "graph adds ~3.5 us, so these spans overstate the kernels slightly)"),
            "work": {"prefill_tflop": w["prefill_flops"] / 1e12,
                     "decode_kv_gb": w["decode_bytes"] / 1e9,
                     "attention_call_tflops": w["attn_flops"] / attn_s / 1e12,
                     "prefill_tflops_over_kernel": w["prefill_flops"] / pre_s / 1e12 if pre_s else None,
                     "decode_gbs_over_kernel": (w["decode_bytes"] / (pre_s if fused else dec_s) / 1e9
                                                if (pre_s if fused else dec_s) else None)},
            "gpu_launches": launches, "launch": "eager" if args.eager else "cuda_graph_replay",
            "wall_s": wall, "clocks": clocks, "e2e": e2e,
            "kernel_source_hashes": {k: kernel_sources_hash(k) for k in KERNEL_SOURCES}}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(spec)
    if rank == 0:
        print(json.dumps(line), flush=True)


def measure_e2e(spec, tens, buf, dev, args, flush, world):
    """Same step through the C ABI with host buffers (``rb_step_host``): inputs copied from
    pinned host memory and the results read back inside the timed region."""
    import torch

    import ragged_mixed_paged_gb300 as rb

    host_in = {
        "token_table": buf.token_table.cpu().pin_memory(),
        "block_table": buf.block_table.cpu().pin_memory(),
        "num_computed": buf.num_computed.cpu().pin_memory(),
        "num_scheduled": buf.num_scheduled.cpu().pin_memory(),
        "q": buf.q.cpu().pin_memory(), "k": buf.k.cpu().pin_memory(),
        "v": buf.v.cpu().pin_memory(), "hidden": buf.hidden.cpu().pin_memory(),
    }
    dst = {"token_table": buf.token_table, "block_table": buf.block_table,
           "num_computed": buf.num_computed, "num_scheduled": buf.num_scheduled,
           "q": buf.q, "k": buf.k, "v": buf.v, "hidden": buf.hidden}
    host_out = {"attn_out": torch.empty_like(buf.attn_out, device="cpu").pin_memory(),
                "rows_out": torch.empty_like(buf.rows_out, device="cpu").pin_memory(),
                "scalars": torch.empty(4, dtype=torch.int32).pin_memory()}
    src_out = {"attn_out": buf.attn_out, "rows_out": buf.rows_out,
               "scalars": buf.meta["scalars"]}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = sum(t.numel() * t.element_size() for t in host_out.values())

    # one rb_step_host call: the C ABI enqueues the host-to-device copies of the step's inputs,
    # the step and the device-to-host copies of its results
    ins = [(dst[k], t) for k, t in host_in.items()]
    outs = [(t, src_out[k]) for k, t in host_out.items()]

    def step():
        rb.run_step_host(buf, ins, outs)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    n = max(3, min(args.steps, 50))
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n)]
    for a, b in ev:
        flush.zero_()
        a.record()
        step()
        b.record()
    torch.cuda.synchronize()
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    ms = reduce_over_ranks(ms, "max", world, dev)
    return {"value": world * spec.num_tokens / (ms / 1000.0), "unit": UNIT, "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "entry": "rb_step_host (C ABI, host buffers)"}


def run_trajectory(args, rank, world, local):
    """The chunked-prefill mix as a stream: every step merges the scheduler's deltas into the
    device-resident persistent batch (packet copy + rb_batch_apply_update), then runs the step
    on the rows it produced.  Eager launches (the shapes change every step)."""
    import dataclasses

    import torch

    import workloads as wl
    import ragged_mixed_paged_gb300 as rb

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device for --impl ours")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    stream = wl.MixedChunkStream(seed=4000 + 7919 * rank)
    d = stream.dims
    dims = rb.Dims.of(d)
    steps = [stream.next_step() for _ in range(args.warmup + args.steps)]
    nmax, rmax = stream.BUDGET, d.max_num_reqs
    g = torch.Generator(device=dev).manual_seed(4000 + rank)
    bf = torch.bfloat16
    rnd = lambda *shape: torch.randn(*shape, generator=g, device=dev, dtype=torch.float32).to(bf)
    q, k, v = (rnd(nmax, d.num_q_heads, d.head_dim), rnd(nmax, d.num_kv_heads, d.head_dim),
               rnd(nmax, d.num_kv_heads, d.head_dim))
    hidden = rnd(nmax, 4096)
    k_cache = torch.empty((d.num_blocks * d.block_size, d.num_kv_heads, d.head_dim), dtype=bf,
                          device=dev).normal_(generator=g)
    v_cache = torch.empty_like(k_cache).normal_(generator=g)
    batch = rb.PersistentBatch(d.max_num_reqs, d.max_model_len, d.max_blocks_per_req, device=dev)
    buf = rb.StepBuffers.allocate(dims, rmax, rmax, nmax, nmax, batch.tables(), q, k, v, hidden,
                                  k_cache, v_cache)
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    E = lambda: torch.cuda.Event(enable_timing=True)
    host_rows = torch.empty((rmax, 4096), dtype=bf).pin_memory()
    host_scalars = torch.empty(4, dtype=torch.int32).pin_memory()
    rec, tokens, h2d, d2h = [], 0, 0, 0
    sampler = ClockSampler(local)
    launches0 = None
    barrier(world)
    for i, step in enumerate(steps):
        if i == args.warmup:
            torch.cuda.synchronize()
            sampler.start()
            launches0 = rb.launch_count()
        flush.zero_()
        ev = [E() for _ in range(5)]
        ev[0].record()
        nbytes = batch.apply(step, copied_event=ev[1])
        ev[2].record()
        R, N = batch.num_reqs, batch.num_tokens_scheduled
        b = dataclasses.replace(buf, num_reqs=R, num_reqs_padded=R, num_tokens=N,
                                num_tokens_padded=N, q=q[:N], k=k[:N], v=v[:N], hidden=hidden[:N],
                                attn_out=buf.attn_out[:N])
        rb.run_step_fused(b)
        ev[3].record()
        host_rows[:R].copy_(b.rows_out[:R], non_blocking=True)
        host_scalars.copy_(b.meta["scalars"], non_blocking=True)
        ev[4].record()
        torch.cuda.synchronize()
        if int(host_scalars[3]) != 0 or int(batch.error_word.item()) != 0:
            raise SystemExit(f"step {i}: error words {int(host_scalars[3]):#x} "
                             f"{int(batch.error_word.item()):#x}")
        if i >= args.warmup:
            rec.append([ev[0].elapsed_time(e) for e in ev[1:]])
            tokens += N
            h2d += nbytes
            d2h += R * 4096 * 2 + 16
    launches = rb.launch_count() - launches0
    clocks = sampler.stop()
    barrier(world)
    rec = list(zip(*rec))  # per mark: copy done | update done | step done | results read
    pack_copy = statistics.mean(rec[0])
    update = statistics.mean(b2 - b1 for b1, b2 in zip(rec[0], rec[1]))
    step_ms = statistics.mean(b3 - b2 for b2, b3 in zip(rec[1], rec[2]))
    e2e_ms = statistics.mean(rec[3])
    dev_ms = update + step_ms
    total = reduce_over_ranks(float(tokens), "sum", world, dev)
    dev_ms = reduce_over_ranks(dev_ms, "max", world, dev)
    e2e_ms = reduce_over_ranks(e2e_ms, "max", world, dev)
    K = args.steps
    # what the update replaces: uploading the whole token and page tables every step
    tt = torch.empty((rmax, d.max_model_len), dtype=torch.int32).pin_memory()
    bt = torch.empty((rmax, d.max_blocks_per_req), dtype=torch.int32).pin_memory()
    gt, gb = torch.empty_like(tt, device=dev), torch.empty_like(bt, device=dev)
    a, z = E(), E()
    a.record()
    for _ in range(5):
        gt.copy_(tt, non_blocking=True)
        gb.copy_(bt, non_blocking=True)
    z.record()
    torch.cuda.synchronize()
    if rank == 0:
        print(json.dumps({
            "metric": METRIC + " (stream of steps with the batch update)",
            "value": total / (dev_ms * K / 1000.0),
            "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
            "ms_per_step": dev_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic request stream",
            "config": {"workload": f"chunked-prefill mix stream, steps {args.warmup}.."
                                   f"{args.warmup + K - 1}", "l2": "512 MiB flush per step",
                       "launch": "eager"},
            "components_ms": {"pack_and_packet_h2d": pack_copy, "batch_update": update,
                              "step": step_ms},
            "e2e": {"value": total / (e2e_ms * K / 1000.0), "unit": UNIT, "ms_per_step": e2e_ms,
                    "h2d_bytes_per_step": h2d / K, "d2h_bytes_per_step": d2h / K},
            "full_table_h2d_ms": a.elapsed_time(z) / 5,
            "full_table_bytes": tt.numel() * 4 + bt.numel() * 4,
            "gpu_launches": launches, "clocks": clocks}), flush=True)

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
    flush = torch.empty(512 << 20, dtype=torch.uint8, device=dev)
    E = lambda: torch.cuda.Event(enable_timing=True)
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
            a, b = E(), E()
            a.record()
            g.replay()
            b.record()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
        res[name] = statistics.mean(times)
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
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=2, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="launch every step from Python instead of replaying a captured graph")
    ap.add_argument("--four-calls", action="store_true",
                    help="time the four separate entry points instead of the one rb_step call")
    ap.add_argument("--manager-ratio", type=int, default=1,
                    help="--config 2/3: page tables of manager blocks of this many kernel pages")
    ap.add_argument("--cascade", action="store_true",
                    help="time one attention call on a shared-prefix batch, plain vs cascade")
    ap.add_argument("--trajectory", action="store_true",
                    help="--config 4 only: time a stream of steps, each with its batch update")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    rank, world, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, rank, world)
    elif args.cascade:
        run_cascade_compare(args, rank, world, local)
    elif args.trajectory:
        if args.config != 4:
            raise SystemExit("--trajectory needs --config 4")
        run_trajectory(args, rank, world, local)
    else:
        run_ours(args, rank, world, local)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
