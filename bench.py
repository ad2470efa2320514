#!/usr/bin/env python3
"""Benchmark of one decode step of paged attention on GB300.

Default workload (the headline): the Llama-3.1-8B-shaped GQA batch -- 256
sequences, 32 query / 8 KV heads, head_dim 128, bf16 K/V, 16-token blocks,
lognormal context lengths (median 1024, clipped to [16, 8192]), shuffled
physical blocks.  --workload selects another synthetic workload (opt13b,
parallel_sampling, long_context with --block-size, tiny).

One step is the whole hot path over the batch: the copy-on-write block copies
(pa_copy_blocks; only parallel_sampling has any), the cache write of the new
tokens (pa_reshape_and_cache), then decode attention over the paged cache
(pa_decode: planning kernel, decode kernel, cross-partition reduce kernel).
pa_copy_blocks is also timed on the parallel-sampling copy list from a CUDA
graph and reported under "rows".

Metric: KV GB/s -- algorithmic bytes (K and V rows of exactly the attended
tokens, the queries, the outputs, the new tokens written, the blocks copied)
per second -- and seq-decode-steps/s.  The KV read per step (1.46 GB for the
headline) is far larger than the 129 MB L2, so no flush is needed between
steps.

--impl reference runs the fp64 CPU oracle on the same workload (a bounded
sample of sequences per step) as the comparison arm.

--workload prefill_llama8b / prefill_opt13b times the prompt phase over a
cached shared prefix instead: one step is the copy-on-write of the shared
partial block, the cache write of every new token and pa_prefill; the metric
is useful attention TFLOP/s (causal pairs only) against the measured bf16
tensor peak.  The default run also reports both prefill workloads under
"rows".
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from paged_kv_cache_132_gb300 import api, metrics, native, sharding, workloads  # noqa: E402

WORKLOAD = "llama8b"
METRIC = "paged decode-attention KV GB/s (% of GB300 HBM peak); seq-decode-steps/s"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_llama8b_ncu.md")
PREFILL_METRIC = "paged prefill attention TFLOP/s (useful, causal pairs; % of GB300 bf16 tensor peak); new tokens/s"
KERNEL_SOURCES = ["decode_mma.cuh", "decode_common.cuh", "decode.cu", "common.cuh", "kernels.h"]
PREFILL_PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "prefill_llama8b_ncu.md")
PREFILL_KERNEL_SOURCES = ["prefill.cuh", "prefill_launch.cuh", "prefill_bf16.cu", "tcgen05.cuh", "decode_common.cuh",
                          "common.cuh"]


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU time of the oracle leg")
    ap.add_argument("--workload", choices=list(workloads.WORKLOADS) + ["beam_search"] + list(workloads.PREFILL_WORKLOADS),
                    default=WORKLOAD,
                    help="which synthetic workload one step runs over (default: the Llama-8B-shaped batch); "
                         "prefill_*: prompt-phase attention over a cached shared prefix")
    ap.add_argument("--block-size", type=int, default=16, help="long_context sweep point (8, 16 or 32)")
    ap.add_argument("--partition-size", type=int, default=None,
                    help="split-KV partition (default: the workload's, else 512)")
    ap.add_argument("--beam-steps", type=int, default=16, help="steps of the beam_search trace")
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="first n sequences only (a smaller case of the same distribution, for profiling)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffer) leg")
    ap.add_argument("--no-rows", action="store_true", help="skip the copy-on-write row timing")
    ap.add_argument("--decode-kernel", choices=["default", "simt"], default="default",
                    help="simt: time the CUDA-core decode kernel instead of the tensor-core one")
    ap.add_argument("--split", choices=["replicas", "heads"], default="replicas",
                    help="N > 1: replicas = each rank runs its own batch (weak scaling); heads = the ranks "
                         "split one batch by KV head, same block tables on every rank (strong scaling)")
    return ap.parse_args(argv)


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def kernel_digest(sources=None) -> str:
    """Digest of a kernel's sources (default: the decode kernel's)."""
    h = hashlib.sha256()
    for f in sources or KERNEL_SOURCES:
        with open(os.path.join(ROOT, "paged_kv_cache_132_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic(summary=PROFILE_SUMMARY, sources=None):
    """DRAM bytes per launch of a kernel from its committed ncu summary (by
    default the decode kernel's), if it was taken on the current kernel
    source (digest line must match)."""
    try:
        with open(summary, encoding="utf-8") as f:
            text = f.read()
    except OSError:
        return None
    digest = traffic = None
    for line in text.splitlines():
        if line.startswith("kernel_digest:"):
            digest = line.split(":", 1)[1].strip()
        if line.startswith("dram_bytes_per_launch:"):
            traffic = float(line.split(":", 1)[1].strip())
    return traffic if digest == kernel_digest(sources) else None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json"), encoding="utf-8") as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0}, "fallback"


def host_cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo, else the
    machine type)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo", encoding="utf-8") as f:
            for line in f:
                if line.startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    import platform

    return platform.machine() or "unknown"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the GPU is busy."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.device_index = device_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.device_index), "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def all_reduce_max(value: float, world: int, device: str = "cuda") -> float:
    """The maximum of `value` over the ranks (each rank's step time)."""
    if world == 1:
        return value
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(world: int, bytes_per_rank_step: float, slowest_step_ms: float) -> float:
    """Whole-job GB/s: every rank processes its own replica of the batch, and
    the job takes as long as the slowest rank."""
    return world * bytes_per_rank_step / (slowest_step_ms * 1e-3) / 1e9


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


# ---------------------------------------------------------------------------
# CPU oracle leg (baseline and reference arm)
# ---------------------------------------------------------------------------
def oracle_setup(w):
    import oracle as O

    def bits(t):
        t = t.detach().contiguous().cpu()
        return t.view(torch.int32).numpy() if t.dtype == torch.float32 else t.view(torch.int16).numpy()

    orc = O.get()
    k = bits(w.k_cache).copy()
    v = bits(w.v_cache).copy()
    if w.copy_pairs.numel():
        orc.copy_blocks([k], [v], w.copy_pairs.cpu().numpy())
    orc.reshape_and_cache(bits(w.new_key), bits(w.new_value), k, v, w.slot_mapping.cpu().numpy())
    code = {torch.float32: O.F32, torch.float16: O.F16, torch.bfloat16: O.BF16}[w.dtype]
    return orc, code, k, v, bits(w.query), w.block_tables.cpu().numpy(), w.context_lens.cpu().numpy()


def oracle_run(setup, w, seqs, threads):
    orc, code, k, v, q, tables, ctx = setup
    t0 = time.perf_counter()
    orc.decode(q[seqs], k, v, code, tables[seqs], ctx[seqs], w.num_kv_heads, w.scale, num_threads=threads)
    dt = time.perf_counter() - t0
    nbytes = metrics.decode_bytes(ctx[seqs].tolist(), w.num_heads, w.num_kv_heads, w.head_dim,
                                  w.query.element_size(), 8)
    return dt, nbytes


def cpu_baseline(w, target_seconds):
    import numpy as np

    import oracle as O

    setup = oracle_setup(w)
    threads = O.get().max_threads()
    all_seqs = np.arange(w.num_seqs)
    total_t = total_b = 0.0
    passes = 0
    while total_t < target_seconds and passes < 50:
        dt, nb = oracle_run(setup, w, all_seqs, threads)
        total_t += dt
        total_b += nb
        passes += 1
    # the same oracle on one thread, on the first sequences of the batch (~2 s)
    one_t = one_b = 0.0
    for s_ in range(w.num_seqs):
        dt, nb = oracle_run(setup, w, np.array([s_]), 1)
        one_t += dt
        one_b += nb
        if one_t >= 2.0:
            break
    return {"value": total_b / total_t / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{passes} full pass(es) of the {w.num_seqs}-sequence batch, fp64, "
                      f"OpenMP over (sequence, KV head), {total_t:.1f} s",
            "single_thread_gbs": one_b / one_t / 1e9, "nproc": os.cpu_count(), "cpu_model": host_cpu_model()}


def prefill_config(st, world):
    """The `config` object of a prefill line, the same for both arms."""
    dt = {torch.float16: "f16", torch.bfloat16: "bf16"}[st.dtype]
    n_pairs = int(st.copy_pairs.shape[0])
    return {"workload": f"{st.name}: {st.num_seqs} requests, prefixes {sorted(set(st.prefix_lens))}, "
                        f"{st.num_tokens} new tokens (max chunk {st.max_query_len}), {st.num_heads} query / "
                        f"{st.num_kv_heads} KV heads, d {st.head_dim}, {dt}, block {st.block_size}, "
                        f"{n_pairs} copy-on-write pairs",
            "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (queries + outputs + pool above 129 MB); no flush",
            "useful_flops_per_step": metrics.prefill_flops(st.attended_pairs(), st.num_heads, st.head_dim),
            "attended_pairs_per_head": st.attended_pairs()}


def run_reference_prefill(args):
    """The oracle's prefill on the same step: each timed step is a bounded
    sample (whole sequences, shortest first) sized so that warm-up + timed
    steps take about two minutes."""
    st = workloads.make_prefill(args.workload, device="cpu", num_seqs=args.num_seqs)
    per_step = max(0.05, 120.0 / max(args.steps + args.warmup, 1))
    for _ in range(args.warmup):
        prefill_cpu_baseline(st, per_step)
    tot_t = tot_f = 0.0
    last = None
    for _ in range(args.steps):
        t0 = time.perf_counter()
        last = prefill_cpu_baseline(st, per_step)
        dt = time.perf_counter() - t0
        tot_t += dt
        tot_f += last["value"] * 1e12 * dt
    value = tot_f / tot_t / 1e12
    print(json.dumps({"impl": "reference", "metric": PREFILL_METRIC, "value": value, "unit": "TFLOP/s",
                      "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
                      "ms_per_step": 1e3 * tot_t / max(args.steps, 1), "higher_is_better": True, "scaling": "weak",
                      "vs_baseline": None, "dtype": "f64", "data": "synthetic",
                      "config": prefill_config(st, max(args.gpus, 1)),
                      "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": last["cores"], "kind": "oracle",
                                       "sample": last["sample"], "nproc": last["nproc"],
                                       "cpu_model": last["cpu_model"]},
                      "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                              "d2h_bytes_per_step": 0}}), flush=True)


def decode_config(args, w, world, part, n_pairs, full_heads=None):
    """The `config` object of a decode line, the same for both arms.
    full_heads: (H, Hkv) of the whole batch when the ranks split it by head."""
    ctx_list = w.context_lens.tolist()
    elem = w.query.element_size()
    dt = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}[w.dtype]
    h, hkv = full_heads or (w.num_heads, w.num_kv_heads)
    bytes_step = (metrics.decode_bytes(ctx_list, w.num_heads, w.num_kv_heads, w.head_dim, elem, 4)
                  + metrics.write_bytes(w.num_tokens, w.num_kv_heads, w.head_dim, elem)
                  + metrics.copy_bytes(n_pairs, 1, w.num_kv_heads, w.block_size, w.head_dim, elem))
    if args.split == "heads":
        parallelism = f"tp{world}: the batch split by KV head ({hkv // world} KV heads per rank, same block tables)"
    else:
        parallelism = f"replicas x{world}"
    return {"workload": f"{args.workload}: {w.num_seqs} seqs, {h} query / {hkv} KV heads, d {w.head_dim}, "
                        f"{dt} K/V, block {w.block_size}, partition {part}, {n_pairs} copy-on-write pairs",
            "parallelism": parallelism,
            "l2": "inputs larger than L2 (KV bytes per step far above the 129 MB L2); no flush",
            "algorithmic_bytes_per_step": bytes_step, "sum_context_tokens": int(sum(ctx_list)),
            "table_and_length_bytes_per_step": metrics.table_bytes(ctx_list, w.block_size)}


def run_reference(args, rank, world):
    if rank != 0:
        return
    if args.workload.startswith("prefill_"):
        run_reference_prefill(args)
        return
    import numpy as np

    import oracle as O

    kw = {"num_seqs": args.num_seqs}
    if args.workload == "long_context":
        kw["block_size"] = args.block_size
    w = workloads.make(args.workload, device="cpu", **kw)
    setup = oracle_setup(w)
    threads = O.get().max_threads()
    # Size the per-step sample so that warm-up + timed steps take about 2 minutes.
    probe = np.arange(min(8, w.num_seqs))
    dt, _ = oracle_run(setup, w, probe, threads)
    per_seq = max(dt / len(probe), 1e-6)
    n = int(max(1, min(w.num_seqs, 120.0 / max(args.steps + args.warmup, 1) / per_seq)))
    rng = np.random.default_rng(0)
    samples = [rng.choice(w.num_seqs, size=n, replace=False) for _ in range(args.steps + args.warmup)]
    for i in range(args.warmup):
        oracle_run(setup, w, samples[i], threads)
    tot_t = tot_b = 0.0
    for i in range(args.steps):
        dt, nb = oracle_run(setup, w, samples[args.warmup + i], threads)
        tot_t += dt
        tot_b += nb
    value = tot_b / tot_t / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot_t / max(args.steps, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": decode_config(args, w, max(args.gpus, 1), partition_for(args, w), int(w.copy_pairs.shape[0])),
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"{n} random sequences of the batch per step",
                             "nproc": os.cpu_count(), "cpu_model": host_cpu_model()},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def make_workload(args, rank, world=1, device="cuda"):
    """Rank `rank`'s batch: its own replica (seed per rank), or with
    --split heads its KV heads of the one batch every rank draws alike."""
    kw = {"num_seqs": args.num_seqs}
    if args.workload == "long_context":
        kw["block_size"] = args.block_size
    replica = 0 if args.split == "heads" else rank
    seed = workloads.SEED_BASE + workloads.WORKLOADS.index(args.workload) + 1000 * replica
    w = workloads.make(args.workload, device=device, seed=seed, **kw)
    if args.split == "heads" and world > 1:
        full = w
        w = sharding.shard_workload(full, world, rank)
        del full
        if device == "cuda":
            torch.cuda.empty_cache()
    return w


def partition_for(args, w):
    """Explicit partition size, so that the number of launches is known."""
    if args.partition_size is not None:
        return args.partition_size
    if w.partition_size:
        return w.partition_size
    return 512


def graph_time_us(fn, reps, stream):
    """Device time of one call of fn, replayed from a CUDA graph of `reps` calls."""
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    with torch.cuda.stream(side):
        fn()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for _ in range(reps):
                fn()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    g.replay()
    e.record(stream)
    torch.cuda.synchronize()
    return 1e3 * s.elapsed_time(e) / reps


def swap_rows(w, stream, pairs_n=2048):
    """Swap-out (GPU -> page-locked host) and swap-in of 2048 random blocks of
    the workload's pool in one pa_swap_blocks launch each, against one
    cudaMemcpyAsync per K and per V block (both timed from CUDA graphs).
    GB/s = bytes moved (each block once) / time."""
    g = torch.Generator().manual_seed(7)
    n = min(pairs_n, w.num_blocks)
    src = torch.randperm(w.num_blocks, generator=g)[:n]
    hk = torch.empty((n,) + tuple(w.k_cache.shape[1:]), dtype=w.k_cache.dtype).pin_memory()
    hv = torch.empty_like(hk).pin_memory()
    out_pairs = torch.stack([src, torch.arange(n)], dim=1).contiguous().cuda()
    in_pairs = torch.stack([torch.arange(n), src], dim=1).contiguous().cuda()
    moved = 2 * n * w.k_cache[0].numel() * w.k_cache.element_size()
    out_us = graph_time_us(lambda: api.swap_blocks([w.k_cache], [w.v_cache], [hk], [hv], out_pairs), 5, stream)
    in_us = graph_time_us(lambda: api.swap_blocks([hk], [hv], [w.k_cache], [w.v_cache], in_pairs), 5, stream)
    src_list = src.tolist()

    def per_block_out():
        for j, b in enumerate(src_list):
            hk[j].copy_(w.k_cache[b], non_blocking=True)
            hv[j].copy_(w.v_cache[b], non_blocking=True)

    memcpy_us = graph_time_us(per_block_out, 1, stream)
    # Reference: the same bytes as two contiguous device -> host copies.
    dk, dv = w.k_cache[:n], w.v_cache[:n]
    contiguous_us = graph_time_us(lambda: (hk.copy_(dk, non_blocking=True), hv.copy_(dv, non_blocking=True)), 5,
                                  stream)
    status, code = api.get_device_error()
    if status != 0:
        raise RuntimeError(f"device error {status} ({code:#x}) in the swap rows")
    return {"swap_out_us": out_us, "swap_out_gbs": moved / (out_us * 1e-6) / 1e9,
            "swap_in_us": in_us, "swap_in_gbs": moved / (in_us * 1e-6) / 1e9,
            "swap_out_per_block_memcpy_us": memcpy_us,
            "swap_out_per_block_memcpy_gbs": moved / (memcpy_us * 1e-6) / 1e9,
            "contiguous_d2h_memcpy_gbs": moved / (contiguous_us * 1e-6) / 1e9, "swap_pairs": n}


def host_call_costs(w, out, ws, max_ctx, part, calls=40):
    """Host time to submit one pa_decode call: through the Python binding
    (argument checks, ctypes), through a prepared call (api.PreparedDecode:
    checks done once) and through ctypes with prepared arguments (the C ABI's
    own cost: argument checks, cached tensor maps, the launches).  A few calls
    at a time, so that the launch queue never fills."""
    import ctypes

    lib = native.load()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(calls):
        api.decode(w.query, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale, out=out,
                   max_context_len=max_ctx, partition_size=part, workspace=ws)
    py_us = 1e6 * (time.perf_counter() - t0) / calls
    torch.cuda.synchronize()
    prepared = api.PreparedDecode(w.query, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale, out=out,
                                  max_context_len=max_ctx, partition_size=part, workspace=ws)
    t0 = time.perf_counter()
    for _ in range(calls):
        prepared()
    prep_us = 1e6 * (time.perf_counter() - t0) / calls
    torch.cuda.synchronize()
    desc = api.cache_desc(w.k_cache)
    args_ = (out.data_ptr(), native.PA_F32, w.query.data_ptr(), w.k_cache.data_ptr(), w.v_cache.data_ptr(),
             ctypes.byref(desc), w.block_tables.data_ptr(), w.block_tables.shape[1], w.context_lens.data_ptr(),
             w.num_seqs, max_ctx, w.num_heads, w.num_kv_heads, ctypes.c_float(w.scale), part, ws.data_ptr(),
             ws.numel(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    t0 = time.perf_counter()
    for _ in range(calls):
        rc = lib.pa_decode(*args_)
    c_us = 1e6 * (time.perf_counter() - t0) / calls
    torch.cuda.synchronize()
    if rc != 0:
        raise RuntimeError(f"pa_decode returned {rc}")
    return {"host_us_per_decode_call_python": py_us, "host_us_per_decode_call_prepared": prep_us,
            "host_us_per_decode_call_c_abi": c_us}


def run_ours(args, rank, world, local_rank):
    torch.cuda.set_device(local_rank)
    native.load()
    w = make_workload(args, rank, world)
    full_heads = (w.num_heads * world, w.num_kv_heads * world) if args.split == "heads" else None
    elem = w.query.element_size()
    ctx_list = w.context_lens.tolist()
    max_ctx = max(ctx_list)
    part = partition_for(args, w)
    pairs = w.copy_pairs
    n_pairs = int(pairs.shape[0])
    decode_b = metrics.decode_bytes(ctx_list, w.num_heads, w.num_kv_heads, w.head_dim, elem, 4)
    write_b = metrics.write_bytes(w.num_tokens, w.num_kv_heads, w.head_dim, elem)
    copy_b = metrics.copy_bytes(n_pairs, 1, w.num_kv_heads, w.block_size, w.head_dim, elem)
    bytes_step = decode_b + write_b + copy_b
    stream = torch.cuda.current_stream()
    out = torch.empty((w.num_seqs, w.num_heads, w.head_dim), dtype=torch.float32, device="cuda")
    ws = torch.empty(api.decode_workspace_size(w.num_seqs, w.num_heads, max_ctx, part, w.head_dim),
                     dtype=torch.uint8, device="cuda")
    # Pre-step copy of the inputs for the oracle leg (the GPU steps write in place).
    cpu_w = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        cpu_w = workloads.Workload(**{**w.__dict__, **{f: getattr(w, f).cpu() for f in (
            "context_lens", "block_tables", "query", "k_cache", "v_cache", "new_key", "new_value",
            "slot_mapping", "copy_pairs")}})

    # The cache write and decode calls of the device-timed steps, checked and
    # marshalled once (api.PreparedCacheWrite / api.PreparedDecode, the
    # binding a serving loop uses for fixed buffers); the end-to-end leg
    # below goes through api.reshape_and_cache and api.decode.
    prepared = api.PreparedDecode(w.query, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale, out=out,
                                  max_context_len=max_ctx, partition_size=part, workspace=ws)
    prepared_write = api.PreparedCacheWrite(w.new_key, w.new_value, w.k_cache, w.v_cache, w.slot_mapping)

    def step(q=w.query, nk=w.new_key, nv=w.new_value, slots=w.slot_mapping, tables=w.block_tables,
             ctx=w.context_lens, prs=pairs, marks=None):
        if marks:
            marks[0].record(stream)
        if n_pairs:
            api.copy_blocks([w.k_cache], [w.v_cache], prs)
        if marks:
            marks[1].record(stream)
        if nk is w.new_key and nv is w.new_value and slots is w.slot_mapping:
            prepared_write()
        else:
            api.reshape_and_cache(nk, nv, w.k_cache, w.v_cache, slots)
        if marks:
            marks[2].record(stream)
        if q is w.query and tables is w.block_tables and ctx is w.context_lens:
            prepared()
        else:
            api.decode(q, w.k_cache, w.v_cache, tables, ctx, w.scale, out=out, max_context_len=max_ctx,
                       partition_size=part, workspace=ws)
        if marks:
            marks[3].record(stream)

    for _ in range(args.warmup):
        step()
    status, code = api.get_device_error()
    if status != 0:
        raise RuntimeError(f"device error {status} ({code:#x}) during warm-up")

    # ---- device-resident timing -----------------------------------------
    k = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(k)]
    sampler = ClockSampler(local_rank)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.2)  # let the sampler start before the timed region
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    # Headline loop: events only at its two ends (an event between two
    # launches would stop the planning kernel overlapping the cache write).
    start.record(stream)
    for i in range(k):
        step()
    end.record(stream)
    # Breakdown loop: the same steps with events around every call, for the
    # per-row times and the decode call's duration in the roofline.
    for i in range(k):
        step(marks=ev[i])
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier(world)
    status, code = api.get_device_error()
    if status != 0:
        raise RuntimeError(f"device error {status} ({code:#x}) in the timed region")
    total_ms = start.elapsed_time(end)
    copy_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    write_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    decode_ms = statistics.mean(e[2].elapsed_time(e[3]) for e in ev)
    step_ms = all_reduce_max(total_ms / k, world)
    decode_ms_max = all_reduce_max(decode_ms, world)
    # Kernels per step: copy-on-write copy (if any pairs), cache write,
    # decode, and -- when a context can span more than one partition -- the
    # planning and cross-partition reduce kernels.
    per_step = (1 if n_pairs else 0) + 2 + (2 if max_ctx > part else 0)
    launches = k * per_step

    e2e_ms, h2d, d2h, launches_e2e, host_us = None, 0, 0, 0, None
    if not args.no_e2e:
        # ---- end to end through the public API with host buffers -----------
        # Every step uploads its inputs from pinned host memory and downloads
        # its output.  Two buffer sets and a copy stream let step i+1's upload
        # and step i's download overlap step i's kernels, as a serving loop
        # would; all copies are inside the timed region.
        names = ["query", "new_key", "new_value", "slot_mapping", "block_tables", "context_lens"]
        if n_pairs:
            names.append("copy_pairs")
        # The step's inputs packed into one pinned staging buffer (one upload
        # per step), each at a 256-byte aligned offset; typed views on both sides.
        layout, off = {}, 0
        for name in names:
            t = getattr(w, name)
            layout[name] = (off, t.dtype, tuple(t.shape))
            off += -(-t.numel() * t.element_size() // 256) * 256
        staging = torch.empty(off, dtype=torch.uint8).pin_memory()
        for name in names:
            o, dt_, shp = layout[name]
            t = getattr(w, name).cpu().contiguous()
            staging[o:o + t.numel() * t.element_size()].copy_(t.view(-1).view(torch.uint8))

        def views(buf):
            out_ = {}
            for name, (o, dt_, shp) in layout.items():
                n = 1
                for x in shp:
                    n *= x
                nbytes = n * torch.tensor([], dtype=dt_).element_size()
                out_[name] = buf[o:o + nbytes].view(dt_).view(shp)
            return out_

        dev_bufs = [torch.empty(off, dtype=torch.uint8, device="cuda") for _ in range(2)]
        dev = [views(b_) for b_ in dev_bufs]
        outs = [torch.empty_like(out) for _ in range(2)]
        out_host = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        h2d = sum(getattr(w, name).numel() * getattr(w, name).element_size() for name in names)
        d2h = out_host[0].numel() * out_host[0].element_size()
        # Separate upload and download streams: on one in-order stream, step
        # i+1's upload would queue behind step i's download, which waits for
        # step i's kernels.
        upload_stream = torch.cuda.Stream()
        download_stream = torch.cuda.Stream()
        inputs_ready = [torch.cuda.Event() for _ in range(2)]
        output_ready = [torch.cuda.Event() for _ in range(2)]
        buffer_free = [torch.cuda.Event() for _ in range(2)]
        download_done = [torch.cuda.Event() for _ in range(2)]
        for ev_ in buffer_free + download_done:
            ev_.record(stream)

        def e2e_step(i):
            b = i % 2
            d = dev[b]
            with torch.cuda.stream(upload_stream):
                upload_stream.wait_event(buffer_free[b])    # step i-2 finished reading this set
                dev_bufs[b].copy_(staging, non_blocking=True)
                inputs_ready[b].record(upload_stream)
            stream.wait_event(inputs_ready[b])
            stream.wait_event(download_done[b])             # step i-2's output has left outs[b]
            if n_pairs:
                api.copy_blocks([w.k_cache], [w.v_cache], d["copy_pairs"])
            api.reshape_and_cache(d["new_key"], d["new_value"], w.k_cache, w.v_cache, d["slot_mapping"])
            api.decode(d["query"], w.k_cache, w.v_cache, d["block_tables"], d["context_lens"], w.scale, out=outs[b],
                       max_context_len=max_ctx, partition_size=part, workspace=ws)
            output_ready[b].record(stream)
            buffer_free[b].record(stream)
            with torch.cuda.stream(download_stream):
                download_stream.wait_event(output_ready[b])
                out_host[b].copy_(outs[b], non_blocking=True)
                download_done[b].record(download_stream)

        k_e2e = max(3, min(k, 500))
        for i in range(3):
            e2e_step(i)
        barrier(world)
        torch.cuda.synchronize()
        s2 = torch.cuda.Event(enable_timing=True)
        e2 = torch.cuda.Event(enable_timing=True)
        s2.record(stream)
        upload_stream.wait_stream(stream)
        download_stream.wait_stream(stream)
        host_t0 = time.perf_counter()
        for i in range(k_e2e):
            e2e_step(i)
        host_us = 1e6 * (time.perf_counter() - host_t0) / k_e2e
        stream.wait_stream(download_stream)  # the last download is inside the timed region
        e2.record(stream)
        torch.cuda.synchronize()
        e2e_ms = all_reduce_max(s2.elapsed_time(e2) / k_e2e, world)
        launches_e2e = k_e2e * per_step

    decode_call = lambda: api.decode(w.query, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale,
                                     out=out, max_context_len=max_ctx, partition_size=part, workspace=ws)
    rows = {"a1_cache_write_us": 1e3 * write_ms, "a2_a6_decode_us": 1e3 * decode_ms,
            "a1_cache_write_median_us": 1e3 * statistics.median(e[1].elapsed_time(e[2]) for e in ev),
            "a2_a6_decode_median_us": 1e3 * statistics.median(e[2].elapsed_time(e[3]) for e in ev),
            "step_graph_us": graph_time_us(step, 20, stream),
            # device time of back-to-back decode calls with no host gap (replayed from a CUDA graph)
            "a2_a6_decode_warm_graph_us": graph_time_us(decode_call, 20, stream),
            "a1_cache_write_graph_us": graph_time_us(
                lambda: api.reshape_and_cache(w.new_key, w.new_value, w.k_cache, w.v_cache, w.slot_mapping), 20,
                stream)}
    rows.update(host_call_costs(w, out, ws, max_ctx, part))
    if not args.no_rows:
        # ---- cold decode calls: L2 flushed (a 2 x L2 buffer written) before each
        flush = torch.empty(2 * 129 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
        cold = []
        for _ in range(20):
            flush.fill_(1.0)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            api.decode(w.query, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale, out=out,
                       max_context_len=max_ctx, partition_size=part, workspace=ws)
            b.record(stream)
            cold.append((a, b))
        torch.cuda.synchronize()
        rows["a2_a6_decode_cold_median_us"] = 1e3 * statistics.median(a.elapsed_time(b) for a, b in cold)
        rows["a2_a6_decode_cold_gbs"] = decode_b / (rows["a2_a6_decode_cold_median_us"] * 1e-6) / 1e9
        # The write-flush leaves ~L2's size of dirty lines, written back to
        # HBM while the call reads; flushing by reading 2 x L2 instead leaves
        # clean lines, so this one measures the call alone from a cold L2.
        cold = []
        sink = torch.empty((), dtype=torch.float32, device="cuda")
        for _ in range(20):
            torch.sum(flush, dim=0, out=sink)
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            api.decode(w.query, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale, out=out,
                       max_context_len=max_ctx, partition_size=part, workspace=ws)
            b.record(stream)
            cold.append((a, b))
        torch.cuda.synchronize()
        rows["a2_a6_decode_cold_clean_median_us"] = 1e3 * statistics.median(a.elapsed_time(b) for a, b in cold)
        rows["a2_a6_decode_cold_clean_gbs"] = decode_b / (rows["a2_a6_decode_cold_clean_median_us"] * 1e-6) / 1e9
        del flush, sink
    if n_pairs:
        rows["a7_copy_blocks_us"] = 1e3 * copy_ms
        rows["a7_copy_blocks_pairs"] = n_pairs
    if not args.no_rows:
        # ---- the copy-on-write row on the parallel-sampling copy list, timed
        # from a CUDA graph (one call is a few microseconds of device time).
        ps = workloads.make("parallel_sampling", device="cuda")
        ck, cv = ps.k_cache.clone(), ps.v_cache.clone()
        copy_us = graph_time_us(lambda: api.copy_blocks([ck], [cv], ps.copy_pairs), 50, stream)
        ps_b = metrics.copy_bytes(ps.copy_pairs.shape[0], 1, ps.num_kv_heads, ps.block_size, ps.head_dim, 2)
        rows["a7_copy_blocks_graph_us"] = copy_us
        rows["a7_copy_blocks_graph_gbs"] = ps_b / (copy_us * 1e-6) / 1e9
        rows["a7_copy_blocks_graph_pairs"] = int(ps.copy_pairs.shape[0])
        del ps, ck, cv
        rows.update(swap_rows(w, stream))
        rows.update(prefill_rows(stream))

    # ---- CPU oracle baseline (rank 0, one GPU only) ------------------------
    cpu = None
    if cpu_w is not None:
        cpu = cpu_baseline(cpu_w, args.cpu_seconds)

    if rank != 0:
        return
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", 6800.0))
    achieved = decode_b / (decode_ms * 1e-3) / 1e9
    traffic = (profiled_traffic() if args.workload == WORKLOAD and args.num_seqs is None and world == 1
               else None)
    dt = {torch.float32: "f32", torch.float16: "f16", torch.bfloat16: "bf16"}[w.dtype]
    config = decode_config(args, w, world, part, n_pairs, full_heads)
    assert config["algorithmic_bytes_per_step"] == bytes_step
    line = {
        "metric": METRIC,
        # one step = the whole hot path (copy-on-write, cache write, decode);
        # decode alone is "decode_gbs" below and the roofline object
        "value": aggregate_throughput(world, bytes_step, step_ms),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": k,
        "warmup": args.warmup,
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "strong" if args.split == "heads" and world > 1 else "weak",
        "vs_baseline": None,
        "dtype": dt,
        "data": "synthetic",
        "config": config,
        "decode_gbs": aggregate_throughput(world, decode_b, decode_ms_max),
        # with --split heads every rank decodes the same sequences (its heads)
        "seq_decode_steps_per_s": (1 if args.split == "heads" else world) * w.num_seqs / (step_ms * 1e-3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "peak_source": f"{peak_kind} hbm_gbs",
                     "kernel": f"pa_decode ({'CUDA-core' if args.decode_kernel == 'simt' else 'tensor-core'} "
                               f"decode kernel + planning + reduce kernels), CUDA events per call"},
        "rows": rows,
        "e2e": None if e2e_ms is None else {
            "value": aggregate_throughput(world, bytes_step, e2e_ms), "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "host_us_per_step": host_us},
        "gpu_launches": launches,
        "gpu_launches_e2e": launches_e2e,
        "clocks": clocks,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# prefill over a cached shared prefix
# ---------------------------------------------------------------------------
def prefill_step_fn(st, k, v, out):
    """The step: copy-on-write, cache write of the new tokens, prefill."""
    def step():
        if st.copy_pairs.numel():
            api.copy_blocks([k], [v], st.copy_pairs)
        api.reshape_and_cache(st.new_key, st.new_value, k, v, st.slot_mapping)
        api.prefill(st.query, st.query_start_loc, k, v, st.block_tables, st.context_lens, st.scale,
                    st.max_query_len, out=out)
    return step


def prefill_rows(stream, names=("prefill_llama8b", "prefill_opt13b")):
    """Each prefill workload's pa_prefill call and whole step, timed from CUDA
    graphs; useful TFLOP/s and its fraction of the measured bf16 peak."""
    peaks, kind = measured_peaks()
    peak = float(peaks.get("bf16_tflops", 1900.0))
    rows = {}
    for name in names:
        st = workloads.make_prefill(name, device="cuda")
        k, v = st.k_cache.clone(), st.v_cache.clone()
        out = torch.empty(st.num_tokens, st.num_heads, st.head_dim, dtype=st.dtype, device="cuda")
        prefill_step_fn(st, k, v, out)()
        call_us = graph_time_us(lambda: api.prefill(st.query, st.query_start_loc, k, v, st.block_tables,
                                                    st.context_lens, st.scale, st.max_query_len, out=out),
                                10, stream)
        step_us = graph_time_us(prefill_step_fn(st, k, v, out), 10, stream)
        status, code = api.get_device_error()
        if status != 0:
            raise RuntimeError(f"device error {status} ({code:#x}) in the {name} row")
        write_us = graph_time_us(lambda: api.reshape_and_cache(st.new_key, st.new_value, k, v, st.slot_mapping),
                                 10, stream)
        write_b = metrics.write_bytes(st.num_tokens, st.num_kv_heads, st.head_dim, st.new_key.element_size())
        hbm = float(peaks.get("hbm_gbs", 6800.0))
        rows[f"{name}_cache_write_us"] = write_us
        rows[f"{name}_cache_write_gbs"] = write_b / (write_us * 1e-6) / 1e9
        rows[f"{name}_cache_write_frac_of_{kind}_hbm"] = write_b / (write_us * 1e-6) / 1e9 / hbm
        tflops = metrics.prefill_flops(st.attended_pairs(), st.num_heads, st.head_dim) / (call_us * 1e-6) / 1e12
        rows[f"{name}_call_us"] = call_us
        rows[f"{name}_tflops"] = tflops
        rows[f"{name}_frac_of_{kind}_bf16_peak"] = tflops / peak
        rows[f"{name}_step_us"] = step_us
        rows[f"{name}_new_tokens_per_s"] = st.num_tokens / (step_us * 1e-6)
        del st, k, v, out
    return rows


def prefill_cpu_baseline(st, target_seconds):
    """The fp64 oracle on whole sequences of the step, as many as fit in
    about target_seconds (at least one)."""
    import numpy as np

    import oracle as O

    def bits(t):
        t = t.detach().contiguous().cpu()
        return t.view(torch.int16).numpy()

    orc = O.get()
    threads = orc.max_threads()
    code = {torch.float16: O.F16, torch.bfloat16: O.BF16}[st.dtype]
    k, v = bits(st.k_cache).copy(), bits(st.v_cache).copy()
    if st.copy_pairs.numel():
        orc.copy_blocks([k], [v], st.copy_pairs.cpu().numpy())
    orc.reshape_and_cache(bits(st.new_key), bits(st.new_value), k, v, st.slot_mapping.cpu().numpy())
    q = bits(st.query)
    qsl = st.query_start_loc.cpu().numpy()
    tables, ctx = st.block_tables.cpu().numpy(), st.context_lens.cpu().numpy()
    total_t, flops, done = 0.0, 0, 0
    order = np.argsort(np.asarray(st.chunk_lens))  # shortest first: several sequences in the budget
    for s in order:
        a, b = int(qsl[s]), int(qsl[s + 1])
        if b == a:
            continue
        t0 = time.perf_counter()
        orc.prefill(q[a:b], np.array([0, b - a], dtype=np.int32), k, v, code, tables[s:s + 1], ctx[s:s + 1],
                    st.num_kv_heads, st.scale, num_threads=threads)
        total_t += time.perf_counter() - t0
        n, pre = st.chunk_lens[s], st.prefix_lens[s]
        flops += metrics.prefill_flops(n * pre + n * (n + 1) // 2, st.num_heads, st.head_dim)
        done += 1
        if total_t >= target_seconds:
            break
    return {"value": flops / total_t / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{done} whole sequence(s) of the step (shortest first), fp64, OpenMP over KV heads, "
                      f"{total_t:.1f} s", "nproc": os.cpu_count(), "cpu_model": host_cpu_model()}


def run_prefill(args, rank, world, local_rank):
    """One step: copy-on-write of the shared partial prefix block, cache write
    of the new tokens, pa_prefill.  value = useful attention TFLOP/s of the
    step (whole job); roofline = the pa_prefill call against the measured
    bf16 tensor peak."""
    torch.cuda.set_device(local_rank)
    native.load()
    st = workloads.make_prefill(args.workload, device="cuda", num_seqs=args.num_seqs,
                                seed=None if rank == 0 else workloads.SEED_BASE + 500 + rank)
    stream = torch.cuda.current_stream()
    k, v = st.k_cache.clone(), st.v_cache.clone()
    out = torch.empty(st.num_tokens, st.num_heads, st.head_dim, dtype=st.dtype, device="cuda")
    step = prefill_step_fn(st, k, v, out)
    flops = metrics.prefill_flops(st.attended_pairs(), st.num_heads, st.head_dim)
    n_pairs = int(st.copy_pairs.shape[0])
    per_step = (1 if n_pairs else 0) + 2
    for _ in range(max(args.warmup, 3)):
        step()
    status, code = api.get_device_error()
    if status != 0:
        raise RuntimeError(f"device error {status} ({code:#x}) during warm-up")
    k_steps = max(1, args.steps)
    sampler = ClockSampler(local_rank)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.2)
    s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(k_steps):
        step()
    e0.record(stream)
    torch.cuda.synchronize()
    # breakdown: the pa_prefill call alone, events around each call
    calls = []
    for _ in range(min(k_steps, 50)):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if n_pairs:
            api.copy_blocks([k], [v], st.copy_pairs)
        api.reshape_and_cache(st.new_key, st.new_value, k, v, st.slot_mapping)
        a.record(stream)
        api.prefill(st.query, st.query_start_loc, k, v, st.block_tables, st.context_lens, st.scale,
                    st.max_query_len, out=out)
        b.record(stream)
        calls.append((a, b))
    torch.cuda.synchronize()
    clocks = sampler.stop()
    status, code = api.get_device_error()
    if status != 0:
        raise RuntimeError(f"device error {status} ({code:#x}) in the timed region")
    step_ms = all_reduce_max(s0.elapsed_time(e0) / k_steps, world)
    call_ms = statistics.median(a.elapsed_time(b) for a, b in calls)

    # end to end: the step's inputs from page-locked host memory, the output
    # back.  Two device buffer sets and separate upload / download streams let
    # step i+1's upload and step i's download overlap step i's kernels, as a
    # serving loop would; every copy is inside the timed region.
    e2e = None
    if not args.no_e2e:
        names = ("query", "new_key", "new_value", "slot_mapping", "query_start_loc", "context_lens", "block_tables")
        host_in = [getattr(st, n).cpu().pin_memory() for n in names]
        dev_in = [[torch.empty_like(getattr(st, n)) for n in names] for _ in range(2)]
        outs = [torch.empty_like(out) for _ in range(2)]
        host_out = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        h2d = sum(t.numel() * t.element_size() for t in host_in)
        d2h = host_out[0].numel() * host_out[0].element_size()
        upload_stream, download_stream = torch.cuda.Stream(), torch.cuda.Stream()
        inputs_ready = [torch.cuda.Event() for _ in range(2)]
        output_ready = [torch.cuda.Event() for _ in range(2)]
        buffer_free = [torch.cuda.Event() for _ in range(2)]
        download_done = [torch.cuda.Event() for _ in range(2)]
        for ev_ in buffer_free + download_done:
            ev_.record(stream)

        def e2e_step(i):
            b = i % 2
            d = dev_in[b]
            with torch.cuda.stream(upload_stream):
                upload_stream.wait_event(buffer_free[b])       # step i-2 finished reading this set
                for h_, d_ in zip(host_in, d):
                    d_.copy_(h_, non_blocking=True)
                inputs_ready[b].record(upload_stream)
            stream.wait_event(inputs_ready[b])
            stream.wait_event(download_done[b])                # step i-2's output has left outs[b]
            q_, nk_, nv_, slots_, qsl_, ctx_, tables_ = d
            if st.copy_pairs.numel():
                api.copy_blocks([k], [v], st.copy_pairs)
            api.reshape_and_cache(nk_, nv_, k, v, slots_)
            api.prefill(q_, qsl_, k, v, tables_, ctx_, st.scale, st.max_query_len, out=outs[b])
            output_ready[b].record(stream)
            buffer_free[b].record(stream)
            with torch.cuda.stream(download_stream):
                download_stream.wait_event(output_ready[b])
                host_out[b].copy_(outs[b], non_blocking=True)
                download_done[b].record(download_stream)

        for i in range(3):
            e2e_step(i)
        torch.cuda.synchronize()
        n_e2e = max(1, min(k_steps, 200))
        s1, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s1.record(stream)
        upload_stream.wait_stream(stream)
        download_stream.wait_stream(stream)
        for i in range(n_e2e):
            e2e_step(i)
        stream.wait_stream(download_stream)  # the last download is inside the timed region
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = all_reduce_max(s1.elapsed_time(e1) / n_e2e, world)
        e2e = {"value": world * flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = prefill_cpu_baseline(st, args.cpu_seconds)
    if rank != 0:
        return
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("bf16_tflops", 1900.0))
    achieved = flops / (call_ms * 1e-3) / 1e12
    # DRAM bytes per pa_prefill launch from the committed ncu summary (the
    # llama8b-shaped workload at full size, current kernel source only)
    traffic = (profiled_traffic(PREFILL_PROFILE_SUMMARY, PREFILL_KERNEL_SOURCES)
               if args.workload == "prefill_llama8b" and args.num_seqs is None else None)
    dt = {torch.float16: "f16", torch.bfloat16: "bf16"}[st.dtype]
    line = {
        "metric": PREFILL_METRIC,
        "value": world * flops / (step_ms * 1e-3) / 1e12,
        "unit": "TFLOP/s",
        "n_gpus": world, "steps": k_steps, "warmup": args.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dt, "data": "synthetic",
        "config": prefill_config(st, world),
        "new_tokens_per_s": world * st.num_tokens / (step_ms * 1e-3),
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                     "traffic": traffic, "peak_source": f"{peak_kind} bf16_tflops (burst)",
                     "kernel": "pa_prefill (tcgen05 kernel), CUDA events per call; bf16 P is split in two halves, "
                               "so the tensor pipe does 1.5x the useful flops"},
        "rows": {"prefill_call_us": 1e3 * call_ms, "step_us": 1e3 * step_ms},
        "e2e": e2e,
        "gpu_launches": k_steps * per_step,
        "clocks": clocks,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


def run_beam(args, rank, world, local_rank):
    """Beam search (64 requests x 4 beams, 1000-token prompts, 16-token
    blocks, llama8b heads): every step forks and frees beams, copies shared
    blocks (copy-on-write), writes one token per beam and decodes.  A timed
    pass replays all steps of the trace; value = the steps' algorithmic bytes
    / their time."""
    torch.cuda.set_device(local_rank)
    native.load()
    t = workloads.beam_search(requests=64, beams=4, prompt_len=1000, steps=args.beam_steps, block_size=16,
                              num_heads=32, num_kv_heads=8, head_dim=128, dtype=torch.bfloat16,
                              seed=workloads.SEED_BASE + 10 + 1000 * rank, device="cuda")
    stream = torch.cuda.current_stream()
    k, v = t.k_cache, t.v_cache
    elem = k.element_size()
    part = args.partition_size or 512
    max_ctx = max(int(st.context_lens.max()) for st in t.steps)
    nseq = t.steps[0].context_lens.numel()
    ws = torch.empty(api.decode_workspace_size(nseq, t.num_heads, max_ctx, part, t.head_dim), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty(nseq, t.num_heads, t.head_dim, device="cuda")
    step_bytes, launches_per_pass, copies = 0, 0, 0
    for st in t.steps:
        n = int(st.copy_pairs.shape[0])
        copies += n
        step_bytes += metrics.decode_bytes(st.context_lens.tolist(), t.num_heads, t.num_kv_heads, t.head_dim, elem, 4)
        step_bytes += metrics.write_bytes(nseq, t.num_kv_heads, t.head_dim, elem)
        step_bytes += metrics.copy_bytes(n, 1, t.num_kv_heads, t.block_size, t.head_dim, elem)
        launches_per_pass += (1 if n else 0) + 2 + (2 if int(st.context_lens.max()) > part else 0)

    # Host-side facts of every step, taken before timing (no device sync in the loop).
    plan = [(st, int(st.context_lens.max()), int(st.copy_pairs.shape[0])) for st in t.steps]

    def one_pass():
        for st, mc, n in plan:
            if n:
                api.copy_blocks([k], [v], st.copy_pairs)
            api.reshape_and_cache(st.new_key, st.new_value, k, v, st.slot_mapping)
            api.decode(st.query, k, v, st.block_tables, st.context_lens, t.scale, out=out,
                       max_context_len=mc, partition_size=part, workspace=ws)

    for _ in range(max(args.warmup // len(t.steps), 3)):
        one_pass()
    status, code = api.get_device_error()
    if status != 0:
        raise RuntimeError(f"device error {status} ({code:#x}) during warm-up")
    passes = max(1, args.steps // len(t.steps))
    sampler = ClockSampler(local_rank)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.2)
    s0, e0 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(passes):
        one_pass()
    e0.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    status, code = api.get_device_error()
    if status != 0:
        raise RuntimeError(f"device error {status} ({code:#x}) in the timed region")
    nsteps = passes * len(t.steps)
    step_ms = all_reduce_max(s0.elapsed_time(e0) / nsteps, world)
    if rank != 0:
        return
    peaks, peak_kind = measured_peaks()
    value = aggregate_throughput(world, step_bytes / len(t.steps), step_ms)
    print(json.dumps({
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": nsteps, "warmup": args.warmup,
        "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"beam_search: 64 requests x 4 beams, 1000-token prompts, {len(t.steps)} steps, "
                               f"d 128, 32/8 heads, bf16, block 16, partition {part}",
                   "copy_on_write_pairs_per_step": copies / len(t.steps), "parallelism": f"replicas x{world}"},
        "seq_decode_steps_per_s": world * nseq / (step_ms * 1e-3),
        "roofline": {"bound": "hbm", "achieved": value / world, "peak": float(peaks.get("hbm_gbs", 6800.0)),
                     "unit": "GB/s", "frac": value / world / float(peaks.get("hbm_gbs", 6800.0)), "traffic": None,
                     "peak_source": f"{peak_kind} hbm_gbs", "kernel": "whole step (copy, write, decode)"},
        "gpu_launches": passes * launches_per_pass, "clocks": clocks}), flush=True)


def main():
    args = parse_args()
    if args.decode_kernel == "simt":
        api.set_option("decode_kernel_simt", True)
    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist

        if args.impl == "reference":
            if rank != 0:
                return
        else:
            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    try:
        if args.workload == "beam_search":
            run_beam(args, rank, world, local_rank)
        elif args.workload.startswith("prefill_"):
            run_prefill(args, rank, world, local_rank)
        else:
            run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
