#!/usr/bin/env python3
"""Benchmark of one decode step of paged attention on GB300.

Workload: the Llama-3.1-8B-shaped GQA batch -- 256 sequences, 32 query / 8 KV
heads, head_dim 128, bf16 K/V, 16-token blocks, lognormal context lengths
(median 1024, clipped to [16, 8192]), shuffled physical blocks.  One step is
the whole hot path over that batch: the cache write of each sequence's new
token (pa_reshape_and_cache), then decode attention over the paged cache
(pa_decode: planning kernel + decode kernel, split-KV and merge included).
The workload has no shared blocks, so no copy-on-write copies occur in its
step; pa_copy_blocks is timed on the parallel-sampling copy list and reported
under "rows".

Metric: KV GB/s -- algorithmic bytes (K and V rows of the attended tokens, the
queries, the outputs, plus the new tokens written) per second -- and
seq-decode-steps/s.  Inputs (1.8 GB of KV) are far larger than L2, so no
flush is needed between steps.

--impl reference runs the fp64 CPU oracle on the same workload (a bounded
sample of sequences per step) as the comparison arm.
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

from paged_kv_cache_132_gb300 import api, metrics, native, workloads  # noqa: E402

WORKLOAD = "llama8b"
METRIC = "paged decode-attention KV GB/s (% of GB300 HBM peak); seq-decode-steps/s"
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "decode_llama8b_ncu.md")
KERNEL_SOURCES = ["decode_mma.cuh", "decode_common.cuh", "decode.cu", "common.cuh"]


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timing leg")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="target CPU time of the oracle leg")
    ap.add_argument("--num-seqs", type=int, default=None,
                    help="first n sequences only (a smaller case of the same distribution, for profiling)")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffer) leg")
    ap.add_argument("--no-rows", action="store_true", help="skip the copy-on-write row timing")
    ap.add_argument("--decode-kernel", choices=["default", "simt"], default="default",
                    help="simt: time the CUDA-core decode kernel instead of the tensor-core one")
    return ap.parse_args()


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def kernel_digest() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "paged_kv_cache_132_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per decode launch from the committed ncu summary, if it was
    taken on the current kernel source (digest line must match)."""
    try:
        with open(PROFILE_SUMMARY, encoding="utf-8") as f:
            text = f.read()
    except OSError:
        return None
    digest = traffic = None
    for line in text.splitlines():
        if line.startswith("kernel_digest:"):
            digest = line.split(":", 1)[1].strip()
        if line.startswith("dram_bytes_per_launch:"):
            traffic = float(line.split(":", 1)[1].strip())
    return traffic if digest == kernel_digest() else None


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json"), encoding="utf-8") as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0}, "fallback"


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


def all_reduce_max(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def step_bytes(w):
    ctx = w.context_lens.tolist()
    decode = metrics.decode_bytes(ctx, w.num_heads, w.num_kv_heads, w.head_dim, w.query.element_size(), 4)
    write = metrics.write_bytes(w.num_tokens, w.num_kv_heads, w.head_dim, w.query.element_size())
    return decode, write


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
    return {"value": total_b / total_t / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": f"{passes} full pass(es) of the {w.num_seqs}-sequence batch, fp64, "
                      f"OpenMP over (sequence, KV head), {total_t:.1f} s"}


def run_reference(args, rank, world):
    if rank != 0:
        return
    import numpy as np

    import oracle as O

    w = workloads.make(WORKLOAD, device="cpu")
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
            "data": "synthetic", "config": {"workload": f"{WORKLOAD} (256 seqs, H32/Hkv8, d128, bf16 K/V, B16)"},
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads, "kind": "oracle",
                             "sample": f"{n} random sequences of the batch per step"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args, rank, world, local_rank):
    torch.cuda.set_device(local_rank)
    native.load()
    w = workloads.make(WORKLOAD, device="cuda", seed=workloads.SEED_BASE + 2 + 1000 * rank, num_seqs=args.num_seqs)
    decode_b, write_b = step_bytes(w)
    stream = torch.cuda.current_stream()
    out = torch.empty((w.num_seqs, w.num_heads, w.head_dim), dtype=torch.float32, device="cuda")
    max_ctx = w.max_context_len
    ws = torch.empty(api.decode_workspace_size(w.num_seqs, w.num_heads, max_ctx, 0, w.head_dim), dtype=torch.uint8,
                     device="cuda")
    # Pre-step pools for the oracle leg (the GPU steps below write in place).
    cpu_w = None
    if not args.no_cpu_baseline and rank == 0 and world == 1:
        cpu_w = workloads.Workload(**{**w.__dict__, **{f: getattr(w, f).cpu() for f in (
            "context_lens", "block_tables", "query", "k_cache", "v_cache", "new_key", "new_value",
            "slot_mapping", "copy_pairs")}})

    def step():
        api.reshape_and_cache(w.new_key, w.new_value, w.k_cache, w.v_cache, w.slot_mapping)
        api.decode(w.query, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale, out=out,
                   max_context_len=max_ctx, workspace=ws)

    for _ in range(args.warmup):
        step()
    status, code = api.get_device_error()
    if status != 0:
        raise RuntimeError(f"device error {status} ({code:#x}) during warm-up")

    # ---- device-resident timing -----------------------------------------
    k = args.steps
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(k)]
    sampler = ClockSampler(local_rank)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.2)  # let the sampler start before the timed region
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(k):
        ev[i][0].record(stream)
        api.reshape_and_cache(w.new_key, w.new_value, w.k_cache, w.v_cache, w.slot_mapping)
        ev[i][1].record(stream)
        api.decode(w.query, w.k_cache, w.v_cache, w.block_tables, w.context_lens, w.scale, out=out,
                   max_context_len=max_ctx, workspace=ws)
        ev[i][2].record(stream)
    end.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier(world)
    status, code = api.get_device_error()
    if status != 0:
        raise RuntimeError(f"device error {status} ({code:#x}) in the timed region")
    total_ms = start.elapsed_time(end)
    write_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    decode_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in ev)
    step_ms = all_reduce_max(total_ms / k, world)
    # Kernels per step: cache write, planning, decode, and (contexts longer
    # than the automatic partition of 512 tokens) the cross-partition reduce.
    per_step = 3 + (1 if max_ctx > 512 else 0)
    launches = k * per_step

    e2e_ms, h2d, d2h, launches_e2e = None, 0, 0, 0
    if not args.no_e2e:
        # ---- end to end through the public API with host buffers -----------
        host = {name: getattr(w, name).cpu().pin_memory() for name in
                ("query", "new_key", "new_value", "slot_mapping", "block_tables", "context_lens")}
        dev = {name: torch.empty_like(getattr(w, name)) for name in host}
        out_host = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = out_host.numel() * out_host.element_size()

        def e2e_step():
            for name, t in host.items():
                dev[name].copy_(t, non_blocking=True)
            api.reshape_and_cache(dev["new_key"], dev["new_value"], w.k_cache, w.v_cache, dev["slot_mapping"])
            api.decode(dev["query"], w.k_cache, w.v_cache, dev["block_tables"], dev["context_lens"], w.scale, out=out,
                       max_context_len=max_ctx, workspace=ws)
            out_host.copy_(out, non_blocking=True)

        k_e2e = max(3, min(k, 500))
        for _ in range(3):
            e2e_step()
        barrier(world)
        torch.cuda.synchronize()
        s2 = torch.cuda.Event(enable_timing=True)
        e2 = torch.cuda.Event(enable_timing=True)
        s2.record(stream)
        for _ in range(k_e2e):
            e2e_step()
        e2.record(stream)
        torch.cuda.synchronize()
        e2e_ms = all_reduce_max(s2.elapsed_time(e2) / k_e2e, world)
        launches_e2e = k_e2e * per_step

    rows = {"a1_cache_write_us": 1e3 * write_ms, "a2_a6_decode_us": 1e3 * decode_ms}
    if not args.no_rows:
        # ---- rows not in this workload's step: copy-on-write copies ----------
        ps = workloads.make("parallel_sampling", device="cuda")
        ck, cv = ps.k_cache.clone(), ps.v_cache.clone()
        for _ in range(5):
            api.copy_blocks([ck], [cv], ps.copy_pairs)
        torch.cuda.synchronize()
        cs = torch.cuda.Event(enable_timing=True)
        ce = torch.cuda.Event(enable_timing=True)
        reps = 200
        cs.record(stream)
        for _ in range(reps):
            api.copy_blocks([ck], [cv], ps.copy_pairs)
        ce.record(stream)
        torch.cuda.synchronize()
        copy_us = 1e3 * cs.elapsed_time(ce) / reps
        copy_b = metrics.copy_bytes(ps.copy_pairs.shape[0], 1, ps.num_kv_heads, ps.block_size, ps.head_dim, 2)
        rows["a7_copy_blocks_us"] = copy_us
        rows["a7_copy_blocks_gbs"] = copy_b / (copy_us * 1e-6) / 1e9
        rows["a7_copy_blocks_pairs"] = int(ps.copy_pairs.shape[0])
        del ps, ck, cv

    # ---- CPU oracle baseline (rank 0, one GPU only) ------------------------
    cpu = None
    if cpu_w is not None:
        cpu = cpu_baseline(cpu_w, args.cpu_seconds)

    if rank != 0:
        return
    peaks, peak_kind = measured_peaks()
    peak = float(peaks.get("hbm_gbs", 6800.0))
    bytes_step = decode_b + write_b
    achieved = decode_b / (decode_ms * 1e-3) / 1e9
    traffic = profiled_traffic()
    line = {
        "metric": METRIC,
        "value": world * bytes_step / (step_ms * 1e-3) / 1e9,
        "unit": "GB/s",
        "n_gpus": world,
        "steps": k,
        "warmup": args.warmup,
        "ms_per_step": step_ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"{WORKLOAD}: {w.num_seqs} seqs, 32 query / 8 KV heads, d 128, bf16 K/V, block 16, "
                               f"lognormal ctx (median 1024, [16, 8192]), shuffled blocks",
                   "parallelism": f"replicas x{world}", "l2": "inputs larger than L2 (1.8 GB of KV per step)",
                   "algorithmic_bytes_per_step": bytes_step, "sum_context_tokens": int(w.context_lens.sum())},
        "seq_decode_steps_per_s": world * w.num_seqs / (step_ms * 1e-3),
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "peak_source": f"{peak_kind} hbm_gbs",
                     "kernel": f"pa_decode ({'CUDA-core' if args.decode_kernel == 'simt' else 'tensor-core'} "
                               f"decode kernel + planning + reduce kernels), CUDA events per call"},
        "rows": rows,
        "e2e": None if e2e_ms is None else {
            "value": world * bytes_step / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms},
        "gpu_launches": launches,
        "gpu_launches_e2e": launches_e2e,
        "clocks": clocks,
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    if args.decode_kernel == "simt":
        os.environ["PA_DECODE_KERNEL"] = "simt"
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
        run_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()


if __name__ == "__main__":
    main()
