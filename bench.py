#!/usr/bin/env python
"""Benchmark of the paged-KV decode step on GB300.

Workload: the continuous-batching mix on the Llama-3-8B attention shape
(32 q heads, 8 kv heads, head_dim 128, bf16, block_size 16), batch 256,
log-normal context lengths (median 1024, sigma 1, clipped to [16, 32768]),
half of the batch sharing a 2048-token prefix with copy-on-write of the last
partial block, shuffled block pool; one appended token and one query per
sequence.  Synthetic data (seeded, see paged_kv_cache_23_gb300.workloads).

One step = copy-on-write block copies + slot mapping + KV append + paged
attention, for one layer, all in libpkv's kernels.  The K/V the step reads
(~1.2 GB unique) is far larger than L2 (126 MB), so no L2 flush is needed
between steps.

Prints ONE JSON line (rank 0).  ``--impl reference`` times the CPU fp64
oracle (the only reference this method has) on the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attention KV GB/s (% of GB300 HBM peak); seq-steps/s at batch 256"
WORKLOAD = "continuous-batching mix, Llama-3-8B attention shape: batch 256, 32 q / 8 kv heads, head_dim 128, " \
           "bf16 KV, block_size 16, log-normal ctx (median 1024, sigma 1, clip [16, 32768]), 50% share a " \
           "2048-token prefix (CoW), q_len 1, 1 appended token/seq"
KERNEL_SOURCES = ["paged_kv_cache_23_gb300/csrc/pkv_attention.cuh",
                  "paged_kv_cache_23_gb300/csrc/pkv_attention_host.cu",
                  "paged_kv_cache_23_gb300/csrc/pkv_common.cuh"]


def kernel_hash() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def load_traffic():
    """DRAM bytes per attention launch from the committed ncu summary, if it
    was taken on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "attention_mix_b256_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        if d.get("kernel_hash") == kernel_hash():
            return float(d["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = device_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return

        def read():
            for line in self.proc.stdout:
                self.rows.append([x.strip() for x in line.split(",")])

        self.thread = threading.Thread(target=read, daemon=True)
        self.thread.start()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return ws, rank, local


def aggregate_max(value: float, world_size: int, device=None) -> float:
    """Max over ranks (the slowest rank sets the job time)."""
    if world_size <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_sum(value: float, world_size: int, device=None) -> float:
    if world_size <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def make_workload(seed: int):
    from paged_kv_cache_23_gb300 import workloads as wl
    return wl.mix(B=256, median=1024, sigma=1.0, clip=(16, 32768), share=0.5, prefix=2048, seed=seed)


def oracle_step_time(w, reps: int = 1):
    """Run the oracle's full step on the host: copy, slots, append, attention."""
    import oracle
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        k = w.k_cache.copy()
        v = w.v_cache.copy()
        oracle.copy_blocks(k, v, w.cow)
        slots, _ = oracle.slot_mapping(w.block_tables, w.seq_lens, w.append_lens, w.block_size, w.num_blocks)
        oracle.kv_append(k, v, w.k_new, w.v_new, slots)
        oracle.attention(w.q, k, v, w.block_tables, w.seq_lens, w.q_lens, w.scale)
        times.append(time.perf_counter() - t0)
    return times


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    from paged_kv_cache_23_gb300 import accounting
    import oracle
    w = make_workload(0)
    b = accounting.step_bytes(w)
    oracle.build()
    # each step: the whole batch (256 sequences); warm-up steps untimed
    oracle_step_time(w, max(0, args.warmup))
    t = oracle_step_time(w, args.steps)
    mean = sum(t) / len(t)
    value = b["step_unique"] / mean / 1e9
    cores = oracle.num_threads()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": 256, "seq_len": "log-normal median 1024",
                       "parallelism": "cpu oracle, rank 0 only", "l2": "n/a (host)"},
            "seq_steps_per_s": 256 / mean,
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": "the whole batch-256 step per step (fp64 C oracle, OpenMP)"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_gpu(args):
    import torch
    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the GPU arm needs a GB300)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    import paged_kv_cache_23_gb300 as pkv
    from paged_kv_cache_23_gb300 import accounting
    from paged_kv_cache_23_gb300.runner import DeviceStep

    w = make_workload(rank)        # weak scaling: each rank owns its own batch of 256 sequences
    b = accounting.step_bytes(w)
    ds = DeviceStep(w, device=device, max_seq_len=32768, partition_tokens=args.partition, flags=args.flags)
    stream = torch.cuda.current_stream(device)

    # parity spot check on this very run: a few sequences against the oracle
    parity = None
    if rank == 0 and not args.no_check:
        parity = spot_check(w, ds, device)
        ds.reset_cache()

    def step():
        ds.cache_ops(stream)
        ds.attention(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()

    # timed region: K steps, per-step attention events on the launching stream
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for i in range(args.steps):
        ds.cache_ops(stream)
        ev[i][0].record(stream)
        ds.attention(stream)
        ev[i][1].record(stream)
    stop.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    total_ms = start.elapsed_time(stop)
    attn_ms = [a.elapsed_time(z) for a, z in ev]
    ms_step = aggregate_max(total_ms, ws, device) / args.steps
    st = int(ds.status.item())
    chosen_P = int(ds.workspace[8:12].view(torch.int32).item())  # partition length the planning kernel used

    # end to end through the public API: pinned host inputs -> device, step, result -> host
    e2e = end_to_end(ds, w, args, stream, device, ws)

    seqs_all = aggregate_sum(w.num_seqs, ws, device)
    bytes_all = aggregate_sum(b["step_unique"], ws, device)
    value = bytes_all / (ms_step / 1e3) / 1e9
    peak, peak_kind = load_peaks()
    attn_avg = sum(attn_ms) / len(attn_ms)
    achieved = b["attention_unique"] / (attn_avg / 1e3) / 1e9
    if rank != 0:
        return 0
    line = {"metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": 256 * ws, "seq_len": "log-normal median 1024",
                       "parallelism": f"replicas x{ws} (independent batches)" if ws > 1 else "single GPU",
                       "l2": "inputs larger than L2 (~1.2 GB unique K/V per step vs 126 MB L2); no flush",
                       "partition_tokens": ds.partition_tokens or f"auto ({chosen_P})", "flags": ds.flags},
            "seq_steps_per_s": seqs_all / (ms_step / 1e3),
            "kv_bytes_per_step": {"unique": b["kv_unique"], "logical": b["kv_logical"],
                                  "step_unique": b["step_unique"]},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": load_traffic(),
                         "kernel": "pkv_paged_attention_decode (plan + attention kernels)",
                         "peak_kind": peak_kind, "attention_ms": attn_avg,
                         "frac_of_nominal_8tbs": achieved / 8000.0},
            "clocks": clocks, "e2e": e2e, "gpu_launches": ds.launches_per_step() * args.steps, "status": st, "parity": parity}
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(w, b)
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def spot_check(w, ds, device):
    """Sampled sequences of this run's output against the oracle."""
    import torch
    import oracle
    from paged_kv_cache_23_gb300 import workloads as wl
    from paged_kv_cache_23_gb300.runner import bf16_to_bits
    ds.step()
    torch.cuda.synchronize()
    k = w.k_cache.copy()
    v = w.v_cache.copy()
    oracle.copy_blocks(k, v, w.cow)
    slots, _ = oracle.slot_mapping(w.block_tables, w.seq_lens, w.append_lens, w.block_size, w.num_blocks)
    oracle.kv_append(k, v, w.k_new, w.v_new, slots)
    pick = np.linspace(0, w.num_seqs - 1, 8).astype(int)
    ref, _ = oracle.attention(w.q[pick], k, v, w.block_tables[pick], w.seq_lens[pick], w.q_lens[pick], w.scale)
    got = wl.bf16_bits_to_f32(bf16_to_bits(ds.out)[pick]).astype(np.float64)
    err = np.abs(got - ref)
    ok = bool(np.all(err <= 1e-2 + 1e-2 * np.abs(ref)))
    return {"sequences": pick.tolist(), "max_abs_err": float(err.max()), "within_tol": ok,
            "status": int(ds.status.item())}


def end_to_end(ds, w, args, stream, device, ws):
    """The step through the public API from pinned host memory: one upload
    of every per-step input, the step, and the output read back."""
    import torch
    host = ds.pinned_inputs()
    out_host = torch.empty(ds.out.shape, dtype=ds.out.dtype, pin_memory=True)
    h2d = host.numel()
    d2h = out_host.numel() * out_host.element_size()
    steps = max(1, args.steps // 2)

    def one():
        ds.upload(host, stream)
        ds.cache_ops(stream)
        ds.attention(stream)
        out_host.copy_(ds.out, non_blocking=True)

    for _ in range(2):
        one()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    z = torch.cuda.Event(enable_timing=True)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(steps):
        one()
    z.record(stream)
    torch.cuda.synchronize()
    ms = aggregate_max(a.elapsed_time(z), ws, device) / steps
    from paged_kv_cache_23_gb300 import accounting
    b = accounting.step_bytes(w)
    bytes_all = aggregate_sum(b["step_unique"], ws, device)
    return {"value": bytes_all / (ms / 1e3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": ms}


def cpu_baseline(w, b):
    import oracle
    oracle.build()
    t = oracle_step_time(w, 2)
    best = min(t)
    return {"value": b["step_unique"] / best / 1e9, "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": "the full batch-256 step (copy, slots, append, fp64 attention), best of 2",
            "seq_steps_per_s": w.num_seqs / best}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--partition", type=int, default=0)
    ap.add_argument("--flags", type=int, default=0)
    ap.add_argument("--no-check", action="store_true")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
