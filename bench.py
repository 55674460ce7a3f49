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


# --workload: the headline mix (default) and the other attention workloads of
# the path; "sample" is the stochastic acceptance kernel alone.
SHAPE = "Llama-3-8B attention shape: 32 q / 8 kv heads, head_dim 128, bf16 KV, block_size 16"
WORKLOADS = {
    "mix": dict(desc=WORKLOAD, batch=256, seq="log-normal median 1024", max_seq_len=32768),
    "decode": dict(desc="8B decode, " + SHAPE + ": batch 64, seq_len ~ U[512, 4096], q_len 1, 1 appended "
                   "token/seq", batch=64, seq="U[512, 4096]", max_seq_len=None),
    "spec": dict(desc="speculative verify, " + SHAPE + ": batch 32, seq_len ~ U[2048, 8192], q_len 5 causal, "
                 "greedy acceptance over logits [32, 6, 128256] fp32", batch=32, seq="U[2048, 8192]",
                 max_seq_len=None),
    "spec6": dict(desc="speculative verify with q_len = k + 1, " + SHAPE + ": batch 32, seq_len ~ U[2048, 8192], "
                  "q_len 6 causal (last accepted token + 5 drafts), greedy acceptance over logits [32, 6, 128256] "
                  "fp32", batch=32, seq="U[2048, 8192]", max_seq_len=None),
    "long": dict(desc="long context + chunk, " + SHAPE + ": 8 decodes of 131072 tokens + one 512-query chunk "
                 "over 8192 + 512, in one call, split-KV partitions of 4096 tokens", batch=9,
                 seq="131072 (x8) and 8704", max_seq_len=None, partition=4096),
    "mix_fp8": dict(desc="continuous-batching mix over an FP8 (e4m3) KV cache with per-kv-head scales, "
                    + SHAPE + ": batch 256, log-normal ctx (median 1024, sigma 1, clip [16, 32768]), 50% share a "
                    "2048-token prefix (CoW), q_len 1, 1 appended token/seq", batch=256,
                    seq="log-normal median 1024", max_seq_len=32768, fp8=True),
    "decode_fp8": dict(desc="8B decode over an FP8 (e4m3) KV cache, " + SHAPE + ": batch 64, seq_len ~ U[512, 4096], "
                       "q_len 1", batch=64, seq="U[512, 4096]", max_seq_len=None, fp8=True),
    "mix_fp8b": dict(desc="continuous-batching mix over an FP8 (e4m3) KV cache with a scale per (block, kv head) tile "
                     "set when the block is opened, " + SHAPE + ": batch 256, log-normal ctx (median 1024, sigma 1, "
                     "clip [16, 32768]), 50% share a 2048-token prefix (CoW), q_len 1, 1 appended token/seq",
                     batch=256, seq="log-normal median 1024", max_seq_len=32768, fp8=True, fmt=0, per_block=True),
    "mix_e5m2": dict(desc="continuous-batching mix over an FP8 (e5m2) KV cache with a scale per (block, kv head) tile "
                     "set when the block is opened, " + SHAPE + ": batch 256, log-normal ctx (median 1024, sigma 1, "
                     "clip [16, 32768]), 50% share a 2048-token prefix (CoW), q_len 1, 1 appended token/seq",
                     batch=256, seq="log-normal median 1024", max_seq_len=32768, fp8=True, fmt=1, per_block=True),
    "prefix": dict(desc="prefix-cache block lookup: batch 256 prompts, log-normal lengths (median 1024, sigma 1, "
                   "clip [16, 32768]), half start with one 2048-token system prompt already cached; block_size 16; "
                   "chained 128-bit block hashes of every full block + batched table lookup", batch=256,
                   seq="log-normal median 1024", max_seq_len=None),
    "sample": dict(desc="stochastic speculative acceptance (modified rejection sampling): batch 32, k 5, "
                   "vocab 128256, p/q fp32 softmax rows, drafts drawn from q", batch=32, seq="n/a",
                   max_seq_len=None),
}


def make_workload(seed: int, name: str = "mix", chunk: int = 512):
    from paged_kv_cache_23_gb300 import workloads as wl
    if name in ("mix", "mix_fp8", "mix_fp8b", "mix_e5m2"):
        return wl.mix(B=256, median=1024, sigma=1.0, clip=(16, 32768), share=0.5, prefix=2048, seed=seed)
    if name == "decode_fp8":
        return wl.decode(64, 512, 4096, seed)
    if name == "decode":
        return wl.decode(64, 512, 4096, seed)
    if name == "spec":
        return wl.spec(32, 2048, 8192, 5, 128256, 0.7, seed)
    if name == "spec6":
        return wl.spec(32, 2048, 8192, 5, 128256, 0.7, seed, q_len=6)
    if name == "long":
        return wl.long_context(8, 131072, chunk, 8192, 4096, seed)
    if name == "sample":
        return wl.spec_sample(B=32, k=5, vocab=128256, seed=seed)
    if name == "prefix":
        return wl.prompts(B=256, seed=seed)
    raise ValueError(name)


def step_bytes_of(w, fp8: bool = False, block_scales: bool = False):
    """Unique bytes of one step: the attention step, plus the logits scan of
    greedy acceptance when the workload carries logits."""
    from paged_kv_cache_23_gb300 import accounting
    b = accounting.step_bytes(w, kv_bytes=1 if fp8 else 2, block_scales=block_scales)
    if w.logits is not None:
        b["accept"] = accounting.accept_greedy_bytes(w)
        b["step_unique"] += b["accept"]
    return b


def _oracle_cache(w, pools=None):
    """The oracle's cache after the step's copy-on-write and append."""
    import oracle
    if pools is None:
        k = w.k_cache.copy()
        v = w.v_cache.copy()
        oracle.copy_blocks(k, v, w.cow)
    else:
        k = pools.k_cache.copy()
        v = pools.v_cache.copy()
        ks, vs = pools.k_scale.copy(), pools.v_scale.copy()
        oracle.copy_blocks_fp8(k, v, ks, vs, w.cow, per_block=pools.per_block)
    slots, _ = oracle.slot_mapping(w.block_tables, w.seq_lens, w.append_lens, w.block_size, w.num_blocks)
    if pools is None:
        oracle.kv_append(k, v, w.k_new, w.v_new, slots)
        return k, v
    oracle.kv_append_fp8_ex(k, v, w.k_new, w.v_new, slots, ks, vs, pools.fmt, pools.per_block)
    return k, v, ks, vs


def _oracle_attention(w, kv, pools):
    import oracle
    if pools is None:
        k, v = kv
        return oracle.attention(w.q, k, v, w.block_tables, w.seq_lens, w.q_lens, w.scale)
    k, v, ks, vs = kv
    return oracle.attention_fp8_ex(w.q, k, v, ks, vs, w.block_tables, w.seq_lens, w.q_lens, w.scale, pools.fmt,
                                   pools.per_block)


def oracle_step_time(w, reps: int = 1, pools=None):
    """Run the oracle's full step on the host: copy, slots, append, attention."""
    import oracle
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        _oracle_attention(w, _oracle_cache(w, pools), pools)
        if w.logits is not None:
            oracle.spec_accept_greedy(w.logits, w.draft)
        times.append(time.perf_counter() - t0)
    return times


def oracle_sample_time(x, reps: int = 1):
    import oracle
    times = []
    for _ in range(reps):
        t0 = time.perf_counter()
        oracle.spec_accept_sample(x.p, x.q, x.draft, x.r, x.s)
        times.append(time.perf_counter() - t0)
    return times


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    from paged_kv_cache_23_gb300 import accounting
    spec = WORKLOADS[args.workload]
    w = make_workload(0, args.workload, args.chunk)
    oracle.build()
    if args.workload == "prefix":
        maxb = w.tokens.shape[1] // PREFIX_BS
        h = oracle.prefix_hash(w.tokens, w.lens, PREFIX_BS, maxb)
        sharer = int(w.meta["sharers"][np.argmax(w.lens[w.meta["sharers"]])])
        nsys = min(int(w.lens[sharer]), w.meta["prefix"]) // PREFIX_BS
        keys = {(int(h[sharer, j, 0]), int(h[sharer, j, 1])): j for j in range(nsys)}
        _, n, _ = _prefix_oracle_step(w, keys)
        nbytes = prefix_bytes(w, int(n.sum()))
        t = []
        for _ in range(max(0, args.warmup) + args.steps):
            t0 = time.perf_counter()
            _prefix_oracle_step(w, keys)
            t.append(time.perf_counter() - t0)
        t = t[max(0, args.warmup):]
        sample = "the whole batch of 256 prompts per step (C hash + Python dict lookup)"
    elif args.workload == "sample":
        acc, _, _ = oracle.spec_accept_sample(w.p, w.q, w.draft, w.r, w.s)
        nbytes = accounting.accept_sample_bytes(w, acc)
        oracle_sample_time(w, max(0, args.warmup))
        t = oracle_sample_time(w, args.steps)
        sample = "the whole batch of 32 sequences per step (C oracle)"
    else:
        from paged_kv_cache_23_gb300 import workloads as wl
        pools = wl.fp8_pools(w, 0, spec.get("fmt", 0), spec.get("per_block", False)) if spec.get("fp8") else None
        L = max(1, args.layers)
        nbytes = step_bytes_of(w, pools is not None, bool(spec.get("per_block")))["step_unique"] * L
        # each step: the whole batch (once per layer); warm-up steps untimed
        oracle_step_time(w, max(0, args.warmup), pools)
        t1 = oracle_step_time(w, args.steps * L, pools)
        t = [sum(t1[i * L:(i + 1) * L]) for i in range(args.steps)]
        sample = f"the whole batch-{spec['batch']} step per step" + (f", {L} layers" if L > 1 else "") + \
                 " (fp64 C oracle, OpenMP)"
    mean = sum(t) / len(t)
    value = nbytes / mean / 1e9
    cores = oracle.num_threads()
    line = {"impl": "reference", "metric": metric_of(args.workload), "value": value, "unit": "GB/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(args, spec, spec["batch"]),
            "parallelism": "cpu oracle, rank 0 only", "l2": "n/a (host)",
            "seq_steps_per_s": spec["batch"] / mean,
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def config_of(args, spec, batch):
    """The workload's config, printed identically by both arms (the GPU arm's
    partition length actually used and its L2 policy are reported outside it)."""
    cfg = {"workload": spec["desc"], "global_batch": batch, "seq_len": spec["seq"]}
    if args.workload not in ("prefix", "sample"):
        cfg["partition_tokens"] = args.partition or spec.get("partition", 0) or "auto"
        cfg["flags"] = args.flags
        if args.workload == "long" and args.chunk != 512:
            cfg["chunk_queries"] = args.chunk
        if args.layers > 1:
            cfg["layers"] = args.layers
    return cfg


def metric_of(name: str) -> str:
    if name == "mix":
        return METRIC
    if name == "sample":
        return "stochastic speculative acceptance GB/s (% of GB300 HBM peak); sequences/s"
    if name == "prefix":
        return "prefix-cache hash + lookup GB/s (% of GB300 HBM peak); prompts/s"
    return f"paged attention KV GB/s (% of GB300 HBM peak); seq-steps/s, {name} workload"


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

    spec = WORKLOADS[args.workload]
    w = make_workload(rank, args.workload, args.chunk)   # weak scaling: each rank owns its own batch
    from paged_kv_cache_23_gb300 import workloads as wl
    pools = wl.fp8_pools(w, rank, spec.get("fmt", 0), spec.get("per_block", False)) if spec.get("fp8") else None
    b = step_bytes_of(w, pools is not None, bool(spec.get("per_block")))
    # the workload's own partition length where its definition fixes one (--partition overrides)
    part = args.partition or spec.get("partition", 0)
    ds = DeviceStep(w, device=device, max_seq_len=spec["max_seq_len"], partition_tokens=part,
                    flags=args.flags, fp8=pools)
    stream = torch.cuda.current_stream(device)

    # parity on this very run: every query row against the oracle
    parity = None
    if rank == 0 and not args.no_check:
        parity = parity_check(w, ds, device, pools)
        ds.reset_cache()
    if args.layers > 1:
        return run_layers(args, w, ds, b, pools, spec, stream, device, ws, rank, local, parity)

    # the plan reads only the lengths: in a step that copies blocks on write
    # it runs on a side stream while the cache ops run, and the attention run
    # waits for it; otherwise the step runs in stream order
    # (DeviceStep.plan_beside_cache_ops)
    plan_stream = torch.cuda.Stream(device)

    def step():
        ds.step(stream, plan_stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()

    # timed region: K whole steps back to back (no events between the kernels
    # of a step, so programmatic launch overlaps them as in real use)
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
        step()
    stop.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    total_ms = start.elapsed_time(stop)
    # roofline of the dominant kernel: the attention run (attention + combine
    # kernels, pkv_paged_attention_run) over this step's plan, bracketed by
    # CUDA events on its stream, one run after another over the same
    # (already appended) cache -- what every layer of a step repeats
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    ds.plan(stream)
    torch.cuda.synchronize()
    for i in range(args.steps):
        ev[i][0].record(stream)
        ds.run(stream=stream)
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    attn_ms = [a.elapsed_time(z) for a, z in ev]
    # the whole call (plan + run) as well, for reference
    evc = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for i in range(args.steps):
        evc[i][0].record(stream)
        ds.attention(stream)
        evc[i][1].record(stream)
    torch.cuda.synchronize()
    call_ms = sum(a.elapsed_time(z) for a, z in evc) / args.steps
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
    line = {"metric": metric_of(args.workload), "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": fp8_dtype(pools),
            "data": "synthetic",
            "config": config_of(args, spec, spec["batch"] * ws),
            "parallelism": f"replicas x{ws} (independent batches)" if ws > 1 else "single GPU",
            "l2": f"inputs larger than L2 ({b['kv_unique'] / 1e9:.2f} GB unique K/V per step vs 126 MB L2); no flush",
            "partition_tokens_used": chosen_P,
            "seq_steps_per_s": seqs_all / (ms_step / 1e3),
            "seq_steps_per_s_attention": seqs_all / (attn_avg / 1e3),
            "kv_bytes_per_step": {"unique": b["kv_unique"], "logical": b["kv_logical"],
                                  "step_unique": b["step_unique"]},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": load_traffic() if args.workload == "mix" else None,
                         "kernel": "pkv_paged_attention_run (attention + combine kernels; the plan is made once "
                                   "per step, " + ("on a side stream beside the cache ops)" if ds.plan_beside_cache_ops()
                                                   else "in stream order after the append)"),
                         "peak_kind": peak_kind, "attention_ms": attn_avg, "call_ms_with_plan": call_ms,
                         "frac_of_nominal_8tbs": achieved / 8000.0},
            "clocks": clocks, "e2e": e2e, "gpu_launches": ds.launches_per_step() * args.steps, "status": st, "parity": parity}
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(w, b, pools)
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def parity_check(w, ds, device, pools=None):
    """This run's output against the oracle: every query row of every
    sequence, element by element; the caches bit for bit; the acceptance
    integers exactly."""
    import torch
    import oracle
    from paged_kv_cache_23_gb300 import workloads as wl
    from paged_kv_cache_23_gb300.runner import bf16_to_bits
    # the step as the timed region runs it (the plan on a side stream where
    # the step copies blocks on write)
    ds.step(torch.cuda.current_stream(device), torch.cuda.Stream(device))
    torch.cuda.synchronize()
    kv = _oracle_cache(w, pools)
    ref, _ = _oracle_attention(w, kv, pools)
    got = wl.bf16_bits_to_f32(bf16_to_bits(ds.out)).astype(np.float64)
    err = np.abs(got - ref)
    ok = bool(np.isfinite(got).all() and np.all(err <= 1e-2 + 1e-2 * np.abs(ref)))
    if pools is None:
        caches = bool(np.array_equal(bf16_to_bits(ds.k_cache), kv[0]) and np.array_equal(bf16_to_bits(ds.v_cache),
                                                                                          kv[1]))
    else:
        caches = bool(np.array_equal(ds.k_cache.cpu().numpy(), kv[0]) and np.array_equal(ds.v_cache.cpu().numpy(),
                                                                                          kv[1])
                      and np.array_equal(ds.k_scale.cpu().numpy(), kv[2])
                      and np.array_equal(ds.v_scale.cpu().numpy(), kv[3]))
    res = {"sequences": f"all {w.num_seqs}", "rows": int(w.total_q), "max_abs_err": float(err.max()),
           "within_tol": ok, "caches_bit_exact": caches, "status": int(ds.status.item())}
    if w.logits is not None:
        acc, nxt, am = oracle.spec_accept_greedy(w.logits, w.draft)
        res["acceptance_bit_exact"] = bool(np.array_equal(ds.accepted.cpu().numpy(), acc)
                                           and np.array_equal(ds.next_token.cpu().numpy(), nxt)
                                           and np.array_equal(ds.argmax.cpu().numpy(), am))
    return res


def fp8_dtype(pools):
    if pools is None:
        return "bf16"
    return ("e5m2" if pools.fmt else "e4m3") + " KV (scale per " + ("block and kv head" if pools.per_block
                                                                    else "kv head") + "), bf16 q/out, f16 MMA"


def run_layers(args, w, ds, b, pools, spec, stream, device, ws, rank, local, parity):
    """A decode step over `layers` layers of the same batch: one plan, then per
    layer its copy-on-write copies, its append and one attention run over its
    own pools (the step's pools copied once per layer), queries and output."""
    import torch
    from paged_kv_cache_23_gb300 import copy_blocks, copy_blocks_fp8, kv_append_fp8, kv_append_paged
    from paged_kv_cache_23_gb300.runner import bf16_to_bits
    L = args.layers
    if pools is not None and (pools.fmt or pools.per_block):
        raise SystemExit("bench.py --layers: bf16 pools or e4m3 pools with per-head scales")
    ds.step()                                   # layer 0's pools hold the appended step
    torch.cuda.synchronize()
    lay = [dict(k=ds.k_cache, v=ds.v_cache, q=ds.q, out=ds.out)]
    for _ in range(1, L):
        lay.append(dict(k=ds.k_cache.clone(), v=ds.v_cache.clone(), q=ds.q.clone(), out=torch.empty_like(ds.out)))
    fp8 = pools is not None

    def layer_ops(x):
        if ds.cow.numel():
            (copy_blocks_fp8 if fp8 else copy_blocks)(x["k"], x["v"], ds.cow, status=ds.status, stream=stream)
        if ds.n_slots:
            if fp8:
                kv_append_fp8(x["k"], x["v"], ds.k_new, ds.v_new, ds.slots, ds.k_scale, ds.v_scale,
                              status=ds.status, stream=stream)
            else:
                kv_append_paged(x["k"], x["v"], ds.k_new, ds.v_new, ds.block_tables, ds.seq_lens, ds.append_lens,
                                ds.slots, status=ds.status, stream=stream)
        ds.run(out=x["out"], q=x["q"], k_cache=x["k"], v_cache=x["v"], stream=stream)

    def step():
        ds.plan(stream)
        for x in lay:
            layer_ops(x)
        ds.accept(stream)

    for _ in range(max(3, args.warmup)):
        step()
    torch.cuda.synchronize()
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if ws > 1:
        torch.distributed.barrier()
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    start.record(stream)
    for _ in range(args.steps):
        step()
    stop.record(stream)
    torch.cuda.synchronize()
    if ws > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    ms_step = aggregate_max(start.elapsed_time(stop) / args.steps, ws, device)
    # the attention runs alone, one after another over the planned workspace
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(L)]
    runs = []
    for _ in range(max(1, args.steps // 10)):
        torch.cuda.synchronize()
        for i, x in enumerate(lay):
            ev[i][0].record(stream)
            ds.run(out=x["out"], q=x["q"], k_cache=x["k"], v_cache=x["v"], stream=stream)
            ev[i][1].record(stream)
        torch.cuda.synchronize()
        runs += [a.elapsed_time(z) for a, z in ev]
    run_ms = sum(runs) / len(runs)
    st = int(ds.status.item())
    # every layer's output equals layer 0's bit for bit (the same data in other buffers)
    o0 = bf16_to_bits(lay[0]["out"])
    same = all(np.array_equal(bf16_to_bits(x["out"]), o0) for x in lay[1:])
    if parity is not None:
        parity = dict(parity, layers_bit_identical=bool(same))
    bytes_step = b["step_unique"] * L
    value = aggregate_sum(bytes_step, ws, device) / (ms_step / 1e3) / 1e9
    peak, peak_kind = load_peaks()
    achieved = b["attention_unique"] / (run_ms / 1e3) / 1e9
    if rank != 0:
        return 0
    line = {"metric": metric_of(args.workload) + f", {L}-layer step (one plan)", "value": value, "unit": "GB/s",
            "n_gpus": ws, "steps": args.steps, "warmup": max(3, args.warmup), "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": fp8_dtype(pools), "data": "synthetic",
            "config": config_of(args, spec, spec["batch"] * ws),
            "parallelism": f"replicas x{ws} (independent batches)" if ws > 1 else "single GPU",
            "l2": "inputs larger than L2; no flush",
            "partition_tokens_used": int(ds.workspace[8:12].view(torch.int32).item()),
            "ms_per_layer": ms_step / L, "attention_run_ms": run_ms,
            "seq_steps_per_s_per_layer": w.num_seqs * ws * L / (ms_step / 1e3),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                         "traffic": None, "kernel": "pkv_paged_attention_run (attention + combine kernels)",
                         "peak_kind": peak_kind},
            "clocks": clocks, "gpu_launches": args.steps * (1 + L * (2 + (1 if ds.cow.numel() else 0)
                                                                     + (1 if ds.n_slots else 0))
                                                           + (2 if ds.spec else 0)),
            "status": st, "parity": parity}
    print(json.dumps(line), flush=True)
    return 0


def end_to_end(ds, w, args, stream, device, ws):
    """The step through the public API from pinned host memory: every step
    uploads all of its inputs (one host -> device copy of the input arena) and
    reads its output back (one device -> host copy), both inside the timed
    region.  As in a serving loop, the copies run on their own streams (the
    host -> device and device -> host copy engines) into double-buffered device
    inputs and outputs, so step n + 1's upload and step n's read-back overlap
    the kernels of step n; a buffer is reused only after the step two back has
    been read back."""
    import torch
    host = ds.pinned_inputs()
    arenas = [ds.arena, torch.empty_like(ds.arena)]
    views = [ds.arena_views(a) for a in arenas]
    outs = [ds.out, torch.empty_like(ds.out)]
    out_hosts = [torch.empty(ds.out.shape, dtype=ds.out.dtype, pin_memory=True) for _ in range(2)]
    h2d = host.numel()
    d2h = out_hosts[0].numel() * out_hosts[0].element_size()
    up_s, dn_s = torch.cuda.Stream(device), torch.cuda.Stream(device)
    plan_stream = torch.cuda.Stream(device)  # the step's streams as in the device-timed step
    up = [torch.cuda.Event() for _ in range(2)]
    done = [torch.cuda.Event() for _ in range(2)]
    free = [torch.cuda.Event() for _ in range(2)]
    for e in free:
        e.record(dn_s)
    steps = max(1, args.steps // 2)

    def one(n):
        i = n & 1
        up_s.wait_event(free[i])
        with torch.cuda.stream(up_s):
            arenas[i].copy_(host, non_blocking=True)
        up[i].record(up_s)
        stream.wait_event(up[i])
        ds.bind(views[i], outs[i])
        ds.step(stream, plan_stream)
        done[i].record(stream)
        dn_s.wait_event(done[i])
        with torch.cuda.stream(dn_s):
            out_hosts[i].copy_(outs[i], non_blocking=True)
        free[i].record(dn_s)

    for n in range(2):
        one(n)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    z = torch.cuda.Event(enable_timing=True)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    a.record(up_s)  # the first timed operation is an upload ...
    for n in range(steps):
        one(n)
    z.record(dn_s)  # ... the last a read-back, after every kernel of the last step
    torch.cuda.synchronize()
    ds.bind(views[0], outs[0])
    ms = aggregate_max(a.elapsed_time(z) / steps, ws, device)
    b = step_bytes_of(w, ds.fp8 is not None)  # the same bytes as the device-timed value
    bytes_all = aggregate_sum(b["step_unique"], ws, device)
    return {"value": bytes_all / (ms / 1e3) / 1e9, "unit": "GB/s", "h2d_bytes_per_step": int(h2d),
            "d2h_bytes_per_step": int(d2h), "ms_per_step": ms,
            "copies": "per step, on copy streams overlapping the previous step's kernels (double-buffered)"}


PREFIX_BS = 16
PREFIX_CAPACITY = 1 << 20


def prefix_bytes(x, nhit):
    """Algorithmic bytes of hash + lookup: the tokens of every full block (4 B),
    each block's key written and read back (16 B each), one 32-byte table
    entry read per probe, and per hit a ref-count update (8 B) and a
    block-table entry (4 B); plus lengths and hit counts."""
    nb = (x.lens // PREFIX_BS).astype(np.int64)
    blocks = int(nb.sum())
    return int(blocks * PREFIX_BS * 4 + blocks * (16 + 16 + 32) + int(nhit) * 12 + len(x.lens) * 8)


def _prefix_oracle_step(x, cache_keys):
    import oracle
    maxb = int(x.tokens.shape[1]) // PREFIX_BS
    h = oracle.prefix_hash(x.tokens, x.lens, PREFIX_BS, maxb)
    cache = oracle.PrefixCache()
    for k, blk in cache_keys.items():
        cache.d[k] = [blk, 1]
    bt = np.full((len(x.lens), maxb), -1, np.int32)
    n = cache.lookup(h, x.lens, PREFIX_BS, bt)
    return h, n, bt


def run_prefix(args):
    """Prefix-cache hash + lookup for a batch of 256 prompts."""
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
    spec = WORKLOADS["prefix"]
    x = make_workload(rank, "prefix")
    B, T = x.tokens.shape
    maxb = T // PREFIX_BS
    tok = torch.from_numpy(x.tokens).to(device)
    lens = torch.from_numpy(x.lens).to(device)
    hashes = torch.zeros((B, maxb, 2), dtype=torch.int64, device=device)
    bt = torch.full((B, maxb), -1, dtype=torch.int32, device=device)
    cached = torch.zeros(B, dtype=torch.int32, device=device)
    st = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    table = pkv.PrefixTable(PREFIX_CAPACITY, device=device)
    # the system prompt is cached: insert the full blocks of the longest sharer
    sharer = int(x.meta["sharers"][np.argmax(x.lens[x.meta["sharers"]])])
    pkv.prefix_hash(hashes, tok, lens, PREFIX_BS)
    nsys = min(int(x.lens[sharer]), x.meta["prefix"]) // PREFIX_BS
    ids = torch.arange(B * maxb, dtype=torch.int32, device=device).view(B, maxb) + 5000
    one = torch.zeros(B, dtype=torch.int32, device=device)
    cnt = torch.zeros(B, dtype=torch.int32, device=device)
    cnt[sharer] = nsys
    res = torch.zeros((B, maxb), dtype=torch.int32, device=device)
    pkv.prefix_insert(table, hashes, ids, one, cnt, res, status=st)
    torch.cuda.synchronize()
    keys = hashes[sharer, :nsys].cpu().numpy().view(np.uint64)
    cache_keys = {(int(k[0]), int(k[1])): 5000 + sharer * maxb + j for j, k in enumerate(keys)}
    flush_buf = torch.ones(64 << 20, dtype=torch.float32, device=device)
    flush_sink = torch.empty(1, dtype=torch.float32, device=device)

    def call():
        pkv.prefix_hash(hashes, tok, lens, PREFIX_BS, stream=stream)
        pkv.prefix_lookup(table, hashes, lens, PREFIX_BS, bt, cached, stream=stream)

    parity = None
    if rank == 0 and not args.no_check:
        call()
        torch.cuda.synchronize()
        h_ref, n_ref, bt_ref = _prefix_oracle_step(x, cache_keys)
        gh = hashes.cpu().numpy().view(np.uint64)
        full = np.arange(maxb)[None, :] < (x.lens // PREFIX_BS)[:, None]
        parity = {"hashes_bit_exact": bool(np.array_equal(gh[full], h_ref[full])),
                  "hits_exact": bool(np.array_equal(cached.cpu().numpy(), n_ref)),
                  "block_tables_exact": bool(np.array_equal(bt.cpu().numpy(), bt_ref)),
                  "hits": int(n_ref.sum())}
    for _ in range(max(3, args.warmup)):
        torch.sum(flush_buf, dim=0, keepdim=True, out=flush_sink)
        call()
    torch.cuda.synchronize()
    nhit = int(cached.sum().item())
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        torch.sum(flush_buf, dim=0, keepdim=True, out=flush_sink)
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = aggregate_max(sum(a.elapsed_time(z) for a, z in ev) / args.steps, ws, device)
    nbytes = prefix_bytes(x, nhit)
    value = aggregate_sum(nbytes, ws, device) / (ms / 1e3) / 1e9
    # latency floor: the same two kernels on one prompt of one full block
    # (launches, the grid-dependency waits and the dependent probe round trips)
    tok1, lens1 = tok[:1, :PREFIX_BS].contiguous(), lens[:1].clone().fill_(PREFIX_BS)
    h1 = torch.zeros((1, 1, 2), dtype=torch.int64, device=device)
    bt1 = torch.full((1, 1), -1, dtype=torch.int32, device=device)
    c1 = torch.zeros(1, dtype=torch.int32, device=device)

    def call1():
        pkv.prefix_hash(h1, tok1, lens1, PREFIX_BS, stream=stream)
        pkv.prefix_lookup(table, h1, lens1, PREFIX_BS, bt1, c1, stream=stream)

    floor_ms = latency_floor(call1, flush_buf, flush_sink, stream, args.steps)
    # end to end: the prompts' tokens and lengths come from pinned host memory
    htok = torch.from_numpy(x.tokens).pin_memory()
    hlen = torch.from_numpy(x.lens).pin_memory()
    hout = torch.empty(B, dtype=torch.int32).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        tok.copy_(htok, non_blocking=True)
        lens.copy_(hlen, non_blocking=True)
        call()
        hout.copy_(cached, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = aggregate_max(e0.elapsed_time(e1) / args.steps, ws, device)
    if rank != 0:
        return 0
    line = {"metric": metric_of("prefix"), "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "u64 hashes, i32 tokens", "data": "synthetic",
            "config": config_of(args, spec, B * ws),
            "parallelism": "single GPU" if ws == 1 else f"replicas x{ws}",
            "l2": "L2 flushed before every call by reading a 256 MB buffer", "table_capacity": PREFIX_CAPACITY,
            "prompts_per_s": B * ws / (ms / 1e3), "bytes_per_call": nbytes, "hits": nhit,
            "roofline": {"bound": "latency", "achieved": ms * 1e3, "peak": floor_ms * 1e3, "unit": "us per call",
                         "frac": floor_ms / ms, "traffic": None,
                         "kernel": "prefix_hash_kernel + prefix_lookup_kernel",
                         "peak_kind": "measured: the same two kernels on one prompt of one block (the chained "
                                      "digests and the dependent table probes, not HBM, bound the call)"},
            "clocks": clocks, "gpu_launches": 2 * args.steps, "status": int(st.item()), "parity": parity,
            "e2e": {"value": nbytes / (ms_e2e / 1e3) / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": int(htok.numel() * 4 + hlen.numel() * 4), "d2h_bytes_per_step": B * 4,
                    "ms_per_step": ms_e2e}}
    t0 = time.perf_counter()
    _prefix_oracle_step(x, cache_keys)
    t_cpu = time.perf_counter() - t0
    line["cpu_baseline"] = {"value": nbytes / t_cpu / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                            "sample": "the whole batch of 256 prompts (C hash + Python dict lookup), one pass"}
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def run_sample(args):
    """Stochastic speculative acceptance alone: batch 32, k 5, vocab 128256."""
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
    spec = WORKLOADS["sample"]
    x = make_workload(rank, "sample")
    B, k1, V = x.p.shape
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(device, dt)
    p, q, d, r, s = (t(x.p, torch.float32), t(x.q, torch.float32), t(x.draft, torch.int32), t(x.r, torch.float32),
                     t(x.s, torch.float32))
    acc = torch.empty(B, dtype=torch.int32, device=device)
    nxt = torch.empty(B, dtype=torch.int32, device=device)
    st = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    # the kernel reads only the rows the draws need (~30 MB of the 180 MB of p
    # and q), the same rows every call, so a read of a 256 MB buffer evicts
    # them from L2 before every call (a read leaves no dirty lines behind)
    flush_buf = torch.ones(64 << 20, dtype=torch.float32, device=device)
    flush_sink = torch.empty(1, dtype=torch.float32, device=device)

    class _Flush:
        @staticmethod
        def zero_():
            torch.sum(flush_buf, dim=0, keepdim=True, out=flush_sink)

    flush = _Flush()

    def call():
        pkv.spec_accept_sample(p, q, d, r, s, acc, nxt, status=st, stream=stream)

    parity = None
    if rank == 0 and not args.no_check:
        import oracle
        call()
        torch.cuda.synchronize()
        ra, rn, rs = oracle.spec_accept_sample(x.p, x.q, x.draft, x.r, x.s)
        parity = {"bit_exact": bool(np.array_equal(acc.cpu().numpy(), ra) and np.array_equal(nxt.cpu().numpy(), rn)),
                  "status": int(st.item()), "oracle_status": int(rs)}
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        call()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    time.sleep(0.3)
    if ws > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        flush.zero_()
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = [a.elapsed_time(z) for a, z in ev]
    ms_step = aggregate_max(sum(ms) / len(ms), ws, device)
    nbytes = accounting.accept_sample_bytes(x, acc.cpu().numpy())
    value = aggregate_sum(nbytes, ws, device) / (ms_step / 1e3) / 1e9
    # latency floor: the same kernel for one sequence, one draft, a 1024-token vocabulary
    V1 = 1024
    p1 = torch.full((1, 2, V1), 1.0 / V1, dtype=torch.float32, device=device)
    q1 = torch.full((1, 1, V1), 1.0 / V1, dtype=torch.float32, device=device)
    d1 = torch.zeros((1, 1), dtype=torch.int32, device=device)
    r1 = torch.full((1, 1), 0.5, dtype=torch.float32, device=device)
    s1 = torch.full((1,), 0.5, dtype=torch.float32, device=device)
    a1 = torch.empty(1, dtype=torch.int32, device=device)
    n1 = torch.empty(1, dtype=torch.int32, device=device)
    floor_ms = latency_floor(lambda: pkv.spec_accept_sample(p1, q1, d1, r1, s1, a1, n1, stream=stream),
                             flush_buf, flush_sink, stream, args.steps)
    # end to end: the uniforms and drafts of a round come from the host each step
    hr = torch.empty_like(r, device="cpu").pin_memory()
    hs = torch.empty_like(s, device="cpu").pin_memory()
    hd = torch.empty_like(d, device="cpu").pin_memory()
    hr.copy_(r.cpu())
    hs.copy_(s.cpu())
    hd.copy_(d.cpu())
    ho = torch.empty(2 * B, dtype=torch.int32).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(args.steps):
        r.copy_(hr, non_blocking=True)
        s.copy_(hs, non_blocking=True)
        d.copy_(hd, non_blocking=True)
        call()
        ho[:B].copy_(acc, non_blocking=True)
        ho[B:].copy_(nxt, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = aggregate_max(e0.elapsed_time(e1) / args.steps, ws, device)
    if rank != 0:
        return 0
    line = {"metric": metric_of("sample"), "value": value, "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
            "warmup": max(3, args.warmup), "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": config_of(args, spec, B * ws),
            "parallelism": "single GPU" if ws == 1 else f"replicas x{ws}",
            "l2": "L2 flushed before every call by reading a 256 MB buffer",
            "sequences_per_s": B * ws / (ms_step / 1e3), "bytes_per_call": nbytes,
            "roofline": {"bound": "latency", "achieved": ms_step * 1e3, "peak": floor_ms * 1e3,
                         "unit": "us per call", "frac": floor_ms / ms_step, "traffic": None,
                         "kernel": "spec_sample_kernel",
                         "peak_kind": "measured: the same kernel for one sequence, one draft, vocab 1024 (dependent "
                                      "rounds of loads and the cluster exchange, not HBM, bound the call)"},
            "clocks": clocks, "gpu_launches": args.steps, "status": int(st.item()), "parity": parity,
            "e2e": {"value": nbytes / (ms_e2e / 1e3) / 1e9, "unit": "GB/s",
                    "h2d_bytes_per_step": int(hr.numel() * 4 + hs.numel() * 4 + hd.numel() * 4),
                    "d2h_bytes_per_step": int(ho.numel() * 4), "ms_per_step": ms_e2e}}
    t_cpu = oracle_sample_time(x, 2)
    line["cpu_baseline"] = {"value": nbytes / min(t_cpu) / 1e9, "unit": "GB/s", "cores": 1, "kind": "oracle",
                            "sample": "the whole batch of 32 sequences (C oracle, one thread), best of 2"}
    print(json.dumps(line), flush=True)
    if ws > 1:
        torch.distributed.destroy_process_group()
    return 0


def latency_floor(call, flush_buf, flush_sink, stream, steps):
    """Mean event-timed duration of `call` (a minimal invocation) with L2
    flushed before each, in ms: the fixed cost of launching the kernels and
    their dependent memory round trips."""
    import torch
    for _ in range(3):
        call()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for i in range(steps):
        torch.sum(flush_buf, dim=0, keepdim=True, out=flush_sink)
        ev[i][0].record(stream)
        call()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(z) for a, z in ev) / steps


def cpu_baseline(w, b, pools=None):
    import oracle
    oracle.build()
    reps = 1 if int(w.seq_lens.max()) > 65536 else 2
    cores = oracle.num_threads()
    t = oracle_step_time(w, reps, pools)
    best = min(t)
    # the same step on one core, when that stays within about 30 s of CPU time
    one = None
    if best * cores <= 30.0:
        oracle.set_num_threads(1)
        try:
            t1 = min(oracle_step_time(w, 1, pools))
        finally:
            oracle.set_num_threads(cores)
        one = {"value": b["step_unique"] / t1 / 1e9, "cores": 1, "seq_steps_per_s": w.num_seqs / t1}
    return {"value": b["step_unique"] / best / 1e9, "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"the full batch-{w.num_seqs} step (copy, slots, append, fp64 attention"
                      f"{', greedy acceptance' if w.logits is not None else ''}), best of {reps}",
            "seq_steps_per_s": w.num_seqs / best,
            "one_core": one if one is not None else "not run: the one-core step would exceed 30 s"}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="pkv", choices=["pkv", "reference"])
    ap.add_argument("--partition", type=int, default=0)
    ap.add_argument("--flags", type=int, default=0)
    ap.add_argument("--workload", default="mix", choices=sorted(WORKLOADS),
                    help="mix (default, the headline), decode, spec, long, or sample (stochastic acceptance)")
    ap.add_argument("--no-check", action="store_true")
    ap.add_argument("--layers", type=int, default=1,
                    help="layers per step: one plan, then per layer copy + append + attention run")
    ap.add_argument("--chunk", type=int, default=512, help="queries of the long workload's prefill chunk")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "sample":
        return run_sample(args)
    if args.workload == "prefix":
        return run_prefix(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
