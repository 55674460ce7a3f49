"""One step of the paged-KV path on the GPU, through the C ABI.

A step over a workload (see ``workloads``) is: copy-on-write block copies,
slot mapping of the appended tokens, KV append, paged attention over the
whole batch, and -- when the workload carries target logits and drafts --
greedy speculative acceptance.  Everything runs in libpkv's kernels on one
CUDA stream; this module only owns the device buffers.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (PKV_ATTN_PLAN_FP8, attention_plan, attention_workspace_bytes, copy_blocks, copy_blocks_fp8,
               copy_blocks_fp8_ex, kv_append, kv_append_fp8, kv_append_fp8_ex, kv_append_paged,
               paged_attention_decode, paged_attention_decode_fp8, paged_attention_decode_fp8_ex,
               paged_attention_run, paged_attention_run_fp8, slot_mapping, spec_accept_greedy)


def to_device_bf16(bits: np.ndarray, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(torch.bfloat16)


def bf16_to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


class DeviceStep:
    """Device-resident inputs of one step, plus outputs and scratch."""

    def __init__(self, w, device="cuda", max_seq_len=None, partition_tokens=None, flags=0, fp8=None):
        """fp8: an FP8 pool set (workloads.Fp8Pools: e4m3 or e5m2, scales per
        kv head or per block) for the workload's structure; the step then
        appends with quantisation and attends over the FP8 pools."""
        self.w = w
        self.device = torch.device(device)
        dev = self.device
        self.fp8 = fp8
        if fp8 is None:
            self.k_cache = to_device_bf16(w.k_cache, dev)
            self.v_cache = to_device_bf16(w.v_cache, dev)
        else:
            self.k_cache = torch.from_numpy(fp8.k_cache).to(dev)
            self.v_cache = torch.from_numpy(fp8.v_cache).to(dev)
            self.k_scale = torch.from_numpy(fp8.k_scale).to(dev)
            self.v_scale = torch.from_numpy(fp8.v_scale).to(dev)
            # the e4m3 per-head pools take the original entry points, the
            # other modes the general ones
            self.fp8_ex = bool(fp8.fmt or fp8.per_block)
            self.fp8_mode = dict(kv_format=int(fp8.fmt), scale_mode=int(bool(fp8.per_block)))
        # the per-step inputs live in one device arena (256-byte aligned
        # slices), so a step's host -> device upload is a single copy
        parts = [("q", w.q, torch.bfloat16), ("k_new", w.k_new, torch.bfloat16),
                 ("v_new", w.v_new, torch.bfloat16), ("block_tables", w.block_tables, torch.int32),
                 ("seq_lens", w.seq_lens, torch.int32), ("q_lens", w.q_lens, torch.int32),
                 ("append_lens", w.append_lens, torch.int32),
                 ("cow", np.ascontiguousarray(w.cow, np.int32).reshape(-1, 2), torch.int32)]
        layout, off = [], 0
        for name, arr, dt in parts:
            nbytes = int(arr.nbytes)
            layout.append((name, off, nbytes, tuple(arr.shape), dt))
            off += (nbytes + 255) // 256 * 256
        self.arena_bytes = max(off, 256)
        host = torch.empty(self.arena_bytes, dtype=torch.uint8)
        hv = host.numpy()
        for (name, o, nbytes, shape, dt), (_, arr, _) in zip(layout, parts):
            hv[o:o + nbytes] = np.ascontiguousarray(arr).view(np.uint8).reshape(-1)
        self.arena = host.to(dev)
        self._layout = layout
        self._host_arena = host
        for name, o, nbytes, shape, dt in layout:
            setattr(self, name, self.arena[o:o + nbytes].view(dt).view(shape))
        self.n_slots = int(w.append_lens.sum())
        self.slots = torch.empty(max(self.n_slots, 1), dtype=torch.int64, device=dev)[: self.n_slots]
        self.out = torch.empty((w.total_q, w.n_q, w.head_dim), dtype=torch.bfloat16, device=dev)
        self.status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.max_seq_len = int(max_seq_len if max_seq_len is not None else max(1, int(w.seq_lens.max())))
        self.max_q_len = max(1, int(w.q_lens.max())) if w.num_seqs else 1  # host bound on every q_len
        self.partition_tokens = int(partition_tokens if partition_tokens is not None else w.partition_tokens)
        self.flags = int(flags)
        nbytes = attention_workspace_bytes(w.num_seqs, w.total_q, w.n_q, w.n_kv, w.head_dim, self.max_seq_len,
                                           self.partition_tokens)
        self.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        self.spec = w.logits is not None
        if self.spec:
            B, k1, V = w.logits.shape
            self.logits = torch.from_numpy(w.logits).to(dev)
            self.draft = torch.from_numpy(w.draft).to(dev)
            self.argmax = torch.empty((B, k1), dtype=torch.int32, device=dev)
            self.accepted = torch.empty(B, dtype=torch.int32, device=dev)
            self.next_token = torch.empty(B, dtype=torch.int32, device=dev)

    def launches_per_step(self) -> int:
        """Kernels one step() launches: copy_blocks (+ the scale copy with
        per-block FP8 scales), the fused slot mapping + append (slot mapping
        and append for FP8 pools, + the block-scale kernel with per-block
        scales), plan + attention + combine, and the two acceptance kernels."""
        pb = self.fp8 is not None and self.fp8.per_block
        n = (1 + (1 if pb else 0) if self.cow.numel() else 0)
        n += ((1 if self.fp8 is None else 2 + (1 if pb else 0)) if self.n_slots else 0)
        n += 3  # plan, attention and the combine kernel, launched on every call
        return n + (2 if self.spec else 0)

    def pinned_inputs(self) -> torch.Tensor:
        """The step's inputs as one pinned host buffer in the arena layout."""
        return self._host_arena.pin_memory()

    def arena_views(self, arena: torch.Tensor) -> dict:
        """The per-step input tensors as views of `arena` (a device buffer of
        arena_bytes in the same layout), for double-buffered inputs."""
        return {name: arena[o:o + nbytes].view(dt).view(shape) for name, o, nbytes, shape, dt in self._layout}

    def bind(self, views: dict, out: torch.Tensor | None = None):
        """Point the step's inputs (and optionally its output) at other buffers."""
        for name, t in views.items():
            setattr(self, name, t)
        if out is not None:
            self.out = out

    def upload(self, host: torch.Tensor, stream=None):
        """One host -> device copy of every per-step input (q, new K/V rows,
        block tables, lengths, copy-on-write pairs)."""
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        with torch.cuda.stream(s):
            self.arena.copy_(host, non_blocking=True)

    def reset_cache(self):
        """Restore the cache to the state before the step (for repeated steps)."""
        if self.fp8 is None:
            self.k_cache.copy_(to_device_bf16(self.w.k_cache, self.device))
            self.v_cache.copy_(to_device_bf16(self.w.v_cache, self.device))
        else:
            self.k_cache.copy_(torch.from_numpy(self.fp8.k_cache))
            self.v_cache.copy_(torch.from_numpy(self.fp8.v_cache))
            self.k_scale.copy_(torch.from_numpy(self.fp8.k_scale))
            self.v_scale.copy_(torch.from_numpy(self.fp8.v_scale))

    def cache_ops(self, stream=None):
        w = self.w
        if self.cow.numel():
            if self.fp8 is not None and self.fp8_ex:
                copy_blocks_fp8_ex(self.k_cache, self.v_cache, self.k_scale, self.v_scale, self.cow,
                                   scale_mode=self.fp8_mode["scale_mode"], status=self.status, stream=stream)
            else:
                (copy_blocks if self.fp8 is None else copy_blocks_fp8)(self.k_cache, self.v_cache, self.cow,
                                                                      status=self.status, stream=stream)
        if self.n_slots:
            if self.fp8 is not None and self.fp8_ex:
                slot_mapping(self.slots, self.block_tables, self.seq_lens, self.append_lens, w.block_size,
                             w.num_blocks, status=self.status, stream=stream)
                kv_append_fp8_ex(self.k_cache, self.v_cache, self.k_scale, self.v_scale, self.k_new, self.v_new,
                                 self.slots, **self.fp8_mode, status=self.status, stream=stream)
            elif self.fp8 is None:
                # slot mapping fused with the append (one launch)
                kv_append_paged(self.k_cache, self.v_cache, self.k_new, self.v_new, self.block_tables,
                                self.seq_lens, self.append_lens, self.slots, status=self.status, stream=stream)
            else:
                slot_mapping(self.slots, self.block_tables, self.seq_lens, self.append_lens, w.block_size,
                             w.num_blocks, status=self.status, stream=stream)
                kv_append_fp8(self.k_cache, self.v_cache, self.k_new, self.v_new, self.slots, self.k_scale,
                              self.v_scale, status=self.status, stream=stream)

    def attention(self, stream=None):
        if self.fp8 is not None and self.fp8_ex:
            paged_attention_decode_fp8_ex(self.out, self.q, self.k_cache, self.v_cache, self.k_scale, self.v_scale,
                                          self.block_tables, self.seq_lens, self.q_lens, self.max_seq_len,
                                          self.w.scale, self.workspace, **self.fp8_mode,
                                          partition_tokens=self.partition_tokens, status=self.status,
                                          stream=stream, max_q_len=self.max_q_len)
            return
        if self.fp8 is not None:
            paged_attention_decode_fp8(self.out, self.q, self.k_cache, self.v_cache, self.k_scale, self.v_scale,
                                       self.block_tables, self.seq_lens, self.q_lens, self.max_seq_len, self.w.scale,
                                       self.workspace, partition_tokens=self.partition_tokens, status=self.status,
                                       stream=stream, max_q_len=self.max_q_len)
            return
        paged_attention_decode(self.out, self.q, self.k_cache, self.v_cache, self.block_tables, self.seq_lens,
                               self.q_lens, self.max_seq_len, self.w.scale, self.workspace,
                               partition_tokens=self.partition_tokens, flags=self.flags, status=self.status,
                               stream=stream, max_q_len=self.max_q_len)

    def plan(self, stream=None):
        """The planning half of attention(): the work list for this step's
        lengths, into the workspace (one plan serves every run() after it)."""
        w = self.w
        attention_plan(self.seq_lens, self.q_lens, w.total_q, w.max_blocks, w.n_q, w.n_kv, w.head_dim, w.block_size,
                       self.max_seq_len, self.workspace, partition_tokens=self.partition_tokens,
                       flags=PKV_ATTN_PLAN_FP8 if self.fp8 is not None else self.flags, status=self.status,
                       stream=stream, max_q_len=self.max_q_len)

    def run(self, out=None, q=None, k_cache=None, v_cache=None, k_scale=None, v_scale=None, stream=None):
        """The attention half over the planned workspace, by default over this
        step's own buffers; another layer passes its own q, pools and out."""
        w = self.w
        out = self.out if out is None else out
        q = self.q if q is None else q
        k_cache = self.k_cache if k_cache is None else k_cache
        v_cache = self.v_cache if v_cache is None else v_cache
        if self.fp8 is not None:
            paged_attention_run_fp8(out, q, k_cache, v_cache, self.k_scale if k_scale is None else k_scale,
                                    self.v_scale if v_scale is None else v_scale, self.block_tables, w.num_seqs,
                                    self.max_seq_len, w.scale, self.workspace,
                                    partition_tokens=self.partition_tokens, status=self.status, stream=stream,
                                    max_q_len=self.max_q_len, **self.fp8_mode)
            return
        paged_attention_run(out, q, k_cache, v_cache, self.block_tables, w.num_seqs, self.max_seq_len, w.scale,
                            self.workspace, partition_tokens=self.partition_tokens, flags=self.flags,
                            status=self.status, stream=stream, max_q_len=self.max_q_len)

    def accept(self, stream=None):
        if self.spec:
            spec_accept_greedy(self.logits, self.draft, self.argmax, self.accepted, self.next_token, stream=stream)

    def plan_beside_cache_ops(self) -> bool:
        """Whether a step's plan runs on a side stream beside its cache ops:
        only when the step copies blocks on write.  Copy plus append are long
        enough to hide the plan and the two cross-stream waits; beside the
        append alone the waits cost more than the overlap saves, and the plan
        runs in stream order, where programmatic launch overlaps each kernel's
        start with the previous one's end."""
        return bool(self.cow.numel())

    def step(self, stream=None, plan_stream=None):
        """One decode step.  With `plan_stream` (and a step that copies blocks
        on write, `plan_beside_cache_ops`), the plan (which reads only the
        lengths) runs there while the cache ops run on `stream`, and the
        attention run waits for it; the plan stream first waits for the work
        already on `stream` (the previous step's kernels still read the
        workspace, and the lengths may have just been uploaded there).
        Otherwise every kernel of the step runs in order on `stream`."""
        if plan_stream is None or not self.plan_beside_cache_ops():
            self.cache_ops(stream)
            self.attention(stream)
            self.accept(stream)
            return
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        plan_stream.wait_stream(s)
        self.plan(plan_stream)
        self.cache_ops(s)
        s.wait_stream(plan_stream)
        self.run(stream=s)
        self.accept(s)


def main(argv=None):
    """Run a few steps of one workload (a small case for profilers):
    ``python -m paged_kv_cache_23_gb300.runner --workload mix --batch 64 --steps 3``."""
    import argparse

    from . import workloads

    ap = argparse.ArgumentParser(description=main.__doc__)
    ap.add_argument("--workload", default="mix", choices=sorted(workloads.FULL))
    ap.add_argument("--batch", type=int, default=0, help="batch size of the mix workload (0 = 256)")
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--partition", type=int, default=0)
    ap.add_argument("--flags", type=int, default=0)
    ap.add_argument("--fp8", action="store_true", help="e4m3 KV pools (random codes, per-head scales)")
    ap.add_argument("--ctx", type=int, default=0, help="decode context of the long workload (0 = 131072)")
    a = ap.parse_args(argv)
    if a.workload == "mix" and a.batch:
        w = workloads.mix(B=a.batch)
    elif a.workload == "long" and a.ctx:
        w = workloads.long_context(ctx=a.ctx)
    else:
        w = workloads.FULL[a.workload]()
    ds = DeviceStep(w, partition_tokens=a.partition or None, flags=a.flags,
                    fp8=workloads.fp8_pools(w) if a.fp8 else None)
    for _ in range(a.steps):
        ds.cache_ops()
        ds.attention()
        ds.accept()
    torch.cuda.synchronize()
    st = int(ds.status.item())
    print(f"{a.workload}: {a.steps} steps, status {st}")
    return 0 if st == 0 else 1


if __name__ == "__main__":
    raise SystemExit(main())
