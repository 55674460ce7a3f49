"""Byte accounting for the roofline: what one step must move, by definition.

"Inference at Scale: KV Cache, Prefill, and Decode", section 03, "Bytes per
token": KV bytes per token = 2 x layers x kv heads x head_dim x bytes per
value (K and V).  Section 02 puts decode attention at about g FLOP per byte
(g = query heads per kv head), far left of any GPU's ridge point, so the
roofline of this path is HBM bandwidth.

Counts here are algorithmic: only bytes the method must read or write (the
visible K/V, Q, O, appended rows, copied blocks, block-table entries), never
workspace or re-reads.
"""
from __future__ import annotations

import numpy as np


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int, bytes_per_value: int = 2) -> int:
    return 2 * num_layers * num_kv_heads * head_dim * bytes_per_value


def step_bytes(w, bytes_per_value: int = 2, kv_bytes: int | None = None, block_scales: bool = False) -> dict:
    """Algorithmic bytes of one step over workload ``w`` (one layer).

    kv_bytes: bytes per cached K/V value (1 for an FP8 pool, section 03 "KV
    cache quantization"); queries, outputs and appended rows stay bf16.
    block_scales: the FP8 pool has a K and a V scale (fp32) per (block, kv
    head) tile, read with the block.

    kv_logical  every sequence's visible K/V, counted once per sequence (the
                query heads of a group share one read)
    kv_unique   distinct (physical block, row) pairs visible to some query,
                so blocks shared between sequences count once
    """
    bs = w.block_size
    kvb = bytes_per_value if kv_bytes is None else kv_bytes
    per_row = w.n_kv * w.head_dim * kvb * 2                      # K and V of one token, all kv heads
    L = w.seq_lens.astype(np.int64)
    kv_logical = int(L.sum()) * per_row
    rows = []
    for b in range(w.num_seqs):
        n = int(L[b])
        if n <= 0:
            continue
        nblk = -(-n // bs)
        ids = w.block_tables[b, :nblk].astype(np.int64)
        cnt = np.full(nblk, bs, np.int64)
        cnt[-1] = n - (nblk - 1) * bs
        rows.append(np.stack([ids, cnt], 1))
    if rows:
        r = np.concatenate(rows)
        # a block's visible rows are a prefix; the union is the longest prefix
        order = np.lexsort((-r[:, 1], r[:, 0]))
        r = r[order]
        first = np.ones(len(r), bool)
        first[1:] = r[1:, 0] != r[:-1, 0]
        kv_unique = int(r[first, 1].sum()) * per_row
        n_unique_blocks = int(first.sum())
    else:
        kv_unique = 0
        n_unique_blocks = 0
    q_bytes = w.total_q * w.n_q * w.head_dim * bytes_per_value
    o_bytes = q_bytes
    tables = int(sum(-(-int(n) // bs) for n in L)) * 4 + 2 * 4 * w.num_seqs
    t_new = int(w.append_lens.sum())
    new_row = w.n_kv * w.head_dim * bytes_per_value * 2
    append = t_new * (new_row + per_row) + t_new * 8  # read new rows, write them (cache format), read slots
    cow = int(w.cow.shape[0]) * 2 * (w.n_kv * bs * w.head_dim * kvb * 2)
    scales_unique = scales_logical = 0
    if block_scales:
        per_blk = w.n_kv * 8                                     # K and V scale, fp32, every kv head
        scales_unique = n_unique_blocks * per_blk
        scales_logical = int(sum(-(-int(n) // bs) for n in L)) * per_blk
        cow += int(w.cow.shape[0]) * 2 * per_blk
        # the append sets the scales of the blocks it opens (positions at a block's row 0)
        A = w.append_lens.astype(np.int64)
        opened = sum(len(range(-(-(int(L[b]) - int(A[b])) // bs) * bs, int(L[b]), bs)) for b in range(w.num_seqs))
        append += int(opened) * per_blk
    attn_unique = kv_unique + q_bytes + o_bytes + tables + scales_unique
    attn_logical = kv_logical + q_bytes + o_bytes + tables + scales_logical
    return dict(kv_logical=kv_logical, kv_unique=kv_unique, q=q_bytes, o=o_bytes, tables=tables,
                append=append, cow=cow, scales=scales_unique, attention_unique=attn_unique,
                attention_logical=attn_logical, step_unique=attn_unique + append + cow,
                step_logical=attn_logical + append + cow)


def accept_greedy_bytes(w) -> int:
    """Greedy acceptance ("Spending the Idle" 12.4): every logits row is
    scanned for its argmax (4 B per score), plus drafts and the outputs."""
    B, k1, V = w.logits.shape
    return B * k1 * V * 4 + B * (k1 - 1) * 4 + B * k1 * 4 + 2 * B * 4


def accept_sample_bytes(x, accepted) -> int:
    """Stochastic acceptance ("Chapter 31 Serving Efficiency" 31.5): per
    sequence the draft, r, p(x) and q(x) of each checked position, and the one
    distribution the draw needs -- p and q rows of the rejected position
    (8 B per token) or the p row after all drafts (4 B per token) -- plus s
    and the two outputs."""
    B, k1, V = x.p.shape
    k = k1 - 1
    acc = np.asarray(accepted, np.int64)
    checked = np.minimum(acc + 1, k)
    rows = np.where(acc < k, 8, 4) * V
    return int((checked * 16).sum() + rows.sum() + B * 12)


def attention_flops(w) -> int:
    """2 FLOP per multiply-add for QK^T and PV over the visible positions."""
    L = w.seq_lens.astype(np.int64)
    ql = w.q_lens.astype(np.int64)
    vis = 0
    for b in range(w.num_seqs):
        # query i of sequence b sees L - ql + i + 1 positions
        n = int(ql[b])
        vis += n * (int(L[b]) - n) + n * (n + 1) // 2
    return 4 * vis * w.n_q * w.head_dim
