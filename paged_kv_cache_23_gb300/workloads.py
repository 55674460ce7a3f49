"""Seeded synthetic inputs for paged-KV decode attention.

This module only builds inputs: random bf16 data, block pools, block tables,
shared prefixes and the copy-on-write pairs a cache manager would emit.  It
computes no step of the attention path (no slot mapping, append, copy,
gather, softmax or acceptance); the CUDA library and the CPU oracle each do
that on their own from what is generated here.

Recipe (common to every workload)
---------------------------------
* Random numbers: numpy PCG64.  One ``SeedSequence(seed)`` per workload;
  its child streams are used in a fixed order: 0 = structure (lengths,
  sharing, pool permutation), 1 = K pool, 2 = V pool, 3 = new K/V rows and Q,
  4 = logits and drafts.  Large fills are drawn in chunks of ``_CHUNK``
  elements, chunk c from grandchild stream c, so the bytes do not depend on
  thread count.
* Values: fp32 standard normal rounded to bf16 (round to nearest even).
* Cache layout: ``[num_blocks][num_kv_heads][block_size][head_dim]`` bf16.
* Pool: ``ceil(1.5 * needed)`` physical blocks, randomly permuted.  Spare
  blocks, and every row of a sequence's last block past its length, hold
  bf16 NaN, so a wrong gather shows up as NaN.
* ``seq_lens`` count the tokens appended in this step; the appended tokens are
  the last ``append_lens[b]`` positions and their rows start out as NaN in the
  cache.  Queries are the last ``q_lens[b]`` positions.
* Block-table padding past a sequence's last block is -1.

A step over a workload is: copy blocks ``cow`` (src -> dst), compute slots for
the appended tokens, append ``k_new``/``v_new``, attend with ``q``; for
speculative workloads, then accept greedily on ``logits``/``draft``.
"""
from __future__ import annotations

import concurrent.futures as _cf
import math
from dataclasses import dataclass, field

import numpy as np

_CHUNK = 1 << 24
BF16_NAN = np.uint16(0x7FC0)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _normal_bf16(ss: np.random.SeedSequence, n: int) -> np.ndarray:
    """n bf16 N(0,1) values, chunk c from ss.spawn(...)[c]."""
    out = np.empty(n, np.uint16)
    nchunks = max(1, -(-n // _CHUNK))
    kids = ss.spawn(nchunks)

    def fill(c):
        lo = c * _CHUNK
        hi = min(n, lo + _CHUNK)
        if hi > lo:
            g = np.random.Generator(np.random.PCG64(kids[c]))
            out[lo:hi] = to_bf16_bits(g.standard_normal(hi - lo, dtype=np.float32))

    if nchunks == 1:
        fill(0)
    else:
        with _cf.ThreadPoolExecutor(max_workers=min(16, nchunks)) as ex:
            list(ex.map(fill, range(nchunks)))
    return out


@dataclass
class Workload:
    name: str
    n_q: int
    n_kv: int
    head_dim: int
    block_size: int
    k_cache: np.ndarray          # uint16 [num_blocks][n_kv][bs][d], state before the step
    v_cache: np.ndarray
    block_tables: np.ndarray     # int32 [B][max_blocks], -1 padded
    seq_lens: np.ndarray         # int32 [B], including this step's appended tokens
    q_lens: np.ndarray           # int32 [B]
    append_lens: np.ndarray      # int32 [B]
    k_new: np.ndarray            # uint16 [sum append_lens][n_kv][d]
    v_new: np.ndarray
    cow: np.ndarray              # int32 [n][2] (src, dst)
    q: np.ndarray                # uint16 [sum q_lens][n_q][d]
    scale: float
    partition_tokens: int = 0    # 0 = library chooses
    logits: np.ndarray | None = None   # float32 [B][k+1][V]
    draft: np.ndarray | None = None    # int32 [B][k]
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_blocks(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def total_q(self) -> int:
        return int(self.q_lens.sum())


class _PoolBuilder:
    """Hands out logical blocks, then maps them to a shuffled physical pool."""

    def __init__(self):
        self.n = 0

    def new(self) -> int:
        self.n += 1
        return self.n - 1


def _finish(name, rng_struct, ss_k, ss_v, ss_new, n_q, n_kv, d, bs, tables_logical, n_logical,
            seq_lens, q_lens, append_lens, cow_logical, valid_rows, scale, partition_tokens,
            rng_q=None, permute=True, pool_factor=1.5, meta=None):
    """Common tail: pool size, permutation, random fill, NaN poisoning.

    valid_rows: dict logical block -> number of leading rows holding data (the
    rest are NaN).  Blocks missing from it are fully NaN (fresh CoW targets).
    """
    num_blocks = max(int(math.ceil(pool_factor * n_logical)), n_logical)
    perm = rng_struct.permutation(num_blocks).astype(np.int32) if permute else np.arange(num_blocks, dtype=np.int32)
    phys = perm[:n_logical]
    B = len(seq_lens)
    max_blocks = max(1, max(len(t) for t in tables_logical))
    bt = np.full((B, max_blocks), -1, np.int32)
    for b, t in enumerate(tables_logical):
        if t:
            bt[b, : len(t)] = phys[np.asarray(t, np.int64)]
    per_block = n_kv * bs * d
    k = _normal_bf16(ss_k, num_blocks * per_block).reshape(num_blocks, n_kv, bs, d)
    v = _normal_bf16(ss_v, num_blocks * per_block).reshape(num_blocks, n_kv, bs, d)
    keep = np.zeros((num_blocks, bs), bool)
    for lb, nrows in valid_rows.items():
        keep[phys[lb], :nrows] = True
    k.transpose(0, 2, 1, 3)[~keep] = BF16_NAN
    v.transpose(0, 2, 1, 3)[~keep] = BF16_NAN
    cow = np.asarray([(phys[s], phys[t]) for s, t in cow_logical], np.int32).reshape(-1, 2)
    g = rng_q if rng_q is not None else np.random.Generator(np.random.PCG64(ss_new))
    seq_lens = np.asarray(seq_lens, np.int32)
    q_lens = np.asarray(q_lens, np.int32)
    append_lens = np.asarray(append_lens, np.int32)
    T = int(append_lens.sum())
    k_new = to_bf16_bits(g.standard_normal((T, n_kv, d), dtype=np.float32))
    v_new = to_bf16_bits(g.standard_normal((T, n_kv, d), dtype=np.float32))
    q = to_bf16_bits(g.standard_normal((int(q_lens.sum()), n_q, d), dtype=np.float32))
    return Workload(name=name, n_q=n_q, n_kv=n_kv, head_dim=d, block_size=bs, k_cache=k, v_cache=v,
                    block_tables=bt, seq_lens=seq_lens, q_lens=q_lens, append_lens=append_lens,
                    k_new=k_new, v_new=v_new, cow=cow, q=q, scale=float(scale),
                    partition_tokens=int(partition_tokens), meta=dict(meta or {}))


def _private_seq(pool, L_cached, L, bs, valid_rows):
    """Blocks for a sequence whose first L_cached positions are cached and
    which ends at L (appended rows start as NaN)."""
    t = []
    for i in range(-(-L // bs)):
        lb = pool.new()
        t.append(lb)
        valid_rows[lb] = max(0, min(bs, L_cached - i * bs))
    return t


def _uniform_decode(name, B, lo, hi, q_len, seed, n_q=32, n_kv=8, d=128, bs=16, partition_tokens=0):
    ss = np.random.SeedSequence(seed)
    s_struct, s_k, s_v, s_new, _ = ss.spawn(5)
    rs = np.random.Generator(np.random.PCG64(s_struct))
    lens = rs.integers(lo, hi + 1, size=B).astype(np.int64)
    pool = _PoolBuilder()
    valid = {}
    tables = [_private_seq(pool, int(L) - q_len, int(L), bs, valid) for L in lens]
    return _finish(name, rs, s_k, s_v, s_new, n_q, n_kv, d, bs, tables, pool.n, lens,
                   [q_len] * B, [q_len] * B, [], valid, 1.0 / math.sqrt(d), partition_tokens,
                   meta=dict(seed=seed, lo=lo, hi=hi))


def tiny(seed: int = 0) -> Workload:
    """1 layer, 4 q / 4 kv heads, head_dim 64, block_size 2; sequences
    A=[10,11,12,13], B=[10,11,12,14], C=[20,21] ("Chapter 31 Serving
    Efficiency", 31.3).  A and B share physical block P0 (positions 0-1); B's
    block 1 is a copy-on-write copy P2 of A's P1, after which B's position 3
    (token 14) is appended.  Blocks P0, P1, P3 are filled in id order from
    PCG64(seed), K then V per block; then B's new row (K, V); then Q for
    A, B, C.  Pool: P0..P3 plus two NaN spares; P2 is NaN until the copy."""
    n, d, bs = 4, 64, 2
    g = np.random.Generator(np.random.PCG64(seed))
    k = np.full((6, n, bs, d), BF16_NAN, np.uint16)
    v = np.full((6, n, bs, d), BF16_NAN, np.uint16)
    for blk in (0, 1, 3):
        k[blk] = to_bf16_bits(g.standard_normal((n, bs, d), dtype=np.float32))
        v[blk] = to_bf16_bits(g.standard_normal((n, bs, d), dtype=np.float32))
    k_new = to_bf16_bits(g.standard_normal((1, n, d), dtype=np.float32))
    v_new = to_bf16_bits(g.standard_normal((1, n, d), dtype=np.float32))
    q = to_bf16_bits(g.standard_normal((3, n, d), dtype=np.float32))
    bt = np.array([[0, 1], [0, 2], [3, -1]], np.int32)
    return Workload(name="tiny", n_q=n, n_kv=n, head_dim=d, block_size=bs, k_cache=k, v_cache=v,
                    block_tables=bt, seq_lens=np.array([4, 4, 2], np.int32),
                    q_lens=np.array([1, 1, 1], np.int32), append_lens=np.array([0, 1, 0], np.int32),
                    k_new=k_new, v_new=v_new, cow=np.array([[1, 2]], np.int32), q=q,
                    scale=1.0 / math.sqrt(d), meta=dict(seed=seed, tokens={"A": [10, 11, 12, 13],
                                                                           "B": [10, 11, 12, 14],
                                                                           "C": [20, 21]}))


def decode(B: int = 64, lo: int = 512, hi: int = 4096, seed: int = 0, **kw) -> Workload:
    """Llama-3-8B-shaped decode layer: 32 q heads, 8 kv heads, head_dim 128,
    block_size 16, seq_len ~ U[lo, hi] (inclusive), q_len 1, one appended
    token per sequence."""
    return _uniform_decode(f"decode_b{B}", B, lo, hi, 1, seed, **kw)


def mix(B: int = 256, median: int = 1024, sigma: float = 1.0, clip=(16, 32768), share: float = 0.5,
        prefix: int = 2048, seed: int = 0, n_q=32, n_kv=8, d=128, bs=16, partition_tokens=0) -> Workload:
    """Continuous-batching mix: seq_len = round(lognormal(ln median, sigma))
    clipped to ``clip``; a random ``share`` fraction of sequences take their
    first min(seq_len - 1, prefix) cached positions from one shared prefix
    (same physical block ids).  When a sharer's appended position falls inside
    a shared block, that block is copied on write to a private block first;
    one appended token per sequence, q_len 1."""
    ss = np.random.SeedSequence(seed)
    s_struct, s_k, s_v, s_new, _ = ss.spawn(5)
    rs = np.random.Generator(np.random.PCG64(s_struct))
    lens = np.clip(np.rint(rs.lognormal(math.log(median), sigma, size=B)), clip[0], clip[1]).astype(np.int64)
    n_share = int(round(share * B))
    sharers = set(rs.choice(B, size=n_share, replace=False).tolist())
    assert prefix % bs == 0
    pool = _PoolBuilder()
    valid = {}
    prefix_blocks = [pool.new() for _ in range(prefix // bs)]
    for lb in prefix_blocks:
        valid[lb] = bs
    tables, cow = [], []
    for b in range(B):
        L = int(lens[b])
        cached = L - 1
        if b not in sharers:
            tables.append(_private_seq(pool, cached, L, bs, valid))
            continue
        shared_pos = min(cached, prefix)
        t = []
        nblk = -(-L // bs)
        for i in range(nblk):
            lo_pos = i * bs
            if lo_pos + bs <= shared_pos:
                t.append(prefix_blocks[i])           # full shared block
            elif lo_pos < shared_pos:
                # partial shared block that will receive the appended token:
                # copy on write into a private block
                lb = pool.new()
                cow.append((prefix_blocks[i], lb))
                t.append(lb)
            else:
                lb = pool.new()
                valid[lb] = max(0, min(bs, cached - lo_pos))
                t.append(lb)
        tables.append(t)
    return _finish(f"mix_b{B}", rs, s_k, s_v, s_new, n_q, n_kv, d, bs, tables, pool.n, lens,
                   [1] * B, [1] * B, cow, valid, 1.0 / math.sqrt(d), partition_tokens,
                   meta=dict(seed=seed, sharers=sorted(sharers), prefix=prefix, median=median,
                             sigma=sigma, clip=tuple(clip)))


def spec(B: int = 32, lo: int = 2048, hi: int = 8192, k: int = 5, vocab: int = 128256,
         alpha: float = 0.7, seed: int = 0, q_len: int | None = None, **kw) -> Workload:
    """Speculative verification: seq_len ~ U[lo, hi] including the new tokens,
    q_len = k by default (the k drafted tokens, causal within the draft) or
    q_len = k + 1 (the last accepted token and the k drafts: one pass yields
    the k + 1 distributions), q_len appended tokens per sequence; target
    logits [B][k+1][vocab] fp32 N(0,1); draft[b][j] equals the row argmax
    (numpy's, first index on ties) with probability alpha, independently per
    position, else a uniform pick among the other ids."""
    ql = k if q_len is None else int(q_len)
    w = _uniform_decode(f"spec_b{B}_k{k}" + ("" if ql == k else f"_q{ql}"), B, lo, hi, ql, seed, **kw)
    ss = np.random.SeedSequence(seed)
    s_logit = ss.spawn(5)[4]
    kids = s_logit.spawn(2)
    rows = B * (k + 1)
    logits = np.empty((rows, vocab), np.float32)
    gl = np.random.Generator(np.random.PCG64(kids[0]))
    for r0 in range(0, rows, 16):
        r1 = min(rows, r0 + 16)
        logits[r0:r1] = gl.standard_normal((r1 - r0, vocab), dtype=np.float32)
    logits = logits.reshape(B, k + 1, vocab)
    gd = np.random.Generator(np.random.PCG64(kids[1]))
    top = logits[:, :k, :].argmax(axis=-1)
    agree = gd.random((B, k)) < alpha
    other = gd.integers(0, vocab - 1, size=(B, k))
    other = other + (other >= top)          # uniform over the vocab minus the argmax
    w.draft = np.where(agree, top, other).astype(np.int32)
    w.logits = logits
    w.meta.update(alpha=alpha, vocab=vocab, k=k)
    return w


@dataclass
class Fp8Pools:
    """An FP8 KV cache holding the same structure as a bf16 workload's pools:
    uint8 codes [num_blocks][n_kv][bs][d] of format fmt (0 = e4m3, 1 = e5m2)
    and fp32 dequantisation scales for K and for V: one per kv head
    ([n_kv]), or one per (block, kv head) tile ([num_blocks][n_kv]) when
    per_block."""
    k_cache: np.ndarray
    v_cache: np.ndarray
    k_scale: np.ndarray
    v_scale: np.ndarray
    fmt: int = 0
    per_block: bool = False


def fp8_pools(w: Workload, seed: int = 0, fmt: int = 0, per_block: bool = False) -> Fp8Pools:
    """Random FP8 contents for the rows the bf16 workload holds (sign random,
    exponent field 4..10 for e4m3 or 12..18 for e5m2 -- magnitudes 2^-3..15
    --, mantissa random; no encoding step), the format's NaN (0x7f) wherever
    the bf16 pool is NaN (unused rows and spare blocks), and scales
    2^-3 * U[0.5, 1.5] per kv head, or per (block, kv head) with per_block."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 8] if fmt == 0 and not per_block
                                                                   else [seed, 8, fmt, int(per_block)])))
    out = []
    for pool in (w.k_cache, w.v_cache):
        sign = g.integers(0, 2, size=pool.shape, dtype=np.uint8) << 7
        if fmt == 0:
            expo = g.integers(4, 11, size=pool.shape, dtype=np.uint8) << 3
            mant = g.integers(0, 8, size=pool.shape, dtype=np.uint8)
        else:
            expo = g.integers(12, 19, size=pool.shape, dtype=np.uint8) << 2
            mant = g.integers(0, 4, size=pool.shape, dtype=np.uint8)
        codes = sign | expo | mant
        codes[(pool & 0x7FFF) > 0x7F80] = 0x7F
        out.append(codes)
    shape = (w.num_blocks, w.n_kv) if per_block else (w.n_kv,)
    ks = (0.125 * g.uniform(0.5, 1.5, size=shape)).astype(np.float32)
    vs = (0.125 * g.uniform(0.5, 1.5, size=shape)).astype(np.float32)
    return Fp8Pools(out[0], out[1], ks, vs, int(fmt), bool(per_block))


@dataclass
class Prompts:
    """Token ids of a batch of prompts: tokens int32 [B][max_len] (0 past each
    length), lens int32 [B]."""
    tokens: np.ndarray
    lens: np.ndarray
    meta: dict = field(default_factory=dict)


def prompts(B: int = 256, median: int = 1024, sigma: float = 1.0, clip=(16, 32768), share: float = 0.5,
            prefix: int = 2048, vocab: int = 128256, seed: int = 0) -> Prompts:
    """Prompt lengths as in the mix (log-normal, clipped); a random ``share`` of
    the batch starts with one common ``prefix``-token system prompt (cut to
    the prompt's length); token ids uniform over the vocabulary."""
    g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 31])))
    lens = np.clip(np.rint(g.lognormal(math.log(median), sigma, size=B)), clip[0], clip[1]).astype(np.int32)
    T = int(lens.max())
    tokens = g.integers(0, vocab, size=(B, T), dtype=np.int32)
    sys_prompt = g.integers(0, vocab, size=prefix, dtype=np.int32)
    sharers = g.choice(B, size=int(round(share * B)), replace=False)
    for b in sharers:
        n = min(prefix, int(lens[b]), T)
        tokens[b, :n] = sys_prompt[:n]
    for b in range(B):
        tokens[b, lens[b]:] = 0
    return Prompts(tokens, lens, dict(B=B, median=median, sigma=sigma, share=share, prefix=prefix, seed=seed,
                                      sharers=np.sort(sharers)))


@dataclass
class SampleInputs:
    """Inputs of stochastic speculative acceptance: target distributions
    p [B][k+1][V], draft distributions q [B][k][V] (fp32, each row sums to 1),
    drafts [B][k] drawn from q, acceptance uniforms r [B][k] and one sampling
    uniform s [B] (fp32 in [0, 1))."""
    p: np.ndarray
    q: np.ndarray
    draft: np.ndarray
    r: np.ndarray
    s: np.ndarray
    meta: dict = field(default_factory=dict)


def _softmax_rows(z: np.ndarray) -> np.ndarray:
    z = z.astype(np.float64)
    z = z - z.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return (e / e.sum(axis=-1, keepdims=True)).astype(np.float32)


def spec_sample(B: int = 32, k: int = 5, vocab: int = 128256, temp: float = 2.0, noise: float = 1.0,
                seed: int = 0) -> SampleInputs:
    """Distributions for stochastic verification: target logits
    temp * N(0, 1) per row, p = softmax; the draft model's logits are the
    target's plus noise * N(0, 1), q = softmax (so p and q overlap the way a
    good small proposer does); each draft is drawn from its q row by inverse
    CDF; r and s uniform in [0, 1)."""
    ss = np.random.SeedSequence([seed, 23])
    g = np.random.Generator(np.random.PCG64(ss))
    z = (temp * g.standard_normal((B, k + 1, vocab), dtype=np.float32)).astype(np.float32)
    p = _softmax_rows(z)
    zq = z[:, :k, :] + (noise * g.standard_normal((B, k, vocab), dtype=np.float32)).astype(np.float32)
    q = _softmax_rows(zq)
    u = g.random((B, k))
    c = np.cumsum(q.astype(np.float64), axis=-1)
    draft = np.empty((B, k), np.int32)
    for b in range(B):
        for j in range(k):
            draft[b, j] = min(int(np.searchsorted(c[b, j], u[b, j] * c[b, j, -1], side="right")), vocab - 1)
    r = g.random((B, k), dtype=np.float32)
    s_ = g.random(B, dtype=np.float32)
    return SampleInputs(p=p, q=q, draft=draft, r=r, s=s_,
                        meta=dict(B=B, k=k, vocab=vocab, temp=temp, noise=noise, seed=seed))


def long_context(B: int = 8, ctx: int = 131072, chunk: int = 512, chunk_prefix: int = 8192,
                 partition_tokens: int = 4096, seed: int = 0, n_q=32, n_kv=8, d=128, bs=16) -> Workload:
    """B decodes of ctx tokens each (q_len 1, one appended token) plus one
    chunked-prefill request of ``chunk`` causal query tokens over a paged
    prefix of ``chunk_prefix`` tokens (seq_len = prefix + chunk, all chunk
    tokens appended in this step), in one batch; split-KV partitions of
    ``partition_tokens``."""
    ss = np.random.SeedSequence(seed)
    s_struct, s_k, s_v, s_new, _ = ss.spawn(5)
    rs = np.random.Generator(np.random.PCG64(s_struct))
    pool = _PoolBuilder()
    valid = {}
    tables = [_private_seq(pool, ctx - 1, ctx, bs, valid) for _ in range(B)]
    Lc = chunk_prefix + chunk
    tables.append(_private_seq(pool, chunk_prefix, Lc, bs, valid))
    lens = [ctx] * B + [Lc]
    ql = [1] * B + [chunk]
    return _finish(f"long_b{B}_ctx{ctx}_chunk{chunk}", rs, s_k, s_v, s_new, n_q, n_kv, d, bs, tables,
                   pool.n, lens, ql, ql, [], valid, 1.0 / math.sqrt(d), partition_tokens,
                   meta=dict(seed=seed, ctx=ctx, chunk=chunk, chunk_prefix=chunk_prefix))


def concat(a: Workload, b: Workload) -> Workload:
    """One batch holding a's sequences then b's, over one pool (b's blocks
    after a's); same head shape and block size.  Acceptance inputs are
    dropped (their shapes differ between workloads)."""
    assert (a.n_q, a.n_kv, a.head_dim, a.block_size) == (b.n_q, b.n_kv, b.head_dim, b.block_size)
    nb = a.num_blocks
    mb = max(a.max_blocks, b.max_blocks)
    bt = np.full((a.num_seqs + b.num_seqs, mb), -1, np.int32)
    bt[: a.num_seqs, : a.max_blocks] = a.block_tables
    bt[a.num_seqs:, : b.max_blocks] = np.where(b.block_tables >= 0, b.block_tables + nb, -1)
    cow = np.concatenate([a.cow.reshape(-1, 2), b.cow.reshape(-1, 2) + nb]).astype(np.int32)
    return Workload(name=f"{a.name}+{b.name}", n_q=a.n_q, n_kv=a.n_kv, head_dim=a.head_dim, block_size=a.block_size,
                    k_cache=np.concatenate([a.k_cache, b.k_cache]), v_cache=np.concatenate([a.v_cache, b.v_cache]),
                    block_tables=bt, seq_lens=np.concatenate([a.seq_lens, b.seq_lens]),
                    q_lens=np.concatenate([a.q_lens, b.q_lens]),
                    append_lens=np.concatenate([a.append_lens, b.append_lens]),
                    k_new=np.concatenate([a.k_new, b.k_new]), v_new=np.concatenate([a.v_new, b.v_new]), cow=cow,
                    q=np.concatenate([a.q, b.q]), scale=a.scale, partition_tokens=a.partition_tokens,
                    meta=dict(parts=[a.name, b.name]))


# The five workloads at full size, by name.
FULL = {
    "tiny": lambda: tiny(0),
    "decode": lambda: decode(64, 512, 4096, 0),
    "mix": lambda: mix(256, 1024, 1.0, (16, 32768), 0.5, 2048, 0),
    "spec": lambda: spec(32, 2048, 8192, 5, 128256, 0.7, 0),
    "long": lambda: long_context(8, 131072, 512, 8192, 4096, 0),
}

# Small versions with the same structure (several tiles, ragged tails,
# sharing, copy-on-write, split partitions), for fast parity tests.
SMALL = {
    "tiny": lambda: tiny(0),
    "decode": lambda: decode(6, 17, 300, 1),
    "mix": lambda: mix(24, 80, 1.0, (16, 1200), 0.5, 128, 2),
    "spec": lambda: spec(4, 40, 260, 5, 1000, 0.7, 3),
    "long": lambda: long_context(2, 5000, 40, 300, 1024, 4),
}
