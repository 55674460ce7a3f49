"""CPU fp64 oracle for paged-KV decode attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
product path (``paged_kv_cache_23_gb300``) never imports it and shares no code
with it: the arithmetic lives in ``pkv_oracle.c`` (plain C, fp64 loops), this
module only compiles it with gcc and marshals numpy arrays through ctypes.

Each wrapper names the passage of the source pages it follows; see the C file
for the definitions written out.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pkv_oracle.c")
_LIB = os.path.join(_HERE, "libpkv_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile pkv_oracle.c with gcc (OpenMP if the compiler has it)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            P = ctypes.c_void_p
            I = ctypes.c_int
            D = ctypes.c_double
            sigs = {
                "oracle_slot_mapping": [P, P, I, P, P, I, I, I],
                "oracle_kv_append": [P, P, P, P, P, I, I, I, I, I],
                "oracle_copy_blocks": [P, P, P, I, I, I, I, I],
                "oracle_gather_kv": [P, P, P, P, P, I, P, I, I, I, I, I],
                "oracle_attention": [P, P, P, P, P, I, P, P, I, I, I, I, I, I, D],
                "oracle_attention_split": [P, P, P, P, I, P, P, P, P, I, P, P, I, I, I, I, I, I, D, I],
                "oracle_spec_accept_greedy": [P, P, P, P, P, I, I, I],
                "oracle_spec_accept_sample": [P, P, P, P, P, P, P, I, I, I],
                "oracle_e4m3_encode": [P, P, ctypes.c_int64],
                "oracle_e4m3_decode": [P, P, ctypes.c_int64],
                "oracle_kv_append_fp8": [P, P, P, P, P, I, I, I, I, I, P, P],
                "oracle_attention_fp8": [P, P, P, P, P, P, P, I, P, P, I, I, I, I, I, I, D],
                "oracle_prefix_hash": [P, P, I, P, I, I, I, ctypes.c_uint64],
                "oracle_fp8_encode": [P, P, ctypes.c_int64, I],
                "oracle_fp8_decode": [P, P, ctypes.c_int64, I],
                "oracle_kv_append_fp8_ex": [P, P, P, P, P, P, P, I, I, I, I, I, I, I],
                "oracle_copy_blocks_fp8": [P, P, P, P, P, I, I, I, I, I, I],
                "oracle_attention_fp8_ex": [P, P, P, P, P, P, P, I, P, P, I, I, I, I, I, I, D, I, I],
                "oracle_num_threads": [],
            }
            for name, argt in sigs.items():
                f = getattr(lib, name)
                f.argtypes = argt
                f.restype = ctypes.c_int
            lib.oracle_block_scale.argtypes = [P, I, I]
            lib.oracle_block_scale.restype = ctypes.c_float
            lib.oracle_set_num_threads.argtypes = [I]
            lib.oracle_set_num_threads.restype = None
            _lib = lib
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    """Threads of the oracle's parallel loops from now on (timing only)."""
    _load().oracle_set_num_threads(int(n))


def slot_mapping(block_tables, seq_lens, append_lens, block_size, num_blocks):
    """Slots of the last append_lens[b] positions of every sequence, packed in
    sequence order ("Inference at Scale: KV Cache, Prefill, and Decode",
    section 05, "The block table").  Returns (slots int64, status)."""
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    al = _c(append_lens, np.int32)
    if bt.shape[0] != len(sl) or len(al) != len(sl):
        raise ValueError("block_tables, seq_lens and append_lens disagree on the batch size")
    n = int(np.clip(al, 0, None).sum())
    slots = np.empty(max(n, 1), np.int64)
    st = _load().oracle_slot_mapping(_p(slots), _p(bt), bt.shape[1], _p(sl), _p(al), len(sl),
                                     block_size, num_blocks)
    return slots[:n], st


def kv_append(k_cache, v_cache, k_new, v_new, slots):
    """Write new K/V rows into their slots, in place (section 02 of "Inference
    at Scale": decode appends one row per new token).  Returns status."""
    assert k_cache.dtype == np.uint16 and k_cache.flags.c_contiguous
    nb, nkv, bs, d = k_cache.shape
    kn = _c(k_new, np.uint16)
    vn = _c(v_new, np.uint16)
    sl = _c(slots, np.int64)
    if kn.shape != (len(sl), nkv, d) or vn.shape != kn.shape:
        raise ValueError("k_new/v_new must be [num_tokens][n_kv][head_dim]")
    return _load().oracle_kv_append(_p(k_cache), _p(v_cache), _p(kn), _p(vn), _p(sl), len(sl),
                                    nb, bs, nkv, d)


def copy_blocks(k_cache, v_cache, src_dst):
    """Copy-on-write block copies, in place ("Chapter 31 Serving Efficiency",
    31.3; "Inference at Scale", section 05).  Returns status."""
    nb, nkv, bs, d = k_cache.shape
    sd = _c(src_dst, np.int32).reshape(-1, 2)
    return _load().oracle_copy_blocks(_p(k_cache), _p(v_cache), _p(sd), sd.shape[0], nb, bs, nkv, d)


def gather_kv(k_cache, v_cache, block_tables, seq_lens):
    """Contiguous [sum seq_len][n_kv][d] K and V read through the block table.
    Returns (k, v, status)."""
    nb, nkv, bs, d = k_cache.shape
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    tot = int(sl.sum())
    ko = np.empty((max(tot, 1), nkv, d), np.uint16)
    vo = np.empty((max(tot, 1), nkv, d), np.uint16)
    st = _load().oracle_gather_kv(_p(ko), _p(vo), _p(k_cache), _p(v_cache), _p(bt), bt.shape[1],
                                  _p(sl), len(sl), nb, bs, nkv, d)
    return ko[:tot], vo[:tot], st


def attention(q, k_cache, v_cache, block_tables, seq_lens, q_lens, scale):
    """fp64 softmax attention through the block table, causal within the new
    tokens (sections 07 and 08 of "Inference at Scale").  q is uint16 bf16
    bits [sum q_len][n_q][d].  Returns (out float64, status)."""
    nb, nkv, bs, d = k_cache.shape
    q = _c(q, np.uint16)
    nq = q.shape[1]
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    ql = _c(q_lens, np.int32)
    if q.shape[0] != int(np.clip(ql, 0, None).sum()) or q.shape[2] != d or nq % nkv:
        raise ValueError("q must be [sum q_lens][n_q][head_dim] with n_q a multiple of n_kv")
    out = np.zeros((max(q.shape[0], 1), nq, d), np.float64)
    st = _load().oracle_attention(_p(out), _p(q), _p(k_cache), _p(v_cache), _p(bt), bt.shape[1],
                                  _p(sl), _p(ql), len(sl), nq, nkv, d, bs, nb, float(scale))
    return out[: q.shape[0]], st


def attention_split(q, k_cache, v_cache, block_tables, seq_lens, q_lens, scale, partition_tokens,
                    want_partials=False):
    """Flash-Decoding split-KV attention with log-sum-exp merge ("Inference at
    Scale", section 07).  Returns (out, status) or, with want_partials,
    (out, status, part_o, part_m, part_l) shaped [rows][n_q][nparts](, d)."""
    nb, nkv, bs, d = k_cache.shape
    q = _c(q, np.uint16)
    nq = q.shape[1]
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    ql = _c(q_lens, np.int32)
    if q.shape[0] != int(np.clip(ql, 0, None).sum()) or q.shape[2] != d or nq % nkv:
        raise ValueError("q must be [sum q_lens][n_q][head_dim] with n_q a multiple of n_kv")
    P = int(partition_tokens)
    if P <= 0:
        raise ValueError("partition_tokens must be positive")
    npm = max(1, -(-int(sl.max(initial=0)) // P))
    rows = max(q.shape[0], 1)
    out = np.zeros((rows, nq, d), np.float64)
    po = pm = pl = None
    if want_partials:
        po = np.zeros((rows, nq, npm, d), np.float64)
        pm = np.zeros((rows, nq, npm), np.float64)
        pl = np.zeros((rows, nq, npm), np.float64)
    st = _load().oracle_attention_split(_p(out), _p(po), _p(pm), _p(pl), npm, _p(q), _p(k_cache),
                                        _p(v_cache), _p(bt), bt.shape[1], _p(sl), _p(ql), len(sl),
                                        nq, nkv, d, bs, nb, float(scale), P)
    n = q.shape[0]
    if want_partials:
        return out[:n], st, po[:n], pm[:n], pl[:n]
    return out[:n], st


def e4m3_encode(x):
    """fp32 -> e4m3 codes (round to nearest even, saturate to 448, NaN kept)."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    _load().oracle_e4m3_encode(_p(out), _p(x), x.size)
    return out


def e4m3_decode(codes):
    """e4m3 codes -> exact fp64 values (NaN for S.1111.111)."""
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().oracle_e4m3_decode(_p(out), _p(c), c.size)
    return out


def kv_append_fp8(k_cache8, v_cache8, k_new, v_new, slots, k_scale, v_scale):
    """Append bf16 rows into e4m3 pools in place ("Inference at Scale" 03, KV
    cache quantization): code = e4m3(x * (1 / scale[head])).  Returns status."""
    nb, nkv, bs, d = k_cache8.shape
    assert k_cache8.dtype == np.uint8 and v_cache8.dtype == np.uint8
    kn = _c(k_new, np.uint16)
    vn = _c(v_new, np.uint16)
    sl = _c(slots, np.int64)
    return _load().oracle_kv_append_fp8(_p(k_cache8), _p(v_cache8), _p(kn), _p(vn), _p(sl), len(sl), nb, bs, nkv, d,
                                        _p(_c(k_scale, np.float32)), _p(_c(v_scale, np.float32)))


def attention_fp8(q, k_cache8, v_cache8, k_scale, v_scale, block_tables, seq_lens, q_lens, scale):
    """attention() over e4m3 pools: K = e4m3(K) * k_scale[kv head], V likewise."""
    qq = _c(q, np.uint16)
    T, n_q, d = qq.shape
    nb, nkv, bs, d2 = k_cache8.shape
    if d2 != d or n_q % nkv or T < int(np.maximum(np.asarray(q_lens), 0).sum()):
        raise ValueError("q must be [sum q_lens][n_q][head_dim] with n_q a multiple of n_kv")
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    ql = _c(q_lens, np.int32)
    out = np.zeros((T, n_q, d), np.float64)
    st = _load().oracle_attention_fp8(_p(out), _p(qq), _p(_c(k_cache8, np.uint8)), _p(_c(v_cache8, np.uint8)),
                                      _p(_c(k_scale, np.float32)), _p(_c(v_scale, np.float32)), _p(bt), bt.shape[1],
                                      _p(sl), _p(ql), len(sl), n_q, nkv, d, bs, nb, float(scale))
    return out, st


E4M3, E5M2 = 0, 1


def fp8_encode(x, fmt=E4M3):
    """fp32 -> e4m3 or e5m2 codes (round to nearest even, saturate to the
    largest finite value, NaN kept as 0x7f)."""
    x = _c(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    _load().oracle_fp8_encode(_p(out), _p(x), x.size, int(fmt))
    return out


def fp8_decode(codes, fmt=E4M3):
    """e4m3 / e5m2 codes -> exact fp64 values."""
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    _load().oracle_fp8_decode(_p(out), _p(c), c.size, int(fmt))
    return out


def block_scale(row, fmt=E4M3):
    """Scale a block's opening row sets for one kv head: the smallest power of
    two s with max|row| <= s * FMAX / 2 (1 for an all-zero or infinite row)."""
    r = _c(row, np.float32).reshape(-1)
    return float(_load().oracle_block_scale(_p(r), r.size, int(fmt)))


def kv_append_fp8_ex(k_cache8, v_cache8, k_new, v_new, slots, k_scale, v_scale, fmt=E4M3, per_block=False):
    """Append bf16 rows into FP8 pools in place ("Inference at Scale" 03, KV
    cache quantization), either format; per_block: scales [num_blocks][n_kv]
    (updated in place: a block's row 0 sets its scales), else [n_kv].
    Returns status."""
    nb, nkv, bs, d = k_cache8.shape
    assert k_cache8.dtype == np.uint8 and v_cache8.dtype == np.uint8
    assert k_scale.dtype == np.float32 and k_scale.flags.c_contiguous and v_scale.flags.c_contiguous
    kn = _c(k_new, np.uint16)
    vn = _c(v_new, np.uint16)
    sl = _c(slots, np.int64)
    return _load().oracle_kv_append_fp8_ex(_p(k_cache8), _p(v_cache8), _p(k_scale), _p(v_scale), _p(kn), _p(vn),
                                           _p(sl), len(sl), nb, bs, nkv, d, int(fmt), int(bool(per_block)))


def copy_blocks_fp8(k_cache8, v_cache8, k_scale, v_scale, src_dst, per_block=False):
    """Copy-on-write block copies in FP8 pools, in place (and the blocks'
    scales with per_block).  Returns status."""
    nb, nkv, bs, d = k_cache8.shape
    sd = _c(src_dst, np.int32).reshape(-1, 2)
    return _load().oracle_copy_blocks_fp8(_p(k_cache8), _p(v_cache8), _p(k_scale), _p(v_scale), _p(sd),
                                          sd.shape[0], nb, bs, nkv, d, int(bool(per_block)))


def attention_fp8_ex(q, k_cache8, v_cache8, k_scale, v_scale, block_tables, seq_lens, q_lens, scale, fmt=E4M3,
                     per_block=False):
    """attention() over FP8 pools of either format: K = fp8(K) * scale of the
    kv head (or of the (block, kv head) tile with per_block), V likewise."""
    qq = _c(q, np.uint16)
    T, n_q, d = qq.shape
    nb, nkv, bs, d2 = k_cache8.shape
    if d2 != d or n_q % nkv or T < int(np.maximum(np.asarray(q_lens), 0).sum()):
        raise ValueError("q must be [sum q_lens][n_q][head_dim] with n_q a multiple of n_kv")
    bt = _c(block_tables, np.int32)
    sl = _c(seq_lens, np.int32)
    ql = _c(q_lens, np.int32)
    out = np.zeros((T, n_q, d), np.float64)
    st = _load().oracle_attention_fp8_ex(_p(out), _p(qq), _p(_c(k_cache8, np.uint8)), _p(_c(v_cache8, np.uint8)),
                                         _p(_c(k_scale, np.float32)), _p(_c(v_scale, np.float32)), _p(bt),
                                         bt.shape[1], _p(sl), _p(ql), len(sl), n_q, nkv, d, bs, nb, float(scale),
                                         int(fmt), int(bool(per_block)))
    return out, st


def spec_accept_sample(p, q, draft, r, s):
    """Modified rejection sampling ("Chapter 31 Serving Efficiency" 31.5,
    Example 31.3; "Spending the Idle" 12.4): accept draft x_j iff
    r_j * q_j(x_j) < p_j(x_j) (fp32), else draw the next token from
    max(0, p_j - q_j) by integer inverse CDF with s_b; all accepted -> draw from
    p_k.  p float32 [B][k+1][V], q float32 [B][k][V], draft int32 [B][k],
    r float32 [B][k], s float32 [B].  Returns (accepted [B], next_token [B],
    status bits)."""
    pp = _c(p, np.float32)
    B, k1, V = pp.shape
    k = k1 - 1
    qq = _c(q, np.float32).reshape(B, k, V)
    dr = _c(draft, np.int32).reshape(B, k)
    rr = _c(r, np.float32).reshape(B, k)
    ss = _c(s, np.float32).reshape(B)
    acc = np.empty(B, np.int32)
    nxt = np.empty(B, np.int32)
    st = _load().oracle_spec_accept_sample(_p(acc), _p(nxt), _p(pp), _p(qq), _p(dr), _p(rr), _p(ss), B, k, V)
    return acc, nxt, int(st)


def spec_accept_greedy(logits, draft):
    """Greedy acceptance ("Spending the Idle" 12.4; "Inference at Scale" 08).
    logits float32 [B][k+1][V], draft int32 [B][k].
    Returns (accepted [B], next_token [B], argmax [B][k+1])."""
    lg = _c(logits, np.float32)
    B, k1, V = lg.shape
    k = k1 - 1
    dr = _c(draft, np.int32).reshape(B, k)
    acc = np.empty(B, np.int32)
    nxt = np.empty(B, np.int32)
    am = np.empty((B, k1), np.int32)
    _load().oracle_spec_accept_greedy(_p(acc), _p(nxt), _p(am), _p(lg), _p(dr), B, k, V)
    return acc, nxt, am


def prefix_hash(tokens, lens, block_size, max_blocks, salt=0):
    """Chained 128-bit block hashes ("Inference at Scale" 05, prefix caching;
    "Chapter 31 Serving Efficiency" 31.3).  tokens int32 [B][max_tokens],
    lens int32 [B].  Returns uint64 [B][max_blocks][2] (zeros past the full
    blocks of each sequence)."""
    tk = _c(tokens, np.int32)
    B, T = tk.shape
    ln = _c(lens, np.int32).reshape(B)
    out = np.zeros((B, max_blocks, 2), np.uint64)
    _load().oracle_prefix_hash(_p(out), _p(tk), T, _p(ln), B, block_size, max_blocks, ctypes.c_uint64(salt & (2**64 - 1)))
    return out


class PrefixCache:
    """The prefix cache's semantics, written plainly over a dict ("Inference at
    Scale" 05: on a hash match a new request bumps the block's ref count and
    skips that part of prefill; only a shared beginning counts, so the first
    miss ends the match, "Chapter 31 Serving Efficiency" 31.3).

    key (lane 0, lane 1) -> [block id, ref count]."""

    def __init__(self):
        self.d = {}

    def lookup(self, hashes, lens, block_size, block_tables):
        """For each sequence the longest run of leading full blocks found;
        their ids go to block_tables[b][:n], each hit's ref count + 1.
        Returns n per sequence."""
        B = hashes.shape[0]
        n = np.zeros(B, np.int32)
        for b in range(B):
            nfull = min(int(lens[b]) // block_size, hashes.shape[1])
            j = 0
            while j < nfull and (int(hashes[b, j, 0]), int(hashes[b, j, 1])) in self.d:
                j += 1
            for i in range(j):
                e = self.d[(int(hashes[b, i, 0]), int(hashes[b, i, 1]))]
                e[1] += 1
                block_tables[b, i] = e[0]
            n[b] = j
        return n

    def insert(self, hashes, block_tables, first, count):
        """Register block_tables[b][j] under hashes[b][j] for j in
        [first[b], first[b] + count[b]).  A key already present keeps its block
        (the caller's block is a duplicate) and gains a reference; a key several
        sequences insert in the same call goes to one of them.  Returns the
        set of keys each (b, j) resolved to, for validation, and the ref counts."""
        claims = {}
        for b in range(hashes.shape[0]):
            for j in range(int(first[b]), int(first[b]) + int(count[b])):
                k = (int(hashes[b, j, 0]), int(hashes[b, j, 1]))
                claims.setdefault(k, []).append((b, j, int(block_tables[b, j])))
        for k, lst in claims.items():
            if k in self.d:
                self.d[k][1] += len(lst)
            else:
                self.d[k] = [None, len(lst)]   # block: any one of lst's (GPU: the first to claim)
                self.d[k].append([c[2] for c in lst])
        return claims

    def release(self, hashes, n):
        for b in range(hashes.shape[0]):
            for j in range(int(n[b])):
                self.d[(int(hashes[b, j, 0]), int(hashes[b, j, 1]))][1] -= 1
