"""paged_kv_cache_23_gb300 -- paged-KV decode attention for GB300 (sm_103a).

A thin ctypes binding over ``libpkv.so`` (C ABI in ``include/pkv.h``).  The
functions here only marshal torch tensors (device pointers, sizes, the current
CUDA stream) into the C calls; every step of the path runs in the library's
CUDA kernels.  There is no CPU fallback: if the library is missing or the
device is not a GB300, calls raise.

Entry points (same names as the C ABI without the ``pkv_`` prefix):
    slot_mapping, kv_append, kv_append_paged, copy_blocks, gather_kv,
    attention_auto_partition, attention_workspace_bytes,
    paged_attention_decode, attention_plan, paged_attention_run,
    spec_accept_greedy, spec_accept_sample, the e4m3 variants, the prefix
    cache and the no-allocation attention
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpkv.so")
_lock = threading.Lock()
_lib = None

PKV_STATUS_BAD_BLOCK = 1
PKV_STATUS_BAD_SEQLEN = 2
PKV_STATUS_BAD_QLEN = 4
PKV_STATUS_BAD_SLOT = 8
PKV_STATUS_TIMEOUT = 32
PKV_STATUS_BAD_PAIR = 64
PKV_STATUS_BAD_TOKEN = 128
PKV_STATUS_BAD_DIST = 256
PKV_STATUS_TABLE_FULL = 512
PKV_STATUS_NOT_FOUND = 1024
PKV_STATUS_BAD_PLAN = 2048
PKV_ATTN_DECODE_CUDA_CORES = 1
PKV_ATTN_NO_TCGEN05 = 2  # multi-query tiles on mma.sync instead of tcgen05
PKV_ATTN_PLAN_FP8 = 4    # attention_plan only: the runs are over FP8 pools
PKV_FP8_E4M3, PKV_FP8_E5M2 = 0, 1
PKV_FP8_SCALE_PER_HEAD, PKV_FP8_SCALE_PER_BLOCK = 0, 1
PKV_ERR_SCRATCH_LIMIT = -8

_P = ctypes.c_void_p
_I = ctypes.c_int
_SIGS = {
    "pkv_version": ([], _I),
    "pkv_error_string": ([_I], ctypes.c_char_p),
    "pkv_status_string": ([_I], ctypes.c_char_p),
    "pkv_slot_mapping": ([_P, _P, _I, _P, _P, _I, _I, _I, _I, _P, _P], _I),
    "pkv_kv_append": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P], _I),
    "pkv_copy_blocks": ([_P, _P, _P, _I, _I, _I, _I, _I, _P, _P], _I),
    "pkv_gather_kv": ([_P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _P, _P], _I),
    "pkv_attention_auto_partition": ([_I, _I, _I, _I], _I),
    "pkv_attention_workspace_bytes": ([_I, _I, _I, _I, _I, _I, _I], ctypes.c_size_t),
    "pkv_paged_attention_decode": ([_P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                                    ctypes.c_float, _I, _I, _P, ctypes.c_size_t, _P, _P], _I),
    "pkv_spec_accept_greedy": ([_P, _P, _I, _I, _I, _P, _P, _P, _P], _I),
    "pkv_spec_accept_sample": ([_P, _P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _P], _I),
    "pkv_prefix_table_bytes": ([_I], ctypes.c_size_t),
    "pkv_prefix_table_init": ([_P, _I, _P], _I),
    "pkv_prefix_hash": ([_P, _P, _I, _P, _I, _I, _I, ctypes.c_uint64, _P], _I),
    "pkv_prefix_lookup": ([_P, _I, _P, _P, _I, _I, _I, _P, _P, _P], _I),
    "pkv_prefix_insert": ([_P, _I, _P, _P, _P, _P, _I, _I, _P, _P, _P], _I),
    "pkv_prefix_release": ([_P, _I, _P, _P, _I, _I, _P, _P], _I),
    "pkv_kv_append_paged": ([_P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P, _P], _I),
    "pkv_kv_append_fp8": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P], _I),
    "pkv_copy_blocks_fp8": ([_P, _P, _P, _I, _I, _I, _I, _I, _P, _P], _I),
    "pkv_paged_attention_decode_fp8": ([_P, _P, _P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                                        _I, ctypes.c_float, _I, _P, ctypes.c_size_t, _P, _P], _I),
    "pkv_attention_plan": ([_P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, ctypes.c_size_t, _P, _P], _I),
    "pkv_paged_attention_run": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float, _I, _I,
                                 _P, ctypes.c_size_t, _P, _P], _I),
    "pkv_paged_attention_run_fp8": ([_P, _P, _P, _P, _P, _P, _I, _I, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                                     ctypes.c_float, _I, _P, ctypes.c_size_t, _P, _P], _I),
    "pkv_kv_append_fp8_ex": ([_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P, _P], _I),
    "pkv_copy_blocks_fp8_ex": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P, _P], _I),
    "pkv_paged_attention_decode_fp8_ex": ([_P, _P, _P, _P, _P, _P, _I, _I, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I,
                                           _I, _I, _I, ctypes.c_float, _I, _P, ctypes.c_size_t, _P, _P], _I),
    "pkv_noalloc_scratch_bytes": ([], ctypes.c_size_t),
    "pkv_wait_selftest": ([ctypes.c_longlong, _P, _P], _I),
    "pkv_paged_attention_decode_noalloc": ([_P, _P, _P, _P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                                            ctypes.c_float, _I, _I, _P, _P], _I),
}


def build(force: bool = False) -> str:
    from . import _build
    return _build.build(force=force)


def lib():
    """The loaded libpkv.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libpkv.so is not built ({LIB_PATH}); run __graft_entry__.build() "
                                   "or python -m paged_kv_cache_23_gb300._build")
            L = ctypes.CDLL(LIB_PATH)
            for name, (argt, rest) in _SIGS.items():
                f = getattr(L, name)
                f.argtypes = argt
                f.restype = rest
            _lib = L
    return _lib


class PkvError(RuntimeError):
    pass


def _check(rc: int, what: str):
    if rc != 0:
        msg = lib().pkv_error_string(rc).decode()
        raise PkvError(f"{what}: {msg} (code {rc})")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _dev(t, name, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise PkvError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise PkvError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise PkvError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def status_bits(code: int):
    return [lib().pkv_status_string(1 << i).decode() for i in range(12) if code & (1 << i)]


def slot_mapping(slots, block_tables, seq_lens, append_lens, block_size, num_blocks, status=None, stream=None):
    """a1: slots[int64, sum(append_lens)] of each sequence's last append_lens[b] positions."""
    _dev(slots, "slots", torch.int64)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    _dev(append_lens, "append_lens", torch.int32)
    rc = lib().pkv_slot_mapping(_ptr(slots), _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
                                _ptr(append_lens), seq_lens.numel(), slots.numel(), block_size, num_blocks,
                                _ptr(status), _stream(stream))
    _check(rc, "pkv_slot_mapping")


def kv_append(k_cache, v_cache, k_new, v_new, slots, status=None, stream=None):
    """a2: write k_new/v_new [T][n_kv][d] (bf16) into the cache rows given by slots."""
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache), ("k_new", k_new), ("v_new", v_new)):
        _dev(t, n, torch.bfloat16)
    _dev(slots, "slots", torch.int64)
    nb, nkv, bs, d = k_cache.shape
    rc = lib().pkv_kv_append(_ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new), _ptr(slots), slots.numel(), nb,
                             bs, nkv, d, _ptr(status), _stream(stream))
    _check(rc, "pkv_kv_append")


def kv_append_paged(k_cache, v_cache, k_new, v_new, block_tables, seq_lens, append_lens, slots, status=None,
                    stream=None):
    """a1 + a2 in one launch: slot mapping fused with the append; slots receives the slots."""
    for n, t in (("k_cache", k_cache), ("v_cache", v_cache), ("k_new", k_new), ("v_new", v_new)):
        _dev(t, n, torch.bfloat16)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    _dev(append_lens, "append_lens", torch.int32)
    _dev(slots, "slots", torch.int64)
    nb, nkv, bs, d = k_cache.shape
    rc = lib().pkv_kv_append_paged(_ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new), _ptr(block_tables),
                                   block_tables.shape[1], _ptr(seq_lens), _ptr(append_lens), seq_lens.numel(),
                                   slots.numel(), nb, bs, nkv, d, _ptr(slots), _ptr(status), _stream(stream))
    _check(rc, "pkv_kv_append_paged")


def copy_blocks(k_cache, v_cache, src_dst, status=None, stream=None):
    """a3: copy-on-write block copies, src_dst int32 [n][2]."""
    _dev(k_cache, "k_cache", torch.bfloat16)
    _dev(v_cache, "v_cache", torch.bfloat16)
    _dev(src_dst, "src_dst", torch.int32)
    nb, nkv, bs, d = k_cache.shape
    rc = lib().pkv_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(src_dst), src_dst.numel() // 2, nb, bs, nkv, d,
                               _ptr(status), _stream(stream))
    _check(rc, "pkv_copy_blocks")


def gather_kv(k_out, v_out, k_cache, v_cache, block_tables, seq_lens, out_offsets, status=None, stream=None):
    """a4 as a utility: contiguous [sum seq_len][n_kv][d] K/V through the block table."""
    for n, t in (("k_out", k_out), ("v_out", v_out), ("k_cache", k_cache), ("v_cache", v_cache)):
        _dev(t, n, torch.bfloat16)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    _dev(out_offsets, "out_offsets", torch.int64)
    nb, nkv, bs, d = k_cache.shape
    rc = lib().pkv_gather_kv(_ptr(k_out), _ptr(v_out), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                             block_tables.shape[1], _ptr(seq_lens), _ptr(out_offsets), seq_lens.numel(), nb, bs, nkv,
                             d, _ptr(status), _stream(stream))
    _check(rc, "pkv_gather_kv")


def attention_auto_partition(num_seqs, total_q, num_kv_heads, max_seq_len) -> int:
    return int(lib().pkv_attention_auto_partition(num_seqs, total_q, num_kv_heads, max_seq_len))


def attention_workspace_bytes(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim, max_seq_len,
                              partition_tokens=0) -> int:
    return int(lib().pkv_attention_workspace_bytes(num_seqs, total_q, num_q_heads, num_kv_heads, head_dim,
                                                   max_seq_len, partition_tokens))


def _max_q(max_q_len, total_q) -> int:
    return int(total_q if max_q_len is None else max_q_len)


def paged_attention_decode(out, q, k_cache, v_cache, block_tables, seq_lens, q_lens, max_seq_len, scale,
                           workspace, partition_tokens=0, flags=0, status=None, stream=None, max_q_len=None):
    """a4-a8: paged attention (decode, speculative verify, prefill chunks) into out [total_q][n_q][d].
    max_q_len: host bound on every q_len (default total_q, always valid)."""
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _dev(t, n, torch.bfloat16)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    _dev(q_lens, "q_lens", torch.int32)
    _dev(workspace, "workspace")
    nb, nkv, bs, d = k_cache.shape
    total_q, nq, _ = q.shape
    rc = lib().pkv_paged_attention_decode(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                          block_tables.shape[1], _ptr(seq_lens), _ptr(q_lens), seq_lens.numel(),
                                          total_q, _max_q(max_q_len, total_q), int(max_seq_len), nq, nkv, d, bs,
                                          nb, float(scale), int(partition_tokens), int(flags), _ptr(workspace),
                                          workspace.numel() * workspace.element_size(), _ptr(status),
                                          _stream(stream))
    _check(rc, "pkv_paged_attention_decode")


def attention_plan(seq_lens, q_lens, total_q, max_blocks, num_q_heads, num_kv_heads, head_dim, block_size,
                   max_seq_len, workspace, partition_tokens=0, flags=0, status=None, stream=None, max_q_len=None):
    """The planning half of paged_attention_decode: the work list for these
    lengths, written into workspace, for any number of paged_attention_run calls."""
    _dev(seq_lens, "seq_lens", torch.int32)
    _dev(q_lens, "q_lens", torch.int32)
    _dev(workspace, "workspace")
    rc = lib().pkv_attention_plan(_ptr(seq_lens), _ptr(q_lens), seq_lens.numel(), int(total_q),
                                  _max_q(max_q_len, total_q), int(max_seq_len), int(max_blocks), int(num_q_heads),
                                  int(num_kv_heads), int(head_dim), int(block_size), int(partition_tokens),
                                  int(flags), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                  _ptr(status), _stream(stream))
    _check(rc, "pkv_attention_plan")


def paged_attention_run(out, q, k_cache, v_cache, block_tables, num_seqs, max_seq_len, scale, workspace,
                        partition_tokens=0, flags=0, status=None, stream=None, max_q_len=None):
    """The attention half of paged_attention_decode over a planned workspace."""
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _dev(t, n, torch.bfloat16)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(workspace, "workspace")
    nb, nkv, bs, d = k_cache.shape
    total_q, nq, _ = q.shape
    rc = lib().pkv_paged_attention_run(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                                       block_tables.shape[1], int(num_seqs), total_q, _max_q(max_q_len, total_q),
                                       int(max_seq_len), nq, nkv, d, bs, nb, float(scale), int(partition_tokens),
                                       int(flags), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _ptr(status), _stream(stream))
    _check(rc, "pkv_paged_attention_run")


def paged_attention_run_fp8(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, num_seqs, max_seq_len, scale,
                            workspace, partition_tokens=0, status=None, stream=None, max_q_len=None,
                            kv_format=PKV_FP8_E4M3, scale_mode=PKV_FP8_SCALE_PER_HEAD):
    """paged_attention_run over FP8 pools (plan made with PKV_ATTN_PLAN_FP8)."""
    _dev(out, "out", torch.bfloat16)
    _dev(q, "q", torch.bfloat16)
    _dev(k_cache, "k_cache", torch.uint8)
    _dev(v_cache, "v_cache", torch.uint8)
    _dev(k_scale, "k_scale", torch.float32)
    _dev(v_scale, "v_scale", torch.float32)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(workspace, "workspace")
    nb, nkv, bs, d = k_cache.shape
    total_q, nq, _ = q.shape
    rc = lib().pkv_paged_attention_run_fp8(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                           _ptr(v_scale), int(kv_format), int(scale_mode), _ptr(block_tables),
                                           block_tables.shape[1], int(num_seqs),
                                           total_q, _max_q(max_q_len, total_q), int(max_seq_len), nq, nkv, d, bs, nb,
                                           float(scale), int(partition_tokens), _ptr(workspace),
                                           workspace.numel() * workspace.element_size(), _ptr(status),
                                           _stream(stream))
    _check(rc, "pkv_paged_attention_run_fp8")


def spec_accept_greedy(logits, draft, argmax_out, accepted, next_token, stream=None):
    """a9: greedy acceptance; logits fp32 [B][k+1][V], draft int32 [B][k]."""
    _dev(logits, "logits", torch.float32)
    _dev(draft, "draft", torch.int32)
    _dev(argmax_out, "argmax_out", torch.int32)
    _dev(accepted, "accepted", torch.int32)
    _dev(next_token, "next_token", torch.int32)
    B, k1, V = logits.shape
    rc = lib().pkv_spec_accept_greedy(_ptr(logits), _ptr(draft), B, k1 - 1, V, _ptr(argmax_out), _ptr(accepted),
                                      _ptr(next_token), _stream(stream))
    _check(rc, "pkv_spec_accept_greedy")


class PrefixTable:
    """A prefix-cache table in device memory (see pkv.h: chained 128-bit
    block keys, open addressing, 32-byte entries)."""

    def __init__(self, capacity: int, device="cuda", stream=None):
        self.capacity = int(capacity)
        nbytes = int(lib().pkv_prefix_table_bytes(self.capacity))
        if nbytes == 0:
            raise ValueError("capacity must be a power of two")
        self.buf = torch.empty(nbytes, dtype=torch.uint8, device=device)
        _check(lib().pkv_prefix_table_init(_ptr(self.buf), self.capacity, _stream(stream)), "pkv_prefix_table_init")

    def entries(self):
        """(keys uint64 [cap][2], block int32 [cap], refs int32 [cap]) on the host."""
        raw = self.buf.view(torch.int64).view(self.capacity, 4).cpu()
        keys = raw[:, :2].numpy().view("uint64")
        br = raw[:, 2:3].contiguous().view(torch.int32).view(self.capacity, 2).numpy()
        return keys, br[:, 0], br[:, 1]


def prefix_hash(hashes, tokens, lens, block_size, salt=0, stream=None):
    """hashes uint64-as-int64 [B][max_blocks][2] out; tokens int32 [B][T]; lens int32 [B]."""
    _dev(hashes, "hashes", torch.int64)
    _dev(tokens, "tokens", torch.int32)
    _dev(lens, "lens", torch.int32)
    B, T = tokens.shape
    rc = lib().pkv_prefix_hash(_ptr(hashes), _ptr(tokens), T, _ptr(lens), B, block_size, hashes.shape[1],
                               ctypes.c_uint64(salt & (2 ** 64 - 1)), _stream(stream))
    _check(rc, "pkv_prefix_hash")


def prefix_lookup(table, hashes, lens, block_size, block_tables, cached_blocks, stream=None):
    _dev(hashes, "hashes", torch.int64)
    _dev(lens, "lens", torch.int32)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(cached_blocks, "cached_blocks", torch.int32)
    B, MB, _ = hashes.shape
    rc = lib().pkv_prefix_lookup(_ptr(table.buf), table.capacity, _ptr(hashes), _ptr(lens), B, block_size, MB,
                                 _ptr(block_tables), _ptr(cached_blocks), _stream(stream))
    _check(rc, "pkv_prefix_lookup")


def prefix_insert(table, hashes, block_tables, first, count, resolved, status=None, stream=None):
    for n, t in (("block_tables", block_tables), ("first", first), ("count", count), ("resolved", resolved)):
        _dev(t, n, torch.int32)
    _dev(hashes, "hashes", torch.int64)
    B, MB, _ = hashes.shape
    rc = lib().pkv_prefix_insert(_ptr(table.buf), table.capacity, _ptr(hashes), _ptr(block_tables), _ptr(first),
                                 _ptr(count), B, MB, _ptr(resolved), _ptr(status), _stream(stream))
    _check(rc, "pkv_prefix_insert")


def prefix_release(table, hashes, count, status=None, stream=None):
    _dev(hashes, "hashes", torch.int64)
    _dev(count, "count", torch.int32)
    B, MB, _ = hashes.shape
    rc = lib().pkv_prefix_release(_ptr(table.buf), table.capacity, _ptr(hashes), _ptr(count), B, MB, _ptr(status),
                                  _stream(stream))
    _check(rc, "pkv_prefix_release")


def kv_append_fp8(k_cache, v_cache, k_new, v_new, slots, k_scale, v_scale, status=None, stream=None):
    """Append bf16 rows into e4m3 pools (uint8 [nb][n_kv][bs][d]) with per-head scales."""
    _dev(k_cache, "k_cache", torch.uint8)
    _dev(v_cache, "v_cache", torch.uint8)
    _dev(k_new, "k_new", torch.bfloat16)
    _dev(v_new, "v_new", torch.bfloat16)
    _dev(slots, "slots", torch.int64)
    _dev(k_scale, "k_scale", torch.float32)
    _dev(v_scale, "v_scale", torch.float32)
    nb, nkv, bs, d = k_cache.shape
    rc = lib().pkv_kv_append_fp8(_ptr(k_cache), _ptr(v_cache), _ptr(k_new), _ptr(v_new), _ptr(slots), _ptr(k_scale),
                                 _ptr(v_scale), slots.numel(), nb, bs, nkv, d, _ptr(status), _stream(stream))
    _check(rc, "pkv_kv_append_fp8")


def copy_blocks_fp8(k_cache, v_cache, src_dst, status=None, stream=None):
    _dev(k_cache, "k_cache", torch.uint8)
    _dev(v_cache, "v_cache", torch.uint8)
    _dev(src_dst, "src_dst", torch.int32)
    nb, nkv, bs, d = k_cache.shape
    rc = lib().pkv_copy_blocks_fp8(_ptr(k_cache), _ptr(v_cache), _ptr(src_dst), src_dst.shape[0], nb, bs, nkv, d,
                                   _ptr(status), _stream(stream))
    _check(rc, "pkv_copy_blocks_fp8")


def paged_attention_decode_fp8(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens, q_lens,
                               max_seq_len, scale, workspace, partition_tokens=0, status=None, stream=None,
                               max_q_len=None):
    """Paged attention over e4m3 pools (uint8 [nb][n_kv][bs][d]) with per-kv-head scales."""
    _dev(out, "out", torch.bfloat16)
    _dev(q, "q", torch.bfloat16)
    _dev(k_cache, "k_cache", torch.uint8)
    _dev(v_cache, "v_cache", torch.uint8)
    _dev(k_scale, "k_scale", torch.float32)
    _dev(v_scale, "v_scale", torch.float32)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    _dev(q_lens, "q_lens", torch.int32)
    _dev(workspace, "workspace")
    nb, nkv, bs, d = k_cache.shape
    total_q, nq, _ = q.shape
    rc = lib().pkv_paged_attention_decode_fp8(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                              _ptr(v_scale), _ptr(block_tables), block_tables.shape[1],
                                              _ptr(seq_lens), _ptr(q_lens), seq_lens.numel(), total_q,
                                              _max_q(max_q_len, total_q), int(max_seq_len), nq, nkv, d, bs, nb,
                                              float(scale),
                                              int(partition_tokens), _ptr(workspace),
                                              workspace.numel() * workspace.element_size(), _ptr(status),
                                              _stream(stream))
    _check(rc, "pkv_paged_attention_decode_fp8")


def _fp8_args(k_cache, v_cache, k_scale, v_scale):
    _dev(k_cache, "k_cache", torch.uint8)
    _dev(v_cache, "v_cache", torch.uint8)
    _dev(k_scale, "k_scale", torch.float32)
    _dev(v_scale, "v_scale", torch.float32)


def kv_append_fp8_ex(k_cache, v_cache, k_scale, v_scale, k_new, v_new, slots, kv_format=PKV_FP8_E4M3,
                     scale_mode=PKV_FP8_SCALE_PER_HEAD, status=None, stream=None):
    """Quantising append into FP8 pools of either format; with per-block scales
    ([num_blocks][n_kv]) the blocks this call opens get their scales set."""
    _fp8_args(k_cache, v_cache, k_scale, v_scale)
    _dev(k_new, "k_new", torch.bfloat16)
    _dev(v_new, "v_new", torch.bfloat16)
    _dev(slots, "slots", torch.int64)
    nb, nkv, bs, d = k_cache.shape
    rc = lib().pkv_kv_append_fp8_ex(_ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(k_new),
                                    _ptr(v_new), _ptr(slots), slots.numel(), nb, bs, nkv, d, int(kv_format),
                                    int(scale_mode), _ptr(status), _stream(stream))
    _check(rc, "pkv_kv_append_fp8_ex")


def copy_blocks_fp8_ex(k_cache, v_cache, k_scale, v_scale, src_dst, scale_mode=PKV_FP8_SCALE_PER_HEAD, status=None,
                       stream=None):
    """Copy-on-write block copies in FP8 pools (and the blocks' scales with per-block scales)."""
    _fp8_args(k_cache, v_cache, k_scale, v_scale)
    _dev(src_dst, "src_dst", torch.int32)
    nb, nkv, bs, d = k_cache.shape
    rc = lib().pkv_copy_blocks_fp8_ex(_ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), _ptr(src_dst),
                                      src_dst.shape[0], nb, bs, nkv, d, int(scale_mode), _ptr(status),
                                      _stream(stream))
    _check(rc, "pkv_copy_blocks_fp8_ex")


def paged_attention_decode_fp8_ex(out, q, k_cache, v_cache, k_scale, v_scale, block_tables, seq_lens, q_lens,
                                  max_seq_len, scale, workspace, kv_format=PKV_FP8_E4M3,
                                  scale_mode=PKV_FP8_SCALE_PER_HEAD, partition_tokens=0, status=None, stream=None,
                                  max_q_len=None):
    """Paged attention over FP8 pools of either format and scale granularity."""
    _dev(out, "out", torch.bfloat16)
    _dev(q, "q", torch.bfloat16)
    _fp8_args(k_cache, v_cache, k_scale, v_scale)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    _dev(q_lens, "q_lens", torch.int32)
    _dev(workspace, "workspace")
    nb, nkv, bs, d = k_cache.shape
    total_q, nq, _ = q.shape
    rc = lib().pkv_paged_attention_decode_fp8_ex(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale),
                                                 _ptr(v_scale), int(kv_format), int(scale_mode), _ptr(block_tables),
                                                 block_tables.shape[1], _ptr(seq_lens), _ptr(q_lens),
                                                 seq_lens.numel(), total_q, _max_q(max_q_len, total_q),
                                                 int(max_seq_len), nq, nkv, d, bs, nb, float(scale),
                                                 int(partition_tokens), _ptr(workspace),
                                                 workspace.numel() * workspace.element_size(), _ptr(status),
                                                 _stream(stream))
    _check(rc, "pkv_paged_attention_decode_fp8_ex")


def spec_accept_sample(p, q, draft, r, s, accepted, next_token, status=None, stream=None):
    """Stochastic acceptance (modified rejection sampling): p fp32 [B][k+1][V],
    q fp32 [B][k][V], draft int32 [B][k], uniforms r fp32 [B][k] and s fp32 [B]."""
    _dev(p, "p", torch.float32)
    _dev(q, "q", torch.float32)
    _dev(draft, "draft", torch.int32)
    _dev(r, "r", torch.float32)
    _dev(s, "s", torch.float32)
    _dev(accepted, "accepted", torch.int32)
    _dev(next_token, "next_token", torch.int32)
    B, k1, V = p.shape
    if tuple(q.shape) != (B, k1 - 1, V) or tuple(draft.shape) != (B, k1 - 1) or tuple(r.shape) != (B, k1 - 1):
        raise ValueError("spec_accept_sample: q [B][k][V], draft and r [B][k] must match p [B][k+1][V]")
    rc = lib().pkv_spec_accept_sample(_ptr(p), _ptr(q), _ptr(draft), _ptr(r), _ptr(s), B, k1 - 1, V, _ptr(accepted),
                                      _ptr(next_token), _ptr(status), _stream(stream))
    _check(rc, "pkv_spec_accept_sample")


def paged_attention_decode_noalloc(out, q, k_cache, v_cache, block_tables, seq_lens, q_lens, max_seq_len, scale,
                                   partition_tokens=0, flags=0, status=None, stream=None, max_q_len=None):
    """paged_attention_decode without a workspace: for callers that cannot
    allocate device memory; the scratch is the library's fixed device array
    (noalloc_scratch_bytes()).  Calls overlapping on the GPU race on it."""
    for n, t in (("out", out), ("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        _dev(t, n, torch.bfloat16)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(seq_lens, "seq_lens", torch.int32)
    _dev(q_lens, "q_lens", torch.int32)
    nb, nkv, bs, d = k_cache.shape
    total_q, nq, _ = q.shape
    rc = lib().pkv_paged_attention_decode_noalloc(_ptr(out), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                                  _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens),
                                                  _ptr(q_lens), seq_lens.numel(), total_q,
                                                  _max_q(max_q_len, total_q), int(max_seq_len), nq, nkv,
                                                  d, bs, nb, float(scale), int(partition_tokens), int(flags),
                                                  _ptr(status), _stream(stream))
    _check(rc, "pkv_paged_attention_decode_noalloc")


def noalloc_scratch_bytes() -> int:
    return int(lib().pkv_noalloc_scratch_bytes())


def wait_selftest(limit_ns: int, status, stream=None):
    """Failure-detection self-test: a device wait on a flag that nothing sets
    must give up after limit_ns and set PKV_STATUS_TIMEOUT in status."""
    _dev(status, "status", torch.int32)
    _check(lib().pkv_wait_selftest(int(limit_ns), _ptr(status), _stream(stream)), "pkv_wait_selftest")
