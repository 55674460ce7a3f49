"""The no-allocation attention entry point, for callers that cannot allocate
device memory on the call path (code inside another runtime's allocator or
pool hooks, latency-critical loops that must not block on the allocator,
plugins handed only their buffers).  It must give the same results as the
workspace entry point, call after call, using only the library's fixed
scratch array.  Collected last on purpose (tests/test_zz_*)."""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_23_gb300 as pkv
from paged_kv_cache_23_gb300 import workloads as wl
from paged_kv_cache_23_gb300.runner import DeviceStep, bf16_to_bits

pytestmark = pytest.mark.gpu


def _noalloc_call(ds, out, status):
    """pkv_paged_attention_decode_noalloc straight through the C ABI."""
    w = ds.w
    L = pkv.lib()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    return L.pkv_paged_attention_decode_noalloc(
        p(out), p(ds.q), p(ds.k_cache), p(ds.v_cache), p(ds.block_tables), w.max_blocks, p(ds.seq_lens),
        p(ds.q_lens), w.num_seqs, w.total_q, ds.max_q_len, ds.max_seq_len, w.n_q, w.n_kv, w.head_dim, w.block_size,
        w.num_blocks, ctypes.c_float(w.scale), ds.partition_tokens, ds.flags, p(status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def _oracle_out(w):
    """The oracle's attention output for the step (copy-on-write, append, attention)."""
    import oracle
    k = w.k_cache.copy()
    v = w.v_cache.copy()
    assert oracle.copy_blocks(k, v, w.cow) == 0
    slots, st = oracle.slot_mapping(w.block_tables, w.seq_lens, w.append_lens, w.block_size, w.num_blocks)
    assert st == 0
    assert oracle.kv_append(k, v, w.k_new, w.v_new, slots) == 0
    ref, st = oracle.attention(w.q, k, v, w.block_tables, w.seq_lens, w.q_lens, w.scale)
    assert st == 0
    return ref


def _check_same(ds):
    ds.cache_ops()
    ds.attention()                                  # workspace entry point
    ref = ds.out.clone()
    out = torch.full_like(ds.out, float("nan"))     # every row must be written
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = _noalloc_call(ds, out, status)
    assert rc == 0, pkv.lib().pkv_error_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0 and int(ds.status.item()) == 0
    # the same kernels on the same inputs: the outputs are identical bit for bit
    # (a tolerance would hide stale scratch that moves only the last bits)
    got = bf16_to_bits(out)
    assert np.array_equal(got, bf16_to_bits(ref))
    # and the oracle, element by element, within the attention tolerance
    a = wl.bf16_bits_to_f32(got).astype(np.float64)
    b = _oracle_out(ds.w)
    assert np.isfinite(a).all()
    assert np.all(np.abs(a - b) <= 1e-2 + 1e-2 * np.abs(b))


def test_noalloc_matches_workspace_entry_two_calls_in_a_row():
    pkv.build()
    # two different problems back to back: split partitions and multi-query
    # tiles on the first, plain decodes on the second, so state left in the
    # shared scratch by one call would show up in the next
    first = DeviceStep(wl.SMALL["long"](), partition_tokens=256)
    second = DeviceStep(wl.SMALL["mix"](), partition_tokens=64)
    need = [pkv.attention_workspace_bytes(d.w.num_seqs, d.w.total_q, d.w.n_q, d.w.n_kv, d.w.head_dim,
                                          d.max_seq_len, d.partition_tokens) for d in (first, second)]
    assert max(need) <= pkv.noalloc_scratch_bytes()
    _check_same(first)
    _check_same(second)


def test_noalloc_rejects_problems_beyond_its_scratch():
    ds = DeviceStep(wl.SMALL["decode"]())
    big = 32768                                    # 4096 sequences up to 32K tokens: GBs of scratch
    assert pkv.attention_workspace_bytes(4096, 4096, 32, 8, 128, big, 512) > pkv.noalloc_scratch_bytes()
    out = torch.empty_like(ds.out)
    L = pkv.lib()
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = L.pkv_paged_attention_decode_noalloc(
        p(out), p(ds.q), p(ds.k_cache), p(ds.v_cache), p(ds.block_tables), ds.w.max_blocks, p(ds.seq_lens),
        p(ds.q_lens), 4096, 4096, 1, big, 32, 8, 128, 16, ds.w.num_blocks, ctypes.c_float(0.1), 512, 0, None,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == pkv.PKV_ERR_SCRATCH_LIMIT
    assert b"scratch" in L.pkv_error_string(rc)
