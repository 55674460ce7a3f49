"""Full-size workloads on the GPU, every output row checked element by element
against the oracle (fp64, OpenMP over sequences: about 0.3 s for the batch-256
mix and under half a minute for the long-context workload on 16 cores), the
caches bit-exact over the whole pool.  Same launch configuration as bench.py."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_23_gb300 as pkv
from paged_kv_cache_23_gb300 import workloads as wl
from paged_kv_cache_23_gb300.runner import DeviceStep, bf16_to_bits

pytestmark = pytest.mark.gpu


def _oracle_cache(w):
    k = w.k_cache.copy()
    v = w.v_cache.copy()
    assert oracle.copy_blocks(k, v, w.cow) == 0
    slots, st = oracle.slot_mapping(w.block_tables, w.seq_lens, w.append_lens, w.block_size, w.num_blocks)
    assert st == 0
    assert oracle.kv_append(k, v, w.k_new, w.v_new, slots) == 0
    return k, v, slots


def _all_rows(w, out_bits, k, v):
    """Every query row of every sequence against the oracle."""
    ref, st = oracle.attention(w.q, k, v, w.block_tables, w.seq_lens, w.q_lens, w.scale)
    assert st == 0
    got = wl.bf16_bits_to_f32(out_bits).astype(np.float64)
    assert got.shape == ref.shape
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    bad = err > 1e-2 + 1e-2 * np.abs(ref)
    assert not bad.any(), f"{bad.sum()} of {bad.size} outside tolerance, max err {err.max():.3e}"
    return float(err.max())


def _auto_target_ok(used: int) -> bool:
    """The automatic mode's target item length: whole 16-token stages, from the
    floor of 512 up to 8192 (each sequence is cut into equal partitions of
    about this length)."""
    return used % 16 == 0 and 512 <= used <= 8192


def _run(w, **kw):
    ds = DeviceStep(w, **kw)
    ds.step()
    torch.cuda.synchronize()
    assert int(ds.status.item()) == 0, pkv.status_bits(int(ds.status.item()))
    if ds.partition_tokens in (None, 0):
        # the length the planning kernel used is the int at byte offset 8 of the workspace
        used = int(ds.workspace[8:12].view(torch.int32).item())
        assert _auto_target_ok(used), used
    return ds


def test_mix_batch256_full_size():
    w = wl.FULL["mix"]()
    ds = _run(w, max_seq_len=32768)       # the bench's configuration
    k, v, slots = _oracle_cache(w)
    assert np.array_equal(ds.slots.cpu().numpy(), slots)
    # caches bit-exact after copy-on-write and append (whole pool)
    assert np.array_equal(bf16_to_bits(ds.k_cache), k)
    assert np.array_equal(bf16_to_bits(ds.v_cache), v)
    _all_rows(w, bf16_to_bits(ds.out), k, v)    # all 256 sequences, 32 heads, 128 dims


def test_decode_batch64_full_size():
    w = wl.FULL["decode"]()
    ds = _run(w)
    k, v, _ = _oracle_cache(w)
    assert np.array_equal(bf16_to_bits(ds.k_cache), k) and np.array_equal(bf16_to_bits(ds.v_cache), v)
    _all_rows(w, bf16_to_bits(ds.out), k, v)    # all 64 sequences


def test_spec_batch32_full_size():
    w = wl.FULL["spec"]()
    ds = _run(w)
    k, v, _ = _oracle_cache(w)
    assert np.array_equal(bf16_to_bits(ds.k_cache), k) and np.array_equal(bf16_to_bits(ds.v_cache), v)
    _all_rows(w, bf16_to_bits(ds.out), k, v)    # all 32 x 5 query rows
    acc, nxt, am = oracle.spec_accept_greedy(w.logits, w.draft)
    assert np.array_equal(ds.argmax.cpu().numpy(), am)
    assert np.array_equal(ds.accepted.cpu().numpy(), acc)
    assert np.array_equal(ds.next_token.cpu().numpy(), nxt)


def test_long_context_with_chunk_full_size():
    w = wl.FULL["long"]()
    ds = _run(w)
    k, v, _ = _oracle_cache(w)
    assert np.array_equal(bf16_to_bits(ds.k_cache), k) and np.array_equal(bf16_to_bits(ds.v_cache), v)
    # all 8 decodes of 131072 positions and all 512 rows of the chunk
    _all_rows(w, bf16_to_bits(ds.out), k, v)
