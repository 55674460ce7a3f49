"""Full-size workloads on the GPU, checked on sampled sequences against the
oracle (which computes only the sampled rows) and with properties that hold at
any size.  Same launch configuration as bench.py for the batch-256 mix."""
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


def _sampled(w, out_bits, k, v, seqs):
    rows = np.concatenate([[0], np.cumsum(w.q_lens)])
    sel = np.concatenate([np.arange(rows[b], rows[b + 1]) for b in seqs])
    ref, st = oracle.attention(w.q[sel], k, v, w.block_tables[seqs], w.seq_lens[seqs], w.q_lens[seqs], w.scale)
    assert st == 0
    got = wl.bf16_bits_to_f32(out_bits[sel]).astype(np.float64)
    assert np.isfinite(got).all()
    err = np.abs(got - ref)
    assert np.all(err <= 1e-2 + 1e-2 * np.abs(ref)), f"max err {err.max():.3e}"


# partition lengths the automatic mode may pick from a floor of 512
AUTO_LADDER = {512, 768, 1024, 1536, 2048, 3072, 4096, 6144, 8192}


def _run(w, **kw):
    ds = DeviceStep(w, **kw)
    ds.step()
    torch.cuda.synchronize()
    assert int(ds.status.item()) == 0, pkv.status_bits(int(ds.status.item()))
    if ds.partition_tokens in (None, 0):
        # the length the planning kernel used is the int at byte offset 8 of the workspace
        used = int(ds.workspace[8:12].view(torch.int32).item())
        assert used in AUTO_LADDER, used
    return ds


def test_mix_batch256_full_size():
    w = wl.FULL["mix"]()
    ds = _run(w, max_seq_len=32768)       # the bench's configuration
    k, v, slots = _oracle_cache(w)
    assert np.array_equal(ds.slots.cpu().numpy(), slots)
    # caches bit-exact after copy-on-write and append (whole pool)
    assert np.array_equal(bf16_to_bits(ds.k_cache), k)
    assert np.array_equal(bf16_to_bits(ds.v_cache), v)
    out = bf16_to_bits(ds.out)
    L = w.seq_lens
    seqs = sorted(set([int(np.argmax(L)), int(np.argmin(L))] + list(range(0, 256, 23))
                      + w.meta["sharers"][:4]))
    _sampled(w, out, k, v, np.array(seqs))
    assert np.isfinite(wl.bf16_bits_to_f32(out)).all()
    # sequences with identical context and query would match; sharers with the
    # same length share every cached position except their own appended row
    # (property at full size: all rows finite, status clean -- checked above)


def test_decode_batch64_full_size():
    w = wl.FULL["decode"]()
    ds = _run(w)
    k, v, _ = _oracle_cache(w)
    out = bf16_to_bits(ds.out)
    _sampled(w, out, k, v, np.arange(0, 64, 9))


def test_spec_batch32_full_size():
    w = wl.FULL["spec"]()
    ds = _run(w)
    k, v, _ = _oracle_cache(w)
    out = bf16_to_bits(ds.out)
    _sampled(w, out, k, v, np.array([0, 7, 31]))
    acc, nxt, am = oracle.spec_accept_greedy(w.logits, w.draft)
    assert np.array_equal(ds.argmax.cpu().numpy(), am)
    assert np.array_equal(ds.accepted.cpu().numpy(), acc)
    assert np.array_equal(ds.next_token.cpu().numpy(), nxt)


def test_long_context_with_chunk_full_size():
    w = wl.FULL["long"]()
    ds = _run(w)
    out = bf16_to_bits(ds.out)
    assert np.isfinite(wl.bf16_bits_to_f32(out)).all()
    # oracle on one long decode and on sampled rows of the chunk
    k, v, _ = _oracle_cache(w)
    _sampled(w, out, k, v, np.array([3]))
    chunk = w.num_seqs - 1
    rows0 = int(w.q_lens[:chunk].sum())
    pick = np.array([0, 1, 255, 256, 511])
    ref, st = oracle.attention(w.q[rows0 + pick], k, v,
                               np.repeat(w.block_tables[chunk:chunk + 1], len(pick), 0),
                               (w.seq_lens[chunk] - w.q_lens[chunk] + pick + 1).astype(np.int32),
                               np.ones(len(pick), np.int32), w.scale)
    assert st == 0
    got = wl.bf16_bits_to_f32(out[rows0 + pick]).astype(np.float64)
    assert np.all(np.abs(got - ref) <= 1e-2 + 1e-2 * np.abs(ref))
