"""Query tiles on the tcgen05 tensor cores vs the CPU oracle (GPU required).

A sequence with q_len * g > 8 (a prefill chunk, a verification) runs as
tiles of 128 (query, q head) rows of one kv head, with 128-token stages, the
scores and the output accumulated in tensor memory.  These cases cover every
head grouping whose g divides 128, ragged last tiles, prefixes that end inside
a block and inside a stage, several partition lengths (split-KV merge of tile
partials), block sizes from 16 to 256, NaN-poisoned cache rows past the
sequence end, bad block ids, and the same rows on the mma.sync path
(PKV_ATTN_NO_TCGEN05).  Tolerance as for every attention output:
|gpu - ref| <= 1e-2 + 1e-2 |ref|.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_23_gb300 as pkv
from paged_kv_cache_23_gb300 import workloads as wl
from paged_kv_cache_23_gb300.runner import DeviceStep, bf16_to_bits

from .test_gpu_parity import assert_close, run_and_check

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    pkv.build()
    torch.cuda.init()


def tiles_used(ds) -> int:
    """Workspace header int 3: 1 when the planning kernel made tcgen05 tiles."""
    return int(ds.workspace[:16].view(torch.int32)[3].item())


def chunk(n_q, n_kv, q_len, prefix, bs=16, decodes=1, ctx=300, P=0, seed=0):
    return wl.long_context(B=decodes, ctx=ctx, chunk=q_len, chunk_prefix=prefix, partition_tokens=P, seed=seed,
                           n_q=n_q, n_kv=n_kv, d=128, bs=bs)


@pytest.mark.parametrize("n_q,n_kv,q_len", [(8, 8, 200), (16, 8, 100), (32, 8, 75), (16, 2, 40), (32, 1, 9),
                                            (64, 1, 2)])
def test_head_groupings_on_tcgen05(n_q, n_kv, q_len):
    # g = 1, 2, 4, 8, 32, 64; the last tile of each sequence is ragged
    ds, _, _ = run_and_check(chunk(n_q, n_kv, q_len, prefix=777, seed=n_q + q_len))
    assert tiles_used(ds) == 1


@pytest.mark.parametrize("P", [128, 256, 640, 768, 0])
def test_partitions_of_tiles(P):
    # P = 128: one stage per partition; 640, 768: partitions of five and six
    # stages (768 is a step of the automatic ladder); 0: automatic
    w = chunk(32, 8, 70, prefix=1000, decodes=2, ctx=900, P=P, seed=P)
    ds, _, _ = run_and_check(w)
    assert tiles_used(ds) == 1


@pytest.mark.parametrize("bs", [16, 32, 64, 256])
def test_block_sizes_on_tcgen05(bs):
    ds, _, _ = run_and_check(chunk(32, 8, 40, prefix=500 + bs // 2, bs=bs, seed=bs))
    assert tiles_used(ds) == 1


@pytest.mark.parametrize("prefix,q_len", [(0, 32), (1, 32), (95, 33), (128, 32), (129, 160)])
def test_stage_edges(prefix, q_len):
    # chunks that start a sequence, end exactly on a stage, or one past it
    ds, _, _ = run_and_check(chunk(32, 8, q_len, prefix=prefix, seed=prefix + q_len), partition_tokens=128)
    assert tiles_used(ds) == 1


def test_partly_filled_tile_and_the_mma_sync_fallbacks():
    # q_len * g = 124 rows: one tile with 4 rows unused; block_size 8 boxes and
    # a partition that is not whole 128-token stages stay on mma.sync
    for w, P, tiles in ((chunk(32, 8, 31, prefix=300), 0, 1), (chunk(32, 8, 64, prefix=300, bs=8), 0, 0),
                        (chunk(32, 8, 64, prefix=300), 48, 0)):
        ds, _, _ = run_and_check(w, partition_tokens=P)
        assert tiles_used(ds) == tiles


def test_tcgen05_and_mma_sync_paths_agree():
    w = chunk(32, 8, 96, prefix=1500, decodes=3, ctx=2000, seed=5)
    a, ref, out_a = run_and_check(w)
    b, _, out_b = run_and_check(w, flags=pkv.PKV_ATTN_NO_TCGEN05)
    assert tiles_used(a) == 1 and tiles_used(b) == 0
    ga = wl.bf16_bits_to_f32(out_a).astype(np.float64)
    gb = wl.bf16_bits_to_f32(out_b).astype(np.float64)
    # both within the oracle's tolerance; against each other within twice it
    assert (np.abs(ga - gb) <= 2 * (1e-2 + 1e-2 * np.abs(ref["out"]))).all()


def test_medium_chunk_many_stages():
    # 256 queries over 2000 cached positions: 18 stages per tile at most
    ds, _, _ = run_and_check(chunk(32, 8, 256, prefix=2000, decodes=1, ctx=100, seed=9), partition_tokens=1024)
    assert tiles_used(ds) == 1


def test_repeated_tile_calls_are_deterministic():
    w = chunk(32, 8, 70, prefix=900, decodes=2, ctx=700, seed=3)
    ds = DeviceStep(w, partition_tokens=256)
    ds.step()
    a = bf16_to_bits(ds.out)
    for _ in range(3):
        ds.reset_cache()
        ds.step()
        assert np.array_equal(a, bf16_to_bits(ds.out))


def test_bad_block_in_a_tile_gives_nan_rows():
    w = chunk(32, 8, 64, prefix=600, decodes=2, ctx=400, seed=4)
    ds = DeviceStep(w, partition_tokens=256)
    ds.cache_ops()
    torch.cuda.synchronize()
    bt = w.block_tables.copy()
    chunk_seq = w.num_seqs - 1
    bt[chunk_seq, 20] = w.num_blocks + 3  # a block of the chunk's prefix
    ds.block_tables.copy_(torch.from_numpy(bt))
    ds.status.zero_()
    ds.attention()
    torch.cuda.synchronize()
    assert tiles_used(ds) == 1
    st = int(ds.status.item())
    assert st & pkv.PKV_STATUS_BAD_BLOCK and not st & pkv.PKV_STATUS_TIMEOUT
    out = wl.bf16_bits_to_f32(bf16_to_bits(ds.out))
    q0 = int(w.q_lens[:chunk_seq].sum())
    # every chunk query sees position 320 (block 20): all its rows are NaN
    assert np.isnan(out[q0:]).all()
    # the decode rows are untouched and correct
    k = w.k_cache.copy()
    v = w.v_cache.copy()
    slots, _ = oracle.slot_mapping(w.block_tables, w.seq_lens, w.append_lens, w.block_size, w.num_blocks)
    oracle.kv_append(k, v, w.k_new, w.v_new, slots)
    ref, _ = oracle.attention(w.q, k, v, w.block_tables, w.seq_lens, w.q_lens, w.scale)
    assert_close(bf16_to_bits(ds.out)[:q0], ref[:q0], "decode rows")


def test_q_len_above_the_host_bound_is_flagged():
    # max_q_len is a host bound: a longer q_len gives NaN rows and BAD_QLEN
    w = chunk(32, 8, 40, prefix=300, decodes=2, ctx=200, seed=6)
    ds = DeviceStep(w, partition_tokens=256)
    ds.cache_ops()
    ds.max_q_len = 39
    ds.status.zero_()
    ds.attention()
    torch.cuda.synchronize()
    st = int(ds.status.item())
    assert st & pkv.PKV_STATUS_BAD_QLEN
    out = wl.bf16_bits_to_f32(bf16_to_bits(ds.out))
    q0 = int(w.q_lens[:-1].sum())
    assert np.isnan(out[q0:]).all() and np.isfinite(out[:q0]).all()


def spec_w(n_q, n_kv, k, lo=200, hi=1500, B=4, bs=16, seed=0):
    return wl.spec(B=B, lo=lo, hi=hi, k=k, vocab=97, seed=seed, n_q=n_q, n_kv=n_kv, d=128, bs=bs)


def test_mixed_batch_of_row_kinds():
    # decode rows, speculative rows (mma.sync) and 128-row tcgen05 tiles in one launch
    a = wl.long_context(B=3, ctx=700, chunk=70, chunk_prefix=600, partition_tokens=256, seed=12, n_q=32, n_kv=8,
                        d=128, bs=16)
    b = spec_w(32, 8, 5, lo=100, hi=900, B=3, seed=13)
    # concatenate the two workloads' sequences over one pool
    ds, _, _ = run_and_check(wl.concat(a, b))
    assert tiles_used(ds) == 1


def test_back_to_back_tile_launches_never_time_out():
    # hundreds of launches with many short tile items per CTA: the MMA warp's
    # barriers must never see a phase run ahead of it (a bounded wait would
    # give up and set PKV_STATUS_TIMEOUT)
    w = chunk(32, 8, 256, prefix=3000, decodes=8, ctx=4000, seed=15)
    ds = DeviceStep(w, partition_tokens=128)
    ds.cache_ops()
    ds.status.zero_()
    for _ in range(300):
        ds.attention()
    torch.cuda.synchronize()
    assert tiles_used(ds) == 1
    assert int(ds.status.item()) == 0, pkv.status_bits(int(ds.status.item()))
