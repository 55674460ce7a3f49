"""CUDA path vs the CPU oracle, element by element (GPU required).

Bit-exact for slot mapping, KV append, copy-on-write copies, gather and the
acceptance integers; attention outputs within |gpu - ref| <= 1e-2 + 1e-2*|ref|
(bf16 in, fp32 accumulate, bf16 out), the stated tolerance of the attention outputs.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_23_gb300 as pkv
from paged_kv_cache_23_gb300 import workloads as wl
from paged_kv_cache_23_gb300.runner import DeviceStep, bf16_to_bits, to_device_bf16

pytestmark = pytest.mark.gpu

ATOL = 1e-2
RTOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    pkv.build()
    torch.cuda.init()


def oracle_step(w):
    k = w.k_cache.copy()
    v = w.v_cache.copy()
    st = oracle.copy_blocks(k, v, w.cow)
    slots, st1 = oracle.slot_mapping(w.block_tables, w.seq_lens, w.append_lens, w.block_size, w.num_blocks)
    st2 = oracle.kv_append(k, v, w.k_new, w.v_new, slots)
    out, st3 = oracle.attention(w.q, k, v, w.block_tables, w.seq_lens, w.q_lens, w.scale)
    return dict(k=k, v=v, slots=slots, out=out, status=st | st1 | st2 | st3)


def assert_close(gpu_bits, ref, what=""):
    g = wl.bf16_bits_to_f32(gpu_bits).astype(np.float64)
    assert np.isfinite(g).all(), f"{what}: non-finite GPU output"
    err = np.abs(g - ref)
    bound = ATOL + RTOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} of {bad.size} outside tolerance, max err {err.max():.3e}"


def run_and_check(w, partition_tokens=None, flags=0, max_seq_len=None):
    ref = oracle_step(w)
    assert ref["status"] == 0
    ds = DeviceStep(w, max_seq_len=max_seq_len, partition_tokens=partition_tokens, flags=flags)
    ds.step()
    torch.cuda.synchronize()
    assert int(ds.status.item()) == 0, pkv.status_bits(int(ds.status.item()))
    assert np.array_equal(ds.slots.cpu().numpy(), ref["slots"])
    assert np.array_equal(bf16_to_bits(ds.k_cache), ref["k"])
    assert np.array_equal(bf16_to_bits(ds.v_cache), ref["v"])
    out = bf16_to_bits(ds.out)
    assert_close(out, ref["out"], w.name)
    return ds, ref, out


@pytest.mark.parametrize("name", ["tiny", "decode", "mix", "spec", "long"])
def test_small_workloads_match_oracle(name):
    w = wl.SMALL[name]()
    ds, ref, out = run_and_check(w)
    if w.logits is not None:
        acc, nxt, am = oracle.spec_accept_greedy(w.logits, w.draft)
        assert np.array_equal(ds.argmax.cpu().numpy(), am)
        assert np.array_equal(ds.accepted.cpu().numpy(), acc)
        assert np.array_equal(ds.next_token.cpu().numpy(), nxt)


@pytest.mark.parametrize("name", ["tiny", "decode", "mix", "spec", "long"])
def test_decode_rows_on_cuda_cores_match_oracle(name):
    run_and_check(wl.SMALL[name](), flags=pkv.PKV_ATTN_DECODE_CUDA_CORES)


@pytest.mark.parametrize("P", [16, 32, 48, 160, 768, 1536, 4096])
def test_partition_sizes(P):
    # many partitions per sequence exercise the split-KV merge; 16 tokens with
    # long sequences takes the many-partition merge path
    run_and_check(wl.SMALL["mix"](), partition_tokens=P)
    run_and_check(wl.SMALL["spec"](), partition_tokens=P)


@pytest.mark.parametrize("bs", [1, 2, 4, 8, 32, 64])
@pytest.mark.parametrize("d", [64, 128])
def test_block_sizes_and_head_dims(bs, d):
    w = wl.decode(B=5, lo=3, hi=140, seed=bs + d, n_q=8, n_kv=2, d=d, bs=bs)
    run_and_check(w, partition_tokens=64)
    w = wl.spec(B=3, lo=10, hi=120, k=3, vocab=300, seed=bs, n_q=8, n_kv=2, d=d, bs=bs)
    run_and_check(w, partition_tokens=48)


@pytest.mark.parametrize("nq,nkv", [(4, 4), (8, 4), (12, 4), (16, 2), (32, 2), (64, 1), (32, 8)])
def test_head_groupings(nq, nkv):
    run_and_check(wl.decode(B=4, lo=1, hi=90, seed=nq, n_q=nq, n_kv=nkv, d=64, bs=16), partition_tokens=32)
    run_and_check(wl.spec(B=3, lo=6, hi=90, k=4, vocab=100, seed=nq, n_q=nq, n_kv=nkv, d=64, bs=16),
                  partition_tokens=32)


def test_one_token_context_returns_v_exactly():
    w = wl.decode(B=3, lo=1, hi=1, seed=3, n_q=8, n_kv=2, d=128, bs=16)
    ds = DeviceStep(w)
    ds.step()
    torch.cuda.synchronize()
    g = w.n_q // w.n_kv
    out = bf16_to_bits(ds.out)
    for b in range(w.num_seqs):
        for h in range(w.n_q):
            # the cache row is the appended token; softmax weight 1 => output == V exactly
            assert np.array_equal(out[b, h], w.v_new[b, h // g])


def test_output_invariant_under_block_permutation():
    w = wl.SMALL["mix"]()
    ds = DeviceStep(w, partition_tokens=64)
    ds.step()
    torch.cuda.synchronize()
    a = bf16_to_bits(ds.out)
    perm = np.random.default_rng(1).permutation(w.num_blocks)
    k2 = np.empty_like(w.k_cache)
    v2 = np.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    w2 = wl.Workload(**{**w.__dict__})
    w2.k_cache, w2.v_cache = k2, v2
    w2.block_tables = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    w2.cow = perm[w.cow].astype(np.int32)
    ds2 = DeviceStep(w2, partition_tokens=64)
    ds2.step()
    torch.cuda.synchronize()
    assert np.array_equal(a, bf16_to_bits(ds2.out))


def test_repeated_calls_are_deterministic():
    w = wl.SMALL["long"]()
    ds = DeviceStep(w)
    ds.step()
    a = bf16_to_bits(ds.out)
    for _ in range(3):
        ds.reset_cache()
        ds.step()
        assert np.array_equal(a, bf16_to_bits(ds.out))


def test_gather_kv_bit_exact():
    w = wl.SMALL["mix"]()
    ref = oracle_step(w)
    ds = DeviceStep(w)
    ds.cache_ops()
    tot = int(w.seq_lens.sum())
    ko = torch.empty((tot, w.n_kv, w.head_dim), dtype=torch.bfloat16, device="cuda")
    vo = torch.empty_like(ko)
    offs = torch.from_numpy(np.concatenate([[0], np.cumsum(w.seq_lens)[:-1]]).astype(np.int64)).cuda()
    pkv.gather_kv(ko, vo, ds.k_cache, ds.v_cache, ds.block_tables, ds.seq_lens, offs, status=ds.status)
    torch.cuda.synchronize()
    kg, vg, st = oracle.gather_kv(ref["k"], ref["v"], w.block_tables, w.seq_lens)
    assert st == 0 and int(ds.status.item()) == 0
    assert np.array_equal(bf16_to_bits(ko), kg)
    assert np.array_equal(bf16_to_bits(vo), vg)


def test_empty_and_zero_query_sequences():
    w = wl.SMALL["decode"]()
    ql = w.q_lens.copy()
    ql[[1, 3]] = 0
    keep = np.repeat(ql > 0, w.q_lens)
    w2 = wl.Workload(**{**w.__dict__})
    w2.q_lens = ql
    w2.q = w.q[keep]
    ref = oracle_step(w2)
    ds = DeviceStep(w2)
    ds.step()
    torch.cuda.synchronize()
    assert int(ds.status.item()) == 0
    assert_close(bf16_to_bits(ds.out), ref["out"], "zero-q")


def test_invalid_inputs_give_nan_rows_and_status():
    w = wl.SMALL["decode"]()
    ds = DeviceStep(w)
    ds.cache_ops()
    torch.cuda.synchronize()
    bt = w.block_tables.copy()
    bt[2, 1] = w.num_blocks + 5           # bad block id inside sequence 2
    sl = w.seq_lens.copy()
    sl[4] = w.max_blocks * w.block_size + 1   # longer than its table
    ds.block_tables.copy_(torch.from_numpy(bt))
    ds.seq_lens.copy_(torch.from_numpy(sl))
    ds.max_seq_len = int(sl.max())
    ds.workspace = torch.empty(pkv.attention_workspace_bytes(w.num_seqs, w.total_q, w.n_q, w.n_kv, w.head_dim,
                                                             ds.max_seq_len, 0), dtype=torch.uint8, device="cuda")
    ds.status.zero_()
    ds.attention()
    torch.cuda.synchronize()
    st = int(ds.status.item())
    assert st & pkv.PKV_STATUS_BAD_BLOCK and st & pkv.PKV_STATUS_BAD_SEQLEN
    out = wl.bf16_bits_to_f32(bf16_to_bits(ds.out))
    assert np.isnan(out[2]).all() and np.isnan(out[4]).all()
    good = [0, 1, 3, 5]
    assert np.isfinite(out[good]).all()


def test_bad_slots_and_pairs_report_status():
    w = wl.SMALL["mix"]()
    ds = DeviceStep(w)
    bad_slots = torch.tensor([-1, w.num_blocks * w.block_size + 3], dtype=torch.int64, device="cuda")
    kn = ds.k_new[:2].contiguous()
    before = ds.k_cache.clone()
    pkv.kv_append(ds.k_cache, ds.v_cache, kn, kn, bad_slots, status=ds.status)
    pairs = torch.tensor([[0, w.num_blocks]], dtype=torch.int32, device="cuda")
    pkv.copy_blocks(ds.k_cache, ds.v_cache, pairs, status=ds.status)
    torch.cuda.synchronize()
    st = int(ds.status.item())
    assert st & pkv.PKV_STATUS_BAD_SLOT and st & pkv.PKV_STATUS_BAD_PAIR
    assert torch.equal(before.view(torch.int16), ds.k_cache.view(torch.int16))


def test_spec_accept_golden_and_nan_rows():
    import json
    import os
    from tests.conftest import GOLDEN
    gold = json.load(open(os.path.join(GOLDEN, "greedy_accept_cases.json")))
    for c in gold["cases"]:
        lg = torch.tensor(np.array(c["logits"], np.float32)[None]).cuda()
        dr = torch.tensor(np.array(c["draft"], np.int32)[None]).cuda()
        am = torch.empty((1, lg.shape[1]), dtype=torch.int32, device="cuda")
        acc = torch.empty(1, dtype=torch.int32, device="cuda")
        nxt = torch.empty(1, dtype=torch.int32, device="cuda")
        pkv.spec_accept_greedy(lg, dr, am, acc, nxt)
        torch.cuda.synchronize()
        assert am[0].tolist() == c["argmax"], c["name"]
        assert int(acc[0]) == c["accepted"] and int(nxt[0]) == c["next_token"], c["name"]


def test_batches_above_1024_sequences():
    # the planning kernel keeps per-sequence records in shared memory up to
    # 1024 sequences and in the workspace beyond; automatic partitions
    run_and_check(wl.decode(1500, 5, 80, 21, n_q=8, n_kv=2, d=64, bs=16))
    run_and_check(wl.spec(B=1100, lo=4, hi=60, k=3, vocab=40, seed=22, n_q=8, n_kv=2, d=64, bs=16))


def test_verification_batch_too_large_for_one_wave():
    # 400 verification sequences: every one-wave length still gives more
    # items than SMs, so the planner falls back to about two items per SM
    run_and_check(wl.spec(B=400, lo=20, hi=400, k=5, vocab=40, seed=23, n_q=32, n_kv=8, d=128, bs=16))


@pytest.mark.parametrize("V", [1, 7, 1000, 128256, 128257])
def test_spec_accept_random_vocab_sizes(V):
    rng = np.random.default_rng(V)
    B, k = 5, 4
    lg = rng.standard_normal((B, k + 1, V)).astype(np.float32)
    if V > 10:
        lg[0, 1, 3] = lg[0, 1, 9] = 100.0    # tie: first index wins
        lg[1, 2, V - 1] = np.nan             # NaN wins
    top = lg.argmax(-1)
    dr = np.where(rng.random((B, k)) < 0.6, top[:, :k], (top[:, :k] + 1) % V).astype(np.int32)
    acc, nxt, am = oracle.spec_accept_greedy(lg, dr)
    lgt = torch.from_numpy(lg).cuda()
    out = [torch.empty((B, k + 1), dtype=torch.int32, device="cuda"), torch.empty(B, dtype=torch.int32, device="cuda"),
           torch.empty(B, dtype=torch.int32, device="cuda")]
    pkv.spec_accept_greedy(lgt, torch.from_numpy(dr).cuda(), *out)
    torch.cuda.synchronize()
    assert np.array_equal(out[0].cpu().numpy(), am)
    assert np.array_equal(out[1].cpu().numpy(), acc)
    assert np.array_equal(out[2].cpu().numpy(), nxt)


@pytest.mark.parametrize("V,shift", [(1004, 0), (128256, 0), (128256, 4), (9000, 2)])
def test_argmax_load_widths_and_ties(V, shift):
    # rows of a multiple of 8 values on a 32-byte boundary take 256-bit loads,
    # a multiple of 4 on a 16-byte boundary 128-bit loads, the rest scalar loads
    # (shift: the logits start `shift` floats into their buffer); ties between a
    # thread's chunks (the first chunk holding the maximum is re-read), between
    # the CTAs of a row, equal zeros of both signs, two NaNs
    rng = np.random.default_rng(V + shift)
    B, k = 6, 3
    lg = rng.standard_normal((B, k + 1, V)).astype(np.float32)
    second = 17 + 8192 if V > 17 + 8192 else V - 20
    lg[0, 0, 17] = lg[0, 0, second] = 50.0        # one thread, chunks 0 and 1 (8-wide loads)
    lg[0, 1, 5] = lg[0, 1, V - 5] = 60.0          # the row's two CTAs
    lg[1, 0, :] = -1.0
    lg[1, 0, 100] = -0.0
    lg[1, 0, 50] = 0.0                            # +0 at 50 before -0 at 100: 50 wins
    lg[2, 2, V // 3] = np.nan
    lg[2, 2, V // 2] = np.nan                     # the first NaN wins
    lg[3, 1, :] = -np.inf                         # all -inf: index 0
    top = lg.argmax(-1)
    dr = np.where(rng.random((B, k)) < 0.7, top[:, :k], (top[:, :k] + 1) % V).astype(np.int32)
    acc, nxt, am = oracle.spec_accept_greedy(lg, dr)
    buf = torch.empty(lg.size + 8, dtype=torch.float32, device="cuda")
    lgt = buf[shift:shift + lg.size].view(lg.shape)
    lgt.copy_(torch.from_numpy(lg))
    out = [torch.empty((B, k + 1), dtype=torch.int32, device="cuda"), torch.empty(B, dtype=torch.int32, device="cuda"),
           torch.empty(B, dtype=torch.int32, device="cuda")]
    pkv.spec_accept_greedy(lgt, torch.from_numpy(dr).cuda(), *out)
    torch.cuda.synchronize()
    assert np.array_equal(out[0].cpu().numpy(), am)
    assert np.array_equal(out[1].cpu().numpy(), acc)
    assert np.array_equal(out[2].cpu().numpy(), nxt)


@pytest.mark.parametrize("g,ql", [(4, 2), (4, 3), (4, 5), (4, 6), (8, 2), (8, 3), (2, 7), (2, 12), (1, 17),
                                  (1, 24), (16, 1), (12, 2), (3, 8)])
@pytest.mark.parametrize("d", [64, 128])
def test_transposed_tiles_of_several_column_tiles(g, ql, d):
    """Short multi-query rows: q_len * g <= 16 run as one transposed tile of up
    to two 8-column n-tiles per kv head, each column with its query's causal
    limit; wider rows as tcgen05 tiles (automatic partitions, head_dim 128) or
    mma.sync row tiles (partitions of 64 tokens, or head_dim 64): partial last
    n-tiles, heads not a power of two, several partitions and a partial last
    stage."""
    n_kv = 2
    w = wl.spec(B=4, lo=ql + 1, hi=300, k=ql, vocab=50, seed=7 * g + ql, n_q=g * n_kv, n_kv=n_kv, d=d, bs=16)
    run_and_check(w, partition_tokens=64)
    run_and_check(w)


@pytest.mark.parametrize("bs", [1, 4, 32])
def test_transposed_wide_tiles_block_sizes(bs):
    w = wl.spec(B=5, lo=6, hi=200, k=5, vocab=50, seed=bs, n_q=32, n_kv=8, d=128, bs=bs)
    run_and_check(w, partition_tokens=48)
