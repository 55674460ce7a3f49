"""FP8 KV caches of the second format and with per-block scales on the GPU vs
the CPU oracle ("Inference at Scale" section 03, KV cache quantization: FP8 as
e4m3 or e5m2).  The pools and the per-block scales after the step's
copy-on-write and quantising append are bit-exact against the oracle's;
attention holds |gpu - ref| <= 1e-2 + 1e-2 |ref| against the oracle's fp64
attention over the dequantised K/V (GPU required)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_23_gb300 as pkv
from paged_kv_cache_23_gb300 import workloads as wl
from paged_kv_cache_23_gb300.runner import DeviceStep, bf16_to_bits

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-2
MODES = [(0, True), (1, False), (1, True)]   # (format, per-block scales): e4m3/block, e5m2/head, e5m2/block


@pytest.fixture(scope="module", autouse=True)
def _built():
    pkv.build()
    torch.cuda.init()


def oracle_step(w, pools):
    k8, v8 = pools.k_cache.copy(), pools.v_cache.copy()
    ks, vs = pools.k_scale.copy(), pools.v_scale.copy()
    st0 = oracle.copy_blocks_fp8(k8, v8, ks, vs, w.cow, per_block=pools.per_block)
    slots, st1 = oracle.slot_mapping(w.block_tables, w.seq_lens, w.append_lens, w.block_size, w.num_blocks)
    st2 = oracle.kv_append_fp8_ex(k8, v8, w.k_new, w.v_new, slots, ks, vs, pools.fmt, pools.per_block)
    out, st3 = oracle.attention_fp8_ex(w.q, k8, v8, ks, vs, w.block_tables, w.seq_lens, w.q_lens, w.scale,
                                       pools.fmt, pools.per_block)
    return k8, v8, ks, vs, out, st0 | st1 | st2 | st3


def run_and_check(w, fmt, per_block, seed=0, partition_tokens=None, max_seq_len=None, pools=None):
    pools = wl.fp8_pools(w, seed, fmt, per_block) if pools is None else pools
    ds = DeviceStep(w, fp8=pools, partition_tokens=partition_tokens, max_seq_len=max_seq_len)
    ds.cache_ops()
    ds.attention()
    torch.cuda.synchronize()
    k8, v8, ks, vs, ref, st = oracle_step(w, pools)
    assert np.array_equal(ds.k_cache.cpu().numpy(), k8)
    assert np.array_equal(ds.v_cache.cpu().numpy(), v8)
    assert np.array_equal(ds.k_scale.cpu().numpy(), ks) and np.array_equal(ds.v_scale.cpu().numpy(), vs)
    got = wl.bf16_bits_to_f32(bf16_to_bits(ds.out)).astype(np.float64)
    bad = np.isnan(ref)
    assert np.array_equal(np.isnan(got), bad)
    err = np.abs(got[~bad] - ref[~bad])
    assert np.all(err <= ATOL + RTOL * np.abs(ref[~bad])), float(err.max())
    assert int(ds.status.item()) == st
    return ds, got, ref


@pytest.mark.parametrize("fmt,per_block", MODES)
@pytest.mark.parametrize("name", ["decode", "mix", "spec", "long"])
def test_small_workloads(name, fmt, per_block):
    run_and_check(wl.SMALL[name](), fmt, per_block)


@pytest.mark.parametrize("fmt,per_block", MODES)
@pytest.mark.parametrize("P", [16, 48, 768, 0])
def test_partitions(P, fmt, per_block):
    run_and_check(wl.SMALL["mix"](), fmt, per_block, partition_tokens=P)


@pytest.mark.parametrize("fmt,per_block", MODES)
@pytest.mark.parametrize("bs", [1, 2, 4, 8, 16, 32, 64])
def test_block_sizes(bs, fmt, per_block):
    """Several blocks per stage (each token its own block's scales), one block
    per stage, and blocks spanning several stages."""
    run_and_check(wl.spec(B=3, lo=10, hi=120, k=3, vocab=300, seed=bs, n_q=8, n_kv=2, d=128, bs=bs), fmt, per_block,
                  seed=bs)
    run_and_check(wl.decode(4, 5, 200, bs, n_q=8, n_kv=4, d=128, bs=bs), fmt, per_block, seed=bs)


@pytest.mark.parametrize("fmt,per_block", MODES)
@pytest.mark.parametrize("nq,nkv", [(8, 8), (16, 4), (32, 8), (12, 4), (6, 2)])
def test_groupings(nq, nkv, fmt, per_block):
    run_and_check(wl.decode(5, 3, 150, nq, n_q=nq, n_kv=nkv, d=128, bs=16), fmt, per_block, seed=nq)


@pytest.mark.parametrize("per_block", [False, True])
def test_e5m2_encoding_edges_bit_exact(per_block):
    """Rounding ties, saturation, infinities and subnormals of the e5m2 append."""
    w = wl.SMALL["decode"]()
    pools = wl.fp8_pools(w, 1, 1, per_block)
    pools.k_scale[:] = 1.0
    pools.v_scale[:] = np.float32(0.75)
    special = np.array([1.125, 1.375, 1.124, 57344.0, 61440.0, 1e30, -1e30, np.inf, -np.inf, 2.0 ** -17,
                        1.5 * 2.0 ** -16, 2.0 ** -16, -0.0, 0.0, 3.0, -3.3, 240.0, 1e-30], np.float32)
    kn = w.k_new.copy()
    flat = kn.reshape(-1)
    bits = (special.view(np.uint32) >> 16).astype(np.uint16)
    flat[: len(bits)] = bits
    w.k_new = kn
    ds = DeviceStep(w, fp8=pools)
    ds.cache_ops()
    torch.cuda.synchronize()
    k8, v8, ks, vs, _, _ = oracle_step(w, pools)
    assert np.array_equal(ds.k_cache.cpu().numpy(), k8)
    assert np.array_equal(ds.k_scale.cpu().numpy(), ks)


def test_blocks_opened_in_the_call_take_their_row_0_scale():
    """A prefill chunk writes whole fresh blocks in one call: every row of a
    block is stored with the scale its row 0 sets, on the GPU as in the oracle."""
    w = wl.long_context(B=1, ctx=300, chunk=96, chunk_prefix=64, partition_tokens=1024, seed=3)
    pools = wl.fp8_pools(w, 2, 0, True)
    ds, _, _ = run_and_check(w, 0, True, pools=pools)
    slots, _ = oracle.slot_mapping(w.block_tables, w.seq_lens, w.append_lens, w.block_size, w.num_blocks)
    opened = {int(s) // w.block_size for s in slots if int(s) % w.block_size == 0}
    assert len(opened) >= 5
    ks = ds.k_scale.cpu().numpy()
    assert not np.array_equal(ks[sorted(opened)], pools.k_scale[sorted(opened)])


@pytest.mark.parametrize("fmt,per_block", MODES)
def test_full_size_mix_every_row(fmt, per_block):
    w = wl.FULL["mix"]()
    run_and_check(w, fmt, per_block, max_seq_len=32768)


@pytest.mark.parametrize("fmt,per_block", MODES)
def test_plan_then_runs_equal_one_call(fmt, per_block):
    w = wl.SMALL["spec"]()
    ds = DeviceStep(w, fp8=wl.fp8_pools(w, 4, fmt, per_block))
    ds.cache_ops()
    ds.attention()
    ref = bf16_to_bits(ds.out)
    ds.out.fill_(float("nan"))
    ds.plan()
    ds.run()
    ds.run()
    torch.cuda.synchronize()
    assert int(ds.status.item()) == 0
    assert np.array_equal(bf16_to_bits(ds.out), ref)
