"""FP8 (e4m3) KV cache on the GPU vs the CPU oracle (GPU required).

Appends and copies are bit-exact against the oracle's whole pools; attention
over e4m3 pools holds |gpu - ref| <= 1e-2 + 1e-2 |ref| against the oracle's
fp64 attention over the dequantised K/V ("Inference at Scale" section 03, KV
cache quantization)."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_23_gb300 as pkv
from paged_kv_cache_23_gb300 import workloads as wl
from paged_kv_cache_23_gb300.runner import DeviceStep, bf16_to_bits, to_device_bf16

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    pkv.build()
    torch.cuda.init()


def oracle_fp8_step(w, pools):
    k8, v8 = pools.k_cache.copy(), pools.v_cache.copy()
    for src, dst in np.asarray(w.cow).reshape(-1, 2):
        k8[dst] = k8[src]
        v8[dst] = v8[src]
    slots, st1 = oracle.slot_mapping(w.block_tables, w.seq_lens, w.append_lens, w.block_size, w.num_blocks)
    st2 = oracle.kv_append_fp8(k8, v8, w.k_new, w.v_new, slots, pools.k_scale, pools.v_scale)
    out, st3 = oracle.attention_fp8(w.q, k8, v8, pools.k_scale, pools.v_scale, w.block_tables, w.seq_lens, w.q_lens,
                                    w.scale)
    return k8, v8, out, st1 | st2 | st3


def run_and_check(w, seed=0, partition_tokens=None, max_seq_len=None):
    pools = wl.fp8_pools(w, seed)
    ds = DeviceStep(w, fp8=pools, partition_tokens=partition_tokens, max_seq_len=max_seq_len)
    ds.cache_ops()
    ds.attention()
    torch.cuda.synchronize()
    k8, v8, ref, st = oracle_fp8_step(w, pools)
    assert np.array_equal(ds.k_cache.cpu().numpy(), k8)
    assert np.array_equal(ds.v_cache.cpu().numpy(), v8)
    got = wl.bf16_bits_to_f32(bf16_to_bits(ds.out)).astype(np.float64)
    bad = np.isnan(ref)
    assert np.array_equal(np.isnan(got), bad)
    err = np.abs(got[~bad] - ref[~bad])
    assert np.all(err <= ATOL + RTOL * np.abs(ref[~bad])), float(err.max())
    assert int(ds.status.item()) == st
    return ds, got, ref


@pytest.mark.parametrize("name", ["decode", "mix", "spec", "long"])
def test_small_workloads(name):
    run_and_check(wl.SMALL[name]())


@pytest.mark.parametrize("P", [16, 48, 512, 768, 0])
def test_partitions(P):
    run_and_check(wl.SMALL["mix"](), partition_tokens=P)


@pytest.mark.parametrize("bs", [1, 2, 4, 8, 16, 32, 64])
def test_block_sizes(bs):
    run_and_check(wl.spec(B=3, lo=10, hi=120, k=3, vocab=300, seed=bs, n_q=8, n_kv=2, d=128, bs=bs), seed=bs)
    run_and_check(wl.decode(4, 5, 200, bs, n_q=8, n_kv=4, d=128, bs=bs), seed=bs)


@pytest.mark.parametrize("nq,nkv", [(8, 8), (8, 4), (16, 4), (32, 8), (16, 2), (32, 2), (12, 4), (6, 2)])
def test_groupings(nq, nkv):
    run_and_check(wl.decode(5, 3, 150, nq, n_q=nq, n_kv=nkv, d=128, bs=16), seed=nq)
    run_and_check(wl.spec(B=3, lo=8, hi=90, k=5, vocab=100, seed=nq, n_q=nq, n_kv=nkv, d=128, bs=16), seed=nq)


def test_encoding_edges_bit_exact():
    """Rounding ties, saturation and subnormals of the quantising append."""
    w = wl.SMALL["decode"]()
    pools = wl.fp8_pools(w, 1)
    pools.k_scale[:] = 1.0
    pools.v_scale[:] = np.float32(0.75)
    special = np.array([1.0625, 1.1875, 1.0624999, 448.0, 460.0, 1e6, -1e6, 2.0 ** -10, 1.5 * 2.0 ** -9, 2.0 ** -9,
                        -0.0, 0.0, 3.0, -3.3, 240.0, 232.0, 1e-30], np.float32)
    kn = w.k_new.copy()
    flat = kn.reshape(-1)
    bits = (special.view(np.uint32) >> 16).astype(np.uint16)   # bf16 truncation keeps these exact or near
    flat[: len(bits)] = bits
    w.k_new = kn
    run_and_check(w)


def test_full_size_mix_every_row():
    w = wl.FULL["mix"]()
    pools = wl.fp8_pools(w, 0)
    ds = DeviceStep(w, fp8=pools, max_seq_len=32768)
    ds.cache_ops()
    ds.attention()
    torch.cuda.synchronize()
    assert int(ds.status.item()) == 0
    k8, v8 = pools.k_cache.copy(), pools.v_cache.copy()
    for src, dst in np.asarray(w.cow).reshape(-1, 2):
        k8[dst] = k8[src]
        v8[dst] = v8[src]
    slots, _ = oracle.slot_mapping(w.block_tables, w.seq_lens, w.append_lens, w.block_size, w.num_blocks)
    oracle.kv_append_fp8(k8, v8, w.k_new, w.v_new, slots, pools.k_scale, pools.v_scale)
    assert np.array_equal(ds.k_cache.cpu().numpy(), k8) and np.array_equal(ds.v_cache.cpu().numpy(), v8)
    # every query row of the batch-256 mix
    ref, st = oracle.attention_fp8(w.q, k8, v8, pools.k_scale, pools.v_scale, w.block_tables, w.seq_lens,
                                   w.q_lens, w.scale)
    assert st == 0
    got = wl.bf16_bits_to_f32(bf16_to_bits(ds.out)).astype(np.float64)
    assert np.isfinite(got).all()
    assert np.all(np.abs(got - ref) <= ATOL + RTOL * np.abs(ref))


def test_bad_block_is_nan_and_status():
    w = wl.SMALL["decode"]()
    w.block_tables = w.block_tables.copy()
    w.block_tables[1, 0] = w.num_blocks + 3
    pools = wl.fp8_pools(w, 2)
    ds = DeviceStep(w, fp8=pools)
    ds.cache_ops()
    ds.attention()
    torch.cuda.synchronize()
    got = wl.bf16_bits_to_f32(bf16_to_bits(ds.out))
    assert np.isnan(got[1]).all() and not np.isnan(got[0]).any()
    assert int(ds.status.item()) & pkv.PKV_STATUS_BAD_BLOCK
