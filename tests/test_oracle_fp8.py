"""Pins of the oracle's FP8 (e4m3) KV cache ("Inference at Scale" section 03,
KV cache quantization) on CPU: the codec against hand-worked values and
torch's float8_e4m3fn, the quantising append against its definition, and
FP8 attention against the bf16 oracle and against torch SDPA on the
dequantised values."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_23_gb300 import workloads as wl
from tests.conftest import GOLDEN

CASES = json.load(open(os.path.join(GOLDEN, "e4m3_cases.json")))


def test_decode_golden_and_torch():
    for c in CASES["decode"]:
        v = oracle.e4m3_decode(np.array([c["code"]], np.uint8))[0]
        assert np.isnan(v) if c["value"] == "nan" else v == c["value"]
    codes = np.arange(256, dtype=np.uint8)
    v = oracle.e4m3_decode(codes)
    t = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(v), np.isnan(t))
    assert np.array_equal(v[~np.isnan(v)], t[~np.isnan(t)])


def test_encode_golden_and_torch():
    for c in CASES["encode"]:
        x = np.float32(np.nan if c["x"] == "nan" else c["x"])
        assert oracle.e4m3_encode(np.array([x], np.float32))[0] == c["code"], c
    g = np.random.default_rng(0)
    x = np.concatenate([g.standard_normal(200000).astype(np.float32) * s for s in (0.003, 0.1, 3.0, 100.0)])
    x = x[np.abs(x) <= 448]
    ours = oracle.e4m3_encode(x)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)
    # saturation: beyond 448 the code stays at +-448
    big = np.array([449, 500, 1e6, 3e38, -449, -1e30], np.float32)
    assert (oracle.e4m3_encode(big) == np.array([126, 126, 126, 126, 254, 254])).all()


def test_encode_is_nearest():
    """Brute force over every finite code: the chosen code is a nearest one."""
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.e4m3_decode(codes)
    fin = ~np.isnan(vals)
    g = np.random.default_rng(1)
    x = (g.uniform(-460, 460, 20000)).astype(np.float32)
    x = np.concatenate([x, (g.standard_normal(20000) * 0.01).astype(np.float32)])
    enc = oracle.e4m3_decode(oracle.e4m3_encode(x))
    best = np.abs(vals[fin][None, :] - np.minimum(np.abs(x.astype(np.float64)), 448)[:, None] *
                  np.sign(x)[:, None]).min(1)
    assert np.allclose(np.abs(enc - np.clip(x, -448, 448)), best, rtol=0, atol=0)


def test_append_fp8_definition():
    w = wl.SMALL["mix"]()
    pools = wl.fp8_pools(w, 3)
    k8, v8 = pools.k_cache.copy(), pools.v_cache.copy()
    slots, st = oracle.slot_mapping(w.block_tables, w.seq_lens, w.append_lens, w.block_size, w.num_blocks)
    assert st == 0
    assert oracle.kv_append_fp8(k8, v8, w.k_new, w.v_new, slots, pools.k_scale, pools.v_scale) == 0
    touched = np.zeros(k8.shape[:3], bool)
    for t, sl in enumerate(slots):
        blk, row = divmod(int(sl), w.block_size)
        touched[blk, :, row] = True
        for h in range(w.n_kv):
            xk = wl.bf16_bits_to_f32(w.k_new[t, h]) * np.float32(np.float32(1.0) / pools.k_scale[h])
            assert np.array_equal(k8[blk, h, row], oracle.e4m3_encode(xk.astype(np.float32)))
            # the dequantised row is within half an e4m3 step of x
            deq = oracle.e4m3_decode(v8[blk, h, row]) * pools.v_scale[h]
            x = wl.bf16_bits_to_f32(w.v_new[t, h]).astype(np.float64)
            assert np.all(np.abs(deq - x) <= np.maximum(np.abs(x) * 2.0 ** -4, 2.0 ** -10 * pools.v_scale[h]) + 1e-12)
    assert np.array_equal(k8[~touched], pools.k_cache[~touched])
    assert np.array_equal(v8[~touched], pools.v_cache[~touched])


def _stepped_pools(w, seed, ks=None, vs=None):
    """fp8 pools after the step's copy-on-write and quantising append."""
    pools = wl.fp8_pools(w, seed)
    ks = pools.k_scale if ks is None else ks
    vs = pools.v_scale if vs is None else vs
    k8, v8 = pools.k_cache.copy(), pools.v_cache.copy()
    for src, dst in np.asarray(w.cow).reshape(-1, 2):
        k8[dst] = k8[src]
        v8[dst] = v8[src]
    slots, st = oracle.slot_mapping(w.block_tables, w.seq_lens, w.append_lens, w.block_size, w.num_blocks)
    assert st == 0 and oracle.kv_append_fp8(k8, v8, w.k_new, w.v_new, slots, ks, vs) == 0
    return k8, v8, ks, vs


def _dequant_bf16_pool(codes, scales):
    """bf16 bit pool holding e4m3 * scale exactly (scales are powers of two)."""
    v = oracle.e4m3_decode(codes) * scales[None, :, None, None].astype(np.float64)
    f = v.astype(np.float32)
    assert np.array_equal(f.astype(np.float64)[~np.isnan(v)], v[~np.isnan(v)])
    return (f.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("name", ["tiny", "decode", "mix", "spec"])
def test_attention_fp8_equals_bf16_oracle_on_exact_values(name):
    w = wl.SMALL[name]()
    ks = (2.0 ** np.arange(-3, -3 - w.n_kv, -1)).astype(np.float32)
    vs = (2.0 ** np.arange(-2, -2 + w.n_kv)).astype(np.float32)
    k8, v8, ks, vs = _stepped_pools(w, 4, ks, vs)
    ref, st = oracle.attention(w.q, _dequant_bf16_pool(k8, ks), _dequant_bf16_pool(v8, vs),
                               w.block_tables, w.seq_lens, w.q_lens, w.scale)
    got, st8 = oracle.attention_fp8(w.q, k8, v8, ks, vs, w.block_tables, w.seq_lens, w.q_lens, w.scale)
    assert st == st8 == 0
    assert not np.isnan(got).any() and not np.isnan(ref).any()
    assert np.allclose(got[~np.isnan(got)], ref[~np.isnan(ref)], rtol=0, atol=1e-12)


def test_attention_fp8_vs_sdpa():
    w = wl.SMALL["decode"]()
    k8, v8, ks, vs = _stepped_pools(w, 5)
    got, st = oracle.attention_fp8(w.q, k8, v8, ks, vs, w.block_tables, w.seq_lens, w.q_lens, w.scale)
    assert st == 0 and not np.isnan(got).any()
    g = w.n_q // w.n_kv
    for b in range(w.num_seqs):
        L = int(w.seq_lens[b])
        blocks = w.block_tables[b, :-(-L // w.block_size)]
        K = oracle.e4m3_decode(k8[blocks]) * ks[None, :, None, None]
        V = oracle.e4m3_decode(v8[blocks]) * vs[None, :, None, None]
        K = torch.from_numpy(K.transpose(1, 0, 2, 3).reshape(w.n_kv, -1, w.head_dim)[:, :L])
        V = torch.from_numpy(V.transpose(1, 0, 2, 3).reshape(w.n_kv, -1, w.head_dim)[:, :L])
        Q = torch.from_numpy(wl.bf16_bits_to_f32(w.q[b]).astype(np.float64))[:, None, :]   # [n_q][1][d]
        ref = torch.nn.functional.scaled_dot_product_attention(
            Q, K.repeat_interleave(g, 0), V.repeat_interleave(g, 0), scale=w.scale)[:, 0].numpy()
        assert np.allclose(got[b], ref, rtol=0, atol=1e-10)
