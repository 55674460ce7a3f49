"""Pins of the oracle's second FP8 format and per-block scales ("Inference at
Scale" section 03, KV cache quantization: FP8 as e4m3 or e5m2) on CPU: the
e5m2 codec against hand-worked values and torch's float8_e5m2, the block-scale
rule against hand-worked cases, the quantising append with per-block scales
against its definition, the copy-on-write of scales, and FP8 attention of
both formats and both scale granularities against torch SDPA on the
dequantised values."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_23_gb300 import workloads as wl
from tests.conftest import GOLDEN

CASES = json.load(open(os.path.join(GOLDEN, "e5m2_cases.json")))


def _f(v):
    return float(v)  # "nan", "inf", "-inf" parse too


def test_e5m2_decode_golden_and_torch():
    for c in CASES["decode"]:
        v = oracle.fp8_decode(np.array([c["code"]], np.uint8), oracle.E5M2)[0]
        want = _f(c["value"])
        assert (np.isnan(v) and np.isnan(want)) or v == want, c
    codes = np.arange(256, dtype=np.uint8)
    v = oracle.fp8_decode(codes, oracle.E5M2)
    t = torch.from_numpy(codes).view(torch.float8_e5m2).to(torch.float64).numpy()
    assert np.array_equal(np.isnan(v), np.isnan(t))
    assert np.array_equal(v[~np.isnan(v)], t[~np.isnan(t)])


def test_e5m2_encode_golden_and_torch():
    for c in CASES["encode"]:
        x = np.float32(_f(c["x"]))
        assert oracle.fp8_encode(np.array([x], np.float32), oracle.E5M2)[0] == c["code"], c
    g = np.random.default_rng(0)
    x = np.concatenate([g.standard_normal(200000).astype(np.float32) * s for s in (1e-4, 0.1, 3.0, 1000.0)])
    x = x[np.abs(x) <= 57344]
    ours = oracle.fp8_encode(x, oracle.E5M2)
    ref = torch.from_numpy(x).to(torch.float8_e5m2).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e5m2_encode_is_nearest():
    """Brute force over every finite code: the chosen code is a nearest one."""
    codes = np.arange(256, dtype=np.uint8)
    vals = oracle.fp8_decode(codes, oracle.E5M2)
    fin = np.isfinite(vals)
    g = np.random.default_rng(1)
    x = np.concatenate([g.uniform(-60000, 60000, 20000), g.standard_normal(20000) * 1e-3]).astype(np.float32)
    enc = oracle.fp8_decode(oracle.fp8_encode(x, oracle.E5M2), oracle.E5M2)
    xc = np.clip(x.astype(np.float64), -57344, 57344)
    best = np.abs(vals[fin][None, :] - xc[:, None]).min(1)
    assert np.array_equal(np.abs(enc - xc), best)


def test_e4m3_through_the_general_codec_is_unchanged():
    g = np.random.default_rng(2)
    x = (g.standard_normal(50000) * 40).astype(np.float32)
    assert np.array_equal(oracle.fp8_encode(x, oracle.E4M3), oracle.e4m3_encode(x))
    codes = np.arange(256, dtype=np.uint8)
    a, b = oracle.fp8_decode(codes, oracle.E4M3), oracle.e4m3_decode(codes)
    assert np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(a[~np.isnan(a)], b[~np.isnan(b)])


def test_block_scale_golden():
    for c in CASES["block_scale"]["cases"]:
        row = np.array([_f(v) for v in c["row"]], np.float32)
        assert oracle.block_scale(row, c["fmt"]) == c["scale"], c


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_block_scale_is_the_smallest_power_of_two(fmt):
    half = 224.0 if fmt == oracle.E4M3 else 28672.0
    g = np.random.default_rng(3)
    for _ in range(500):
        row = (g.standard_normal(64) * 10.0 ** g.uniform(-6, 6)).astype(np.float32)
        s = oracle.block_scale(row, fmt)
        amax = float(np.abs(row.astype(np.float64)).max())
        m, e = np.frexp(s)
        assert m == 0.5                            # a power of two
        assert amax <= s * half                    # the row fits in half the range
        assert amax > s / 2 * half                 # and no smaller power of two does


def _append_case(fmt):
    """A small mix whose appended rows include fresh blocks opened in this
    call: row 0 of a block sets its scales."""
    w = wl.SMALL["mix"]()
    pools = wl.fp8_pools(w, 5, fmt, per_block=True)
    slots, st = oracle.slot_mapping(w.block_tables, w.seq_lens, w.append_lens, w.block_size, w.num_blocks)
    assert st == 0
    return w, pools, slots


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_append_with_block_scales_definition(fmt):
    w, pools, slots = _append_case(fmt)
    k8, v8 = pools.k_cache.copy(), pools.v_cache.copy()
    ks, vs = pools.k_scale.copy(), pools.v_scale.copy()
    assert oracle.kv_append_fp8_ex(k8, v8, w.k_new, w.v_new, slots, ks, vs, fmt, True) == 0
    opened = {int(s) // w.block_size for s in slots if int(s) % w.block_size == 0}
    for blk in range(w.num_blocks):
        if blk not in opened:
            assert np.array_equal(ks[blk], pools.k_scale[blk]) and np.array_equal(vs[blk], pools.v_scale[blk])
    touched = np.zeros(k8.shape[:3], bool)
    for t, sl in enumerate(slots):
        blk, row = divmod(int(sl), w.block_size)
        touched[blk, :, row] = True
        for h in range(w.n_kv):
            xk = wl.bf16_bits_to_f32(w.k_new[t, h])
            if row == 0:
                assert ks[blk, h] == oracle.block_scale(xk, fmt)
            q = (xk * np.float32(np.float32(1.0) / ks[blk, h])).astype(np.float32)
            assert np.array_equal(k8[blk, h, row], oracle.fp8_encode(q, fmt))
    assert np.array_equal(k8[~touched], pools.k_cache[~touched])
    assert np.array_equal(v8[~touched], pools.v_cache[~touched])
    assert len(opened) > 0


def test_rows_appended_with_their_opening_row_use_its_scale():
    """Three rows of one fresh block in one call: rows 1 and 2 are stored with
    the scale row 0 sets, even when their own magnitude is larger."""
    nb, nkv, bs, d = 4, 1, 4, 8
    k8 = np.zeros((nb, nkv, bs, d), np.uint8)
    v8 = np.zeros_like(k8)
    ks = np.full((nb, nkv), 0.5, np.float32)
    vs = np.full((nb, nkv), 0.5, np.float32)
    x = np.array([[1.0] * d, [3.0] * d, [500.0] * d], np.float32)     # rows 0, 1, 2 of block 2
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)[:, None, :]
    slots = np.array([2 * bs + 0, 2 * bs + 1, 2 * bs + 2], np.int64)
    assert oracle.kv_append_fp8_ex(k8, v8, bits, bits, slots, ks, vs, oracle.E4M3, True) == 0
    assert ks[2, 0] == 2.0 ** -7 and vs[2, 0] == 2.0 ** -7              # from row 0 (amax 1)
    assert ks[0, 0] == ks[1, 0] == ks[3, 0] == 0.5                       # other blocks untouched
    deq = oracle.fp8_decode(k8[2, 0, :3], oracle.E4M3) * 2.0 ** -7
    assert np.all(deq[0] == 1.0) and np.all(deq[1] == 3.0)
    assert np.all(deq[2] == 448.0 * 2.0 ** -7)                           # 500 * 2^7 > 448: saturated


def test_copy_blocks_fp8_copies_the_block_scales():
    w, pools, _ = _append_case(oracle.E4M3)
    k8, v8 = pools.k_cache.copy(), pools.v_cache.copy()
    ks, vs = pools.k_scale.copy(), pools.v_scale.copy()
    pairs = np.array([[1, 5], [7, 2]], np.int32)
    assert oracle.copy_blocks_fp8(k8, v8, ks, vs, pairs, per_block=True) == 0
    for src, dst in pairs:
        assert np.array_equal(k8[dst], pools.k_cache[src]) and np.array_equal(v8[dst], pools.v_cache[src])
        assert np.array_equal(ks[dst], pools.k_scale[src]) and np.array_equal(vs[dst], pools.v_scale[src])
    bad = np.array([[0, w.num_blocks]], np.int32)
    assert oracle.copy_blocks_fp8(k8, v8, ks, vs, bad, per_block=True) == 64


def _sdpa_check(w, k8, v8, ks, vs, fmt, per_block, got):
    g = w.n_q // w.n_kv
    q0 = np.concatenate([[0], np.cumsum(w.q_lens)])
    for b in range(w.num_seqs):
        L, ql = int(w.seq_lens[b]), int(w.q_lens[b])
        blocks = w.block_tables[b, :-(-L // w.block_size)]
        sk = ks[blocks][:, :, None, None] if per_block else ks[None, :, None, None]
        sv = vs[blocks][:, :, None, None] if per_block else vs[None, :, None, None]
        K = oracle.fp8_decode(k8[blocks], fmt) * sk
        V = oracle.fp8_decode(v8[blocks], fmt) * sv
        K = torch.from_numpy(K.transpose(1, 0, 2, 3).reshape(w.n_kv, -1, w.head_dim)[:, :L])
        V = torch.from_numpy(V.transpose(1, 0, 2, 3).reshape(w.n_kv, -1, w.head_dim)[:, :L])
        Q = torch.from_numpy(wl.bf16_bits_to_f32(w.q[q0[b]:q0[b + 1]]).astype(np.float64)).transpose(0, 1)
        # causal within the new tokens: query i sees positions 0 .. L - ql + i
        mask = torch.arange(L)[None, :] <= (L - ql + torch.arange(ql))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            Q, K.repeat_interleave(g, 0), V.repeat_interleave(g, 0), attn_mask=mask, scale=w.scale)
        assert np.allclose(got[q0[b]:q0[b + 1]], ref.transpose(0, 1).numpy(), rtol=0, atol=1e-10)


def stepped(w, pools):
    """FP8 pools (and scales) after the step's copy-on-write and quantising append."""
    k8, v8 = pools.k_cache.copy(), pools.v_cache.copy()
    ks, vs = pools.k_scale.copy(), pools.v_scale.copy()
    assert oracle.copy_blocks_fp8(k8, v8, ks, vs, w.cow, per_block=pools.per_block) == 0
    slots, st = oracle.slot_mapping(w.block_tables, w.seq_lens, w.append_lens, w.block_size, w.num_blocks)
    assert st == 0
    assert oracle.kv_append_fp8_ex(k8, v8, w.k_new, w.v_new, slots, ks, vs, pools.fmt, pools.per_block) == 0
    return k8, v8, ks, vs


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
@pytest.mark.parametrize("per_block", [False, True])
@pytest.mark.parametrize("name", ["decode", "spec", "mix"])
def test_attention_fp8_ex_vs_sdpa(fmt, per_block, name):
    w = wl.SMALL[name]()
    k8, v8, ks, vs = stepped(w, wl.fp8_pools(w, 6, fmt, per_block))
    got, st = oracle.attention_fp8_ex(w.q, k8, v8, ks, vs, w.block_tables, w.seq_lens, w.q_lens, w.scale, fmt,
                                      per_block)
    assert st == 0 and not np.isnan(got).any()
    _sdpa_check(w, k8, v8, ks, vs, fmt, per_block, got)


def test_attention_fp8_ex_per_head_mode_is_the_e4m3_attention():
    w = wl.SMALL["mix"]()
    k8, v8, ks, vs = stepped(w, wl.fp8_pools(w, 7))
    a, sa = oracle.attention_fp8(w.q, k8, v8, ks, vs, w.block_tables, w.seq_lens, w.q_lens, w.scale)
    b, sb = oracle.attention_fp8_ex(w.q, k8, v8, ks, vs, w.block_tables, w.seq_lens, w.q_lens, w.scale,
                                    oracle.E4M3, False)
    assert sa == sb == 0 and not np.isnan(a).any() and np.array_equal(a, b)
    # per-block scales that repeat the per-head ones give the same result
    kb = np.repeat(ks[None, :], w.num_blocks, 0)
    vb = np.repeat(vs[None, :], w.num_blocks, 0)
    c, sc = oracle.attention_fp8_ex(w.q, k8, v8, kb, vb, w.block_tables, w.seq_lens, w.q_lens, w.scale,
                                    oracle.E4M3, True)
    assert sc == 0 and np.array_equal(a, c)


def test_append_per_head_mode_is_the_e4m3_append():
    w = wl.SMALL["mix"]()
    pools = wl.fp8_pools(w, 8)
    slots, _ = oracle.slot_mapping(w.block_tables, w.seq_lens, w.append_lens, w.block_size, w.num_blocks)
    a = (pools.k_cache.copy(), pools.v_cache.copy())
    b = (pools.k_cache.copy(), pools.v_cache.copy())
    assert oracle.kv_append_fp8(a[0], a[1], w.k_new, w.v_new, slots, pools.k_scale, pools.v_scale) == 0
    ks, vs = pools.k_scale.copy(), pools.v_scale.copy()
    assert oracle.kv_append_fp8_ex(b[0], b[1], w.k_new, w.v_new, slots, ks, vs, oracle.E4M3, False) == 0
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    assert np.array_equal(ks, pools.k_scale)                           # per-head scales are read only
