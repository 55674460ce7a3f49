"""Pins of the CPU oracle to things other than itself (no GPU needed).

Each test checks the oracle against something the pages or the mathematics
fix: a library routine (torch SDPA in fp64, numpy argmax), a closed form, a
worked example printed on the pages (tests/golden), an invariant of paging,
or an independent restatement of a different algorithm.  A plausible slip in
the oracle (wrong kv head, off-by-one in the causal limit, a dropped
rescale, a transposed gather) fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_23_gb300 import workloads as wl
from tests.conftest import GOLDEN

f32 = wl.bf16_bits_to_f32


def _step_cache(w):
    """Cache after the step's copy-on-write and append, via the oracle."""
    k = w.k_cache.copy()
    v = w.v_cache.copy()
    assert oracle.copy_blocks(k, v, w.cow) == 0
    slots, st = oracle.slot_mapping(w.block_tables, w.seq_lens, w.append_lens, w.block_size, w.num_blocks)
    assert st == 0
    assert oracle.kv_append(k, v, w.k_new, w.v_new, slots) == 0
    return k, v


def _contig(k, v, bt, L, bs):
    """Contiguous [L][n_kv][d] K, V of one sequence via numpy fancy indexing."""
    pos = np.arange(L)
    blk = bt[pos // bs]
    return k[blk, :, pos % bs, :], v[blk, :, pos % bs, :]


def _sdpa_reference(w, k, v):
    """torch scaled_dot_product_attention in fp64 per sequence, causal
    within the new tokens, GQA by repeating kv heads."""
    g = w.n_q // w.n_kv
    out = np.zeros((w.total_q, w.n_q, w.head_dim))
    r = 0
    for b in range(w.num_seqs):
        L, ql = int(w.seq_lens[b]), int(w.q_lens[b])
        if ql == 0:
            continue
        kb, vb = _contig(k, v, w.block_tables[b], L, w.block_size)
        K = torch.from_numpy(f32(kb).astype(np.float64)).permute(1, 0, 2)   # [n_kv][L][d]
        V = torch.from_numpy(f32(vb).astype(np.float64)).permute(1, 0, 2)
        K = K.repeat_interleave(g, 0)
        V = V.repeat_interleave(g, 0)
        Q = torch.from_numpy(f32(w.q[r:r + ql]).astype(np.float64)).permute(1, 0, 2)  # [n_q][ql][d]
        i = torch.arange(ql)[:, None]
        t = torch.arange(L)[None, :]
        mask = t <= (L - ql + i)
        o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=w.scale)
        out[r:r + ql] = o.permute(1, 0, 2).numpy()
        r += ql
    return out


@pytest.mark.parametrize("name", ["tiny", "decode", "mix", "spec", "long"])
def test_attention_matches_torch_sdpa_fp64(name):
    w = wl.SMALL[name]()
    if name == "long":  # keep the CPU run short: drop to 1 long decode + the chunk
        w = wl.long_context(B=1, ctx=3000, chunk=40, chunk_prefix=300, partition_tokens=1024, seed=4)
    k, v = _step_cache(w)
    out, st = oracle.attention(w.q, k, v, w.block_tables, w.seq_lens, w.q_lens, w.scale)
    assert st == 0
    ref = _sdpa_reference(w, k, v)
    assert np.isfinite(out).all()
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_one_token_context_is_v():
    """Closed form: with one visible position, softmax weight is 1 and the
    output is V_0 exactly."""
    rng = np.random.default_rng(7)
    nb, nkv, bs, d, nq = 3, 2, 4, 32, 6
    k = wl.to_bf16_bits(rng.standard_normal((nb, nkv, bs, d), dtype=np.float32))
    v = wl.to_bf16_bits(rng.standard_normal((nb, nkv, bs, d), dtype=np.float32))
    q = wl.to_bf16_bits(rng.standard_normal((1, nq, d), dtype=np.float32))
    bt = np.array([[2]], np.int32)
    out, st = oracle.attention(q, k, v, bt, np.array([1], np.int32), np.array([1], np.int32), 0.3)
    assert st == 0
    g = nq // nkv
    for h in range(nq):
        assert np.array_equal(out[0, h], f32(v[2, h // g, 0]).astype(np.float64))


def test_equal_keys_give_mean_of_v():
    """Closed form: equal scores give uniform weights, the output is the mean
    of the visible V rows."""
    rng = np.random.default_rng(8)
    nb, nkv, bs, d = 4, 1, 4, 16
    krow = wl.to_bf16_bits(rng.standard_normal(d, dtype=np.float32))
    k = np.broadcast_to(krow, (nb, nkv, bs, d)).copy()
    v = wl.to_bf16_bits(rng.standard_normal((nb, nkv, bs, d), dtype=np.float32))
    q = wl.to_bf16_bits(rng.standard_normal((3, 2, d), dtype=np.float32))
    bt = np.array([[3, 0, 1]], np.int32)
    L, ql = 11, 3
    out, st = oracle.attention(q, k, v, bt, np.array([L], np.int32), np.array([ql], np.int32), 0.125)
    assert st == 0
    _, vb = _contig(k, v, bt[0], L, bs)
    vf = f32(vb).astype(np.float64)[:, 0]
    for i in range(ql):
        n = L - ql + i + 1
        for h in range(2):
            np.testing.assert_allclose(out[i, h], vf[:n].mean(0), rtol=1e-13, atol=1e-14)


def _example_31_2_inputs():
    """Scores ln 4, ln 2, 0, 0 (weights 4, 2, 1, 1) and scalar values 1, 3, 0, 2
    carried in component 0 of V; scale = ln 2 and q = e_0, K_t[0] in {2, 1, 0, 0}
    make the scores exact multiples of ln 2."""
    d, bs = 8, 2
    k = np.zeros((2, 1, bs, d), np.float32)
    v = np.zeros((2, 1, bs, d), np.float32)
    k[:, 0, :, 0] = np.array([[2, 1], [0, 0]], np.float32)
    v[:, 0, :, 0] = np.array([[1, 3], [0, 2]], np.float32)
    q = np.zeros((1, 1, d), np.float32)
    q[0, 0, 0] = 1.0
    return (wl.to_bf16_bits(q), wl.to_bf16_bits(k), wl.to_bf16_bits(v),
            np.array([[0, 1]], np.int32), np.array([4], np.int32), np.array([1], np.int32), math.log(2.0))


def test_example_31_2_tile_statistics():
    """Chapter 31 Serving Efficiency, Example 31.2: combining tile statistics
    gives 1.5; averaging the tile outputs gives the wrong 4/3."""
    gold = json.load(open(os.path.join(GOLDEN, "tile_combine_example_31_2.json")))
    q, k, v, bt, sl, ql, scale = _example_31_2_inputs()
    out, st = oracle.attention(q, k, v, bt, sl, ql, scale)
    assert st == 0
    assert out[0, 0, 0] == pytest.approx(gold["merged"], abs=1e-14)
    out2, st, po, pm, pl = oracle.attention_split(q, k, v, bt, sl, ql, scale, 2, want_partials=True)
    assert st == 0
    assert out2[0, 0, 0] == pytest.approx(gold["merged"], abs=1e-14)
    # the page's unnormalised tile denominators are l_k * exp(m_k), numerators o_k times that
    den = pl[0, 0] * np.exp(pm[0, 0])
    num = po[0, 0, :, 0] * den
    np.testing.assert_allclose(den, gold["tile_denominators"], rtol=1e-13)
    np.testing.assert_allclose(num, gold["tile_numerators"], rtol=1e-13)
    wrong = po[0, 0, :, 0].mean()
    assert wrong == pytest.approx(gold["wrong_equal_average"], abs=1e-13)
    assert abs(wrong - out2[0, 0, 0]) > 0.1


@pytest.mark.parametrize("P", [2, 16, 48, 1000])
def test_split_merge_equals_plain(P):
    """Flash-Decoding's partition + log-sum-exp merge reaches the plain
    softmax result (including partitions a causal query cannot see)."""
    for name in ["mix", "spec"]:
        w = wl.SMALL[name]()
        k, v = _step_cache(w)
        a, st = oracle.attention(w.q, k, v, w.block_tables, w.seq_lens, w.q_lens, w.scale)
        b, st2 = oracle.attention_split(w.q, k, v, w.block_tables, w.seq_lens, w.q_lens, w.scale, P)
        assert st == 0 and st2 == 0
        np.testing.assert_allclose(b, a, rtol=1e-12, atol=1e-13)


def test_split_empty_partition_has_zero_weight():
    """A partition past a causal query's last visible position has m = -inf,
    l = 0 and must not change the result."""
    w = wl.SMALL["spec"]()
    k, v = _step_cache(w)
    P = 8
    out, st, po, pm, pl = oracle.attention_split(w.q, k, v, w.block_tables, w.seq_lens, w.q_lens, w.scale,
                                                 P, want_partials=True)
    assert st == 0
    # first sequence, first draft query: positions past L-ql are invisible
    L, ql = int(w.seq_lens[0]), int(w.q_lens[0])
    last = L - ql
    npm = pm.shape[2]
    for kk in range(npm):
        if kk * P > last:
            assert pm[0, 0, kk] == -np.inf and pl[0, 0, kk] == 0.0
    assert np.isfinite(out).all()


def test_online_softmax_fp32_restatement_agrees():
    """An fp32 numpy restatement of the FlashAttention loop ("Inference at
    Scale", section 07: per block S, m', P, l, O rescale, final O/l) agrees
    with the fp64 oracle to fp32 rounding (the page's code sample 3a shows
    errors near 1e-6)."""
    w = wl.SMALL["mix"]()
    k, v = _step_cache(w)
    ref, st = oracle.attention(w.q, k, v, w.block_tables, w.seq_lens, w.q_lens, w.scale)
    g = w.n_q // w.n_kv
    for b in range(w.num_seqs):
        L = int(w.seq_lens[b])
        kb, vb = _contig(k, v, w.block_tables[b], L, w.block_size)
        for h in range(w.n_q):
            qv = f32(w.q[b, h]).astype(np.float32)
            K = f32(kb[:, h // g]).astype(np.float32)
            V = f32(vb[:, h // g]).astype(np.float32)
            m = np.float32(-np.inf)
            l = np.float32(0)
            o = np.zeros(w.head_dim, np.float32)
            for j in range(0, L, 16):
                s = (K[j:j + 16] @ qv) * np.float32(w.scale)
                mn = np.maximum(m, s.max())
                p = np.exp(s - mn)
                c = np.exp(m - mn)
                l = l * c + p.sum()
                o = o * c + p @ V[j:j + 16]
                m = mn
            o = o / l
            np.testing.assert_allclose(o, ref[b, h], rtol=2e-5, atol=2e-5)


def test_paged_layout_invariant_under_block_permutation():
    """Moving physical blocks (and rewriting the tables) leaves the oracle's
    output bit-identical: the result depends on logical contents only."""
    w = wl.SMALL["mix"]()
    k, v = _step_cache(w)
    a, _ = oracle.attention(w.q, k, v, w.block_tables, w.seq_lens, w.q_lens, w.scale)
    perm = np.random.default_rng(11).permutation(w.num_blocks)
    k2 = np.empty_like(k)
    v2 = np.empty_like(v)
    k2[perm] = k
    v2[perm] = v
    bt2 = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    b, _ = oracle.attention(w.q, k2, v2, bt2, w.seq_lens, w.q_lens, w.scale)
    assert np.array_equal(a, b)


def test_tiny_shared_prefix_sees_identical_kv():
    """Chapter 31, 31.3: A=[10,11,12,13] and B=[10,11,12,14] share three
    positions; after the copy-on-write and B's append their gathered K/V are
    bit-identical at positions 0..2 and differ at position 3."""
    w = wl.tiny()
    k, v = _step_cache(w)
    kg, vg, st = oracle.gather_kv(k, v, w.block_tables, w.seq_lens)
    assert st == 0
    A = slice(0, 4)
    B = slice(4, 8)
    assert np.array_equal(kg[A][:3], kg[B][:3]) and np.array_equal(vg[A][:3], vg[B][:3])
    assert not np.array_equal(kg[A][3], kg[B][3])
    assert np.array_equal(kg[B][3], w.k_new[0]) and np.array_equal(vg[B][3], w.v_new[0])
    toks = w.meta["tokens"]
    shared = 0
    while toks["A"][shared] == toks["B"][shared]:
        shared += 1
    assert shared == 3
    assert not np.isnan(f32(kg)).any()


def test_causal_draft_equals_sequential_decodes():
    """Query i of a q_len = k verification equals a plain decode whose
    context ends at position L - k + i ("Inference at Scale", 08: the
    verify pass is like a short prefill)."""
    w = wl.SMALL["spec"]()
    k, v = _step_cache(w)
    out, _ = oracle.attention(w.q, k, v, w.block_tables, w.seq_lens, w.q_lens, w.scale)
    r = 0
    for b in range(w.num_seqs):
        L, ql = int(w.seq_lens[b]), int(w.q_lens[b])
        for i in range(ql):
            o1, st = oracle.attention(w.q[r + i:r + i + 1], k, v, w.block_tables[b:b + 1],
                                      np.array([L - ql + i + 1], np.int32), np.array([1], np.int32), w.scale)
            assert st == 0
            assert np.array_equal(o1[0], out[r + i])
        r += ql


def test_slot_mapping_golden():
    gold = json.load(open(os.path.join(GOLDEN, "slot_mapping_cases.json")))
    for c in gold["cases"]:
        slots, st = oracle.slot_mapping(np.array(c["block_tables"], np.int32), np.array(c["seq_lens"], np.int32),
                                        np.array(c["append_lens"], np.int32), c["block_size"], c["num_blocks"])
        assert st == 0, c["name"]
        assert slots.tolist() == c["slots"], c["name"]


def test_kv_append_then_gather_roundtrip_and_untouched_bytes():
    w = wl.SMALL["spec"]()
    k0, v0 = w.k_cache.copy(), w.v_cache.copy()
    slots, st = oracle.slot_mapping(w.block_tables, w.seq_lens, w.append_lens, w.block_size, w.num_blocks)
    k, v = k0.copy(), v0.copy()
    assert oracle.kv_append(k, v, w.k_new, w.v_new, slots) == 0
    # bytes outside the written slots are untouched
    flat = np.zeros((w.num_blocks, w.block_size), bool)
    flat.reshape(-1)[slots] = True
    mask = np.broadcast_to(flat[:, None, :, None], k.shape)
    assert np.array_equal(k[~mask], k0[~mask]) and np.array_equal(v[~mask], v0[~mask])
    # the appended rows sit at the last positions of each sequence
    kg, vg, st = oracle.gather_kv(k, v, w.block_tables, w.seq_lens)
    assert st == 0
    o = 0
    r = 0
    for b in range(w.num_seqs):
        L, A = int(w.seq_lens[b]), int(w.append_lens[b])
        assert np.array_equal(kg[o + L - A:o + L], w.k_new[r:r + A])
        assert np.array_equal(vg[o + L - A:o + L], w.v_new[r:r + A])
        o += L
        r += A
    assert not np.isnan(f32(kg)).any()


def test_kv_append_skip_and_bad_slot():
    k = np.zeros((2, 1, 2, 4), np.uint16)
    v = np.zeros_like(k)
    kn = np.arange(12, dtype=np.uint16).reshape(3, 1, 4) + 1
    st = oracle.kv_append(k, v, kn, kn, np.array([3, -1, 4], np.int64))
    assert st == 8
    assert np.array_equal(k[1, 0, 1], kn[0, 0]) and k.sum() == kn[0].sum()


def test_copy_blocks_copies_and_reports_bad_pairs():
    rng = np.random.default_rng(3)
    k = rng.integers(0, 60000, (5, 2, 4, 8)).astype(np.uint16)
    v = rng.integers(0, 60000, (5, 2, 4, 8)).astype(np.uint16)
    k0, v0 = k.copy(), v.copy()
    st = oracle.copy_blocks(k, v, np.array([[1, 3], [4, 0], [2, 9]], np.int32))
    assert st == 64
    assert np.array_equal(k[3], k0[1]) and np.array_equal(v[0], v0[4])
    assert np.array_equal(k[[1, 2, 4]], k0[[1, 2, 4]])


def test_gather_identity_table_is_pool_transpose():
    """With block table [0, 1, ..., n-1] the gather is the pool read in block
    order: [n][n_kv][bs][d] transposed to [n*bs][n_kv][d]."""
    rng = np.random.default_rng(4)
    nb, nkv, bs, d = 3, 2, 4, 8
    k = rng.integers(0, 60000, (nb, nkv, bs, d)).astype(np.uint16)
    v = rng.integers(0, 60000, (nb, nkv, bs, d)).astype(np.uint16)
    kg, vg, st = oracle.gather_kv(k, v, np.array([[0, 1, 2]], np.int32), np.array([12], np.int32))
    assert st == 0
    assert np.array_equal(kg, k.transpose(0, 2, 1, 3).reshape(12, nkv, d))
    assert np.array_equal(vg, v.transpose(0, 2, 1, 3).reshape(12, nkv, d))


def test_attention_flags_invalid_inputs():
    w = wl.tiny()
    k, v = _step_cache(w)
    bt = w.block_tables.copy()
    bt[2, 0] = 99                          # C's block id outside the pool
    sl = w.seq_lens.copy()
    ql = w.q_lens.copy()
    sl[1] = 5                              # B longer than its table allows
    out, st = oracle.attention(w.q, k, v, bt, sl, ql, w.scale)
    assert st & 1 and st & 2
    assert np.isnan(out[1]).all() and np.isnan(out[2]).all() and np.isfinite(out[0]).all()
    ql2 = ql.copy()
    ql2[0] = 5                             # more queries than positions
    out, st = oracle.attention(np.concatenate([w.q, w.q, w.q[:1]]), k, v, w.block_tables, w.seq_lens, ql2, w.scale)
    assert st & 4


def test_greedy_accept_golden_cases():
    gold = json.load(open(os.path.join(GOLDEN, "greedy_accept_cases.json")))
    for c in gold["cases"]:
        lg = np.array(c["logits"], np.float32)[None]
        dr = np.array(c["draft"], np.int32)[None]
        acc, nxt, am = oracle.spec_accept_greedy(lg, dr)
        assert am[0].tolist() == c["argmax"], c["name"]
        assert int(acc[0]) == c["accepted"], c["name"]
        assert int(nxt[0]) == c["next_token"], c["name"]


def test_greedy_argmax_matches_numpy():
    rng = np.random.default_rng(5)
    lg = rng.standard_normal((7, 4, 3001)).astype(np.float32)
    lg[0, 1, 100] = np.nan
    lg[0, 1, 50] = np.nan
    lg[2, 0, :] = 1.0
    lg[3, 2, 7] = lg[3, 2, 9] = 50.0
    dr = rng.integers(0, 3001, (7, 3)).astype(np.int32)
    acc, nxt, am = oracle.spec_accept_greedy(lg, dr)
    assert np.array_equal(am, np.argmax(lg, axis=-1))


def test_expected_tokens_per_round_closed_form_matches_pages():
    """The pages print the expected tokens per verification pass; the closed
    form (1 - a^(k+1)) / (1 - a) reproduces every printed value."""
    gold = json.load(open(os.path.join(GOLDEN, "expected_tokens_per_round.json")))
    for row in gold["printed"]:
        a, k = row["alpha"], row["k"]
        e = (1 - a ** (k + 1)) / (1 - a)
        # the pages print truncated or rounded figures: within one unit of the last digit
        assert abs(e - row["tokens"]) < 10.0 ** -row["digits"], (row, e)
        # and, where the print is precise enough, the off-by-one readings (k or
        # k+2 terms instead of k+1) do not fit
        if row["digits"] == 2 and k <= 8:
            for kk in (k - 1, k + 1):
                assert abs((1 - a ** (kk + 1)) / (1 - a) - row["tokens"]) >= 10.0 ** -row["digits"]


def test_greedy_acceptance_statistics_are_geometric():
    """With drafts agreeing with the argmax independently at rate a, the
    oracle's accepted length is truncated-geometric: P(A = j) = a^j (1 - a)
    for j < k, P(A = k) = a^k, so E[A + 1] = (1 - a^(k+1)) / (1 - a)
    ("Spending the Idle" 12.4; "Inference at Scale" 08).  Checks the
    acceptance count and the draft generator together."""
    w = wl.spec(B=3000, lo=8, hi=8, k=4, vocab=64, alpha=0.7, seed=9, n_q=1, n_kv=1, d=8, bs=4)
    acc, nxt, am = oracle.spec_accept_greedy(w.logits, w.draft)
    k, a = 4, 0.7
    mean = acc.mean() + 1
    assert mean == pytest.approx((1 - a ** (k + 1)) / (1 - a), abs=0.08)
    hist = np.bincount(acc, minlength=k + 1) / len(acc)
    expect = np.array([a ** j * (1 - a) for j in range(k)] + [a ** k])
    np.testing.assert_allclose(hist, expect, atol=0.035)
    # next token is the argmax at the first rejected (or bonus) position
    assert np.array_equal(nxt, am[np.arange(len(acc)), acc])
