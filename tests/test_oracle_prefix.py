"""Pins of the oracle's prefix-cache block hashes and cache semantics ("Inference
at Scale" section 05, prefix caching; "Chapter 31 Serving Efficiency" 31.3 and
exercise 4), on CPU."""
import json
import os

import numpy as np
import pytest

import oracle
from tests.conftest import GOLDEN

EX = json.load(open(os.path.join(GOLDEN, "prefix_cache_31_3.json")))


def _pad(seqs):
    T = max(len(s) for s in seqs)
    tok = np.zeros((len(seqs), T), np.int32)
    for i, s in enumerate(seqs):
        tok[i, :len(s)] = s
    return tok, np.array([len(s) for s in seqs], np.int32)


def test_example_31_3():
    names = ["A", "B", "C"]
    tok, lens = _pad([EX["sequences"][n] for n in names])
    bs = EX["block_size"]
    h = oracle.prefix_hash(tok, lens, bs, 2)
    assert (h[0, 0] == h[1, 0]).all()            # shared first block
    assert (h[0, 1] != h[1, 1]).any()            # 13 vs 14
    assert (h[2, 0] != h[0, 0]).any()
    cache = oracle.PrefixCache()
    bt = np.array([[100, 101], [-1, -1], [-1, -1]], np.int32)
    cache.insert(h[:1], bt[:1], np.array([0]), np.array([2]))
    for k, e in cache.d.items():
        e[0] = e[2][0]
    got = cache.lookup(h, lens, bs, bt)
    assert [int(got[i]) for i in range(3)] == [EX["expected_hits"][n] for n in names]
    assert bt[1, 0] == 100


def test_prefix_property_and_parent_dependence():
    g = np.random.default_rng(0)
    bs, nb = 16, 12
    base = g.integers(0, 128000, size=bs * nb).astype(np.int32)
    seqs = []
    for p in [0, 1, 15, 16, 17, 64, 100, bs * nb]:
        s = base.copy()
        if p < len(s):
            s[p:] = g.integers(0, 128000, size=len(s) - p)
        seqs.append(s)
    tok = np.stack(seqs)
    h = oracle.prefix_hash(tok, np.full(len(seqs), bs * nb, np.int32), bs, nb)
    ref = oracle.prefix_hash(base[None], np.array([bs * nb], np.int32), bs, nb)[0]
    for s, p in zip(h, [0, 1, 15, 16, 17, 64, 100, bs * nb]):
        same = np.all(s == ref, axis=1)
        assert same[: p // bs].all() and not same[p // bs:].any()
    # same block content after a different parent: a different key
    t2 = base.copy()
    t2[0] += 1
    h2 = oracle.prefix_hash(t2[None], np.array([bs * nb], np.int32), bs, nb)[0]
    assert not np.any(np.all(h2 == ref, axis=1))


def test_salt_order_and_partial_blocks():
    g = np.random.default_rng(1)
    tok = g.integers(0, 50000, size=(1, 40)).astype(np.int32)
    h0 = oracle.prefix_hash(tok, np.array([40]), 8, 6, salt=0)
    h1 = oracle.prefix_hash(tok, np.array([40]), 8, 6, salt=7)
    assert not np.any(np.all(h0[0, :5] == h1[0, :5], axis=1))      # another computation version
    assert np.array_equal(h0, oracle.prefix_hash(tok, np.array([40]), 8, 6, salt=0))
    sw = tok.copy()
    sw[0, [2, 3]] = sw[0, [3, 2]]                                   # same words, another order (exercise 4)
    hs = oracle.prefix_hash(sw, np.array([40]), 8, 6)
    assert not np.any(np.all(hs[0, :5] == h0[0, :5], axis=1))
    assert (h0[0, 5] == 0).all()                                    # only full blocks are hashed
    hl = oracle.prefix_hash(tok, np.array([39]), 8, 6)
    assert np.array_equal(hl[0, :4], h0[0, :4]) and (hl[0, 4] == 0).all()
    tail = tok.copy()
    tail[0, 39] += 5                                                # a token past the full blocks of len 39
    assert np.array_equal(oracle.prefix_hash(tail, np.array([39]), 8, 6), hl)
    # reserved keys: lane 1 of a real key is never 0 with lane 0 < 2
    g2 = oracle.prefix_hash(g.integers(0, 9, size=(64, 64)).astype(np.int32), np.full(64, 64), 4, 16)
    assert not np.any((g2[..., 1] == 0) & (g2[..., 0] < 2))


def test_lookup_stops_at_first_miss_and_counts_refs():
    g = np.random.default_rng(2)
    bs = 4
    base = g.integers(0, 1000, size=32).astype(np.int32)
    other = base.copy()
    other[9] += 1                                                   # differs in block 2
    tok = np.stack([base, other])
    h = oracle.prefix_hash(tok, np.array([32, 32]), bs, 8)
    cache = oracle.PrefixCache()
    bt = np.arange(16, dtype=np.int32).reshape(2, 8) + 50
    cache.insert(h[:1], bt[:1], np.array([0]), np.array([8]))
    for e in cache.d.values():
        e[0] = e[2][0]
    # remove block 5 of base's chain: a later block cannot match without it
    k5 = (int(h[0, 5, 0]), int(h[0, 5, 1]))
    del cache.d[k5]
    out = np.full((2, 8), -1, np.int32)
    n = cache.lookup(h, np.array([32, 32]), bs, out)
    assert list(n) == [5, 2]
    assert list(out[0, :5]) == list(bt[0, :5]) and (out[0, 5:] == -1).all()
    assert cache.d[(int(h[0, 0, 0]), int(h[0, 0, 1]))][1] == 1 + 2   # insert + two hits
    cache.release(h, n)
    assert cache.d[(int(h[0, 0, 0]), int(h[0, 0, 1]))][1] == 1
