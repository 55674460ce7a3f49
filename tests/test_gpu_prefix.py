"""Prefix-cache block lookup on the GPU vs the oracle ("Inference at Scale"
section 05, prefix caching; "Chapter 31 Serving Efficiency" 31.3).  Hashes,
hit counts, block tables and ref counts are integers, compared exactly; where
several sequences insert one new key in a call, any one of their blocks is a
correct winner, and every one of them must be told that winner."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_23_gb300 as pkv
from tests.conftest import GOLDEN

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _built():
    pkv.build()
    torch.cuda.init()


def t32(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(DEV)


def gpu_hash(tokens, lens, bs, max_blocks, salt=0):
    h = torch.full((len(lens), max_blocks, 2), 0x5A5A, dtype=torch.int64, device=DEV)
    pkv.prefix_hash(h, t32(tokens), t32(lens), bs, salt=salt)
    torch.cuda.synchronize()
    return h.cpu().numpy().view(np.uint64)


@pytest.mark.parametrize("bs,maxb,salt", [(16, 64, 0), (2, 40, 5), (1, 2500, 2 ** 63 + 11), (32, 16, 77)])
def test_hash_matches_oracle(bs, maxb, salt):
    g = np.random.default_rng(bs)
    B = 37
    T = bs * maxb
    tokens = g.integers(-2 ** 31, 2 ** 31 - 1, size=(B, T), dtype=np.int64).astype(np.int32)
    tokens[: B // 2, : T // 3] = tokens[0, : T // 3]          # shared prefixes
    lens = g.integers(0, T + 1, size=B).astype(np.int32)
    lens[0] = T
    got = gpu_hash(tokens, lens, bs, maxb, salt)
    ref = oracle.prefix_hash(tokens, lens, bs, maxb, salt)
    for b in range(B):
        n = lens[b] // bs
        assert np.array_equal(got[b, :n], ref[b, :n]), b
        assert (got[b, n:] == 0x5A5A).all()                    # past the full blocks: untouched


def test_example_31_3():
    ex = json.load(open(os.path.join(GOLDEN, "prefix_cache_31_3.json")))
    names = ["A", "B", "C"]
    seqs = [ex["sequences"][n] for n in names]
    tok = np.zeros((3, 4), np.int32)
    for i, s in enumerate(seqs):
        tok[i, :len(s)] = s
    lens = np.array([len(s) for s in seqs], np.int32)
    bs = ex["block_size"]
    h = torch.from_numpy(gpu_hash(tok, lens, bs, 2).view(np.int64)).to(DEV)
    table = pkv.PrefixTable(64)
    bt = t32([[100, 101], [-1, -1], [-1, -1]])
    res = t32(np.zeros((3, 2)))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.prefix_insert(table, h[:1], bt[:1], t32([0]), t32([2]), res[:1], status=st)
    cached = t32(np.zeros(3))
    pkv.prefix_lookup(table, h, t32(lens), bs, bt, cached)
    torch.cuda.synchronize()
    assert cached.cpu().tolist() == [ex["expected_hits"][n] for n in names]
    assert bt.cpu().numpy()[1, 0] == 100 and int(st.item()) == 0


def _table_dict(table):
    keys, blk, refs = table.entries()
    used = ~(((keys[:, 0] == 0) | (keys[:, 0] == 1)) & (keys[:, 1] == 0))
    return {(int(k[0]), int(k[1])): (int(b), int(r)) for k, b, r in zip(keys[used], blk[used], refs[used])}


def test_scenario_against_oracle():
    g = np.random.default_rng(3)
    bs, maxb, B = 4, 24, 48
    T = bs * maxb
    roots = g.integers(0, 500, size=(4, T)).astype(np.int32)
    tokens = np.empty((B, T), np.int32)
    for b in range(B):
        tokens[b] = roots[b % 4]
        cut = g.integers(0, T)
        tokens[b, cut:] = g.integers(0, 500, size=T - cut)
    lens = g.integers(bs, T + 1, size=B).astype(np.int32)
    hashes = oracle.prefix_hash(tokens, lens, bs, maxb)
    gh = gpu_hash(tokens, lens, bs, maxb)
    full = (np.arange(maxb)[None, :] < (lens // bs)[:, None])
    assert np.array_equal(gh[full], hashes[full])
    h_dev = torch.from_numpy(hashes.view(np.int64)).to(DEV)
    table = pkv.PrefixTable(1024)
    cache = oracle.PrefixCache()
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    # phase 1: the first half inserts all of its full blocks (many shared keys)
    half = B // 2
    blocks = (np.arange(B * maxb, dtype=np.int32) + 1000).reshape(B, maxb)
    first = np.zeros(B, np.int32)
    count = np.where(np.arange(B) < half, lens // bs, 0).astype(np.int32)
    res = t32(np.full((B, maxb), -9))
    pkv.prefix_insert(table, h_dev, t32(blocks), t32(first), t32(count), res, status=st)
    torch.cuda.synchronize()
    claims = cache.insert(hashes, blocks, first, count)
    gt = _table_dict(table)
    r = res.cpu().numpy()
    for k, lst in claims.items():
        blk, refs = gt[k]
        assert blk in [c[2] for c in lst] and refs == len(lst)
        assert all(r[b, j] == blk for b, j, _ in lst)
        cache.d[k][0] = blk
    assert len(gt) == len(cache.d) and int(st.item()) == 0
    # phase 2: everyone looks up; hits stop at the first miss
    bt_gpu = t32(np.full((B, maxb), -1))
    cached = t32(np.zeros(B))
    pkv.prefix_lookup(table, h_dev, t32(lens), bs, bt_gpu, cached)
    bt_ref = np.full((B, maxb), -1, np.int32)
    n_ref = cache.lookup(hashes, lens, bs, bt_ref)
    torch.cuda.synchronize()
    assert np.array_equal(cached.cpu().numpy(), n_ref)
    assert np.array_equal(bt_gpu.cpu().numpy(), bt_ref)
    # phase 3: the second half finishes; ref counts drop
    rel = np.where(np.arange(B) >= half, n_ref, 0).astype(np.int32)
    pkv.prefix_release(table, h_dev, t32(rel), status=st)
    cache.release(hashes, rel)
    torch.cuda.synchronize()
    gt = _table_dict(table)
    assert {k: v[1] for k, v in gt.items()} == {k: v[1] for k, v in cache.d.items()}
    assert int(st.item()) == 0


def test_table_full_and_not_found():
    g = np.random.default_rng(4)
    tokens = g.integers(0, 1000, size=(2, 64)).astype(np.int32)
    lens = np.array([64, 64], np.int32)
    h = torch.from_numpy(gpu_hash(tokens, lens, 4, 16).view(np.int64)).to(DEV)
    table = pkv.PrefixTable(8)
    res = t32(np.zeros((2, 16)))
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    pkv.prefix_insert(table, h, t32(np.arange(32).reshape(2, 16)), t32([0, 0]), t32([16, 16]), res, status=st)
    torch.cuda.synchronize()
    r = res.cpu().numpy()
    assert int(st.item()) & pkv.PKV_STATUS_TABLE_FULL
    assert (r == -1).sum() == 32 - 8 and len(_table_dict(table)) == 8
    st.zero_()
    other = torch.from_numpy(gpu_hash(tokens + 1, lens, 4, 16).view(np.int64)).to(DEV)
    big = pkv.PrefixTable(64)
    pkv.prefix_release(big, other, t32([1, 0]), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & pkv.PKV_STATUS_NOT_FOUND
