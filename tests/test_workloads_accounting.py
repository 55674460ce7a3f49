"""Input generators and byte accounting (CPU only)."""
import json
import math
import os

import numpy as np
import pytest

from paged_kv_cache_23_gb300 import accounting
from paged_kv_cache_23_gb300 import workloads as wl
from tests.conftest import GOLDEN


def test_kv_bytes_per_token_matches_pages():
    gold = json.load(open(os.path.join(GOLDEN, "kv_bytes_per_token.json")))
    for m in gold["models"]:
        b = accounting.kv_bytes_per_token(m["layers"], m["n_kv"], m["head_dim"], gold["bytes_per_value"])
        assert b / 1024 == m["kib_per_token"], m["name"]
        if "gib_at_128k" in m:
            assert round(b * 131072 / 2 ** 30, 2) == m["gib_at_128k"], m["name"]
    per_tok = accounting.kv_bytes_per_token(32, 8, 128, 2)
    for row in gold["llama31_8b_kv_per_seq_gb"]:
        assert round(per_tok * row["context"] / 1e9, 2) == row["gb"]
    # one layer of the 8B shape: 4096 bytes per token
    assert accounting.kv_bytes_per_token(1, 8, 128, 2) == 4096


def test_tiny_layout():
    w = wl.tiny()
    assert w.block_tables.tolist() == [[0, 1], [0, 2], [3, -1]]
    assert w.cow.tolist() == [[1, 2]]
    nan = w.k_cache == wl.BF16_NAN
    assert nan[2].all() and nan[4].all() and nan[5].all()
    assert not nan[[0, 1, 3]].any()
    assert w.scale == 0.125
    b = accounting.step_bytes(w)
    per_row = 4 * 64 * 2 * 2
    assert b["kv_logical"] == 10 * per_row
    assert b["kv_unique"] == 8 * per_row        # A and B read P0 once


def test_generators_are_deterministic():
    a = wl.SMALL["mix"]()
    b = wl.SMALL["mix"]()
    for f in ("k_cache", "v_cache", "block_tables", "seq_lens", "cow", "q", "k_new"):
        assert np.array_equal(getattr(a, f), getattr(b, f)), f


@pytest.mark.parametrize("name", ["decode", "mix", "spec", "long"])
def test_pool_structure(name):
    w = wl.SMALL[name]()
    bs = w.block_size
    used = set()
    for b in range(w.num_seqs):
        L = int(w.seq_lens[b])
        n = -(-L // bs)
        ids = w.block_tables[b, :n]
        assert (ids >= 0).all() and (ids < w.num_blocks).all()
        assert (w.block_tables[b, n:] == -1).all()
        used.update(ids.tolist())
        # rows past the length in the last block are NaN poison
        last = int(ids[-1])
        r = L - (n - 1) * bs
        assert (w.k_cache[last, :, r:] == wl.BF16_NAN).all()
    used.update(w.cow[:, 1].tolist())
    assert w.num_blocks == math.ceil(1.5 * len(used))
    spare = sorted(set(range(w.num_blocks)) - used)
    assert (w.k_cache[spare] == wl.BF16_NAN).all()
    assert w.q.shape == (w.total_q, w.n_q, w.head_dim)
    assert w.k_new.shape == (int(w.append_lens.sum()), w.n_kv, w.head_dim)


def test_mix_sharing_and_copy_on_write():
    w = wl.mix(B=40, median=60, sigma=1.0, clip=(16, 600), share=0.5, prefix=64, seed=5)
    bs = w.block_size
    sharers = w.meta["sharers"]
    assert len(sharers) == 20
    prefix_ids = None
    n_cow = 0
    for b in sharers:
        L = int(w.seq_lens[b])
        cached = L - 1
        full = min(cached, 64) // bs
        ids = w.block_tables[b, :full].tolist()
        if prefix_ids is None or len(ids) > len(prefix_ids):
            if prefix_ids is not None:
                assert ids[:len(prefix_ids)] == prefix_ids
            prefix_ids = ids
        else:
            assert ids == prefix_ids[:len(ids)]
        if cached < 64 and cached % bs:
            n_cow += 1
            dst = int(w.block_tables[b, cached // bs])
            assert [prefix_ids_src for prefix_ids_src, d in w.cow.tolist() if d == dst]
    assert n_cow == w.cow.shape[0]
    lens = w.seq_lens
    assert lens.min() >= 16 and lens.max() <= 600


def test_spec_draft_agreement_rate():
    w = wl.spec(B=400, lo=10, hi=10, k=5, vocab=50, alpha=0.7, seed=1, n_q=1, n_kv=1, d=8, bs=4)
    top = w.logits[:, :5].argmax(-1)
    rate = (w.draft == top).mean()
    assert abs(rate - 0.7) < 0.04
    assert ((w.draft >= 0) & (w.draft < 50)).all()


def test_step_bytes_full_mix_is_in_expected_range():
    """The headline workload moves about 1.7 GB of logical K/V (sigma = 1
    log-normal around 1024 tokens, 4096 bytes per token per layer) and
    fewer unique bytes because half the batch shares a 2048-token prefix."""
    w = wl.mix(B=256, median=1024, sigma=1.0, clip=(16, 32768), share=0.5, prefix=2048, seed=0,
               n_q=32, n_kv=8, d=8, bs=16)   # tiny head_dim: structure only
    b = accounting.step_bytes(w)
    scale = 128 / 8
    logical = b["kv_logical"] * scale
    unique = b["kv_unique"] * scale
    assert 1.2e9 < logical < 2.6e9
    assert unique < logical
