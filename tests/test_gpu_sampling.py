"""Stochastic speculative acceptance on the GPU vs the CPU oracle (GPU
required).  Every result is an integer decided by fp32 comparisons and an
integer inverse CDF that both sides define identically, so accepted lengths
and drawn tokens are compared bit-exactly."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_23_gb300 as pkv
from paged_kv_cache_23_gb300 import workloads as wl
from tests.conftest import GOLDEN

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    pkv.build()
    torch.cuda.init()


def gpu_sample(p, q, draft, r, s):
    dev = torch.device("cuda")
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).to(dev, dt)
    B = p.shape[0]
    acc = torch.full((B,), -7, dtype=torch.int32, device=dev)
    nxt = torch.full((B,), -7, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    pkv.spec_accept_sample(t(p, torch.float32), t(q, torch.float32), t(draft, torch.int32), t(r, torch.float32),
                           t(s, torch.float32), acc, nxt, status=st)
    torch.cuda.synchronize()
    return acc.cpu().numpy(), nxt.cpu().numpy(), int(st.item())


def check(p, q, draft, r, s):
    ra, rn, rs = oracle.spec_accept_sample(p, q, draft, r, s)
    ga, gn, gs = gpu_sample(p, q, draft, r, s)
    assert np.array_equal(ga, ra), np.nonzero(ga != ra)[0][:10]
    assert np.array_equal(gn, rn), np.nonzero(gn != rn)[0][:10]
    assert gs == rs
    return ga, gn


def test_pages_examples_grid():
    """Example 31.3 and exercise 3 ("Chapter 31 Serving Efficiency"): every
    (draft, r, s) of a grid gives the oracle's integers."""
    cases = json.load(open(os.path.join(GOLDEN, "rejection_sampling_examples.json")))["cases"]
    N = 64
    g = ((np.arange(N) + 0.5) / N).astype(np.float32)
    for c in cases:
        pr = np.array(c["p"], np.float32)
        qr = np.array(c["q"], np.float32)
        xs, rs, ss = np.meshgrid(np.arange(2), g, g, indexing="ij")
        B = xs.size
        p = np.tile(np.stack([pr, pr]), (B, 1, 1))
        q = np.tile(qr[None], (B, 1, 1))
        acc, nxt = check(p, q, xs.reshape(B, 1).astype(np.int32), rs.reshape(B, 1), ss.reshape(B))
        # Lyon (x = 1) is always accepted; a rejected Paris always becomes Lyon
        x = xs.reshape(B)
        assert (acc[x == 1] == 1).all()
        assert (nxt[(x == 0) & (acc == 0)] == 1).all()


@pytest.mark.parametrize("B,k,V,seed", [(64, 5, 1000, 0), (37, 3, 1001, 1), (16, 1, 4, 2), (8, 40, 300, 3),
                                        (300, 2, 64, 4), (5, 5, 1, 5), (20, 4, 4099, 6)])
def test_random_matches_oracle(B, k, V, seed):
    x = wl.spec_sample(B=B, k=k, vocab=V, seed=seed)
    check(x.p, x.q, x.draft, x.r, x.s)


def test_full_size():
    """The spec workload's shape: 32 sequences, k = 5, vocab 128256."""
    x = wl.spec_sample(B=32, k=5, vocab=128256, seed=0)
    acc, nxt = check(x.p, x.q, x.draft, x.r, x.s)
    assert 0 < acc.mean() < 5


def test_edges():
    g = np.random.default_rng(9)
    V = 257
    x = wl.spec_sample(B=12, k=3, vocab=V, seed=9)
    p, q, d, r, s = x.p.copy(), x.q.copy(), x.draft.copy(), x.r.copy(), x.s.copy()
    d[0, 0] = V            # bad token at the first position
    d[1, 1] = -1           # bad token after an accepted one (if accepted)
    r[1, 0] = 0.0
    q[2, 0] = p[2, 0] * 0.5  # residual has weight everywhere p > q
    p[3] = 0.0
    r[3, 0] = 0.5            # p = 0 at the draft: rejected, nothing positive anywhere
    s[4] = 0.0
    s[5] = np.float32(0.99999994)
    p[6, 0, :] = np.nan      # NaN target row: rejected, residual weights 0 -> fallback to p (also 0)
    r[7, :] = 0.0            # r = 0 accepts whenever p(x) > 0
    check(p, q, d, r, s)


def test_deterministic():
    x = wl.spec_sample(B=48, k=4, vocab=5000, seed=12)
    a1 = gpu_sample(x.p, x.q, x.draft, x.r, x.s)
    a2 = gpu_sample(x.p, x.q, x.draft, x.r, x.s)
    assert all(np.array_equal(u, v) for u, v in zip(a1[:2], a2[:2]))
