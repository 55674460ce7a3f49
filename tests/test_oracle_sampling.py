"""Pins of the oracle's stochastic speculative acceptance (modified rejection
sampling) to the pages' worked examples and to the mathematics, on CPU.

The oracle is used as a black box: the acceptance probability is measured
over a grid of uniforms r, the residual distribution over a grid of s, and
the output distribution of the first token is assembled from them and
compared with the target p ("Chapter 31 Serving Efficiency" 31.5, Example
31.3; exercise 3; "Inference at Scale" section 08: the output is distributed
exactly as p).
"""
import json
import os

import numpy as np
import pytest

import oracle
from paged_kv_cache_23_gb300 import workloads as wl
from tests.conftest import GOLDEN

N = 4096  # grid points per uniform
GRID = ((np.arange(N) + 0.5) / N).astype(np.float32)


def _accept_rate(p, q, x):
    """Fraction of the r grid for which draft x (k = 1) is accepted."""
    V = len(p)
    P = np.tile(np.array([p, p], np.float32), (N, 1, 1))
    Q = np.tile(np.array([q], np.float32), (N, 1, 1))
    acc, _, st = oracle.spec_accept_sample(P, Q, np.full((N, 1), x, np.int32), GRID.reshape(N, 1),
                                           np.zeros(N, np.float32))
    assert st == 0
    return acc.mean()


def _residual_dist(p, q):
    """Distribution of the replacement token after a forced rejection."""
    V = len(p)
    # a draft with p(x) < q(x) and r just below 1 is always rejected
    x = int(np.argmax(np.array(q) - np.array(p)))
    P = np.tile(np.array([p, p], np.float32), (N, 1, 1))
    Q = np.tile(np.array([q], np.float32), (N, 1, 1))
    acc, nxt, st = oracle.spec_accept_sample(P, Q, np.full((N, 1), x, np.int32),
                                             np.full((N, 1), 0.99999994, np.float32), GRID)
    assert st == 0 and (acc == 0).all()
    return np.bincount(nxt, minlength=V) / N


def _output_dist(p, q):
    V = len(p)
    A = np.array([_accept_rate(p, q, x) for x in range(V)])
    R = _residual_dist(p, q)
    q = np.array(q, np.float64)
    out = q * A + (q * (1 - A)).sum() * R
    return A, R, out


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "rejection_sampling_examples.json")))["cases"],
                         ids=lambda c: c["name"])
def test_pages_examples(case):
    A, R, out = _output_dist(case["p"], case["q"])
    assert np.allclose(A, case["acceptance"], atol=2.0 / N)
    assert np.allclose(np.array(case["q"]) * A, case["accepted_mass"], atol=2.0 / N)
    assert np.allclose(R, case["residual"], atol=2.0 / N)
    assert np.allclose(out, case["final"], atol=3.0 / N)
    if "wrong_resample_from_p_first" in case:
        # the wrong rule (resample from p) lands elsewhere; ours does not
        assert abs(out[0] - case["wrong_resample_from_p_first"]) > 0.1


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_output_distribution_is_target(seed):
    """Random small distributions: acceptance = min(1, p/q), residual =
    norm(max(0, p - q)), and the first output token is distributed as p."""
    g = np.random.default_rng(seed)
    V = 6
    p = g.dirichlet(np.ones(V)).astype(np.float32)
    q = g.dirichlet(np.ones(V)).astype(np.float32)
    A, R, out = _output_dist(p, q)
    p64, q64 = p.astype(np.float64), q.astype(np.float64)
    assert np.allclose(A, np.minimum(1.0, p64 / q64), atol=2.0 / N)
    res = np.maximum(0.0, p64 - q64)
    assert np.allclose(R, res / res.sum(), atol=2.0 / N)
    assert np.allclose(out, p64, atol=4.0 / N)


def test_one_hot_reduces_to_greedy():
    """With one-hot p and q the rule is greedy acceptance ("Inference at
    Scale" 08): compare with the greedy oracle on the same argmaxes."""
    g = np.random.default_rng(5)
    B, k, V = 64, 4, 9
    top = g.integers(0, V, size=(B, k + 1))
    agree = g.random((B, k)) < 0.6
    draft = np.where(agree, top[:, :k], (top[:, :k] + 1 + g.integers(0, V - 1, size=(B, k))) % V).astype(np.int32)
    p = np.zeros((B, k + 1, V), np.float32)
    np.put_along_axis(p, top[..., None], 1.0, axis=-1)
    q = np.zeros((B, k, V), np.float32)
    np.put_along_axis(q, draft[..., None].astype(np.int64), 1.0, axis=-1)
    acc, nxt, st = oracle.spec_accept_sample(p, q, draft, g.random((B, k), dtype=np.float32),
                                             g.random(B, dtype=np.float32))
    acc_g, nxt_g, _ = oracle.spec_accept_greedy(p, draft)
    assert st == 0
    assert (acc == acc_g).all() and (nxt == nxt_g).all()


def test_expected_accepted_matches_independent_positions():
    """Each position accepts with probability alpha_j = sum min(p_j, q_j);
    positions are independent given the drafts' and uniforms' independence, so
    E[accepted] = sum_j prod_{i<=j} alpha_i -- the pages' expected-tokens
    argument ("Inference at Scale" 08, "Serving": (1 - a^{k+1}) / (1 - a) - 1
    for equal a)."""
    x = wl.spec_sample(B=6000, k=3, vocab=50, temp=1.5, noise=0.8, seed=11)
    acc, nxt, st = oracle.spec_accept_sample(x.p, x.q, x.draft, x.r, x.s)
    assert st == 0
    alpha = np.minimum(x.p[:, :3].astype(np.float64), x.q).sum(-1)          # [B][k]
    expect = np.cumprod(alpha, axis=1).sum(1)                              # per row
    diff = acc.mean() - expect.mean()
    sd = acc.std() / np.sqrt(len(acc))
    assert abs(diff) < 4 * sd + 1e-3, (acc.mean(), expect.mean())
    # equal-alpha closed form on the same machinery
    a = 0.7
    assert abs(((1 - a ** 4) / (1 - a) - 1) - sum(a ** j for j in range(1, 4))) < 1e-12


@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "rejection_sampling_examples.json")))[
    "inverse_cdf_cases"], ids=lambda c: c["name"])
def test_inverse_cdf_cases(case):
    """All drafts accepted -> the next token is drawn from p_k with s."""
    V = len(case["p"])
    p = np.array([[[1.0] + [0.0] * (V - 1), case["p"]]], np.float32)
    q = np.array([[[1.0] + [0.0] * (V - 1)]], np.float32)
    acc, nxt, st = oracle.spec_accept_sample(p, q, np.array([[0]], np.int32), np.array([[0.5]], np.float32),
                                             np.array([case["s"]], np.float32))
    assert st == 0 and acc[0] == 1 and nxt[0] == case["next"]


def test_bad_draft_and_degenerate_distributions():
    V = 4
    p = np.array([[[0.1, 0.2, 0.3, 0.4], [0.25] * 4]], np.float32)
    q = np.array([[[0.25] * 4]], np.float32)
    # draft outside the vocab: rejected at that position, status bit 128
    acc, nxt, st = oracle.spec_accept_sample(p, q, np.array([[V]], np.int32), np.array([[0.0]], np.float32),
                                             np.array([0.0], np.float32))
    assert st & 128 and acc[0] == 0 and 0 <= nxt[0] < V
    # residual with no positive part falls back to p
    p2 = np.array([[[0.05, 0.05, 0.05, 0.05], [0.25] * 4]], np.float32)
    acc, nxt, st = oracle.spec_accept_sample(p2, q, np.array([[2]], np.int32), np.array([[0.9]], np.float32),
                                             np.array([0.6], np.float32))
    assert st == 0 and acc[0] == 0 and nxt[0] == 2
    # nothing positive at all: next = -1, status bit 256
    p3 = np.zeros((1, 2, V), np.float32)
    acc, nxt, st = oracle.spec_accept_sample(p3, q, np.array([[1]], np.int32), np.array([[0.5]], np.float32),
                                             np.array([0.5], np.float32))
    assert st & 256 and acc[0] == 0 and nxt[0] == -1
