"""Pins of the oracle's greedy acceptance and commit (oracle/accept.py).

* hand-worked cases (tests/golden/accept_hand_examples.json), one slot each;
* the same cases as one ragged batch (plus an empty slot) give the same
  per-slot results;
* brute force: argmax by a plain Python scan (first strict maximum) on small
  vocabularies, including many ties;
* invariants on random batches: 0 <= a <= T - 1, committed = ctx_len - (T-1-a),
  drafts equal to the argmax chain are all accepted, a wrong first draft
  accepts nothing.
"""
import json
import os

import numpy as np
import pytest

from oracle.accept import argmax_lowest, greedy_accept

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "accept_hand_examples.json")
CASES = json.load(open(GOLDEN))["cases"]


def _one(case):
    lg = np.array(case["logits"], np.float64)
    T = lg.shape[0]
    return greedy_accept(lg, [0], [T], np.array(case["tokens"], np.int32), [case["ctx_len"]])


@pytest.mark.parametrize("case", CASES, ids=lambda c: c["name"][:40])
def test_hand_examples(case):
    a, nxt, com = _one(case)
    assert [int(a[0]), int(nxt[0]), int(com[0])] == case["expect"]


def test_ragged_batch_matches_solo():
    lgs, toks, offs, nq, ctx = [], [], [], [], []
    r = 0
    for i, case in enumerate(CASES):
        if i == 3:                                   # an empty slot in the middle
            offs.append(r); nq.append(0); ctx.append(17)
        lg = np.array(case["logits"], np.float64)
        lgs.append(lg); toks += case["tokens"]
        offs.append(r); nq.append(lg.shape[0]); ctx.append(case["ctx_len"])
        r += lg.shape[0]
    a, nxt, com = greedy_accept(np.concatenate(lgs), offs, nq, np.array(toks, np.int32), ctx)
    got = [[int(a[b]), int(nxt[b]), int(com[b])] for b in range(len(nq)) if nq[b] > 0]
    assert got == [c["expect"] for c in CASES]
    empty = nq.index(0)
    assert (int(a[empty]), int(nxt[empty]), int(com[empty])) == (0, -1, 17)


def _scan_argmax(row):
    best, idx = None, -1
    for i, v in enumerate(row):
        if best is None or v > best:
            best, idx = v, i
    return idx


def test_argmax_brute_force_with_ties():
    rng = np.random.default_rng(0)
    for _ in range(300):
        V = int(rng.integers(1, 40))
        row = rng.integers(-3, 4, size=V).astype(np.float64)     # many ties
        assert argmax_lowest(row) == _scan_argmax(list(row))


def test_invariants_random():
    rng = np.random.default_rng(1)
    S, V = 9, 50
    nq = rng.integers(0, 9, size=S)
    offs = np.concatenate([[0], np.cumsum(nq)[:-1]])
    rows = int(nq.sum())
    lg = rng.standard_normal((rows, V))
    ctx = rng.integers(20, 1000, size=S)
    g = lg.argmax(axis=1)
    # drafts: follow the argmax chain for a random prefix, then a wrong token
    toks = np.zeros(rows, np.int32)
    want_a = np.zeros(S, np.int64)
    for b in range(S):
        T = int(nq[b])
        if T == 0:
            continue
        k = int(rng.integers(0, T))                  # accepted drafts we plant
        r0 = offs[b]
        toks[r0] = int(rng.integers(0, V))
        for j in range(1, T):
            toks[r0 + j] = g[r0 + j - 1] if j <= k else (g[r0 + j - 1] + 1) % V
        want_a[b] = min(k, T - 1)
    a, nxt, com = greedy_accept(lg, offs, nq, toks, ctx)
    for b in range(S):
        T = int(nq[b])
        if T == 0:
            assert (a[b], nxt[b], com[b]) == (0, -1, ctx[b])
            continue
        assert 0 <= a[b] <= T - 1
        assert a[b] == want_a[b]
        assert nxt[b] == g[offs[b] + a[b]]
        assert com[b] == ctx[b] - (T - 1 - a[b])


# ----------------------------------------------------------------------------- sampled acceptance
from oracle.accept import gumbel_keys, noise_uniform, sample_accept, splitmix64_at, target_prob


def test_splitmix64_published_outputs():
    # the reference generator's first outputs for seed 0
    assert splitmix64_at(0, 0) == 0xE220A8397B1DCDAF
    assert splitmix64_at(0, 1) == 0x6E789E6AA1B965F4
    assert splitmix64_at(0, 2) == 0x06C45D188009454F


def test_noise_uniform_matches_scalar_definition():
    seed, row = 12345, 7
    toks = np.array([0, 1, 2, 1000, 248319])
    got = noise_uniform(seed, row, toks)
    for t, g in zip(toks, got):
        z = splitmix64_at(seed, row * (1 << 32) + int(t))
        assert g == ((z >> 41) + 0.5) / (1 << 23)
        assert np.float32(g) == g                      # exact in float32
    assert np.all((got > 0) & (got < 1))


def test_two_token_hand_case():
    # logits (0, ln 3), tau 1: p(token 1) = 3/4; the residual after rejecting
    # token 1 has one token left, so the replacement is 0 whatever the noise
    lg = np.array([[0.0, np.log(3.0)], [5.0, 0.0]])
    assert abs(target_prob(lg[0], 1.0, 1) - 0.75) < 1e-15
    a, nxt, com = sample_accept(lg, [0], [2], np.array([0, 1]), [9], 1.0, np.array([0.70, 0.5]), seed=3)
    assert int(a[0]) == 1 and int(com[0]) == 9            # accepted; bonus drawn from row 1
    a, nxt, com = sample_accept(lg, [0], [2], np.array([0, 1]), [9], 1.0, np.array([0.80, 0.5]), seed=3)
    assert (int(a[0]), int(nxt[0]), int(com[0])) == (0, 0, 8)


def test_gumbel_max_samples_the_softmax():
    # empirical frequencies of argmax(logit/tau + G) over many independent rows
    lg = np.array([1.0, 0.0, -1.0, 2.0, 0.5])
    tau = 0.7
    n = 40000
    counts = np.zeros(5)
    for row in range(n):
        counts[int(np.argmax(gumbel_keys(lg, tau, 99, row)))] += 1
    p = np.exp(lg / tau - (lg / tau).max())
    p /= p.sum()
    assert np.max(np.abs(counts / n - p)) < 0.012


def test_low_temperature_reduces_to_greedy():
    rng = np.random.default_rng(4)
    nq = [5, 1, 0, 7]
    offs = np.concatenate([[0], np.cumsum(nq)[:-1]])
    rows = sum(nq)
    lg = rng.standard_normal((rows, 30))
    g = lg.argmax(axis=1)
    toks = rng.integers(0, 30, size=rows).astype(np.int32)
    toks[1:3] = g[0:2]                                 # slot 0 accepts 2 drafts greedily
    ctx = [50, 60, 70, 80]
    u = rng.uniform(0.001, 0.999, size=rows)
    want = greedy_accept(lg, offs, nq, toks, ctx)
    got = sample_accept(lg, offs, nq, toks, ctx, 1e-4, u, seed=1)
    for w_, g_ in zip(want, got):
        assert np.array_equal(w_, g_)


# ----------------------------------------------------------------------------- top-p nucleus
from oracle.accept import nucleus_cut, sample_accept_nucleus


def test_nucleus_hand_cases():
    lg = np.log(np.array([0.5, 0.3, 0.2]))
    assert nucleus_cut(lg, 1.0, 0.6) == (lg[1], pytest.approx(0.8))       # {0, 1}
    assert nucleus_cut(lg, 1.0, 0.5)[0] == lg[0]                           # {0}: 0.5 >= 0.5
    assert nucleus_cut(lg, 1.0, 0.81)[0] == lg[2]                          # everything
    assert nucleus_cut(lg, 1.0, 1.0)[0] == -np.inf
    # ties at the cut are all kept
    cut, mass = nucleus_cut(np.array([1.0, 1.0, 0.0, 0.0, -1.0]), 1.0, 0.1)
    assert cut == 1.0 and mass == pytest.approx(2 * np.e / (2 * np.e + 2 + np.exp(-1)))


def test_nucleus_matches_sorted_prefix_without_ties():
    rng = np.random.default_rng(5)
    for _ in range(200):
        V = int(rng.integers(2, 60))
        l = rng.standard_normal(V) * 2
        tau = float(rng.uniform(0.3, 2.0))
        top_p = float(rng.uniform(0.05, 0.99))
        p = np.exp(l / tau - np.max(l / tau))
        p /= p.sum()
        order = np.argsort(-l, kind="stable")
        c = np.cumsum(p[order])
        k = int(np.searchsorted(c, top_p))              # first prefix reaching top_p
        want = set(order[: min(k, V - 1) + 1].tolist())
        cut, mass = nucleus_cut(l, tau, top_p)
        got = set(np.flatnonzero(l >= cut).tolist())
        assert got == want
        assert abs(mass - p[list(got)].sum()) < 1e-12


def test_nucleus_acceptance_hand_case():
    # row 0: p = (0.5, 0.3, 0.2), top_p 0.6 -> q = (0.625, 0.375, 0)
    lg = np.log(np.array([[0.5, 0.3, 0.2], [0.2, 0.3, 0.5]]))
    run = lambda toks, u: sample_accept_nucleus(lg, [0], [2], np.array(toks), [7], 1.0, 0.6, np.array([u, 0.5]), 11)
    a, n, c = run([0, 1], 0.37)
    assert int(a[0]) == 1 and int(c[0]) == 7 and int(n[0]) in (1, 2)      # accepted; bonus from row 1's nucleus {2, 1}
    a, n, c = run([0, 1], 0.38)
    assert (int(a[0]), int(n[0]), int(c[0])) == (0, 0, 6)                 # rejected: the residual nucleus is {0}
    a, n, c = run([0, 2], 1e-9)
    assert int(a[0]) == 0 and int(n[0]) in (0, 1)                          # outside the nucleus: always rejected


def test_top_p_one_is_plain_sampling():
    rng = np.random.default_rng(6)
    nq = [4, 0, 6, 1]
    offs = np.concatenate([[0], np.cumsum(nq)[:-1]])
    rows = sum(nq)
    lg = rng.standard_normal((rows, 40))
    toks = rng.integers(0, 40, size=rows).astype(np.int32)
    u = rng.uniform(0.001, 0.999, size=rows)
    ctx = [10, 20, 30, 40]
    want = sample_accept(lg, offs, nq, toks, ctx, 0.8, u, seed=2)
    got = sample_accept_nucleus(lg, offs, nq, toks, ctx, 0.8, 1.0, u, seed=2)
    for w_, g_ in zip(want, got):
        assert np.array_equal(w_, g_)


def test_gumbel_max_over_the_nucleus_samples_the_filtered_distribution():
    lg = np.array([1.0, 0.0, -1.0, 2.0, 0.5, -3.0])
    tau, top_p = 0.9, 0.7
    cut, mass = nucleus_cut(lg, tau, top_p)
    p = np.exp(lg / tau - np.max(lg / tau))
    p /= p.sum()
    q = np.where(lg >= cut, p, 0.0) / mass
    counts = np.zeros(6)
    n = 40000
    for row in range(n):
        keys = gumbel_keys(lg, tau, 5, row)
        keys[lg < cut] = -np.inf
        counts[int(np.argmax(keys))] += 1
    assert np.max(np.abs(counts / n - q)) < 0.012
    assert counts[lg < cut].sum() == 0
