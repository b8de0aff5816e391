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
