"""Greedy acceptance of a verify step and the commit (rollback) of the cache length.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Source: the "Quasar" (q27) engine wiki -- the sampler paragraph of "Serving"
(temperature 0, greedy argmax, is the default every determinism gate assumes),
the "Model tool protocol" bullet (greedy speculative decode by default), and
the attention-KV bullet of the prefix-cache discussion (attention rows below the
point where the drafts diverge are append-only and stay valid in place, so a
rejected draft is undone by shortening the length).  The pages give the
behaviour, not the bookkeeping; the reading taken here:

* A slot's step verifies T = 1 + d query tokens: t_0 (the last committed
  token, whose K/V the step appends) and the drafts d_1 .. d_d.  The verify
  pass yields one row of logits per query token; row j predicts the token after
  query token j.
* g_j = argmax of row j; on equal maxima the lowest vocabulary index wins.
* Drafts are accepted in order while d_{j+1} == g_j; a is the number accepted
  (0 <= a <= d).  The token after the accepted prefix is g_a (the correction
  when a < d, the bonus token when every draft was accepted).
* The cache held ctx_len positions after the step's append (t_0 and all d
  drafts); the committed length keeps t_0 and the a accepted drafts:
  committed = ctx_len - (d - a).  Rows past it are stale and are overwritten
  by the next append.
* A slot with T = 0 accepts nothing: a = 0, next = -1, committed = ctx_len.
"""
from __future__ import annotations

import numpy as np


def argmax_lowest(row: np.ndarray) -> int:
    """Index of the largest value; the lowest such index on ties (np.argmax's rule)."""
    return int(np.argmax(np.asarray(row)))


def greedy_accept(logits: np.ndarray, q_offsets, n_q, tokens, ctx_len):
    """Greedy acceptance for every slot.

    logits    [rows, vocab] (the values the kernel compares, as float64 or float32)
    q_offsets slot b's rows start at q_offsets[b]
    n_q       T_b query tokens of slot b
    tokens    [rows] the query tokens (t_0, d_1 .. d_d per slot)
    ctx_len   cache length of slot b after the step's append

    Returns (n_accepted, next_token, committed_len), int32 arrays of the slot count.
    """
    S = len(n_q)
    n_acc = np.zeros(S, np.int32)
    nxt = np.full(S, -1, np.int32)
    committed = np.array(ctx_len, np.int64).astype(np.int32)
    for b in range(S):
        T = int(n_q[b])
        if T <= 0:
            continue
        r0 = int(q_offsets[b])
        g = [argmax_lowest(logits[r0 + j]) for j in range(T)]
        a = 0
        while a < T - 1 and int(tokens[r0 + a + 1]) == g[a]:
            a += 1
        n_acc[b] = a
        nxt[b] = g[a]
        committed[b] = int(ctx_len[b]) - (T - 1 - a)
    return n_acc, nxt, committed
