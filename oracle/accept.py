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


# ----------------------------------------------------------------------------- sampled acceptance
# The pages' sampled speculative decode ("Model tool protocol" bullet: Gumbel-max
# sampling with rejection-sampled acceptance, seeded and reproducible; greedy
# unchanged).  Reading taken here (the top-p nucleus filter is not modelled):
#
# * target distribution of row j: p_j = softmax(logits_j / tau);
# * the drafts are point masses (a deterministic drafter), so draft d_{j+1} is
#   accepted with probability min(1, p_j(d)/1) = p_j(d): accepted iff the
#   given uniform u_j (one per row, passed in) is below p_j(d_{j+1});
# * at the first rejection (row a) the replacement is drawn from the residual
#   max(0, p_a - delta_d) / norm, i.e. p_a without the rejected token, by
#   Gumbel-max over the other tokens; if every draft is accepted the bonus token
#   is drawn from p_{T-1} the same way;
# * Gumbel noise G(row, x) = -log(-log U) with U from a counter-based
#   SplitMix64 stream (published definition: state += 0x9E3779B97F4A7C15, then
#   the 64-bit mix below): U = ((z >> 41) + 0.5) / 2^23 (exact in float32 and
#   float64) with z the output of counter k = row * 2^32 + x of the stream
#   seeded with `seed`.

MASK64 = (1 << 64) - 1
GOLDEN_GAMMA = 0x9E3779B97F4A7C15


def splitmix64_at(seed: int, k: int) -> int:
    """Output number k (0-based) of the SplitMix64 stream seeded with `seed`."""
    z = (seed + (k + 1) * GOLDEN_GAMMA) & MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def noise_uniform(seed: int, row: int, tokens: np.ndarray) -> np.ndarray:
    """U(row, x) in (0, 1) for the given token ids (exact 24-bit values, float64)."""
    tokens = np.asarray(tokens, np.uint64)
    with np.errstate(over="ignore"):
        k = np.uint64(row) * np.uint64(1 << 32) + tokens
        z = np.uint64(seed) + (k + np.uint64(1)) * np.uint64(GOLDEN_GAMMA)
        z = (z ^ (z >> np.uint64(30))) * np.uint64(0xBF58476D1CE4E5B9)
        z = (z ^ (z >> np.uint64(27))) * np.uint64(0x94D049BB133111EB)
        z = z ^ (z >> np.uint64(31))
    return ((z >> np.uint64(41)).astype(np.float64) + 0.5) / float(1 << 23)


def gumbel_keys(logits_row: np.ndarray, tau: float, seed: int, row: int) -> np.ndarray:
    """logit / tau + G(row, x) for every token x (float64)."""
    x = np.arange(logits_row.shape[0])
    return np.asarray(logits_row, np.float64) / tau - np.log(-np.log(noise_uniform(seed, row, x)))


def target_prob(logits_row: np.ndarray, tau: float, token: int) -> float:
    """p(token) under softmax(logits_row / tau), float64."""
    l = np.asarray(logits_row, np.float64) / tau
    m = l.max()
    e = np.exp(l - m)
    return float(e[token] / e.sum()) if 0 <= token < l.shape[0] else 0.0


def sample_accept(logits: np.ndarray, q_offsets, n_q, tokens, ctx_len, tau: float, uniforms, seed: int):
    """Rejection-sampled acceptance for every slot; returns (n_accepted, next_token, committed_len)."""
    S = len(n_q)
    n_acc = np.zeros(S, np.int32)
    nxt = np.full(S, -1, np.int32)
    committed = np.array(ctx_len, np.int64).astype(np.int32)
    V = logits.shape[1]
    for b in range(S):
        T = int(n_q[b])
        if T <= 0:
            continue
        r0 = int(q_offsets[b])
        a = 0
        while a < T - 1 and float(uniforms[r0 + a]) < target_prob(logits[r0 + a], tau, int(tokens[r0 + a + 1])):
            a += 1
        keys = gumbel_keys(logits[r0 + a], tau, seed, r0 + a)
        if a < T - 1:                                  # residual: the rejected token is excluded
            d = int(tokens[r0 + a + 1])
            if 0 <= d < V:
                keys[d] = -np.inf
        n_acc[b] = a
        nxt[b] = int(np.argmax(keys))
        committed[b] = int(ctx_len[b]) - (T - 1 - a)
    return n_acc, nxt, committed


# ----------------------------------------------------------------------------- top-p nucleus
# The pages' sampled speculative decode filters each target distribution to its
# top-p nucleus before the Gumbel-max draw and the rejection test ("Model tool
# protocol" bullet), on the temperature-scaled distribution (the sampler
# paragraph of "Serving": q27 filters after temperature).  Reading taken here,
# a threshold rule on the logits (the pages do not say how ties at the cut are
# broken; this keeps all of them):
#
# * p_j = softmax(l_j / tau); for a logit value t, mass(t) = sum of p_j(x) over
#   the tokens with l_x >= t;
# * l* = the largest logit value of the row with mass(l*) >= top_p; the nucleus
#   is {x : l_x >= l*} (every token tied with the cut is in);
# * the filtered distribution is p_j restricted to the nucleus, renormalised;
#   top_p >= 1 keeps every token (the plain sampled acceptance).
# The draft test, the residual and the bonus draw are those of sample_accept
# with the filtered distribution: a draft outside the nucleus is always
# rejected, and the Gumbel-max argmax runs over the nucleus only.


def nucleus_cut(logits_row: np.ndarray, tau: float, top_p: float):
    """(l*, mass of the nucleus) of one row; l* = -inf keeps every token."""
    l = np.asarray(logits_row, np.float64)
    p = np.exp(l / tau - np.max(l / tau))
    p /= p.sum()
    if top_p >= 1.0:
        return -np.inf, 1.0
    vals = np.unique(l)[::-1]                          # distinct logits, largest first
    for t in vals:
        m = float(p[l >= t].sum())
        if m >= top_p:
            return float(t), m
    return float(vals[-1]), 1.0


def sample_accept_nucleus(logits: np.ndarray, q_offsets, n_q, tokens, ctx_len, tau: float, top_p: float,
                          uniforms, seed: int):
    """Rejection-sampled acceptance with top-p nucleus filtering; returns (n_accepted, next_token, committed_len)."""
    S = len(n_q)
    n_acc = np.zeros(S, np.int32)
    nxt = np.full(S, -1, np.int32)
    committed = np.array(ctx_len, np.int64).astype(np.int32)
    V = logits.shape[1]
    for b in range(S):
        T = int(n_q[b])
        if T <= 0:
            continue
        r0 = int(q_offsets[b])

        def filtered_prob(j, d):
            row = np.asarray(logits[r0 + j], np.float64)
            cut, mass = nucleus_cut(row, tau, top_p)
            if not (0 <= d < V) or row[d] < cut:
                return 0.0
            return target_prob(row, tau, d) / mass

        a = 0
        while a < T - 1 and float(uniforms[r0 + a]) < filtered_prob(a, int(tokens[r0 + a + 1])):
            a += 1
        row = np.asarray(logits[r0 + a], np.float64)
        cut, _ = nucleus_cut(row, tau, top_p)
        keys = gumbel_keys(row, tau, seed, r0 + a)
        keys[row < cut] = -np.inf
        if a < T - 1:
            d = int(tokens[r0 + a + 1])
            if 0 <= d < V:
                keys[d] = -np.inf
        n_acc[b] = a
        nxt[b] = int(np.argmax(keys))
        committed[b] = int(ctx_len[b]) - (T - 1 - a)
    return n_acc, nxt, committed
