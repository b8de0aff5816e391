"""Multi-token causal verify attention (oracle; test infrastructure only).

Source: "Quasar" (q27 wiki), "Self-speculation as the whole design" bullet -- the
drafted tokens of a step are checked in "one shared-KV MMA verify"; "Width-12
verify" bullet -- up to 12 tokens per step; "Continuous batching" bullet --
concurrent slots go through one fused round.  The pages fix none of the
arithmetic below; it is the plain reading of attention over a rotated,
quantised cache:

For one slot with N cached positions before the step and T new tokens
(appended first, so the cache holds L = N + T positions), query token t in
[0, T), query head h, kv head g = h // group (contiguous GQA groups):

    q'      = H q                                   (float64, exact rotation)
    s_p     = q' . k_hat_p / sqrt(256)              for p in [0, N + t]
    P       = softmax(s)                            (masked positions excluded)
    out     = H ( sum_p P_p v_hat_p )               (back to the unrotated basis)

k_hat and v_hat are the exactly dequantised rotated vectors ((q - 3.5) * s),
so no float32 rounding enters the reference result.  Everything is float64.
"""
from __future__ import annotations

import numpy as np

from .wht import rotate_f64

SOFTMAX_SCALE = 1.0 / 16.0   # 1/sqrt(head_dim), head_dim = 256


def causal_limit(n_ctx: int, t: int) -> int:
    """Number of positions query token t may see: [0, n_ctx + t]."""
    return n_ctx + t + 1


def scores_rotated(q_rot: np.ndarray, k_hat: np.ndarray) -> np.ndarray:
    """q_rot [R, D] . k_hat [L, D]^T / 16, float64 [R, L]."""
    return (np.asarray(q_rot, np.float64) @ np.asarray(k_hat, np.float64).T) * SOFTMAX_SCALE


def verify_attention(q: np.ndarray, k_hat: np.ndarray, v_hat: np.ndarray, n_ctx: int, group: int) -> np.ndarray:
    """Verify attention of one slot at one layer.

    q      raw queries, [T, Hq, D]
    k_hat  dequantised rotated keys, [Hkv, L, D] with L >= n_ctx + T
    v_hat  dequantised rotated values, same shape
    returns float64 [T, Hq, D] in the unrotated basis.
    """
    q = np.asarray(q, np.float64)
    T, Hq, D = q.shape
    q_rot = rotate_f64(q)
    o_rot = np.zeros((T, Hq, D), dtype=np.float64)
    for h in range(Hq):
        g = h // group
        for t in range(T):
            lim = causal_limit(n_ctx, t)
            s = scores_rotated(q_rot[t, h][None, :], k_hat[g, :lim])[0]
            m = np.max(s)
            e = np.exp(s - m)
            o_rot[t, h] = (e @ np.asarray(v_hat[g, :lim], np.float64)) / np.sum(e)
    return rotate_f64(o_rot)


def partial_state(s: np.ndarray, v_hat: np.ndarray):
    """Flash-decode partial of one position range: (m, l, o) for scores s [R, n] (-inf = masked)."""
    m = np.max(s, axis=1)
    finite = np.isfinite(m)
    e = np.where(finite[:, None], np.exp(s - np.where(finite, m, 0.0)[:, None]), 0.0)
    return m, e.sum(axis=1), e @ np.asarray(v_hat, np.float64)


def merge_partials(parts):
    """Combine partials of disjoint position ranges: o = sum e^(m_i - M) o_i / sum e^(m_i - M) l_i."""
    ms = np.stack([p[0] for p in parts])
    M = np.max(ms, axis=0)
    w = np.where(np.isfinite(ms), np.exp(ms - np.where(np.isfinite(M), M, 0.0)[None, :]), 0.0)
    l = sum(wi * p[1] for wi, p in zip(w, parts))
    o = sum(wi[:, None] * p[2] for wi, p in zip(w, parts))
    return o / l[:, None]
