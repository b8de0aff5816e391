"""Pins of the oracle's verify attention.

* brute force on a tiny case: scores, mask and softmax in pure Python (math.fsum,
  math.exp) over scipy's Hadamard matrix, no numpy reductions;
* constant V: the output is H v whatever Q and N are;
* T = 1, N = 0: only position 0 is visible, output = H v_0;
* causality: positions after N + t never change row t; position N + t does;
* GQA mapping: q heads 8g..8g+7 read kv head g;
* split invariance of the flash-decode merge rule, including fully masked rows;
* the scores are rotation invariant: (Hq).(k_rot) = q.(H k_rot).
* a prefill-sized case equals torch's scaled_dot_product_attention (float64,
  explicit bottom-right causal mask, repeated kv heads).
"""
import math

import numpy as np
import scipy.linalg

from oracle import attention
from oracle.wht import rotate_f64


def _brute(q, kh, vh, n_ctx, group):
    Hs = scipy.linalg.hadamard(256).astype(float) / 16.0
    T, Hq, D = q.shape
    out = np.zeros((T, Hq, D))
    for t in range(T):
        for h in range(Hq):
            g = h // group
            qr = [math.fsum(Hs[i, j] * q[t, h, j] for j in range(D)) for i in range(D)]
            vis = n_ctx + t + 1
            s = [math.fsum(qr[i] * kh[g, p, i] for i in range(D)) / 16.0 for p in range(vis)]
            m = max(s)
            e = [math.exp(x - m) for x in s]
            z = math.fsum(e)
            o = [math.fsum(e[p] * vh[g, p, i] for p in range(vis)) / z for i in range(D)]
            out[t, h] = [math.fsum(Hs[i, j] * o[j] for j in range(D)) for i in range(D)]
    return out


def _case(rng, T, n_ctx, Hkv=2, group=8, scale=1.0):
    L = n_ctx + T
    q = rng.standard_normal((T, Hkv * group, 256))
    kh = rng.standard_normal((Hkv, L, 256)) * scale
    vh = rng.standard_normal((Hkv, L, 256)) * scale
    return q, kh, vh


def test_brute_force_tiny():
    rng = np.random.default_rng(0)
    q, kh, vh = _case(rng, T=2, n_ctx=3, Hkv=2, group=2)
    got = attention.verify_attention(q, kh, vh, 3, 2)
    want = _brute(q, kh, vh, 3, 2)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_constant_v():
    rng = np.random.default_rng(1)
    q, kh, vh = _case(rng, T=5, n_ctx=40, scale=3.0)
    vconst = rng.standard_normal(256)
    vh[:] = vconst
    out = attention.verify_attention(q * 7, kh, vh, 40, 8)
    want = rotate_f64(vconst)
    np.testing.assert_allclose(out, np.broadcast_to(want, out.shape), rtol=0, atol=1e-12)


def test_single_visible_position():
    rng = np.random.default_rng(2)
    q, kh, vh = _case(rng, T=1, n_ctx=0)
    out = attention.verify_attention(q, kh, vh, 0, 8)
    for h in range(16):
        np.testing.assert_allclose(out[0, h], rotate_f64(vh[h // 8, 0]), rtol=0, atol=1e-12)


def test_causality():
    rng = np.random.default_rng(3)
    T, n = 4, 20
    q, kh, vh = _case(rng, T=T, n_ctx=n)
    base = attention.verify_attention(q, kh, vh, n, 8)
    for t in range(T):
        kh2, vh2 = kh.copy(), vh.copy()
        kh2[:, n + t + 1:] += 5.0
        vh2[:, n + t + 1:] -= 3.0
        out = attention.verify_attention(q, kh2, vh2, n, 8)
        np.testing.assert_array_equal(out[t], base[t])
        vh3 = vh.copy()
        vh3[:, n + t] += 1.0
        out3 = attention.verify_attention(q, kh, vh3, n, 8)
        assert np.all(np.abs(out3[t] - base[t]).max(axis=-1) > 1e-9)


def test_gqa_mapping():
    rng = np.random.default_rng(4)
    q, kh, vh = _case(rng, T=2, n_ctx=10)
    c0, c1 = rng.standard_normal(256), rng.standard_normal(256)
    vh[0] = c0
    vh[1] = c1
    out = attention.verify_attention(q, kh, vh, 10, 8)
    for h in range(16):
        want = rotate_f64(c0 if h < 8 else c1)
        np.testing.assert_allclose(out[:, h], np.broadcast_to(want, (2, 256)), atol=1e-12)


def test_split_merge_invariance():
    rng = np.random.default_rng(5)
    R, L = 6, 300
    s = rng.standard_normal((R, L)) * 4.6
    s[0, 100:] = -np.inf          # row 0 sees only [0, 100): the last split is fully masked for it
    v = rng.standard_normal((L, 256)) * 4.6
    whole = attention.merge_partials([attention.partial_state(s, v)])
    for cuts in ([0, 150, 300], [0, 1, 2, 299, 300], [0, 100, 200, 300], list(range(0, 301, 25))):
        parts = [attention.partial_state(s[:, a:b], v[a:b]) for a, b in zip(cuts[:-1], cuts[1:])]
        np.testing.assert_allclose(attention.merge_partials(parts), whole, rtol=0, atol=1e-12)
    direct = np.exp(s - s.max(1, keepdims=True))
    np.testing.assert_allclose(whole, (direct @ v) / direct.sum(1, keepdims=True), atol=1e-12)


def test_scores_rotation_invariant():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((3, 256))
    k_rot = rng.standard_normal((7, 256))
    a = attention.scores_rotated(rotate_f64(q), k_rot)
    b = q @ rotate_f64(k_rot).T / 16.0
    np.testing.assert_allclose(a, b, atol=1e-12)


def test_prefill_shape_equals_library_attention():
    # A prefill-sized case (300 new tokens over 200 cached positions) against
    # torch's scaled_dot_product_attention in float64 on the CPU (a library
    # routine): queries rotated by scipy's Hadamard matrix, kv head repeated
    # over its 8 q heads, row t allowed positions [0, 200 + t], output rotated
    # back.
    torch = __import__("torch")
    rng = np.random.default_rng(7)
    T, n_ctx = 300, 200
    q, kh, vh = _case(rng, T=T, n_ctx=n_ctx, scale=2.0)
    got = attention.verify_attention(q, kh, vh, n_ctx, 8)
    Hs = torch.from_numpy(scipy.linalg.hadamard(256).astype(np.float64) / 16.0)
    qr = torch.from_numpy(q).permute(1, 0, 2) @ Hs.T                       # [Hq, T, 256]
    k = torch.from_numpy(kh).repeat_interleave(8, dim=0)                    # [Hq, L, 256]
    v = torch.from_numpy(vh).repeat_interleave(8, dim=0)
    allowed = torch.arange(n_ctx + T)[None, :] <= (n_ctx + torch.arange(T))[:, None]
    o = torch.nn.functional.scaled_dot_product_attention(qr, k, v, attn_mask=allowed, scale=1.0 / 16.0)
    want = (o @ Hs.T).permute(1, 0, 2).numpy()
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-11)
