"""Walsh-Hadamard rotation (oracle; test infrastructure only).

Source: "Quasar" (q27 wiki), "KV cache" bullet -- turbo3 stores "WHT-rotated"
blocks, and turbo5k uses "the same WHT rotation".  The pages do not say which
Hadamard ordering, normalisation or sign pattern; this library reads it as the
plain Sylvester matrix, orthonormal, with no random sign flips:

    H[i, j] = (-1)**popcount(i & j) / sqrt(n),   n = 256  (so 1/16).

Two forms are given:

* ``hadamard_matrix`` -- the dense definition, float64, exact;
* ``fwht_f32``        -- the pinned float32 evaluation order the codec uses:
  radix-2 butterflies over index bits 0,1,...,7 (stride 1, 2, ..., 128), each
  stage mapping (a, b) -> (a + b, a - b) in float32 round-to-nearest-even,
  where a has the lower index, then one multiplication by 0.0625 (exact).
  Codes must be bit-exact, so the order of the float32 additions is part of the
  codec's definition.
"""
from __future__ import annotations

import numpy as np

N = 256


def hadamard_matrix(n: int = N) -> np.ndarray:
    """Dense orthonormal Sylvester-Hadamard matrix, float64 [n, n]."""
    i = np.arange(n, dtype=np.int64)
    bits = i[:, None] & i[None, :]
    # popcount parity of i & j
    parity = np.zeros_like(bits)
    b = bits.copy()
    while np.any(b):
        parity ^= b & 1
        b >>= 1
    return np.where(parity == 1, -1.0, 1.0) / np.sqrt(float(n))


def fwht_f32(x: np.ndarray) -> np.ndarray:
    """Rotate the last axis (length 256) by H in the pinned float32 order."""
    y = np.array(x, dtype=np.float32, copy=True)
    lead = y.shape[:-1]
    n = y.shape[-1]
    if n != N:
        raise ValueError("head_dim must be 256")
    h = 1
    while h < n:
        v = y.reshape(lead + (n // (2 * h), 2, h))
        a = v[..., 0, :]
        b = v[..., 1, :]
        y = np.stack([a + b, a - b], axis=-2).reshape(lead + (n,))
        h *= 2
    return y * np.float32(0.0625)


def rotate_f64(x: np.ndarray) -> np.ndarray:
    """H @ x along the last axis in float64 (used for queries and outputs)."""
    return np.asarray(x, dtype=np.float64) @ hadamard_matrix(x.shape[-1]).T
