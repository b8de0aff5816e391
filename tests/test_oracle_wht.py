"""Pins of the oracle's Walsh-Hadamard rotation against things other than itself.

* the dense matrix against scipy's Sylvester construction (a library routine);
* H H = I exactly, and closed forms for a unit vector and the all-ones vector;
* exactness on integer inputs, where float32 never rounds;
* the pinned float32 evaluation order against an independent evaluation of the
  Sylvester recursion H_2n = [[H_n, H_n], [H_n, -H_n]] (sub-transforms first);
* the orthogonality invariant (Hq).(Hk) = q.k.
"""
import numpy as np
import pytest
import scipy.linalg

from oracle.wht import fwht_f32, hadamard_matrix, rotate_f64


def test_dense_matches_scipy_sylvester():
    H = hadamard_matrix(256)
    assert np.array_equal(H * 16.0, scipy.linalg.hadamard(256).astype(np.float64))


def test_involution_exact():
    H = hadamard_matrix(256)
    assert np.array_equal(H @ H, np.eye(256))
    assert np.array_equal(H, H.T)


def test_closed_forms():
    e0 = np.zeros(256, np.float32)
    e0[0] = 1.0
    assert np.array_equal(fwht_f32(e0), np.full(256, 1.0 / 16, np.float32))
    ones = np.ones(256, np.float32)
    want = np.zeros(256, np.float32)
    want[0] = 16.0
    assert np.array_equal(fwht_f32(ones), want)
    # column j of H: row i of H e_j is (-1)^popcount(i & j) / 16
    ej = np.zeros(256, np.float32)
    ej[0b10110] = 1.0
    i = np.arange(256)
    sign = np.array([(-1.0) ** bin(k & 0b10110).count("1") for k in i])
    assert np.array_equal(fwht_f32(ej), (sign / 16).astype(np.float32))


def test_integer_inputs_are_exact():
    rng = np.random.default_rng(5)
    x = rng.integers(-4096, 4097, size=(64, 256)).astype(np.float32)
    want = x.astype(np.float64) @ (scipy.linalg.hadamard(256).T / 16.0)
    assert np.array_equal(fwht_f32(x).astype(np.float64), want)


def _sylvester_recursive_f32(x):
    n = x.shape[-1]
    if n == 1:
        return x
    a = _sylvester_recursive_f32(x[..., : n // 2])
    b = _sylvester_recursive_f32(x[..., n // 2:])
    return np.concatenate([a + b, a - b], axis=-1)


def test_pinned_float32_order_bit_exact():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal((512, 256)) * np.exp(rng.uniform(-3, 3, (512, 256)))).astype(np.float32)
    want = _sylvester_recursive_f32(x) * np.float32(0.0625)
    got = fwht_f32(x)
    assert got.dtype == np.float32
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    # a different stage order (highest index bit first) rounds differently somewhere
    y = x.copy()
    h = 128
    while h >= 1:
        v = y.reshape(512, 256 // (2 * h), 2, h)
        y = np.stack([v[:, :, 0] + v[:, :, 1], v[:, :, 0] - v[:, :, 1]], axis=2).reshape(512, 256)
        h //= 2
    assert not np.array_equal((y * np.float32(0.0625)).view(np.uint32), got.view(np.uint32))


def test_float32_close_to_dense():
    rng = np.random.default_rng(11)
    x = rng.standard_normal((128, 256)).astype(np.float32)
    dense = x.astype(np.float64) @ hadamard_matrix().T
    err = np.abs(fwht_f32(x) - dense)
    bound = 8 * 2.0 ** -24 * np.sum(np.abs(x), axis=1, keepdims=True) / 16 * 2
    assert np.all(err <= bound)


def test_orthogonality_invariant():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((32, 256))
    k = rng.standard_normal((32, 256)) * 10 ** rng.uniform(0, 1, 256)
    np.testing.assert_allclose(np.sum(rotate_f64(q) * rotate_f64(k), axis=1), np.sum(q * k, axis=1), rtol=1e-12, atol=1e-10)
    np.testing.assert_allclose(np.linalg.norm(rotate_f64(k), axis=1), np.linalg.norm(k, axis=1), rtol=1e-13)


def test_wrong_length_rejected():
    with pytest.raises(ValueError):
        fwht_f32(np.zeros((2, 128), np.float32))
