"""Pins for the Walsh-Hadamard construction (Needle .cact page §一: normalised WHT)."""

import numpy as np
import pytest
import scipy.linalg

from oracle import fwht_butterfly, sylvester_hadamard


@pytest.mark.parametrize("g", [1, 2, 4, 8, 16, 32, 64, 128])
def test_orthogonal_and_symmetric(g):
    Hu = sylvester_hadamard(g)
    assert np.array_equal(Hu @ Hu, g * np.eye(g))
    assert np.array_equal(Hu, Hu.T)
    H = Hu / np.sqrt(g)
    assert np.allclose(H @ H, np.eye(g), atol=1e-14)


def test_matches_library_sylvester():
    # scipy.linalg.hadamard builds the Sylvester-order matrix independently.
    assert np.array_equal(sylvester_hadamard(128), scipy.linalg.hadamard(128).astype(np.float64))


def test_butterfly_columns_equal_dense():
    Hu = sylvester_hadamard(128)
    for k in range(128):
        e = np.zeros(128)
        e[k] = 1.0
        assert np.array_equal(fwht_butterfly(e), Hu[:, k])


def test_butterfly_exact_on_small_integers():
    rng = np.random.default_rng(1)
    v = rng.integers(-127, 128, size=(50, 128)).astype(np.float64)
    assert np.array_equal(fwht_butterfly(v), v @ sylvester_hadamard(128))
    # self-inverse up to g
    assert np.array_equal(fwht_butterfly(fwht_butterfly(v)), 128 * v)


def test_rejects_non_power_of_two():
    with pytest.raises(ValueError):
        sylvester_hadamard(96)
    with pytest.raises(ValueError):
        fwht_butterfly(np.zeros(96))
