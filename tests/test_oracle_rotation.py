"""Pins for the oracle's rotation: the normalised Sylvester Hadamard matrix
against scipy.linalg.hadamard, orthonormality and symmetry, the sign
generator against published SplitMix64 outputs, and the round trip of the
randomized Hadamard transform."""
import os

import numpy as np
import pytest
from scipy.linalg import hadamard as sylvester

GOLD = os.path.join(os.path.dirname(__file__), "golden")


@pytest.mark.parametrize("D", [2, 4, 8, 16, 32, 64, 128, 256])
def test_hadamard_orthonormal_symmetric(orc, D):
    H = orc.hadamard(D)
    assert np.array_equal(H, sylvester(D) / np.sqrt(D))
    assert np.array_equal(H, H.T)
    assert np.max(np.abs(H @ H - np.eye(D))) < 1e-12


def test_signs_splitmix64_reference(orc):
    """s_i = -1 exactly when the top bit of SplitMix64 output i is set."""
    outs = [int(l, 16) for l in open(os.path.join(GOLD, "splitmix64_seed0.txt"))
            if l.strip() and not l.startswith("#")]
    s = orc.signs(3, seed=0)
    assert list(s) == [-1 if (o >> 63) else 1 for o in outs]


def test_signs_shape_and_balance(orc):
    s = orc.signs(128, 42)
    assert s.dtype == np.int8 and set(np.unique(s)) <= {-1, 1}
    big = orc.signs(1 << 16, 42)
    assert abs(big.astype(np.int64).sum()) < 4 * np.sqrt(1 << 16)
    assert not np.array_equal(orc.signs(128, 42), orc.signs(128, 42 + 1337))


def test_rht_round_trip_and_parseval(orc):
    rng = np.random.default_rng(0)
    D = 128
    H = orc.hadamard(D)
    s = orc.signs(D, 42).astype(np.float64)
    for _ in range(20):
        x = rng.normal(size=D) * rng.uniform(0.1, 10)
        y = H @ (s * x)
        assert abs(np.linalg.norm(y) - np.linalg.norm(x)) < 1e-12 * np.linalg.norm(x)
        back = s * (H @ y)
        assert np.max(np.abs(back - x)) < 1e-12 * np.linalg.norm(x)
