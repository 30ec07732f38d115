"""Pins for the oracle's rotation: the normalised Sylvester Hadamard matrix
against scipy.linalg.hadamard, orthonormality and symmetry, the sign
generator against published SplitMix64 outputs, the round trip of the
randomized Hadamard transform, and the store's pre-quantisation coordinates
for one-hot and two-hot keys, which fix the order "signs, then transform"
("turboquant-plus.md", Background: a random sign vector followed by a
Walsh-Hadamard transform)."""
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


def _store_y(orc, k, preset=2):
    L = orc.layout(preset)
    s = orc.signs(128, 42)
    c32, m32 = orc.codebook(128, L["key_bits"])
    _, y = orc.store_one(preset, np.asarray(k, np.float32), np.zeros(128, np.float32), s, c32, m32)
    return y.astype(np.float64), s.astype(np.float64)


@pytest.mark.parametrize("j", [0, 1, 5, 64, 127])
def test_store_rotation_one_hot(orc, j):
    """k = a e_j gives y = H (s . k) / ||k|| = s_j H[:, j], with H from scipy
    (not the oracle's own matrix).  Rotating first and flipping signs after
    (s . H k) or leaving the signs out gives another vector for some j."""
    H = sylvester(128) / np.sqrt(128)
    k = np.zeros(128)
    k[j] = 3.0
    y, s = _store_y(orc, k)
    want = s[j] * H[:, j]
    assert np.max(np.abs(y - want)) < 1e-7
    assert abs(np.linalg.norm(y) - 1) < 1e-6


@pytest.mark.parametrize("i,j", [(0, 1), (3, 70), (12, 127)])
def test_store_rotation_two_hot(orc, i, j):
    """k = a e_i + b e_j: y = (a s_i H[:, i] + b s_j H[:, j]) / sqrt(a^2 + b^2).
    With the sign vector's entries of opposite sign at i and j (checked), a
    rotation taken in the other order, s . (H k) / ||k||, lands elsewhere."""
    H = sylvester(128) / np.sqrt(128)
    s = orc.signs(128, 42).astype(np.float64)
    assert s[i] != s[j]
    a, b = 2.0, -0.5
    k = np.zeros(128)
    k[i], k[j] = a, b
    y, _ = _store_y(orc, k)
    want = (a * s[i] * H[:, i] + b * s[j] * H[:, j]) / np.hypot(a, b)
    assert np.max(np.abs(y - want)) < 1e-7
    other = s * (H @ k) / np.hypot(a, b)
    assert np.max(np.abs(other - want)) > 1e-2
