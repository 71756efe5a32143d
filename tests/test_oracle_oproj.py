"""Pins for the oracle's output projection (out = y w_o^T, nn.Linear without bias):
brute force over the definition's sum, the identity and a permutation weight."""
import numpy as np

import oracle


def test_matches_brute_force_sum():
    r = np.random.default_rng(0)
    y = r.standard_normal((3, 5))
    w = r.standard_normal((4, 5))
    out = oracle.o_proj(y, w)
    ref = np.array([[sum(y[i, c] * w[n, c] for c in range(5)) for n in range(4)] for i in range(3)])
    assert np.allclose(out, ref, rtol=1e-14, atol=1e-14)


def test_identity_and_permutation():
    y = np.random.default_rng(1).standard_normal((6, 8)).astype(np.float32)
    assert np.array_equal(oracle.o_proj(y, np.eye(8)), y.astype(np.float64))
    perm = np.random.default_rng(2).permutation(8)
    assert np.array_equal(oracle.o_proj(y, np.eye(8)[perm]), y.astype(np.float64)[:, perm])
