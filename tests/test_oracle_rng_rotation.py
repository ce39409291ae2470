"""Pins for the oracle's random streams and seeded matrices (CPU only)."""
import json
import os

import numpy as np
import pytest

from oracle import rng, rotation


def test_splitmix64_known_answers():
    # Published reference outputs of splitmix64.c (Vigna) started from state 0.
    out = rng.splitmix64(0, 3)
    assert [int(x) for x in out] == [0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4, 0x06C45D188009454F]


def test_splitmix64_fourth_output_and_gaussian_known_answers():
    """Box-Muller pairing pinned by known answers (tests/golden/gaussians_seed0.json): the
    first four published SplitMix64 outputs of state 0, the uniforms they give and the
    four Gaussians of stream 0.  Swapping cos and sin, taking u1 instead of 1 - u1, or
    pairing other than consecutive outputs changes these values."""
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "gaussians_seed0.json")))
    assert [int(x) for x in rng.splitmix64(0, 4)] == [int(x, 16) for x in g["splitmix64_outputs"]]
    u = rng.uniforms(0, 4)
    assert [float(x) for x in u] == [g["pairs"][0]["u1"], g["pairs"][0]["u2"], g["pairs"][1]["u1"], g["pairs"][1]["u2"]]
    got = rng.gaussians(0, 4)
    assert np.max(np.abs(got - np.array(g["gaussians"]))) <= g["tolerance"]
    # an odd count is the prefix of the even one
    assert np.array_equal(rng.gaussians(0, 3), got[:3])


def test_splitmix64_is_counter_based():
    # output i depends only on seed + (i+1)*gamma: a window equals the tail of a longer run
    a = rng.splitmix64(12345, 100)
    b = rng.splitmix64(12345, 40, start=60)
    assert np.array_equal(a[60:], b)


def test_uniform_and_gaussian_moments():
    n = 2_000_000
    u = rng.uniforms(7, n)
    assert u.min() >= 0.0 and u.max() < 1.0
    assert abs(u.mean() - 0.5) < 5 * np.sqrt(1 / 12 / n)
    g = rng.gaussians(7, n)
    se = 1 / np.sqrt(n)
    assert abs(g.mean()) < 5 * se
    assert abs(g.var() - 1.0) < 5 * np.sqrt(2) * se
    assert abs(np.mean(g ** 4) - 3.0) < 5 * np.sqrt(96) * se
    # P(|g| < 1) for N(0,1)
    p = np.mean(np.abs(g) < 1.0)
    assert abs(p - 0.6826894921370859) < 5 * np.sqrt(p * (1 - p) / n)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_rotation_orthogonal(d):
    Pi = rotation.haar_rotation(d, seed=0)
    assert np.max(np.abs(Pi.T @ Pi - np.eye(d))) <= 1e-12
    assert np.max(np.abs(Pi @ Pi.T - np.eye(d))) <= 1e-12


@pytest.mark.parametrize("d", [8, 128])
def test_rotation_is_sign_fixed_q_factor(d):
    # Pi must be the Q of G = Q R with a positive diagonal of R: Pi^T G is upper
    # triangular with a positive diagonal (this rules out Q^T, unfixed signs, wrong stream).
    seed = 3
    G = rotation.gaussian_matrix(rng.rotation_stream_seed(seed), d, d)
    R = rotation.haar_rotation(d, seed).T @ G
    scale = np.max(np.abs(G))
    assert np.max(np.abs(np.tril(R, -1))) <= 1e-12 * scale * d
    assert np.all(np.diag(R) > 0)


def test_rotation_haar_statistics():
    # Haar O(d) is invariant under sign flips of rows and columns: E[Pi_ij] = 0 and
    # E[Pi_ij^2] = 1/d.  A QR without the sign fix leaves the diagonal biased.
    d, n = 4, 3000
    diag = np.array([rotation.haar_rotation(d, s)[0, 0] for s in range(n)])
    sd = np.sqrt(1.0 / d / n)
    assert abs(diag.mean()) < 5 * sd
    assert abs(np.mean(diag ** 2) - 1.0 / d) < 0.05


def test_qjl_matrix_moments_and_streams():
    S = rotation.qjl_matrix(256, 256, seed=0)
    n = S.size
    assert abs(S.mean()) < 5 / np.sqrt(n)
    assert abs(S.var() - 1) < 5 * np.sqrt(2 / n)
    # the two streams differ (S is not the rotation's Gaussian matrix)
    G = rotation.gaussian_matrix(rng.rotation_stream_seed(0), 256, 256)
    assert not np.allclose(S, G)
    assert np.array_equal(S, rotation.qjl_matrix(256, 256, seed=0))
