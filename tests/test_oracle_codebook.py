"""Pins for the oracle's Lloyd-Max codebooks (CPU only)."""
import math

import numpy as np
import pytest
from scipy import integrate, optimize

from oracle import codebook as cb

CASES = [(d, L) for d in (64, 128, 256) for L in (2, 4, 8, 16, 32)]


@pytest.mark.parametrize("L", [2, 4, 8, 16, 32])
def test_d3_is_uniform_quantizer(L):
    # d = 3: a coordinate of a uniform point on the 2-sphere is uniform on [-1, 1]
    # (Archimedes), whose Lloyd-Max quantizer is the uniform one with MSE (2/L)^2 / 12.
    c, t, _ = cb.lloyd_max(3, L)
    k = np.arange(L)
    assert np.max(np.abs(c - (-1 + (2 * k + 1) / L))) <= 1e-12
    assert np.max(np.abs(t - (-1 + 2 * np.arange(1, L) / L))) <= 1e-12
    assert abs(cb.distortion(c, t, 3) - (2.0 / L) ** 2 / 12) <= 1e-13


@pytest.mark.parametrize("d", [5, 64, 128, 256])
def test_one_bit_closed_form(d):
    # two cells split at 0: c = +-E|Y| = +-Gamma(d/2) / (sqrt(pi) Gamma((d+1)/2))
    c, t, _ = cb.lloyd_max(d, 2)
    e = math.exp(math.lgamma(d / 2) - math.lgamma((d + 1) / 2)) / math.sqrt(math.pi)
    assert abs(c[1] - e) <= 1e-14 and abs(c[0] + e) <= 1e-14 and t[0] == 0.0


def _quad_cell(a, b, d):
    al = (d - 3) / 2
    f = lambda x: (1 - x * x) ** al
    m0 = integrate.quad(f, a, b, epsabs=0, epsrel=2e-14, limit=200)[0]
    m1 = integrate.quad(lambda x: x * f(x), a, b, epsabs=0, epsrel=2e-14, limit=200)[0]
    return m1 / m0


@pytest.mark.parametrize("d,L", CASES)
def test_fixed_point_by_independent_quadrature(d, L):
    c, t, _ = cb.lloyd_max(d, L)
    edges = np.concatenate(([-1.0], t, [1.0]))
    for k in range(L):
        assert abs(c[k] - _quad_cell(edges[k], edges[k + 1], d)) <= 1e-12
    assert np.max(np.abs(t - 0.5 * (c[:-1] + c[1:]))) == 0.0


@pytest.mark.parametrize("d,L", [(128, 4), (128, 8), (64, 16)])
def test_generic_root_finder_agrees(d, L):
    # Solve the Lloyd-Max conditions with a generic root-finder and quadrature, from a
    # perturbed start; the optimum is unique (log-concave density), so it must coincide.
    c0, _, _ = cb.lloyd_max(d, L)
    half = L // 2

    def resid(xpos):
        c = np.concatenate((-xpos[::-1], xpos))
        t = 0.5 * (c[:-1] + c[1:])
        edges = np.concatenate(([-1.0], t, [1.0]))
        return np.array([_quad_cell(edges[half + k], edges[half + k + 1], d) - c[half + k]
                         for k in range(half)])

    sol = optimize.root(resid, c0[half:] * 1.07, method="hybr", tol=1e-14)
    assert np.max(np.abs(resid(sol.x))) <= 1e-14
    assert np.max(np.abs(sol.x - c0[half:])) <= 1e-12


@pytest.mark.parametrize("d,L", CASES)
def test_symmetry_and_middle_boundary(d, L):
    c, t, _ = cb.lloyd_max(d, L)
    assert np.array_equal(c, -c[::-1])
    assert np.all(np.diff(c) > 0)
    assert t[L // 2 - 1] == 0.0


@pytest.mark.parametrize("d", [64, 128, 256])
def test_distortion_falls_and_sits_in_band(d):
    # d*D(bits) between the Gaussian rate-distortion bound 4^-bits and the high-resolution
    # (Panter-Dite) constant sqrt(3) pi / 2 ~ 2.72 times it.
    prev = np.inf
    for bits in range(1, 6):
        c, t, _ = cb.lloyd_max(d, 2 ** bits)
        dd = d * cb.distortion(c, t, d)
        assert dd < prev
        assert 4.0 ** -bits <= dd <= math.sqrt(3) * math.pi / 2 * 4.0 ** -bits
        prev = dd


def test_gaussian_limit_matches_max_1960():
    # Large d: sqrt(d) Y -> N(0,1); Max (1960) tables of the Gaussian Lloyd-Max quantizer.
    d = 4096
    s = math.sqrt(d)
    c1, t1, _ = cb.lloyd_max(d, 2)
    assert abs(c1[1] * s - 0.7979) < 2e-3
    c2, t2, _ = cb.lloyd_max(d, 4)
    assert abs(c2[2] * s - 0.4528) < 2e-3 and abs(c2[3] * s - 1.510) < 3e-3
    assert abs(t2[2] * s - 0.9816) < 3e-3
    for bits, mse in ((1, 0.3634), (2, 0.1175), (3, 0.03455), (4, 0.009497)):
        c, t, _ = cb.lloyd_max(d, 2 ** bits)
        assert abs(d * cb.distortion(c, t, d) / mse - 1) < 3e-3


@pytest.mark.parametrize("d,L", [(128, 4), (64, 8), (256, 16)])
def test_distortion_matches_monte_carlo(d, L):
    c, t, _ = cb.lloyd_max(d, L)
    rs = np.random.default_rng(11)
    x = rs.standard_normal((20000, d))
    u = x / np.linalg.norm(x, axis=1, keepdims=True)
    err = (u - c[cb.encode(u, t)]) ** 2
    per_vec = err.sum(axis=1)
    D = cb.distortion(c, t, d)
    assert abs(per_vec.mean() - d * D) < 5 * per_vec.std() / np.sqrt(len(per_vec))


def test_encode_is_nearest_centroid():
    c, t, _ = cb.lloyd_max(128, 8)
    y = np.random.default_rng(5).standard_normal(200000) * 0.12
    brute = np.argmin(np.abs(y[:, None] - c[None, :]), axis=1)
    assert np.array_equal(cb.encode(y, t), brute)
    # a value equal to a boundary takes the upper cell
    assert np.array_equal(cb.encode(t, t), np.arange(1, len(c)))
