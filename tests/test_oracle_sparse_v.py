"""Pins of the oracle's Sparse V (oracle.decode.attend_sparse_v; [3BITS] llama.cpp section:
positions with low attention weights are skipped during decoding).

Reading pinned here: with p_t = exp(l_t - max l), positions with p_t < theta leave the
numerator of the attention average, and the denominator keeps every position.
"""
import math

import numpy as np

from oracle import decode as dec
from oracle import params


def _tokens(p, T, rng, mse_only=False):
    d = p.Pi.shape[0]
    tk = dict(idx=rng.integers(0, len(p.cb_k[0]), (T, d)), n=rng.random(T) + 0.5,
              sigma=None if mse_only else rng.integers(0, 2, (T, d)),
              gamma=None if mse_only else rng.random(T) * 0.3)
    tv = dict(idx=rng.integers(0, len(p.cb_v[0]), (T, d)), n=rng.random(T) + 0.5)
    return tk, tv


def test_theta_zero_is_dense_attention():
    p = params.make(64, 3)
    rng = np.random.default_rng(0)
    tk, tv = _tokens(p, 300, rng)
    q = rng.standard_normal(64) * 3
    o, lg = dec.attend_route_a(q, tk, tv, p.Pi, p.S, p.cb_k, p.cb_v)
    os_, lgs, skipped = dec.attend_sparse_v(q, tk, tv, p.Pi, p.S, p.cb_k, p.cb_v, 0.0)
    assert np.array_equal(lg, lgs) and skipped == 0.0
    assert np.allclose(os_, o, rtol=1e-14, atol=1e-15)


def test_one_dominant_key_closed_form():
    # keys of norm 0 score exactly 0 (no QJL term either: gamma 0); token 0 scores L > 0.
    # Every theta in (exp(-L), 1] keeps token 0 alone, and the denominator still counts the
    # other T - 1 positions: out = v^_0 / (1 + (T - 1) e^{-L}).  (A numerator-and-
    # denominator skip would give v^_0 itself.)
    d, T = 32, 9
    p = params.make(d, 3)
    rng = np.random.default_rng(1)
    tk, tv = _tokens(p, T, rng)
    tk["n"][1:] = 0.0
    tk["gamma"][:] = 0.0
    q = rng.standard_normal(d)
    _, lg = dec.attend_route_a(q, tk, tv, p.Pi, p.S, p.cb_k, p.cb_v)
    q = q * (3.0 / lg[0])   # the logit is linear in q: token 0 now scores 3
    _, lg = dec.attend_route_a(q, tk, tv, p.Pi, p.S, p.cb_k, p.cb_v)
    L = lg[0]
    assert abs(L - 3.0) < 1e-12 and np.all(lg[1:] == 0.0)
    vhat0 = (tv["n"][0] * (p.Pi.T @ p.cb_v[0][tv["idx"][0]]))
    want = vhat0 / (1.0 + (T - 1) * math.exp(-L))
    for theta in (math.exp(-L) * 1.0001, 0.5, 1.0):
        out, _, skipped = dec.attend_sparse_v(q, tk, tv, p.Pi, p.S, p.cb_k, p.cb_v, theta)
        assert np.allclose(out, want, rtol=1e-13, atol=1e-15), theta
        assert skipped > 0.0


def test_dropping_the_smallest_weight_removes_exactly_its_term():
    # theta just above the smallest weight drops that one position: the change against the
    # dense output is its weighted value, e_min v^_min / sum e, and equals the bound
    p = params.make(64, 4)
    rng = np.random.default_rng(2)
    tk, tv = _tokens(p, 50, rng, mse_only=True)
    q = rng.standard_normal(64) * 4
    dense, lg = dec.attend_route_a(q, tk, tv, p.Pi, p.S, p.cb_k, p.cb_v)
    e = np.exp(lg - lg.max())
    i = int(np.argmin(e))
    e_sorted = np.sort(e)
    theta = 0.5 * (e_sorted[0] + e_sorted[1])
    out, _, skipped = dec.attend_sparse_v(q, tk, tv, p.Pi, p.S, p.cb_k, p.cb_v, theta)
    vhat_i = tv["n"][i] * (p.Pi.T @ p.cb_v[0][tv["idx"][i]])
    diff = dense - out
    assert np.allclose(diff, e[i] * vhat_i / e.sum(), rtol=1e-9, atol=1e-16)
    assert math.isclose(skipped, np.linalg.norm(diff), rel_tol=1e-9)


def test_bound_and_monotone_in_theta():
    p = params.make(128, 3)
    rng = np.random.default_rng(3)
    tk, tv = _tokens(p, 400, rng)
    q = rng.standard_normal(128) * 6   # peaky: a wide spread of logits
    dense, _ = dec.attend_route_a(q, tk, tv, p.Pi, p.S, p.cb_k, p.cb_v)
    last = 0.0
    for theta in (1e-9, 1e-6, 1e-3, 1e-1):
        out, _, skipped = dec.attend_sparse_v(q, tk, tv, p.Pi, p.S, p.cb_k, p.cb_v, theta)
        assert np.linalg.norm(out - dense) <= skipped * (1 + 1e-12) + 1e-15
        assert skipped >= last
        last = skipped
