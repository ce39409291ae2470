"""Pins of the oracle's compressed inner-product scan (oracle.decode.ip_topk; [BLOG] 6.4)."""
import numpy as np

from oracle import decode as dec
from oracle import params, quant


def _keys(p, T, rng):
    d = p.Pi.shape[0]
    return dict(idx=rng.integers(0, len(p.cb_k[0]), (T, d)), n=rng.random(T) + 0.5,
                sigma=rng.integers(0, 2, (T, d)), gamma=rng.random(T) * 0.3)


def test_estimates_are_the_attention_logits_times_sqrt_d():
    # the scan ranks by the decode's own score: logit = <q, k^> / sqrt(d)
    p = params.make(64, 3)
    rng = np.random.default_rng(0)
    tk = _keys(p, 200, rng)
    tv = dict(idx=rng.integers(0, len(p.cb_v[0]), (200, 64)), n=rng.random(200))
    q = rng.standard_normal(64)
    _, lg = dec.attend_route_a(q, tk, tv, p.Pi, p.S, p.cb_k, p.cb_v)
    slots, est = dec.ip_topk(q, tk, p.Pi, p.S, p.cb_k, 200)
    assert np.allclose(est, lg[slots] * 8.0, rtol=1e-13, atol=1e-13)
    assert sorted(slots.tolist()) == list(range(200))          # k = T: a permutation
    assert np.all(np.diff(est) <= 0)                          # by decreasing estimate


def test_ties_go_to_the_lower_slot_and_k_truncates():
    p = params.make(32, 3)
    rng = np.random.default_rng(1)
    tk = _keys(p, 6, rng)
    for f in ("idx", "sigma"):   # slots 1, 3 and 4 hold the same key
        tk[f][3] = tk[f][1]
        tk[f][4] = tk[f][1]
    for f in ("n", "gamma"):
        tk[f][3] = tk[f][1]
        tk[f][4] = tk[f][1]
    q = rng.standard_normal(32)
    khat = quant.reconstruct_keys_any(tk, p.Pi, p.S, p.cb_k[0])
    q = q if khat[1] @ q > 0 else -q       # make the repeated key score positively
    tk["n"][[0, 2, 5]] = 0.0                # the others score exactly zero (no norm, no residual)
    tk["gamma"][[0, 2, 5]] = 0.0
    slots, est = dec.ip_topk(q, tk, p.Pi, p.S, p.cb_k, 4)
    assert slots.tolist() == [1, 3, 4, 0]   # the three equal best in slot order, then the lowest zero
    assert est[0] == est[1] == est[2] > 0 and est[3] == 0.0
    assert dec.ip_topk(q, tk, p.Pi, p.S, p.cb_k, 0)[0].size == 0
