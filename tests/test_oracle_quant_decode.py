"""Pins for the oracle's quantizer, page format and decode (CPU only)."""
import json
import math
import os

import numpy as np
import pytest

from oracle import codebook as cb
from oracle import decode as dec
from oracle import pagefmt, params, quant, rotation

HERE = os.path.dirname(os.path.abspath(__file__))


def _bf16_like(x):
    """Round fp64 values to bf16 precision (what the inputs are)."""
    import torch
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def test_stage1_reconstruction_mse():
    # E ||u - u~||^2 over random directions equals d * D(L): the codebook density is the
    # exact law of a rotated coordinate.  A transposed Pi in DEQUANT gives ~2 instead.
    d, L = 128, 4
    p = params.make(d, 3)
    X = _bf16_like(np.random.default_rng(1).standard_normal((20000, d)))
    idx, n, _ = quant.mse_stage(X, p.Pi, *p.cb_k)
    xt = quant.dequant_mse(idx, n, p.Pi, p.cb_k[0])
    rel = np.sum((X - xt) ** 2, axis=1) / n ** 2
    D = cb.distortion(*p.cb_k, d)
    assert abs(rel.mean() - d * D) < 5 * rel.std() / np.sqrt(len(rel))


def test_residual_norm_is_rotation_invariant():
    p = params.make(64, 4)
    X = _bf16_like(np.random.default_rng(2).standard_normal((500, 64)) * 3)
    k = quant.quantize_keys(X, p.Pi, p.S, p.cb_k)
    g_rot = k["n64"] * np.linalg.norm(k["yhat"] - p.cb_k[0][k["idx"]], axis=1)
    assert np.max(np.abs(k["gamma64"] - g_rot) / k["gamma64"]) < 1e-12


def test_zero_vector():
    p = params.make(128, 3)
    k = quant.quantize_keys(np.zeros((2, 128)), p.Pi, p.S, p.cb_k)
    assert np.all(k["idx"] == 2) and np.all(k["n"] == 0) and np.all(k["gamma"] == 0)
    assert np.all(k["sigma"] == 1)
    v = quant.quantize_values(np.zeros((1, 128)), p.Pi, p.cb_v)
    assert np.all(v["idx"] == 4)


def test_qjl_estimator_unbiased_with_closed_form_variance():
    # d = m = 8, fixed x, q and Pi; 10^4 independent Gaussian S.  The QJL-corrected inner
    # product must average to the exact <q, x> (brute force); its variance has the closed
    # form [(pi/2) gamma^2 ||q||^2 - <q, r>^2] / m.
    d = m = 8
    rs = np.random.default_rng(3)
    x = _bf16_like(rs.standard_normal(d)[None, :])
    q = rs.standard_normal(d)
    Pi = rotation.haar_rotation(d, 0)
    cbk = cb.codebook(d, 4)
    idx, n, _ = quant.mse_stage(x, Pi, *cbk)
    xt = quant.dequant_mse(idx, n, Pi, cbk[0])[0]
    r = x[0] - xt
    gamma = np.linalg.norm(r)
    exact = float(sum(q[i] * x[0, i] for i in range(d)))
    N = 10000
    est = np.empty(N)
    for s in range(N):
        S = rotation.qjl_matrix(m, d, seed=1000 + s)
        sig, g, _ = quant.qjl_stage(x, idx, n, Pi, S, cbk[0])
        khat = quant.reconstruct_keys(idx, n, sig, g, Pi, S, cbk[0])[0]
        est[s] = khat @ q
    var = ((math.pi / 2) * gamma ** 2 * (q @ q) - (q @ r) ** 2) / m
    assert abs(est.mean() - exact) < 4 * math.sqrt(var / N)
    assert abs(est.var() / var - 1) < 0.08


def test_qjl_key_reconstruction_error():
    # E ||rhat - r||^2 = gamma^2 (pi d / (2 m) - 1 / m) for the sign sketch of r.
    d = m = 16
    r = np.random.default_rng(4).standard_normal(d)
    gamma = np.linalg.norm(r)
    N = 4000
    errs = np.empty(N)
    for s in range(N):
        S = rotation.qjl_matrix(m, d, seed=50000 + s)
        sig = (S @ r >= 0).astype(np.float64)
        rhat = gamma * quant.QJL_CONST / m * ((2 * sig - 1) @ S)
        errs[s] = np.sum((rhat - r) ** 2) / gamma ** 2
    target = math.pi * d / (2 * m) - 1.0 / m
    assert abs(errs.mean() - target) < 5 * errs.std() / math.sqrt(N)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("b", [2, 3, 4, 5])
def test_pack_round_trip(d, b):
    rs = np.random.default_rng(d * 10 + b)
    P = pagefmt.P
    kidx = rs.integers(0, 2 ** (b - 1), (P, d))
    vidx = rs.integers(0, 2 ** b, (P, d))
    sigma = rs.integers(0, 2, (P, d)).astype(np.uint8)
    nk, gm, nv = (rs.standard_normal(P).astype(np.float32) for _ in range(3))
    buf = pagefmt.pack_page(d, b, d, kidx, sigma, nk, gm, vidx, nv)
    assert len(buf) == pagefmt.page_bytes(d, b, d)
    u = pagefmt.unpack_page(d, b, d, buf)
    assert np.array_equal(u["kidx"], kidx) and np.array_equal(u["vidx"], vidx)
    assert np.array_equal(u["sigma"], sigma)
    for a, e in ((u["nk"], nk), (u["gamma"], gm), (u["nv"], nv)):
        assert np.array_equal(a.view(np.uint32), e.view(np.uint32))


def test_positions_are_bijective():
    for D in (64, 128, 256):
        w, bit = pagefmt.coord_position(np.arange(D), D)
        assert len(set(zip(w.tolist(), bit.tolist()))) == D and w.max() == D // 32 - 1
    w, bit = pagefmt.token_position(np.arange(128))
    assert len(set(zip(w.tolist(), bit.tolist()))) == 128


def test_hand_built_page_d32_b2():
    g = json.load(open(os.path.join(HERE, "golden", "page_d32_b2.json")))
    d, b, m, P = 32, 2, 32, 128
    kidx = np.zeros((P, d), dtype=np.int64)
    j = np.arange(d)
    kidx[0] = j & 1
    kidx[1] = (j < 16).astype(np.int64)
    kidx[2] = (j < 4).astype(np.int64)
    kidx[3, 31] = 1
    sigma = np.zeros((P, m), dtype=np.uint8)
    sigma[5, 20] = 1
    vidx = np.zeros((P, d), dtype=np.int64)
    vidx[5, 7] |= 1          # plane 0, coordinate 7, slot 5
    vidx[127, 0] |= 2        # plane 1, coordinate 0, slot 127
    vidx[0:32, 31] |= 1      # plane 0, coordinate 31, slots 0..31
    nk = np.zeros(P, dtype=np.float32)
    nk[2] = 1.5
    z = np.zeros(P, dtype=np.float32)
    buf = pagefmt.pack_page(d, b, m, kidx, sigma, nk, z, vidx, z)
    assert len(buf) == g["page_bytes"]
    words = buf.view("<u4")
    expected = np.zeros_like(words)
    for case in g["cases"]:
        expected[case["offset"] // 4] = int(case["u32"], 16)
    assert np.array_equal(words, expected)


@pytest.mark.parametrize("name", ["page_d128_b3.json", "page_d256_b2.json"])
def test_hand_built_pages_wide(name):
    """Hand-derived words at d = 128 and 256, where the key/sign map's 2*kb term and its
    D-dependent stride (2*D/32 per c) take values that d = 32 never reaches."""
    g = json.load(open(os.path.join(HERE, "golden", name)))
    d, b, m, P = g["d"], g["b"], g["m"], 128
    arrays = dict(kidx=np.zeros((P, d), dtype=np.int64), sigma=np.zeros((P, m), dtype=np.uint8),
                  vidx=np.zeros((P, d), dtype=np.int64), nk=np.zeros(P, dtype=np.float32),
                  gamma=np.zeros(P, dtype=np.float32), nv=np.zeros(P, dtype=np.float32))
    for inp in g["inputs"]:
        a = arrays[inp["field"]]
        if a.ndim == 1:
            a[inp["slot"]] = inp["value"]
        elif "coords" in inp:
            lo, hi = inp["coords"]
            a[inp["slot"], lo:hi + 1] = inp["value"]
        else:
            a[inp["slot"], inp["coord"]] = inp["value"]
    buf = pagefmt.pack_page(d, b, m, arrays["kidx"], arrays["sigma"], arrays["nk"], arrays["gamma"],
                            arrays["vidx"], arrays["nv"])
    assert len(buf) == g["page_bytes"]
    words = buf.view("<u4")
    expected = np.zeros_like(words)
    for case in g["cases"]:
        expected[case["offset"] // 4] = int(case["u32"], 16)
    assert np.array_equal(words, expected), np.nonzero(words != expected)
    # and the unpacker reads the hand-derived page back to the same fields
    u = pagefmt.unpack_page(d, b, m, expected.view(np.uint8))
    for key, a in arrays.items():
        assert np.array_equal(np.asarray(u[key]), a), key


def _random_tokens(p, T, rs, scale=1.0):
    Xk = _bf16_like(rs.standard_normal((T, p.d)) * scale)
    Xv = _bf16_like(rs.standard_normal((T, p.d)))
    k = quant.quantize_keys(Xk, p.Pi, p.S, p.cb_k)
    v = quant.quantize_values(Xv, p.Pi, p.cb_v)
    return (dict(idx=k["idx"], n=k["n"], sigma=k["sigma"], gamma=k["gamma"]),
            dict(idx=v["idx"], n=v["n"]))


def test_routes_agree():
    p = params.make(64, 3)
    rs = np.random.default_rng(6)
    tk, tv = _random_tokens(p, 300, rs, scale=2.0)
    for _ in range(4):
        q = rs.standard_normal(64)
        oa, la = dec.attend_route_a(q, tk, tv, p.Pi, p.S, p.cb_k, p.cb_v)
        ob, lb = dec.attend_route_b(q, tk, tv, p.Pi, p.S, p.cb_k, p.cb_v)
        assert np.max(np.abs(la - lb)) <= 1e-12 * np.max(np.abs(la))
        assert np.max(np.abs(oa - ob)) <= 1e-12 * np.max(np.abs(oa))


def test_decode_is_textbook_attention_over_reconstructed_cache():
    # Brute force with explicit loops: logits <q, khat_t>/sqrt(d), softmax, weighted vhat;
    # query head h reads kv head h // G.
    p = params.make(64, 4)
    rs = np.random.default_rng(7)
    B, Hkv, G, T = 2, 2, 3, 40
    toks = {(bb, g): _random_tokens(p, T, rs) for bb in range(B) for g in range(Hkv)}
    q = rs.standard_normal((B, Hkv * G, 64))
    out, logits = dec.decode(q, lambda bb, g: toks[(bb, g)], Hkv, p.Pi, p.S, p.cb_k, p.cb_v)
    for bb in range(B):
        for h in range(Hkv * G):
            tk, tv = toks[(bb, h // G)]
            K = quant.reconstruct_keys(tk["idx"], tk["n"], tk["sigma"], tk["gamma"], p.Pi, p.S, p.cb_k[0])
            V = quant.reconstruct_values(tv["idx"], tv["n"], p.Pi, p.cb_v[0])
            lg = [sum(q[bb, h, j] * K[t, j] for j in range(64)) / 8.0 for t in range(T)]
            w = [math.exp(x) for x in lg]
            tot = sum(w)
            o = [sum(w[t] / tot * V[t, j] for t in range(T)) for j in range(64)]
            assert np.max(np.abs(np.array(lg) - logits[bb][h])) < 1e-10
            assert np.max(np.abs(np.array(o) - out[bb, h])) < 1e-10


def test_empty_sequence_gives_zero():
    p = params.make(64, 3)
    e = dict(idx=np.zeros((0, 64), dtype=np.int64), n=np.zeros(0), sigma=np.zeros((0, 64)), gamma=np.zeros(0))
    o, lg = dec.attend_route_a(np.ones(64), e, dict(idx=e["idx"], n=e["n"]), p.Pi, p.S, p.cb_k, p.cb_v)
    assert np.all(o == 0) and len(lg) == 0


def test_unpack_tokens_across_pages():
    p = params.make(64, 3)
    rs = np.random.default_rng(8)
    T, n_pages = 300, 3
    tk, tv = _random_tokens(p, T, rs)
    pb = pagefmt.page_bytes(64, 3, 64)
    cache = np.zeros(2 * n_pages * pb, dtype=np.uint8)        # batch 1, kv heads 2
    for pg in range(n_pages):
        lo, hi = pg * 128, min(T, pg * 128 + 128)
        pad = lambda a: np.concatenate([a[lo:hi], np.zeros((128 - (hi - lo),) + a.shape[1:], a.dtype)])
        page = pagefmt.pack_page(64, 3, 64, pad(tk["idx"]), pad(tk["sigma"]), pad(tk["n"]),
                                 pad(tk["gamma"]), pad(tv["idx"]), pad(tv["n"]))
        base = (1 * n_pages + pg) * pb
        cache[base:base + pb] = page
    u = pagefmt.unpack_tokens(64, 3, 64, cache, n_pages, 0, 1, T, 2)
    assert np.array_equal(u["kidx"], tk["idx"]) and np.array_equal(u["vidx"], tv["idx"])
    assert np.array_equal(u["nk"], tk["n"])
