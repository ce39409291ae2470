"""Pins for the oracle's generalised formats (CPU only): separate key and value widths and
keys without the QJL stage ([3BITS] "Python + HuggingFace": a cache object with key_bits and
value_bits, a stage-1-only quantizer with bits; the QJL remark of the same page)."""
import math

import numpy as np
import pytest

from oracle import codebook as cb
from oracle import decode as dec
from oracle import pagefmt, params, quant

P = pagefmt.P


def _bf16_like(x):
    import torch
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("d,kb,vb,m,per_token", [
    (128, 2, 3, 128, 32 + 16 + 4 + 4 + 48 + 4),   # version 1, b = 3: 108 B per token
    (128, 4, 2, 0, 64 + 4 + 32 + 4),              # key_bits 4 (no QJL), value_bits 2
    (128, 3, 3, 0, 48 + 4 + 48 + 4),              # 3-bit keys and values, QJL off
    (128, 2, 4, 128, 32 + 16 + 4 + 4 + 64 + 4),   # key_bits 3 with QJL, value_bits 4
    (64, 2, 2, 0, 16 + 4 + 16 + 4),
    (256, 1, 5, 256, 32 + 32 + 4 + 4 + 160 + 4),
])
def test_page_sizes_by_hand(d, kb, vb, m, per_token):
    assert pagefmt.page_bytes_kv(d, kb, vb, m) == P * per_token
    off = pagefmt.region_offsets_kv(d, kb, vb, m)
    assert off["signs"] == kb * d * P // 8 and off["vcodes"] - off["nk"] == (8 if m else 4) * P
    assert off["end"] - off["nv"] == 4 * P and off["nv"] - off["vcodes"] == vb * d * P // 8


def _random_page(d, kb, vb, m, rs):
    kidx = rs.integers(0, 2 ** kb, (P, d))
    vidx = rs.integers(0, 2 ** vb, (P, d))
    sigma = rs.integers(0, 2, (P, m)).astype(np.uint8) if m else None
    nk, gm, nv = (rs.standard_normal(P).astype(np.float32) for _ in range(3))
    return kidx, sigma, nk, (gm if m else None), vidx, nv


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("kb,vb,qjl", [(1, 2, False), (3, 2, False), (4, 5, False), (2, 4, True), (3, 2, True),
                                       (1, 5, True)])
def test_round_trip(d, kb, vb, qjl):
    m = d if qjl else 0
    rs = np.random.default_rng(100 * d + 10 * kb + vb)
    kidx, sigma, nk, gm, vidx, nv = _random_page(d, kb, vb, m, rs)
    buf = pagefmt.pack_page_kv(d, kb, vb, m, kidx, sigma, nk, gm, vidx, nv)
    assert len(buf) == pagefmt.page_bytes_kv(d, kb, vb, m)
    u = pagefmt.unpack_page_kv(d, kb, vb, m, buf)
    assert np.array_equal(u["kidx"], kidx) and np.array_equal(u["vidx"], vidx)
    assert np.array_equal(u["nk"].view(np.uint32), nk.view(np.uint32))
    assert np.array_equal(u["nv"].view(np.uint32), nv.view(np.uint32))
    if qjl:
        assert np.array_equal(u["sigma"], sigma) and np.array_equal(u["gamma"].view(np.uint32), gm.view(np.uint32))
    else:
        assert u["sigma"] is None and u["gamma"] is None


@pytest.mark.parametrize("d,b", [(64, 2), (128, 3), (256, 4)])
def test_mse_only_page_is_version_1_without_sign_and_gamma(d, b):
    # The version-1 layout is pinned by the hand-built page; a key format without QJL must be
    # that page with regions 2 (signs) and 4 (gamma) cut out, every other byte unchanged.
    rs = np.random.default_rng(d + b)
    kidx, sigma, nk, gm, vidx, nv = _random_page(d, b - 1, b, d, rs)
    v1 = pagefmt.pack_page(d, b, d, kidx, sigma, nk, gm, vidx, nv)
    o = pagefmt.region_offsets(d, b, d)
    cut = np.concatenate([v1[:o["signs"]], v1[o["nk"]:o["gamma"]], v1[o["vcodes"]:]])
    v2 = pagefmt.pack_page_kv(d, b - 1, b, 0, kidx, None, nk, None, vidx, nv)
    assert np.array_equal(v2, cut)
    assert np.array_equal(pagefmt.pack_page_kv(d, b - 1, b, d, kidx, sigma, nk, gm, vidx, nv), v1)


def test_constants_of_each_format():
    d = 64
    a = params.make_kv(d, 4, 2, qjl=False)
    assert (a.kb, a.vb, a.m, a.S) == (4, 2, 0, None)
    assert len(a.cb_k[0]) == 16 and len(a.cb_v[0]) == 4
    w = params.make_kv(d, 4, 2, qjl=True)
    assert (w.kb, w.m) == (3, d) and len(w.cb_k[0]) == 8
    v1 = params.make(d, 3)
    s = params.make_kv(d, 3, 3, qjl=True)
    assert np.array_equal(s.Pi, v1.Pi) and np.array_equal(s.S, v1.S)
    assert all(np.array_equal(x, y) for x, y in zip(s.cb_k + s.cb_v, v1.cb_k + v1.cb_v))
    with pytest.raises(ValueError):
        params.make_kv(d, 1, 2, qjl=True)


@pytest.mark.parametrize("kb", [1, 2, 3])
def test_mse_only_inner_product_shrinks_by_one_minus_distortion(kb):
    # Over Haar rotations Pi, E[n Pi^T c(Pi x / n)] = (1 - d D) x exactly: by rotation
    # invariance the mean is parallel to x, and its length is E<y, c(y)> = d E[c(Y)^2] =
    # d (E[Y^2] - D) = 1 - d D, because a Lloyd-Max centroid is the conditional mean of its
    # cell.  (At one bit and large d the factor tends to 2/pi.)  A transposed Pi, a shifted
    # cell index or a dropped norm breaks the identity.
    d, N = 16, 4000
    rs = np.random.default_rng(11 + kb)
    x = _bf16_like(rs.standard_normal(d) * 2.0)
    q = rs.standard_normal(d)
    c, t = cb.codebook(d, 2 ** kb)
    samples = np.empty(N)
    for i in range(N):
        Q, R = np.linalg.qr(rs.standard_normal((d, d)))
        Pi = Q * np.where(np.diag(R) < 0, -1.0, 1.0)          # Haar (sign-fixed QR)
        idx, n, _ = quant.mse_stage(x[None, :], Pi, c, t)
        samples[i] = quant.dequant_mse(idx, n, Pi, c)[0] @ q
    expect = (1.0 - d * cb.distortion(c, t, d)) * (x @ q)
    assert abs(samples.mean() - expect) < 4.0 * samples.std() / math.sqrt(N)


def _tokens(p, T, rs, qjl):
    Xk = _bf16_like(rs.standard_normal((T, p.d)) * 2.0)
    Xv = _bf16_like(rs.standard_normal((T, p.d)))
    k = quant.quantize_keys(Xk, p.Pi, p.S, p.cb_k) if qjl else quant.quantize_keys_mse(Xk, p.Pi, p.cb_k)
    v = quant.quantize_values(Xv, p.Pi, p.cb_v)
    return (dict(idx=k["idx"], n=k["n"], sigma=k["sigma"], gamma=k["gamma"]), dict(idx=v["idx"], n=v["n"]))


@pytest.mark.parametrize("key_bits,value_bits,qjl", [(4, 2, False), (3, 3, False), (4, 2, True), (2, 4, True)])
def test_routes_agree(key_bits, value_bits, qjl):
    p = params.make_kv(64, key_bits, value_bits, qjl=qjl)
    rs = np.random.default_rng(key_bits * 10 + value_bits)
    tk, tv = _tokens(p, 300, rs, qjl)
    for _ in range(3):
        q = rs.standard_normal(64)
        oa, la = dec.attend_route_a(q, tk, tv, p.Pi, p.S, p.cb_k, p.cb_v)
        ob, lb = dec.attend_route_b(q, tk, tv, p.Pi, p.S, p.cb_k, p.cb_v)
        assert np.max(np.abs(la - lb)) <= 1e-12 * np.max(np.abs(la))
        assert np.max(np.abs(oa - ob)) <= 1e-12 * np.max(np.abs(oa))


def test_mse_only_decode_is_textbook_attention():
    # Brute force with explicit loops over the stage-1 reconstruction n Pi^T c[idx] of keys
    # and values (no QJL term); query head h reads kv head h // G.
    p = params.make_kv(32, 3, 2, qjl=False)
    rs = np.random.default_rng(21)
    B, Hkv, G, T, d = 2, 2, 2, 30, 32
    toks = {(bb, g): _tokens(p, T, rs, False) for bb in range(B) for g in range(Hkv)}
    q = rs.standard_normal((B, Hkv * G, d))
    out, logits = dec.decode(q, lambda bb, g: toks[(bb, g)], Hkv, p.Pi, p.S, p.cb_k, p.cb_v)
    ck, cv = p.cb_k[0], p.cb_v[0]
    for bb in range(B):
        for h in range(Hkv * G):
            tk, tv = toks[(bb, h // G)]
            K = [[float(tk["n"][t]) * sum(ck[tk["idx"][t, i]] * p.Pi[i, j] for i in range(d)) for j in range(d)]
                 for t in range(T)]
            V = [[float(tv["n"][t]) * sum(cv[tv["idx"][t, i]] * p.Pi[i, j] for i in range(d)) for j in range(d)]
                 for t in range(T)]
            lg = [sum(q[bb, h, j] * K[t][j] for j in range(d)) / math.sqrt(d) for t in range(T)]
            mx = max(lg)
            w = [math.exp(x - mx) for x in lg]
            tot = sum(w)
            o = [sum(w[t] / tot * V[t][j] for t in range(T)) for j in range(d)]
            assert np.max(np.abs(np.array(lg) - logits[bb][h])) < 1e-10
            assert np.max(np.abs(np.array(o) - out[bb, h])) < 1e-10


def test_mse_only_zero_vector_and_cache_round_trip():
    d, kb, vb = 64, 2, 3
    p = params.make_kv(d, kb, vb, qjl=False)
    k = quant.quantize_keys_mse(np.zeros((1, d)), p.Pi, p.cb_k)
    assert np.all(k["idx"] == 2 ** (kb - 1)) and k["n"][0] == 0 and k["sigma"] is None
    # a two-page cache of one (batch, kv head) read back through unpack_tokens_kv
    rs = np.random.default_rng(31)
    T = 200
    tk, tv = _tokens(p, T, rs, False)
    pages = []
    for pg in range(2):
        sl = slice(pg * P, min(T, (pg + 1) * P))
        n = sl.stop - sl.start
        pad = lambda a: np.concatenate([a, np.zeros((P - n,) + a.shape[1:], dtype=a.dtype)])
        pages.append(pagefmt.pack_page_kv(d, kb, vb, 0, pad(tk["idx"][sl]), None, pad(tk["n"][sl]), None,
                                          pad(tv["idx"][sl]), pad(tv["n"][sl])))
    u = pagefmt.unpack_tokens_kv(d, kb, vb, 0, np.concatenate(pages), 2, 0, 0, T, 1)
    assert np.array_equal(u["kidx"], tk["idx"]) and np.array_equal(u["vidx"], tv["idx"])
    assert u["sigma"] is None and u["gamma"] is None
