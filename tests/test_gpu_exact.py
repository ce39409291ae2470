"""Quantizer decisions next to a boundary, on every quantizer kernel.

The oracle screens a large pool of seeded N(0,1) bf16 vectors and keeps those with a rotated
coordinate within 2^-19 of a Lloyd-Max boundary (keys and values, [BLOG] §1.2 stage 1), or
with a projection (S r)_i within 2^-15 ||r|| of zero (keys, stage 2).  Those decisions lie
inside the band where the library's fast fp32 / tensor-core arithmetic cannot settle them,
so every selected row goes through the double-float re-evaluation.  The pages must then hold
exactly the oracle's codes and signs.
"""
import numpy as np
import pytest
import torch

import kv_cache_vector_19_b300 as tq
from oracle import params, quant

import parity as P

pytestmark = pytest.mark.gpu

BAND_CODE = 2.0 ** -19
BAND_SIGN = 2.0 ** -15


def _pool(d, n, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((n, d), dtype=np.float32)
    return torch.from_numpy(x).to(torch.bfloat16)


def _near_code_rows(X, p, book, want):
    """Indices of rows with a coordinate within BAND_CODE of a boundary of ``book``."""
    Xd = X.double().numpy()
    n = np.linalg.norm(Xd, axis=1)
    yhat = (Xd @ p.Pi.T) / n[:, None]
    t = np.asarray(book[1])
    dist = np.min(np.abs(yhat[..., None] - t), axis=(1, 2))
    return np.nonzero(dist < BAND_CODE)[0][:want]


def _near_sign_rows(X, p, want):
    Xd = X.double().numpy()
    ok = quant.quantize_keys(Xd, p.Pi, p.S, p.cb_k)
    g = ok["gamma64"]
    near = np.min(np.abs(ok["z"]), axis=1) < BAND_SIGN * g
    return np.nonzero(near & (g > 0))[0][:want]


def _selected(d, b, n_rows):
    """K rows (three quarters near a key boundary, one quarter near a zero projection) and V
    rows (near a value boundary), n_rows each, from seeded pools."""
    p = params.make(d, b)
    pool = _pool(d, {64: 1 << 19, 128: 1 << 18, 256: 1 << 17}[d], seed=1000 + d + b)
    n_sign = n_rows // 4
    kc = _near_code_rows(pool, p, p.cb_k, n_rows - n_sign)
    ks = _near_sign_rows(pool[: 1 << 17], p, n_rows - len(kc))
    vc = _near_code_rows(pool, p, p.cb_v, n_rows)
    assert len(kc) + len(ks) == n_rows and len(vc) == n_rows, (len(kc), len(ks), len(vc))
    k = torch.cat([pool[torch.from_numpy(kc)], pool[torch.from_numpy(ks)]])
    v = pool[torch.from_numpy(vc)]
    return k, v


def _check(run, k, v, n):
    cache = run.cache_np()
    got = run.tokens(cache, 0, 0, n)
    res = P.compare_sequence(run, P.to64(k), P.to64(v), got)
    assert res["kmis"] == 0 and res["vmis"] == 0 and res["smis"] == 0, (res["kmis"], res["vmis"], res["smis"])
    P.assert_quantize_ok(res)


@pytest.mark.parametrize("d,b", [(128, 2), (128, 3), (128, 5), (64, 3), (256, 3), (256, 5)])
def test_boundary_rows_bulk(d, b):
    n = 512
    k, v = _selected(d, b, n)
    run = P.Run(d, b, 1, 1, 1, n)
    run.quantize(k.view(1, 1, n, d), v.view(1, 1, n, d), [0])
    assert run.status() == tq.TQ_OK
    _check(run, k, v, n)


@pytest.mark.parametrize("d,b", [(128, 3), (64, 4), (256, 2)])
def test_boundary_rows_appends(d, b):
    n = 64
    k, v = _selected(d, b, n)
    run = P.Run(d, b, 1, 1, 1, n)
    for t in range(0, n, 4):   # 4 tokens per call: the few-token kernel
        run.quantize(k[t:t + 4].reshape(1, 1, 4, d).contiguous(), v[t:t + 4].reshape(1, 1, 4, d).contiguous(), [t])
    assert run.status() == tq.TQ_OK
    _check(run, k, v, n)
