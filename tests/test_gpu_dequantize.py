"""tq_dequantize_kv against the oracle's reconstruction on the GPU's own pages, plus the
reconstruction error statistics the method predicts (codebook distortion; for keys the QJL
residual estimate's closed-form variance)."""
import numpy as np
import pytest
import torch

import kv_cache_vector_19_b300 as tq
from oracle import codebook as ocb
from oracle import quant

import parity as P

pytestmark = pytest.mark.gpu


def _setup(d, b, B=2, H=2, N=300, maxT=512, seed=3):
    run = P.Run(d, b, B, H, H, maxT)
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(B, H, N, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, H, N, d, generator=g).to(torch.bfloat16)
    run.quantize(k, v, [0] * B)
    return run, k, v


@pytest.mark.parametrize("d,b", [(128, 3), (64, 2), (256, 5), (128, 4)])
def test_dequantize_matches_oracle_reconstruction(d, b):
    run, k, v = _setup(d, b)
    B, H, N = k.shape[:3]
    start = [0, 37]
    n = 200
    kout = torch.full((B, H, n, d), float("nan"), device="cuda")
    vout = torch.full((B, H, n, d), float("nan"), device="cuda")
    sp = torch.tensor(start, dtype=torch.int32, device="cuda")
    run.ctx.dequantize_kv(run.cache, sp, B, H, n, run.max_tokens, kout, vout)
    assert run.status() == tq.TQ_OK
    kout, vout = kout.cpu().double().numpy(), vout.cpu().double().numpy()
    cache = run.cache_np()
    p = run.p
    for bb in range(B):
        for h in range(H):
            tok = run.tokens(cache, bb, h, N)
            sl = slice(start[bb], start[bb] + n)
            kref = quant.reconstruct_keys(tok["kidx"][sl], tok["nk"][sl].astype(np.float64), tok["sigma"][sl],
                                          tok["gamma"][sl].astype(np.float64), p.Pi, p.S, p.cb_k[0])
            vref = quant.reconstruct_values(tok["vidx"][sl], tok["nv"][sl].astype(np.float64), p.Pi, p.cb_v[0])
            for got, ref in ((kout[bb, h], kref), (vout[bb, h], vref)):
                err = np.linalg.norm(got - ref, axis=1) / np.maximum(np.linalg.norm(ref, axis=1), 1e-30)
                assert np.max(err) < 2e-5, np.max(err)


def test_dequantize_one_side_and_bounds():
    run, k, v = _setup(128, 3, B=1, H=1, N=130)
    out = torch.zeros(1, 1, 130, 128, device="cuda")
    sp = torch.zeros(1, dtype=torch.int32, device="cuda")
    run.ctx.dequantize_kv(run.cache, sp, 1, 1, 130, run.max_tokens, v_out=out)   # keys skipped
    assert run.status() == tq.TQ_OK and torch.isfinite(out).all()
    bad = torch.tensor([run.max_tokens - 10], dtype=torch.int32, device="cuda")
    untouched = torch.full((1, 1, 130, 128), 7.0, device="cuda")
    run.ctx.dequantize_kv(run.cache, bad, 1, 1, 130, run.max_tokens, k_out=untouched)
    assert run.status() == tq.TQ_EBOUNDS
    assert torch.all(untouched == 7.0)


@pytest.mark.parametrize("d,b", [(128, 3), (64, 4)])
def test_reconstruction_error_matches_distortion(d, b):
    """Normalized MSE of values = d * D(b bits); of keys = d * D(b-1 bits) * (pi/2 - 1/d) at
    m = d (stage-1 distortion times the QJL estimate's variance factor)."""
    B, H, N = 2, 4, 1000
    run, k, v = _setup(d, b, B=B, H=H, N=N, maxT=1024, seed=9)
    kout = torch.empty(B, H, N, d, device="cuda")
    vout = torch.empty(B, H, N, d, device="cuda")
    sp = torch.zeros(B, dtype=torch.int32, device="cuda")
    run.ctx.dequantize_kv(run.cache, sp, B, H, N, run.max_tokens, kout, vout)
    assert run.status() == tq.TQ_OK
    kx, vx = k.float().cuda(), v.float().cuda()
    mse_k = ((kout - kx).pow(2).sum(-1) / kx.pow(2).sum(-1)).mean().item()
    mse_v = ((vout - vx).pow(2).sum(-1) / vx.pow(2).sum(-1)).mean().item()
    ck, tk = ocb.codebook(d, 2 ** (b - 1))
    cv, tv = ocb.codebook(d, 2 ** b)
    exp_v = d * ocb.distortion(cv, tv, d)
    exp_k = d * ocb.distortion(ck, tk, d) * (np.pi / 2 - 1.0 / d)
    assert abs(mse_v / exp_v - 1) < 0.05, (mse_v, exp_v)
    assert abs(mse_k / exp_k - 1) < 0.08, (mse_k, exp_k)
