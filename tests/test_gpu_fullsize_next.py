"""The "next" rows at the long-context benchmark's full size (4 sequences x 8 KV heads x 131,072
tokens, 32 query heads, b = 3, the benchmark's seeded inputs):

* the paged pool through a shuffled block table decodes bit-identically to the contiguous cache
  (outputs and logits), after the same prefill and an append;
* the scan's top-k of sampled query heads equals an exact sort of the same fp32 estimates;
* Sparse V with peaked queries stays within the oracle's skipped-mass bound of the oracle's
  sparse output on a sampled KV head, recomputed in full from the GPU's pages.
"""
import math

import numpy as np
import pytest
import torch

import kv_cache_vector_19_b300 as tq
from kv_cache_vector_19_b300 import workloads
from oracle import decode as odec

import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def longctx():
    w = workloads.preset("longctx")
    data = workloads.generate(w)
    run = P.Run(w.d, w.b, w.batch, w.kv_heads, w.q_heads, w.max_tokens, seed=w.seed)
    run.quantize(data["k"], data["v"], [0] * w.batch)
    run.quantize(data["k_new"][0], data["v_new"][0], [w.tokens] * w.batch)
    return w, data, run


def test_paged_pool_full_size(longctx):
    w, data, run = longctx
    B, H, T = w.batch, w.kv_heads, w.max_tokens
    max_blocks = (T + 127) // 128
    n_blocks = B * max_blocks
    perm = torch.randperm(n_blocks, generator=torch.Generator().manual_seed(9))
    table = perm.to(torch.int32).reshape(B, max_blocks).cuda()
    pool = run.ctx.alloc_pool(H, n_blocks)
    zero = torch.zeros(B, dtype=torch.int32, device="cuda")
    run.ctx.quantize_kv_paged(data["k"].cuda(), data["v"].cuda(), zero, pool, n_blocks, table)
    at = torch.full((B,), w.tokens, dtype=torch.int32, device="cuda")
    run.ctx.quantize_kv_paged(data["k_new"][0].cuda(), data["v_new"][0].cuda(), at, pool, n_blocks, table)
    q = data["q"][0].cuda().contiguous()
    lens = torch.full((B,), w.tokens + 1, dtype=torch.int32, device="cuda")
    Tw = 128 * max_blocks
    ws = run.ctx.alloc_workspace(B, w.q_heads, H, Tw)
    out_c, out_p = torch.empty_like(q), torch.empty_like(q)
    lg_c = torch.zeros(B, w.q_heads, T, device="cuda")
    lg_p = torch.zeros(B, w.q_heads, Tw, device="cuda")
    run.ctx.attn_decode(q, run.cache, lens, H, T, out_c, run.ws, logits=lg_c)
    run.ctx.attn_decode_paged(q, pool, n_blocks, table, lens, H, out_p, ws, logits=lg_p)
    assert run.status() == tq.TQ_OK
    assert torch.equal(out_c, out_p)
    n = w.tokens + 1
    assert torch.equal(lg_c[:, :, :n], lg_p[:, :, :n])


def test_scan_full_size(longctx):
    w, data, run = longctx
    B, H, T, k = w.batch, w.kv_heads, w.max_tokens, 100
    q = data["q"][0].cuda().contiguous()
    lens = torch.full((B,), w.tokens + 1, dtype=torch.int32, device="cuda")
    idx, sc = run.ctx.ip_topk(q, run.cache, lens, H, T, k)
    lg = torch.zeros(B, w.q_heads, T, device="cuda")
    out = torch.empty_like(q)
    run.ctx.attn_decode(q, run.cache, lens, H, T, out, run.ws, logits=lg)
    assert run.status() == tq.TQ_OK
    scale = np.float32(math.sqrt(w.d))
    n = w.tokens + 1
    for bb, hq in [(0, 0), (1, 13), (3, 31)]:
        est = (lg[bb, hq, :n].cpu().numpy().astype(np.float32) * scale).astype(np.float32)
        want = np.lexsort((np.arange(n), -est.astype(np.float64)))[:k]
        assert np.array_equal(idx[bb, hq].cpu().numpy(), want), (bb, hq)
        assert np.array_equal(sc[bb, hq].cpu().numpy(), est[want]), (bb, hq)


def test_sparse_v_full_size(longctx):
    w, data, run = longctx
    B, H, T, G, theta = w.batch, w.kv_heads, w.max_tokens, w.group, 1e-3
    q = (data["q"][0] * 4).cuda().contiguous()   # peaked attention
    lens = torch.full((B,), w.tokens + 1, dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    run.ctx.set_sparse_v(theta)
    run.ctx.attn_decode(q, run.cache, lens, H, T, out, run.ws)
    run.ctx.set_sparse_v(0.0)
    assert run.status() == tq.TQ_OK
    out = out.cpu().numpy()
    cache = run.cache_np()
    bb, h, n = 2, 5, w.tokens + 1
    tok = run.tokens(cache, bb, h, n)
    tk = dict(idx=tok["kidx"], n=tok["nk"].astype(np.float64), sigma=tok["sigma"],
              gamma=tok["gamma"].astype(np.float64))
    tv = dict(idx=tok["vidx"], n=tok["nv"].astype(np.float64))
    qc = q.cpu()
    for hq in (h * G, h * G + G - 1):
        o, _, skipped = odec.attend_sparse_v(qc[bb, hq].double().numpy(), tk, tv, run.p.Pi, run.p.S, run.p.cb_k,
                                             run.p.cb_v, theta)
        assert skipped > 0.0
        assert np.linalg.norm(out[bb, hq] - o) <= skipped + 2e-3 * np.linalg.norm(o), hq
