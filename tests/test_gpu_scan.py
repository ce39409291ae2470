"""GPU tests of the compressed inner-product scan (tq_ip_topk; [BLOG] 6.4: vector search and the
compression of RAG indexes).

* The selection is exact: against the decode logits of the same call (read back), each query
  head's slots equal an exact argsort by (estimate descending, slot ascending), and the returned
  estimates equal logit * sqrt(d) in fp32 — including rows whose keys repeat (ties), rows with
  one key almost everywhere (the coarse bin of the k-th key overflows shared memory and the exact
  radix select takes over), rows shorter than k (padding -1 / -inf), and k = 1 and TQ_TOPK_MAX.
* Against the oracle's scan (oracle.decode.ip_topk on the GPU's own pages, fp64): every returned estimate is within
  the score bar of the oracle's, every returned slot's oracle estimate is within twice that of
  the oracle's k-th best, and every slot that beats the k-th best by more than that is returned.
"""
import math

import numpy as np
import pytest
import torch

import kv_cache_vector_19_b300 as tq
from oracle import decode as odec
import parity as P

pytestmark = pytest.mark.gpu


def _exact_topk(scores, k):
    order = np.lexsort((np.arange(len(scores)), -scores.astype(np.float64)))
    return order[:k]


def _run(d, b, B, H, G, T, k, seq, keys="normal", seed=0):
    run = P.Run(d, b, B, H, G * H, T, seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    kk = torch.randn(B, H, T, d, generator=g)
    vv = torch.randn(B, H, T, d, generator=g)
    if keys == "dup":      # every key repeated in 8 slots: equal codes, equal estimates (ties)
        kk = kk[:, :, ::8].repeat_interleave(8, dim=2)[:, :, :T].contiguous()
    elif keys == "equal":  # one key everywhere but a few slots: one bin far over the buffer, all ties
        base = kk[:, :, :1].clone()
        kk[:, :, 5:] = base
    elif keys == "narrow":  # one key plus small noise: distinct scores, all within one coarse bin
        kk = kk[:, :, :1] + 1e-3 * kk
    run.quantize(kk.to(torch.bfloat16), vv.to(torch.bfloat16), [0] * B)
    q = torch.randn(B, G * H, d, generator=g).cuda()
    sl = torch.as_tensor(seq, dtype=torch.int32, device="cuda")
    idx, sc = run.ctx.ip_topk(q, run.cache, sl, H, T, k)
    # the decode's own logits of the same queries
    out = torch.empty_like(q)
    lg = torch.full((B, G * H, T), float("nan"), device="cuda")
    run.ctx.attn_decode(q, run.cache, sl, H, T, out, run.ws, logits=lg)
    assert run.status() == tq.TQ_OK
    return run, q.cpu(), idx.cpu().numpy(), sc.cpu().numpy(), lg.cpu().numpy()


@pytest.mark.parametrize("k,keys,T", [(1, "normal", 3000), (10, "normal", 3000), (100, "dup", 3000),
                                      (1024, "normal", 3000), (100, "equal", 9000), (1024, "equal", 9000),
                                      (100, "narrow", 9000), (1000, "narrow", 9000)])
def test_topk_selection_is_exact(k, keys, T):
    d, b, B, H, G = 128, 3, 2, 2, 4
    seq = [T, 700]
    run, q, idx, sc, lg = _run(d, b, B, H, G, T, k, seq, keys=keys)
    scale = np.float32(math.sqrt(d))
    for bb in range(B):
        for hq in range(G * H):
            n = seq[bb]
            est = (lg[bb, hq, :n].astype(np.float32) * scale).astype(np.float32)
            want = _exact_topk(est, min(k, n))
            got = idx[bb, hq]
            assert np.array_equal(got[:len(want)], want), (bb, hq)
            assert np.array_equal(sc[bb, hq, :len(want)], est[want]), (bb, hq)
            assert np.all(got[len(want):] == -1) and np.all(np.isneginf(sc[bb, hq, len(want):]))


def test_topk_matches_oracle_ranking():
    d, b, B, H, G, T, k = 128, 3, 1, 2, 4, 2048, 50
    run, q, idx, sc, lg = _run(d, b, B, H, G, T, k, [T], seed=7)
    cache = run.cache_np()
    # each estimate is within the score bar of the oracle's, so the k-th best moves by at most
    # that much too: a slot can be misranked only within twice the bar of the k-th best
    tol = 2 * P.LOGIT_ATOL * math.sqrt(d)
    for h in range(H):
        tok = run.tokens(cache, 0, h, T)
        tk = dict(idx=tok["kidx"], n=tok["nk"].astype(np.float64), sigma=tok["sigma"],
                  gamma=tok["gamma"].astype(np.float64))
        for gh in range(G):
            hq = h * G + gh
            slots_o, est_o = odec.ip_topk(q[0, hq].double().numpy(), tk, run.p.Pi, run.p.S, run.p.cb_k, T)
            est = np.empty(T)
            est[slots_o] = est_o   # the oracle's estimate of every slot
            kth = np.sort(est)[::-1][k - 1]
            got = idx[0, hq]
            assert len(set(got.tolist())) == k
            assert np.all(est[got] >= kth - tol), hq
            must = np.nonzero(est > kth + tol)[0]
            assert set(must.tolist()) <= set(got.tolist()), hq
            assert np.all(np.abs(sc[0, hq] - est[got]) < tol / 2), hq


def test_topk_rejects_bad_arguments():
    run = P.Run(128, 3, 1, 1, 4, 256)
    q = torch.zeros(1, 4, 128, device="cuda")
    sl = torch.tensor([256], dtype=torch.int32, device="cuda")
    for k in (0, tq.binding.TQ_TOPK_MAX + 1):
        with pytest.raises(tq.TQError):
            run.ctx.ip_topk(q, run.cache, sl, 1, 256, k)
