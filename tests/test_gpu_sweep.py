"""The bit/dim sweep at its own size, checked against the oracle point by point: b in
{2, 3, 4, 5}, head_dim in {64, 128, 256}, m = head_dim, one KV head, 65,536 tokens of N(0,1),
16 queries (as 16 query heads of the KV head, the benchmark's sweep configuration).

For every point the oracle recomputes, from the same seeded inputs:
  * the quantizer over all 65,536 tokens: code and sign mismatch rate and its boundary rule;
  * every logit of the 16 queries against route A on the GPU's own pages;
  * every output against route A on the GPU's pages and against its own quantize + decode.
"""
import numpy as np
import pytest
import torch

import kv_cache_vector_19_b300 as tq
from kv_cache_vector_19_b300 import workloads

import parity as P

pytestmark = pytest.mark.gpu

POINTS = [(d, b) for d in (64, 128, 256) for b in (2, 3, 4, 5)]


@pytest.mark.parametrize("d,b", POINTS, ids=[f"d{d}_b{b}" for d, b in POINTS])
def test_sweep_point_full_size(d, b):
    w = workloads.sweep_point(d, b)
    data = workloads.generate(w)
    T, nq = w.tokens, w.extra["n_queries"]
    run = P.Run(d, b, 1, 1, nq, T, seed=w.seed)
    run.quantize(data["k"], data["v"], [0])
    q = data["q"][0].reshape(1, nq, d)
    out, lg = run.decode(q, [T], logits=True)
    assert run.status() == tq.TQ_OK
    out, lg = out.cpu().numpy(), lg.cpu().numpy()
    assert np.all(np.isfinite(out))
    cache = run.cache_np()
    tok = run.tokens(cache, 0, 0, T)
    res = P.compare_sequence(run, P.to64(data["k"][0, 0]), P.to64(data["v"][0, 0]), tok)
    P.assert_quantize_ok(res)
    for h in range(nq):
        qrow = q[0, h].double().numpy()
        o_pages, l_pages = P.oracle_logits_on_pages(run, qrow, tok)
        assert np.max(np.abs(lg[0, h, :T] - l_pages)) < P.LOGIT_ATOL, (d, b, h)
        assert P.rel_l2(out[0, h], o_pages) < P.OUT_ON_PAGES_REL_L2, (d, b, h)
        o_e2e, _ = P.oracle_end_to_end(run, qrow, res["oracle_k"], res["oracle_v"])
        assert P.rel_l2(out[0, h], o_e2e) < P.OUT_REL_L2, (d, b, h)
