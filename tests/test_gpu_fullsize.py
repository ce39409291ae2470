"""Full-size workloads in the configuration the benchmark runs (same seeded inputs, same
automatic kernel choice and launch plan), checked on sampled (batch, KV head) sequences that
the oracle recomputes in full: every logit of their query heads, their outputs, and the
quantizer's code / sign mismatch rate over the whole sequence.

  longctx   batch 4, 8 KV / 32 query heads, 131,072 tokens + one appended token, b=3
  llama8b   batch 1, 8 KV / 32 query heads, 32,768 tokens, b=4, log-normal channels
  llama70b  batch 16, 8 KV / 64 query heads, 32,768 tokens, b=3, K outlier tokens
"""
import numpy as np
import pytest
import torch

import kv_cache_vector_19_b300 as tq
from kv_cache_vector_19_b300 import workloads

import parity as P

pytestmark = pytest.mark.gpu

CASES = [("longctx", [(0, 3), (3, 7)]), ("llama8b", [(0, 0), (0, 5)]), ("llama70b", [(0, 2), (15, 7)])]


@pytest.mark.parametrize("name,sampled", CASES, ids=[c[0] for c in CASES])
def test_full_size_sampled(name, sampled):
    w = workloads.preset(name)
    data = workloads.generate(w)
    run = P.Run(w.d, w.b, w.batch, w.kv_heads, w.q_heads, w.max_tokens, seed=w.seed)
    run.quantize(data["k"], data["v"], [0] * w.batch)
    seq_len = w.tokens
    if w.decode_steps > 1:            # the first decode step's appended token, as the bench does
        run.quantize(data["k_new"][0], data["v_new"][0], [w.tokens] * w.batch)
        seq_len += 1
    q = data["q"][0]
    out, lg = run.decode(q, [seq_len] * w.batch, logits=True)
    assert run.status() == tq.TQ_OK
    out = out.cpu().numpy()
    assert np.all(np.isfinite(out))
    cache = run.cache_np()
    G = w.group
    for i, (bb, h) in enumerate(sampled):
        tok = run.tokens(cache, bb, h, seq_len)
        lg_rows = lg[bb, h * G:(h + 1) * G, :seq_len].cpu().numpy()
        for j, hq in enumerate(range(h * G, (h + 1) * G)):
            qrow = q[bb, hq].double().numpy()
            o_pages, l_pages = P.oracle_logits_on_pages(run, qrow, tok)
            assert np.max(np.abs(lg_rows[j] - l_pages)) < P.LOGIT_ATOL, (name, bb, hq)
            assert P.rel_l2(out[bb, hq], o_pages) < P.OUT_ON_PAGES_REL_L2, (name, bb, hq)
        if i == 0:
            # the quantizer over the whole sequence, and quantize + decode end to end
            xk = P.to64(data["k"][bb, h])
            xv = P.to64(data["v"][bb, h])
            if seq_len > w.tokens:
                xk = np.concatenate([xk, P.to64(data["k_new"][0, bb, h])])
                xv = np.concatenate([xv, P.to64(data["v_new"][0, bb, h])])
            res = P.compare_sequence(run, xk, xv, tok)
            P.assert_quantize_ok(res)
            hq = h * G
            o_e2e, _ = P.oracle_end_to_end(run, q[bb, hq].double().numpy(), res["oracle_k"], res["oracle_v"])
            assert P.rel_l2(out[bb, hq], o_e2e) < P.OUT_REL_L2, name
