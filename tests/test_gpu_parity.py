"""GPU parity of tq_quantize_kv and tq_attn_decode against the fp64 oracle, at sizes the
oracle finishes in seconds (several pages, ragged tails, unaligned start slots) and on
every (d, b) the library supports.  All calls go through the C ABI."""
import numpy as np
import pytest
import torch

import kv_cache_vector_19_b300 as tq
from kv_cache_vector_19_b300 import workloads
from oracle import pagefmt

import parity as P

pytestmark = pytest.mark.gpu

ALL_DB = [(d, b) for d in (64, 128, 256) for b in (2, 3, 4, 5)]


def _inputs(batch, heads, n, d, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    k = (torch.randn(batch, heads, n, d, generator=g) * scale).to(torch.bfloat16)
    v = torch.randn(batch, heads, n, d, generator=g).to(torch.bfloat16)
    return k, v


@pytest.mark.parametrize("d,b", ALL_DB)
def test_quantize_small_all_formats(d, b):
    B, H, N, maxT = 2, 2, 300, 512
    run = P.Run(d, b, B, H, 4 * H, maxT)
    run.cache.fill_(0xA5)
    k, v = _inputs(B, H, N, d, seed=d * 10 + b, scale=2.0)
    starts = [0, 77]
    run.quantize(k, v, starts)
    assert run.status() == tq.TQ_OK
    cache = run.cache_np()
    blank = pagefmt.unpack_page(d, b, d, np.full(pagefmt.page_bytes(d, b, d), 0xA5, np.uint8))
    for bb in range(B):
        for h in range(H):
            s0 = starts[bb]
            got_all = run.tokens(cache, bb, h, maxT)
            got = {key: val[s0:s0 + N] for key, val in got_all.items()}
            res = P.compare_sequence(run, P.to64(k[bb, h]), P.to64(v[bb, h]), got)
            P.assert_quantize_ok(res)
            # slots outside [s0, s0 + N) keep their previous bytes, bit for bit
            for t in list(range(0, s0)) + list(range(s0 + N, maxT)):
                sl = t % 128
                for key in ("kidx", "sigma", "vidx"):
                    assert np.array_equal(got_all[key][t], blank[key][sl]), (key, t)
                for key in ("nk", "gamma", "nv"):
                    assert got_all[key][t].view(np.uint32) == blank[key][sl].view(np.uint32)
            # a fully written page re-packs to identical bytes
            page = 1
            pg = {key: val[page * 128:(page + 1) * 128] for key, val in got_all.items()}
            assert P.repack_matches(run, cache, bb, h, page, pg)


def _check_decode(d, b, G, path="auto"):
    B, H, maxT = 2, 2, 700
    N = 650
    run = P.Run(d, b, B, H, G * H, maxT, decode_path=path)
    k, v = _inputs(B, H, N, d, seed=100 + d + b, scale=1.5)
    run.quantize(k, v, [0, 0])
    q = torch.randn(B, G * H, d, generator=torch.Generator().manual_seed(7))
    seq_lens = [N, 257]
    out, lg = run.decode(q, seq_lens, logits=True)
    assert run.status() == tq.TQ_OK
    out, lg = out.cpu().numpy(), lg.cpu().numpy()
    cache = run.cache_np()
    for bb in range(B):
        for h in range(H):
            T = seq_lens[bb]
            tok = run.tokens(cache, bb, h, T)
            res = P.compare_sequence(run, P.to64(k[bb, h, :T]), P.to64(v[bb, h, :T]), tok)
            for hq in range(h * G, (h + 1) * G):
                qrow = q[bb, hq].double().numpy()
                o_pages, l_pages = P.oracle_logits_on_pages(run, qrow, tok)
                assert np.max(np.abs(lg[bb, hq, :T] - l_pages)) < P.LOGIT_ATOL
                assert P.rel_l2(out[bb, hq], o_pages) < P.OUT_ON_PAGES_REL_L2
                o_e2e, _ = P.oracle_end_to_end(run, qrow, res["oracle_k"], res["oracle_v"])
                assert P.rel_l2(out[bb, hq], o_e2e) < P.OUT_REL_L2


@pytest.mark.parametrize("d,b,G", [(64, 2, 1), (128, 3, 4), (128, 4, 8), (256, 5, 16), (256, 3, 2),
                                   (64, 5, 16), (128, 2, 3), (64, 3, 4), (64, 4, 4), (256, 2, 4)])
def test_decode_small(d, b, G):
    _check_decode(d, b, G)


# every decode kernel on its own, whatever the automatic choice would be
@pytest.mark.parametrize("path,d,b,G", [
    ("simt", 64, 2, 1), ("simt", 128, 3, 4), ("simt", 256, 5, 16),
    ("mma", 64, 2, 1), ("mma", 128, 3, 4), ("mma", 128, 4, 8), ("mma", 128, 3, 16), ("mma", 128, 2, 3),
    ("mma", 128, 5, 2), ("mma", 256, 4, 1),
    ("tc", 128, 3, 4), ("tc", 128, 3, 8), ("tc", 128, 3, 16), ("tc", 128, 2, 3), ("tc", 128, 2, 16),
    ("tc", 128, 3, 1), ("tc", 128, 3, 2), ("tc", 128, 3, 6), ("tc", 128, 2, 12),
    ("tc4", 128, 3, 4), ("tc4", 128, 3, 8), ("tc4", 128, 2, 3), ("tc4", 128, 3, 1), ("tc4", 128, 3, 2),
    ("tc4", 128, 2, 8), ("tc4", 128, 3, 6), ("tc4", 128, 2, 5),
    # 4-bit codes: two query heads per pass, a KV head of 4 or 8 as 2 or 4 virtual ones
    ("tc4", 128, 4, 1), ("tc4", 128, 4, 2), ("tc4", 128, 4, 4), ("tc4", 128, 4, 8),
    # 16 query heads per KV head: four virtual KV heads of four
    ("tc4", 128, 3, 16), ("tc4", 128, 2, 16)])
def test_decode_small_each_kernel(path, d, b, G):
    _check_decode(d, b, G, path)


def test_decode_path_selection():
    ctx = tq.Context(64, 4)
    with pytest.raises(tq.TQError) as e:
        ctx.set_decode_path("tc")          # head dim 64 has no tcgen05 kernel
    assert e.value.status == tq.TQ_EUNSUPPORTED
    assert tq.lib().tq_ctx_set_decode_path(ctx.handle, 7) == tq.TQ_EINVAL
    for path in ("simt", "mma", "auto"):
        ctx.set_decode_path(path)
        assert ctx.workspace_bytes(2, 8, 2, 700) > 0


@pytest.mark.parametrize("path,d,b", [("tc4", 128, 3), ("tc4", 128, 4), ("tc", 128, 3), ("mma", 128, 3),
                                      ("simt", 128, 3), ("auto", 64, 3), ("auto", 256, 2)])
def test_decode_long_sequences_each_kernel(path, d, b):
    """Sequences of ~120 pages, so that every CTA of the bit-plane kernels streams far more
    pages than its shared-memory ring holds (ring refills, many segments), checked on two
    heads against the oracle on the GPU's own pages."""
    G, B, H, maxT = 4, 2, 8, 15360
    run = P.Run(d, b, B, H, G * H, maxT, decode_path=path)
    gen = torch.Generator().manual_seed(11)
    for bb in range(B):   # quantize one sequence at a time to keep host memory small
        k = (torch.randn(1, H, maxT, d, generator=gen) * 1.3).to(torch.bfloat16)
        v = torch.randn(1, H, maxT, d, generator=gen).to(torch.bfloat16)
        run.ctx.quantize_kv(k.cuda(), v.cuda(), torch.zeros(1, dtype=torch.int32, device="cuda"),
                            run.cache[bb * H * run.n_pages * run.ctx.page_bytes:], maxT)
    q = torch.randn(B, G * H, d, generator=gen)
    seq_lens = [maxT, 14001]
    out, lg = run.decode(q, seq_lens, logits=True)
    assert run.status() == tq.TQ_OK
    out, lg = out.cpu().numpy(), lg.cpu().numpy()
    cache = run.cache_np()
    for bb, h in [(0, 3), (1, 7)]:
        T = seq_lens[bb]
        tok = run.tokens(cache, bb, h, T)
        for hq in (h * G, h * G + G - 1):
            o_pages, l_pages = P.oracle_logits_on_pages(run, q[bb, hq].double().numpy(), tok)
            assert np.max(np.abs(lg[bb, hq, :T] - l_pages)) < P.LOGIT_ATOL
            assert P.rel_l2(out[bb, hq], o_pages) < P.OUT_ON_PAGES_REL_L2
    assert np.all(np.isfinite(out))


def test_append_one_token_at_a_time_matches_bulk():
    """Appends (one token per call: the few-token kernel) against one bulk call (the page-tile
    kernel): the slots written before the appends are untouched, and the appended tokens meet
    the same oracle bars as bulk-quantized ones (codes may differ only at a boundary)."""
    d, b, B, H, maxT = 128, 3, 2, 2, 300
    k, v = _inputs(B, H, 260, d, seed=5)
    bulk = P.Run(d, b, B, H, 8, maxT)
    bulk.quantize(k, v, [0, 0])
    step = P.Run(d, b, B, H, 8, maxT)
    step.quantize(k[:, :, :250].contiguous(), v[:, :, :250].contiguous(), [0, 0])
    for t in range(250, 260):
        step.quantize(k[:, :, t:t + 1].contiguous(), v[:, :, t:t + 1].contiguous(), [t, t])
    assert step.status() == tq.TQ_OK
    a, c = bulk.cache_np(), step.cache_np()
    for bb in range(B):
        for h in range(H):
            ta, tc = bulk.tokens(a, bb, h, 260), step.tokens(c, bb, h, 260)
            for key in ta:
                assert np.array_equal(ta[key][:250], tc[key][:250]), key
            sl = slice(250, 260)
            got = {key: val[sl] for key, val in tc.items()}
            res = P.compare_sequence(step, P.to64(k[bb, h, sl]), P.to64(v[bb, h, sl]), got)
            P.assert_quantize_ok(res)
            for key in ("kidx", "vidx", "sigma"):   # exact decisions on both paths
                assert np.array_equal(tc[key][sl], ta[key][sl]), key
            for key in ("nk", "nv", "gamma"):
                assert np.allclose(tc[key][sl], ta[key][sl], rtol=1e-5, atol=1e-30), key


def test_few_token_appends_every_format():
    """The few-token kernel at every (d, b): appends of 1..8 tokens at unaligned slots."""
    for d, b in ALL_DB:
        run = P.Run(d, b, 1, 2, 2, 400)
        k, v = _inputs(1, 2, 140, d, seed=30 + d + b)
        run.quantize(k[:, :, :100].contiguous(), v[:, :, :100].contiguous(), [0])
        t = 100
        for n in (1, 3, 8, 5, 2, 1, 8, 8, 4):
            run.quantize(k[:, :, t:t + n].contiguous(), v[:, :, t:t + n].contiguous(), [t])
            t += n
        assert run.status() == tq.TQ_OK
        cache = run.cache_np()
        for h in range(2):
            tok = run.tokens(cache, 0, h, 140)
            res = P.compare_sequence(run, P.to64(k[0, h]), P.to64(v[0, h]), tok)
            P.assert_quantize_ok(res)


def test_zero_vectors_and_tiny_sequences():
    d, b = 128, 3
    run = P.Run(d, b, 3, 1, 4, 256)
    k = torch.zeros(3, 1, 5, d, dtype=torch.bfloat16)
    v = torch.zeros(3, 1, 5, d, dtype=torch.bfloat16)
    k[1, 0, 2] = 1.0
    run.quantize(k, v, [0, 0, 0])
    cache = run.cache_np()
    tok = run.tokens(cache, 0, 0, 5)
    assert np.all(tok["kidx"] == 2) and np.all(tok["vidx"] == 4) and np.all(tok["sigma"] == 1)
    assert np.all(tok["nk"] == 0) and np.all(tok["gamma"] == 0) and np.all(tok["nv"] == 0)
    q = torch.randn(3, 4, d)
    out, lg = run.decode(q, [0, 1, 5], logits=True)
    assert run.status() == tq.TQ_OK
    out = out.cpu().numpy()
    assert np.all(out[0] == 0)                        # empty sequence -> zero rows
    assert np.all(np.isfinite(out))
    assert np.all(np.isnan(lg.cpu().numpy()[0]))       # no logit written for seq_len 0
    tok1 = run.tokens(cache, 1, 0, 1)
    for hq in range(4):
        o_ref, _ = P.oracle_logits_on_pages(run, q[1, hq].double().numpy(), tok1)
        assert P.rel_l2(out[1, hq], o_ref) < P.OUT_ON_PAGES_REL_L2


def test_device_bounds_are_reported_not_faulted():
    d, b = 64, 3
    run = P.Run(d, b, 2, 1, 2, 256)
    run.cache.fill_(0)
    k, v = _inputs(2, 1, 10, d, seed=9)
    run.quantize(k, v, [250, 3])                 # sequence 0 would overrun: skipped
    assert run.status() == tq.TQ_EBOUNDS
    assert run.status() == tq.TQ_OK              # the flag is cleared by reading it
    cache = run.cache_np()
    pb = pagefmt.page_bytes(d, b, d)
    assert not cache[:2 * pb].any()              # sequence 0 untouched
    assert cache[2 * pb:].any()                  # sequence 1 written
    q = torch.randn(2, 2, d)
    out, _ = run.decode(q, [300, 13])            # 300 > max_tokens: clamped and reported
    assert run.status() == tq.TQ_EBOUNDS
    assert torch.isfinite(out).all()


def test_host_rejects_bad_arguments():
    run = P.Run(128, 3, 1, 2, 8, 256)
    k, v = _inputs(1, 2, 4, 128, seed=1)
    kd, vd = k.cuda(), v.cuda()
    start = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(tq.TQError) as e:
        run.ctx.quantize_kv(kd, vd, start, run.cache[1:], 256)      # misaligned cache
    assert e.value.status == tq.TQ_EINVAL
    q = torch.randn(1, 6, 128, device="cuda")
    with pytest.raises(tq.TQError) as e:                               # 6 % 2 == 0 but
        run.ctx.attn_decode(q, run.cache, start, 4, 256, torch.empty_like(q), run.ws)   # 6 % 4 != 0
    assert e.value.status == tq.TQ_EINVAL
    q = torch.randn(1, 34, 128, device="cuda")
    with pytest.raises(tq.TQError) as e:                               # group of 17 > 16
        run.ctx.attn_decode(q, run.cache, start, 2, 256, torch.empty_like(q), run.ws)
    assert e.value.status == tq.TQ_EUNSUPPORTED
    with pytest.raises(tq.TQError) as e:                               # workspace too small
        run.ctx.attn_decode(q[:, :8], run.cache, start, 2, 256, torch.empty(1, 8, 128, device="cuda"),
                            run.ws[:256])
    assert e.value.status == tq.TQ_ENOMEM
    # n_tokens == 0 is a no-op
    run.ctx.quantize_kv(kd[:, :, :0], vd[:, :, :0], start, run.cache, 256)
    assert run.status() == tq.TQ_OK


def test_tiny_workload_full():
    """Tiny single head: d=128, 4096 keys and values with 4 outlier channels x20, b=3,
    16 fp32 queries, seed 0 - every output compared."""
    w = workloads.preset("tiny")
    data = workloads.generate(w)
    run = P.Run(w.d, w.b, w.batch, w.kv_heads, w.q_heads, w.max_tokens, seed=w.seed)
    run.quantize(data["k"], data["v"], [0])
    q = data["q"][0]
    out, lg = run.decode(q, [w.tokens], logits=True)
    assert run.status() == tq.TQ_OK
    out, lg = out.cpu().numpy(), lg.cpu().numpy()
    cache = run.cache_np()
    tok = run.tokens(cache, 0, 0, w.tokens)
    res = P.compare_sequence(run, P.to64(data["k"][0, 0]), P.to64(data["v"][0, 0]), tok)
    P.assert_quantize_ok(res)
    for hq in range(w.q_heads):
        qrow = q[0, hq].double().numpy()
        o_pages, l_pages = P.oracle_logits_on_pages(run, qrow, tok)
        assert np.max(np.abs(lg[0, hq] - l_pages)) < P.LOGIT_ATOL
        o_e2e, _ = P.oracle_end_to_end(run, qrow, res["oracle_k"], res["oracle_v"])
        assert P.rel_l2(out[0, hq], o_e2e) < P.OUT_REL_L2


def test_bounded_wait_times_out_and_reports():
    """A device-side wait that can never complete gives up after its limit: the kernel
    returns, the sticky status reads TQ_ETIMEOUT once, and the context stays usable."""
    import time
    run = P.Run(128, 3, 1, 1, 4, 256)
    t0 = time.time()
    assert tq.lib().tq_selftest_bounded_wait(run.ctx.handle, binding_stream()) == tq.TQ_OK
    assert run.status() == tq.TQ_ETIMEOUT
    assert time.time() - t0 < 30
    assert run.status() == tq.TQ_OK            # the flag is cleared by the read
    k, v = _inputs(1, 1, 20, 128, seed=1)
    run.quantize(k, v, [0])                    # the context still works
    out, _ = run.decode(torch.randn(1, 4, 128), [20])
    assert run.status() == tq.TQ_OK and torch.isfinite(out).all()


def binding_stream():
    from kv_cache_vector_19_b300 import binding
    return binding._stream_handle(None)
