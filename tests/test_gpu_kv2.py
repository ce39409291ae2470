"""GPU parity of format version 2: separate key and value widths, keys with or without the QJL
stage ([3BITS] "Python + HuggingFace": a cache built with key_bits and value_bits, a stage-1
quantizer alone returning indices and norms).  Every case goes through the C ABI
(tq_ctx_create_kv) and is checked against the oracle's version-2 functions: identical codes
and signs, the oracle's packer re-packing the GPU's pages to identical bytes, logits within
2e-3 of route A on the GPU's own pages, outputs within 2e-3 there and 1e-2 end to end."""
import numpy as np
import pytest
import torch

import kv_cache_vector_19_b300 as tq
from oracle import decode as odec
from oracle import pagefmt, params, quant

import parity as P

pytestmark = pytest.mark.gpu

# (d, key_bits, value_bits, qjl): K3V4, K4V2 without QJL, K2V3 with QJL and more shapes
FORMATS = [(128, 3, 4, True), (128, 4, 2, False), (128, 2, 3, True), (128, 1, 3, False), (64, 3, 3, False),
           (256, 2, 4, True), (128, 5, 5, False)]


def _ids(f):
    d, kb, vb, q = f
    return f"d{d}_K{kb}V{vb}{'_qjl' if q else ''}"


class Run2:
    def __init__(self, d, key_bits, value_bits, qjl, batch, kv_heads, q_heads, max_tokens, seed=0):
        self.d, self.batch, self.kv_heads, self.q_heads, self.max_tokens = d, batch, kv_heads, q_heads, max_tokens
        self.ctx = tq.Context(d, key_bits=key_bits, value_bits=value_bits, qjl=qjl, seed=seed)
        self.p = params.make_kv(d, key_bits, value_bits, qjl=qjl, seed=seed)
        self.kb, self.vb, self.m = self.p.kb, self.p.vb, self.p.m
        self.cache = self.ctx.alloc_cache(batch, kv_heads, max_tokens)
        self.ws = self.ctx.alloc_workspace(batch, q_heads, kv_heads, max_tokens)
        self.n_pages = (max_tokens + 127) // 128

    def quantize(self, k, v, start_pos):
        start = torch.as_tensor(start_pos, dtype=torch.int32, device="cuda")
        self.ctx.quantize_kv(k.cuda().contiguous(), v.cuda().contiguous(), start, self.cache, self.max_tokens)

    def tokens(self, cache_np, bb, h, n):
        return pagefmt.unpack_tokens_kv(self.d, self.kb, self.vb, self.m, cache_np, self.n_pages, bb, h, n,
                                        self.kv_heads)

    def oracle(self, X_k, X_v):
        p = self.p
        ok = quant.quantize_keys(X_k, p.Pi, p.S, p.cb_k) if self.m > 0 else quant.quantize_keys_mse(X_k, p.Pi, p.cb_k)
        ov = quant.quantize_values(X_v, p.Pi, p.cb_v)
        return ok, ov


def _inputs(batch, heads, n, d, seed):
    g = torch.Generator().manual_seed(seed)
    k = (torch.randn(batch, heads, n, d, generator=g) * 2.0).to(torch.bfloat16)
    v = torch.randn(batch, heads, n, d, generator=g).to(torch.bfloat16)
    return k, v


@pytest.mark.parametrize("fmt", FORMATS, ids=[_ids(f) for f in FORMATS])
def test_kv2_quantize_pages(fmt):
    d, kbits, vbits, qjl = fmt
    B, H, N, maxT = 2, 2, 300, 512
    run = Run2(d, kbits, vbits, qjl, B, H, 4 * H, maxT, seed=7)
    assert run.ctx.page_bytes == pagefmt.page_bytes_kv(d, run.kb, run.vb, run.m)
    run.cache.fill_(0xA5)
    k, v = _inputs(B, H, N, d, seed=d + 10 * kbits + vbits)
    starts = [0, 77]
    run.quantize(k, v, starts)
    assert run.ctx.device_status() == tq.TQ_OK
    torch.cuda.synchronize()
    cache = run.cache.cpu().numpy()
    blank = pagefmt.unpack_page_kv(d, run.kb, run.vb, run.m,
                                   np.full(pagefmt.page_bytes_kv(d, run.kb, run.vb, run.m), 0xA5, np.uint8))
    for bb in range(B):
        for h in range(H):
            s0 = starts[bb]
            allt = run.tokens(cache, bb, h, maxT)
            got = {key: (None if val is None else val[s0:s0 + N]) for key, val in allt.items()}
            ok, ov = run.oracle(P.to64(k[bb, h]), P.to64(v[bb, h]))
            assert np.array_equal(got["kidx"], ok["idx"])
            assert np.array_equal(got["vidx"], ov["idx"])
            assert np.max(np.abs(got["nk"] - ok["n64"]) / np.maximum(ok["n64"], 1e-30)) < 2e-6
            assert np.max(np.abs(got["nv"] - ov["n64"]) / np.maximum(ov["n64"], 1e-30)) < 2e-6
            if run.m > 0:
                assert np.array_equal(got["sigma"], ok["sigma"])
                assert np.max(np.abs(got["gamma"] - ok["gamma64"]) / np.maximum(ok["gamma64"], 1e-30)) < 1e-4
            else:
                assert got["sigma"] is None and got["gamma"] is None
            # slots outside [s0, s0 + N) keep their bytes
            for t in list(range(0, s0)) + list(range(s0 + N, maxT)):
                sl = t % 128
                for key in ("kidx", "vidx") + (("sigma",) if run.m > 0 else ()):
                    assert np.array_equal(allt[key][t], blank[key][sl]), (key, t)
            # a fully written page re-packs to identical bytes
            page = 1
            pb = pagefmt.page_bytes_kv(d, run.kb, run.vb, run.m)
            base = ((bb * H) + h) * run.n_pages * pb + page * pb
            pg = {key: (None if val is None else val[page * 128:(page + 1) * 128]) for key, val in allt.items()}
            again = pagefmt.pack_page_kv(d, run.kb, run.vb, run.m, pg["kidx"], pg["sigma"], pg["nk"], pg["gamma"],
                                         pg["vidx"], pg["nv"])
            assert np.array_equal(cache[base:base + pb], again)


@pytest.mark.parametrize("fmt", FORMATS, ids=[_ids(f) for f in FORMATS])
def test_kv2_decode(fmt):
    d, kbits, vbits, qjl = fmt
    B, H, G, maxT, N = 2, 2, 4, 700, 650
    run = Run2(d, kbits, vbits, qjl, B, H, G * H, maxT, seed=3)
    k, v = _inputs(B, H, N, d, seed=5 + d)
    run.quantize(k, v, [0, 0])
    seq = [N, 333]
    g = torch.Generator().manual_seed(11)
    q = torch.randn(B, G * H, d, generator=g)
    qd = q.cuda().contiguous()
    out = torch.empty_like(qd)
    lg = torch.full((B, G * H, maxT), float("nan"), device="cuda")
    sl = torch.as_tensor(seq, dtype=torch.int32, device="cuda")
    run.ctx.attn_decode(qd, run.cache, sl, H, maxT, out, run.ws, logits=lg)
    assert run.ctx.device_status() == tq.TQ_OK
    out, lg = out.cpu().numpy(), lg.cpu().numpy()
    cache = run.cache.cpu().numpy()
    p = run.p
    for bb in range(B):
        for h in range(H):
            tok = run.tokens(cache, bb, h, seq[bb])
            tk = dict(idx=tok["kidx"], n=tok["nk"].astype(np.float64), sigma=tok["sigma"],
                      gamma=None if tok["gamma"] is None else tok["gamma"].astype(np.float64))
            tv = dict(idx=tok["vidx"], n=tok["nv"].astype(np.float64))
            ok, ov = run.oracle(P.to64(k[bb, h, :seq[bb]]), P.to64(v[bb, h, :seq[bb]]))
            ek = dict(idx=ok["idx"], n=ok["n"].astype(np.float64), sigma=ok["sigma"],
                      gamma=None if ok["gamma"] is None else ok["gamma"].astype(np.float64))
            ev = dict(idx=ov["idx"], n=ov["n"].astype(np.float64))
            for gh in range(G):
                hq = h * G + gh
                qrow = q[bb, hq].double().numpy()
                o_pg, l_pg = odec.attend_route_a(qrow, tk, tv, p.Pi, p.S, p.cb_k, p.cb_v)
                assert np.max(np.abs(lg[bb, hq, :seq[bb]] - l_pg)) < P.LOGIT_ATOL, (bb, hq)
                assert P.rel_l2(out[bb, hq], o_pg) < P.OUT_ON_PAGES_REL_L2, (bb, hq)
                o_e2e, _ = odec.attend_route_a(qrow, ek, ev, p.Pi, p.S, p.cb_k, p.cb_v)
                assert P.rel_l2(out[bb, hq], o_e2e) < P.OUT_REL_L2, (bb, hq)


@pytest.mark.parametrize("fmt", [(128, 3, 4, True), (128, 4, 2, False)], ids=_ids)
def test_kv2_appends_match_bulk(fmt):
    d, kbits, vbits, qjl = fmt
    B, H, maxT = 2, 2, 300
    k, v = _inputs(B, H, 260, d, seed=99)
    bulk = Run2(d, kbits, vbits, qjl, B, H, 8, maxT)
    bulk.quantize(k, v, [0, 0])
    step = Run2(d, kbits, vbits, qjl, B, H, 8, maxT)
    step.quantize(k[:, :, :250].contiguous(), v[:, :, :250].contiguous(), [0, 0])
    for t in range(250, 260):
        step.quantize(k[:, :, t:t + 1].contiguous(), v[:, :, t:t + 1].contiguous(), [t, t])
    assert step.ctx.device_status() == tq.TQ_OK
    torch.cuda.synchronize()
    a, c = bulk.cache.cpu().numpy(), step.cache.cpu().numpy()
    for bb in range(B):
        for h in range(H):
            ta, tc = bulk.tokens(a, bb, h, 260), step.tokens(c, bb, h, 260)
            for key in ("kidx", "vidx", "sigma"):
                if ta[key] is not None:
                    assert np.array_equal(ta[key], tc[key]), key
            for key in ("nk", "nv", "gamma"):
                if ta[key] is not None:
                    assert np.allclose(ta[key], tc[key], rtol=1e-5, atol=1e-30), key


@pytest.mark.parametrize("fmt", [(128, 3, 4, True), (64, 3, 3, False)], ids=_ids)
def test_kv2_dequantize(fmt):
    d, kbits, vbits, qjl = fmt
    B, H, N = 1, 2, 200
    run = Run2(d, kbits, vbits, qjl, B, H, 2, N)
    k, v = _inputs(B, H, N, d, seed=1234)
    run.quantize(k, v, [0])
    zero = torch.zeros(B, dtype=torch.int32, device="cuda")
    khat = torch.empty(B, H, N, d, device="cuda")
    vhat = torch.empty(B, H, N, d, device="cuda")
    run.ctx.dequantize_kv(run.cache, zero, B, H, N, N, khat, vhat)
    assert run.ctx.device_status() == tq.TQ_OK
    cache = run.cache.cpu().numpy()
    p = run.p
    for h in range(H):
        tok = run.tokens(cache, 0, h, N)
        tk = dict(idx=tok["kidx"], n=tok["nk"].astype(np.float64), sigma=tok["sigma"],
                  gamma=None if tok["gamma"] is None else tok["gamma"].astype(np.float64))
        kref = quant.reconstruct_keys_any(tk, p.Pi, p.S, p.cb_k[0])
        vref = quant.reconstruct_values(tok["vidx"], tok["nv"].astype(np.float64), p.Pi, p.cb_v[0])
        kg, vg = khat[0, h].cpu().double().numpy(), vhat[0, h].cpu().double().numpy()
        assert np.max(np.abs(kg - kref)) / np.max(np.abs(kref)) < 2e-5
        assert np.max(np.abs(vg - vref)) / np.max(np.abs(vref)) < 2e-5


def test_kv2_rejects_and_routes():
    with pytest.raises(tq.TQError):
        tq.Context(128, key_bits=1, value_bits=3, qjl=True)   # no Lloyd-Max bit left for keys
    with pytest.raises(tq.TQError):
        tq.Context(96, key_bits=3, value_bits=3, qjl=False)
    c = tq.Context(128, key_bits=3, value_bits=4, qjl=False)
    with pytest.raises(tq.TQError):
        c.set_decode_path("tc4")                              # version 2 decodes on CUDA cores
    c.set_decode_path("simt")
    # qjl with equal widths is format version 1
    v1 = tq.Context(128, key_bits=3, value_bits=3, qjl=True)
    assert v1.page_bytes == pagefmt.page_bytes(128, 3, 128)
