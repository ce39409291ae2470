"""GPU tests of the paged (block-table) cache: tq_quantize_kv_paged, tq_attn_decode_paged and
tq_dequantize_kv_paged ([BLOG] 3.5, vLLM / PagedAttention; [3BITS] "vLLM").

The paged calls run the contiguous calls' kernels with another page address, so the tests
hold them to identity with the contiguous path on the same inputs, which the parity suites tie
to the oracle:
* after the same prefill and appends, the oracle's gather of the pool through its table equals
  the contiguous cache byte for byte, for every quantizer kernel (tensor-core prefill,
  few-token appends, CUDA cores at d = 64 / 256, format version 2) — including the bytes of
  slots no call wrote — and blocks outside the table keep their bytes;
* decode outputs and logits are bit-identical to the contiguous decode for every decode kernel
  (e2m1 and f8f6f4 tcgen05, mma.sync, CUDA cores, format version 2), and within the bars of
  the oracle's route A on the gathered pages;
* dequantized vectors and the scan's top-k are bit-identical;
* a block id outside the pool is clamped and reported as TQ_EBOUNDS; bad table arguments are
  rejected on the host.
"""
import math

import numpy as np
import pytest
import torch

import kv_cache_vector_19_b300 as tq
from oracle import decode as odec
from oracle import pagefmt, params

pytestmark = pytest.mark.gpu


class Pair:
    """The same context with a contiguous cache and a paged pool that starts as its image."""

    def __init__(self, d, B, H, max_blocks, bits=None, kv=None, extra=3, seed=0, path="auto"):
        if kv is not None:
            self.ctx = tq.Context(d, key_bits=kv[0], value_bits=kv[1], qjl=kv[2], seed=seed, decode_path=path)
        else:
            self.ctx = tq.Context(d, bits, seed=seed, decode_path=path)
        self.d, self.B, self.H, self.max_blocks = d, B, H, max_blocks
        self.T = 128 * max_blocks
        self.n_blocks = B * max_blocks + extra
        rng = np.random.default_rng(seed + 11)
        perm = rng.permutation(self.n_blocks)
        self.table_np = perm[:B * max_blocks].reshape(B, max_blocks).astype(np.int32)
        self.spare = perm[B * max_blocks:]
        self.pb = tq.lib().tq_page_bytes(self.ctx._ctx)
        pool0 = rng.integers(0, 256, self.n_blocks * H * self.pb, dtype=np.uint8)
        self.pool0 = pool0
        self.pool = torch.from_numpy(pool0.copy()).cuda()
        cache0 = pagefmt.gather_paged(pool0, self.table_np, B, H, self.pb, max_blocks)
        self.cache = torch.from_numpy(cache0).cuda()
        self.table = torch.from_numpy(self.table_np).cuda()

    def quantize(self, k, v, start):
        st = torch.as_tensor(start, dtype=torch.int32, device="cuda")
        k, v = k.cuda().contiguous(), v.cuda().contiguous()
        self.ctx.quantize_kv(k, v, st, self.cache, self.T)
        self.ctx.quantize_kv_paged(k, v, st, self.pool, self.n_blocks, self.table)

    def gathered(self):
        torch.cuda.synchronize()
        return pagefmt.gather_paged(self.pool.cpu().numpy(), self.table_np, self.B, self.H, self.pb,
                                    self.max_blocks)

    def status(self):
        return self.ctx.device_status()


def _kv(B, H, N, d, seed):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(B, H, N, d, generator=g).to(torch.bfloat16),
            torch.randn(B, H, N, d, generator=g).to(torch.bfloat16))


QUANT_CASES = [
    dict(d=128, bits=3),                      # tensor-core prefill + few-token appends
    dict(d=128, bits=4),
    dict(d=64, bits=3),                       # CUDA cores
    dict(d=256, bits=2),
    dict(d=128, kv=(3, 4, True)),             # format version 2
    dict(d=64, kv=(4, 2, False)),
]


@pytest.mark.parametrize("case", QUANT_CASES, ids=lambda c: f"d{c['d']}_{c.get('bits') or c.get('kv')}")
def test_paged_quantize_equals_contiguous(case):
    d, B, H, max_blocks = case["d"], 2, 2, 5
    pr = Pair(d, B, H, max_blocks, bits=case.get("bits"), kv=case.get("kv"))
    k, v = _kv(B, H, 300, d, 1)
    pr.quantize(k, v, [0, 40])                 # prefill, ragged start: partial first and last pages
    for i, n in enumerate((1, 3, 8)):          # appends
        ka, va = _kv(B, H, n, d, 10 + i)
        pos = [300 + 12 * i, 340 + 12 * i]
        pr.quantize(ka, va, pos)
    assert pr.status() == tq.TQ_OK
    got = pr.gathered()
    want = pr.cache.cpu().numpy()
    assert np.array_equal(got, want)
    pool = pr.pool.cpu().numpy()
    for blk in pr.spare:   # blocks outside the table are untouched
        lo = pagefmt.paged_page_offset(int(blk), 0, H, pr.pb)
        assert np.array_equal(pool[lo:lo + H * pr.pb], pr.pool0[lo:lo + H * pr.pb])


DECODE_CASES = [
    dict(d=128, bits=3, G=4, path="auto"),     # e2m1 tcgen05
    dict(d=128, bits=3, G=8, path="auto"),     # e2m1 tcgen05, four token-warp sets
    dict(d=128, bits=2, G=16, path="auto"),    # f8f6f4 tcgen05
    dict(d=128, bits=4, G=4, path="auto"),     # e2m1 tcgen05, two virtual KV heads per KV head
    dict(d=128, bits=4, G=4, path="mma"),      # mma.sync
    dict(d=64, bits=3, G=2, path="auto"),
    dict(d=256, bits=3, G=4, path="simt"),     # CUDA cores
    dict(d=128, kv=(3, 4, True), G=4, path="auto"),   # format version 2
]


@pytest.mark.parametrize("case", DECODE_CASES,
                         ids=lambda c: f"d{c['d']}_{c.get('bits') or c.get('kv')}_G{c['G']}_{c['path']}")
def test_paged_decode_equals_contiguous(case):
    d, B, H, max_blocks, G = case["d"], 2, 2, 6, case["G"]
    pr = Pair(d, B, H, max_blocks, bits=case.get("bits"), kv=case.get("kv"), path=case["path"])
    T = pr.T
    k, v = _kv(B, H, T, d, 2)
    pr.quantize(k, v, [0, 0])
    Hq = G * H
    q = torch.randn(B, Hq, d, generator=torch.Generator().manual_seed(3)).cuda()
    sl = torch.tensor([T - 61, 300], dtype=torch.int32, device="cuda")
    ws = pr.ctx.alloc_workspace(B, Hq, H, T)
    out_c, out_p = torch.empty_like(q), torch.empty_like(q)
    lg_c = torch.full((B, Hq, T), float("nan"), device="cuda")
    lg_p = torch.full((B, Hq, T), float("nan"), device="cuda")
    pr.ctx.attn_decode(q, pr.cache, sl, H, T, out_c, ws, logits=lg_c)
    pr.ctx.attn_decode_paged(q, pr.pool, pr.n_blocks, pr.table, sl, H, out_p, ws, logits=lg_p)
    assert pr.status() == tq.TQ_OK
    assert torch.equal(out_c, out_p)
    assert torch.equal(torch.nan_to_num(lg_c, nan=7.0), torch.nan_to_num(lg_p, nan=7.0))


def test_paged_decode_matches_oracle_on_gathered_pages():
    d, b, B, H, G, max_blocks = 128, 3, 1, 2, 4, 4
    pr = Pair(d, B, H, max_blocks, bits=b, seed=5)
    T = pr.T
    k, v = _kv(B, H, T, d, 4)
    pr.quantize(k, v, [0])
    q = torch.randn(B, G * H, d, generator=torch.Generator().manual_seed(6))
    n = T - 17
    sl = torch.tensor([n], dtype=torch.int32, device="cuda")
    ws = pr.ctx.alloc_workspace(B, G * H, H, T)
    out = torch.empty(B, G * H, d, device="cuda")
    lg = torch.full((B, G * H, T), float("nan"), device="cuda")
    pr.ctx.attn_decode_paged(q.cuda(), pr.pool, pr.n_blocks, pr.table, sl, H, out, ws, logits=lg)
    assert pr.status() == tq.TQ_OK
    cache = pr.gathered()
    p = params.make(d, b, seed=5)
    out, lg = out.cpu().numpy(), lg.cpu().numpy()
    for h in range(H):
        tok = pagefmt.unpack_tokens(d, b, d, cache, max_blocks, 0, h, n, H)
        tk = dict(idx=tok["kidx"], n=tok["nk"].astype(np.float64), sigma=tok["sigma"],
                  gamma=tok["gamma"].astype(np.float64))
        tv = dict(idx=tok["vidx"], n=tok["nv"].astype(np.float64))
        for gh in range(G):
            hq = h * G + gh
            o, lo = odec.attend_route_a(q[0, hq].double().numpy(), tk, tv, p.Pi, p.S, p.cb_k, p.cb_v)
            assert np.max(np.abs(lg[0, hq, :n] - lo)) < 2e-3
            assert np.linalg.norm(out[0, hq] - o) <= 2e-3 * np.linalg.norm(o)


def test_paged_dequantize_equals_contiguous():
    d, B, H, max_blocks = 128, 2, 2, 3
    pr = Pair(d, B, H, max_blocks, bits=3)
    k, v = _kv(B, H, 200, d, 8)
    pr.quantize(k, v, [10, 100])
    st = torch.tensor([10, 100], dtype=torch.int32, device="cuda")
    kc, vc = (torch.empty(B, H, 200, d, device="cuda") for _ in range(2))
    kp, vp = (torch.empty(B, H, 200, d, device="cuda") for _ in range(2))
    pr.ctx.dequantize_kv(pr.cache, st, B, H, 200, pr.T, k_out=kc, v_out=vc)
    pr.ctx.dequantize_kv_paged(pr.pool, pr.n_blocks, pr.table, st, B, H, 200, k_out=kp, v_out=vp)
    assert pr.status() == tq.TQ_OK
    assert torch.equal(kc, kp) and torch.equal(vc, vp)


def test_paged_scan_equals_contiguous():
    d, B, H, G, max_blocks = 128, 2, 2, 4, 4
    pr = Pair(d, B, H, max_blocks, bits=3, seed=4)
    k, v = _kv(B, H, pr.T, d, 12)
    pr.quantize(k, v, [0, 0])
    q = torch.randn(B, G * H, d, generator=torch.Generator().manual_seed(13)).cuda()
    sl = torch.tensor([pr.T - 5, 200], dtype=torch.int32, device="cuda")
    ic, sc = pr.ctx.ip_topk(q, pr.cache, sl, H, pr.T, 64)
    ip, sp = pr.ctx.ip_topk_paged(q, pr.pool, pr.n_blocks, pr.table, sl, H, 64)
    assert pr.status() == tq.TQ_OK
    assert torch.equal(ic, ip) and torch.equal(sc, sp)


def test_block_id_outside_the_pool_is_clamped_and_reported():
    d, B, H, max_blocks = 128, 1, 1, 2
    pr = Pair(d, B, H, max_blocks, bits=3, extra=0)
    bad = pr.table.clone()
    bad[0, 1] = pr.n_blocks + 5          # clamped to the last block
    k, v = _kv(B, H, 200, d, 9)
    st = torch.zeros(B, dtype=torch.int32, device="cuda")
    pr.ctx.quantize_kv_paged(k.cuda(), v.cuda(), st, pr.pool, pr.n_blocks, bad)
    assert pr.status() == tq.TQ_EBOUNDS
    bad[0, 1] = -1                       # clamped to block 0
    q = torch.randn(B, 4, d, device="cuda")
    ws = pr.ctx.alloc_workspace(B, 4, H, pr.T)
    out = torch.empty_like(q)
    sl = torch.tensor([200], dtype=torch.int32, device="cuda")
    pr.ctx.attn_decode_paged(q, pr.pool, pr.n_blocks, bad, sl, H, out, ws)
    assert pr.status() == tq.TQ_EBOUNDS
    assert pr.status() == tq.TQ_OK       # the flag is cleared by the read


def test_paged_rejects_bad_table_arguments():
    d, B, H = 128, 1, 1
    pr = Pair(d, B, H, 2, bits=3)
    k, v = _kv(B, H, 16, d, 3)
    st = torch.zeros(B, dtype=torch.int32, device="cuda")
    lib = tq.lib()
    kd, vd = k.cuda(), v.cuda()
    for n_blocks, table, max_blocks in ((0, pr.table, 2), (pr.n_blocks, None, 2), (pr.n_blocks, pr.table, 0)):
        tp = table.data_ptr() if table is not None else None
        rc = lib.tq_quantize_kv_paged(pr.ctx._ctx, kd.data_ptr(), vd.data_ptr(), B, H, 16,
                                      st.data_ptr(), pr.pool.data_ptr(), n_blocks, tp, max_blocks, None)
        assert rc == tq.TQ_EINVAL
    assert math.isclose(lib.tq_paged_pool_bytes(pr.ctx._ctx, H, pr.n_blocks), pr.pool.numel())
