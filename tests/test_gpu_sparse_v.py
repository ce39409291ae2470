"""GPU tests of Sparse V (tq_ctx_set_sparse_v; [3BITS] llama.cpp section: positions with low
attention weights are skipped during decoding).

The kernels apply the rule with their running maximum, which never exceeds the true one, so
they keep every position the oracle's rule (oracle.decode.attend_sparse_v, true maximum)
keeps and possibly more.  Each decode kernel is therefore held, on the GPU's own pages, to
  |out - oracle_sparse| <= skipped + 2e-3 |oracle_sparse|,
  |out - out_dense|     <= skipped (1 + 1e-3) + 2e-3 |out_dense|,
with skipped the oracle's bound (dropped mass sum p_t |v^_t| / sum p_t), and the logits are
those of the dense call bit for bit.  Queries are scaled up so that attention is peaked and
the threshold drops most positions.
"""
import numpy as np
import pytest
import torch

import kv_cache_vector_19_b300 as tq
from oracle import decode as odec

import parity as P

pytestmark = pytest.mark.gpu

CASES = [
    dict(d=128, b=3, G=4, path="auto"),    # e2m1 tcgen05
    dict(d=128, b=3, G=8, path="auto"),    # e2m1 tcgen05, four token-warp sets
    dict(d=128, b=2, G=16, path="auto"),   # f8f6f4 tcgen05
    dict(d=128, b=4, G=4, path="auto"),    # e2m1 tcgen05, two virtual KV heads per KV head
    dict(d=128, b=4, G=4, path="mma"),     # mma.sync
    dict(d=64, b=3, G=4, path="simt"),     # CUDA cores
]


def _check_case(run, G, H, T, theta, qscale, seed):
    d = run.d
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(1, H, T, d, generator=g).to(torch.bfloat16)
    v = torch.randn(1, H, T, d, generator=g).to(torch.bfloat16)
    run.quantize(k, v, [0])
    q = torch.randn(1, G * H, d, generator=g) * qscale
    dense, lg_d = run.decode(q, [T], logits=True)
    run.ctx.set_sparse_v(theta)
    sparse, lg_s = run.decode(q, [T], logits=True)
    run.ctx.set_sparse_v(0.0)
    assert run.status() == tq.TQ_OK
    assert torch.equal(lg_d, lg_s)
    dense, sparse = dense.cpu().numpy(), sparse.cpu().numpy()
    cache = run.cache_np()
    total_skipped = 0.0
    for h in range(H):
        tok = run.tokens(cache, 0, h, T)
        tk = dict(idx=tok["kidx"], n=tok["nk"].astype(np.float64), sigma=tok["sigma"],
                  gamma=tok["gamma"].astype(np.float64))
        tv = dict(idx=tok["vidx"], n=tok["nv"].astype(np.float64))
        for gh in range(G):
            hq = h * G + gh
            o, _, skipped = odec.attend_sparse_v(q[0, hq].double().numpy(), tk, tv, run.p.Pi, run.p.S,
                                                 run.p.cb_k, run.p.cb_v, theta)
            total_skipped += skipped
            assert np.linalg.norm(sparse[0, hq] - o) <= skipped + 2e-3 * np.linalg.norm(o), hq
            assert (np.linalg.norm(sparse[0, hq] - dense[0, hq])
                    <= skipped * (1 + 1e-3) + 2e-3 * np.linalg.norm(dense[0, hq])), hq
    return dense, sparse, total_skipped


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"d{c['d']}_b{c['b']}_G{c['G']}_{c['path']}")
def test_sparse_v_within_the_skipped_mass(case):
    d, b, G, H, T = case["d"], case["b"], case["G"], 2, 1500
    run = P.Run(d, b, 1, H, G * H, T, seed=3, decode_path=case["path"])
    dense, sparse, skipped = _check_case(run, G, H, T, theta=1e-3, qscale=4.0, seed=4)
    assert skipped > 0.0
    assert not np.array_equal(dense, sparse)   # the threshold took effect


def test_sparse_v_format_version_2():
    d, G, H, T = 128, 4, 1, 900
    ctx = tq.Context(d, key_bits=3, value_bits=4, qjl=True, seed=2)
    cache = ctx.alloc_cache(1, H, T)
    ws = ctx.alloc_workspace(1, G * H, H, T)
    g = torch.Generator().manual_seed(5)
    k = torch.randn(1, H, T, d, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(1, H, T, d, generator=g).to(torch.bfloat16).cuda()
    ctx.quantize_kv(k, v, torch.zeros(1, dtype=torch.int32, device="cuda"), cache, T)
    q = (torch.randn(1, G * H, d, generator=g) * 4).cuda()
    sl = torch.tensor([T], dtype=torch.int32, device="cuda")
    dense, sparse = torch.empty_like(q), torch.empty_like(q)
    ctx.attn_decode(q, cache, sl, H, T, dense, ws)
    ctx.set_sparse_v(1e-3)
    ctx.attn_decode(q, cache, sl, H, T, sparse, ws)
    assert ctx.device_status() == tq.TQ_OK
    diff = torch.linalg.norm(sparse - dense, dim=-1)
    assert torch.all(diff <= 0.05 * torch.linalg.norm(dense, dim=-1)) and torch.any(diff > 0)


def test_threshold_zero_is_dense_and_bad_thresholds_are_rejected():
    run = P.Run(128, 3, 1, 1, 4, 512, seed=1)
    g = torch.Generator().manual_seed(0)
    run.quantize(torch.randn(1, 1, 512, 128, generator=g).to(torch.bfloat16),
                 torch.randn(1, 1, 512, 128, generator=g).to(torch.bfloat16), [0])
    q = torch.randn(1, 4, 128, generator=g) * 4
    a, _ = run.decode(q, [512])
    run.ctx.set_sparse_v(0.0)
    b, _ = run.decode(q, [512])
    assert torch.equal(a, b)
    for bad in (-1e-3, 1.5, float("nan")):
        with pytest.raises(tq.TQError):
            run.ctx.set_sparse_v(bad)
