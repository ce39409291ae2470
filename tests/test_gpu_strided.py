"""GPU tests of strided quantize input (tq_quantize_kv_strided, tq_quantize_kv_paged_strided):
a prefill's projection output, token-major [batch][tokens][kv heads][d], goes into the
compressed cache without a transpose.  The strided call must write the same bytes as the
contiguous call on the transposed copy, for every quantizer kernel (tensor-core prefill,
few-token appends, CUDA cores at d = 64 / 256, format version 2), contiguous and paged.
"""
import numpy as np
import pytest
import torch

import kv_cache_vector_19_b300 as tq
from oracle import pagefmt

pytestmark = pytest.mark.gpu

CASES = [dict(d=128, bits=3, n=300), dict(d=128, bits=3, n=5), dict(d=128, bits=4, n=200),
         dict(d=64, bits=3, n=250), dict(d=256, bits=2, n=130), dict(d=128, kv=(3, 4, True), n=260),
         dict(d=64, kv=(4, 2, False), n=7)]


def _ctx(case):
    if "kv" in case:
        kb, vb, qjl = case["kv"]
        return tq.Context(case["d"], key_bits=kb, value_bits=vb, qjl=qjl, seed=3)
    return tq.Context(case["d"], case["bits"], seed=3)


def _token_major(B, N, H, d, seed):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(B, N, H, d, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(B, N, H, d, generator=g).to(torch.bfloat16).cuda()
    return k, v   # [B, N, H, d]; the quantizer's view is k.permute(0, 2, 1, 3)


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"d{c['d']}_{c.get('bits') or c.get('kv')}_n{c['n']}")
def test_strided_equals_contiguous(case):
    d, B, H, N, T = case["d"], 2, 3, case["n"], 640
    ctx = _ctx(case)
    k, v = _token_major(B, N, H, d, 1)
    kv_view, vv_view = k.permute(0, 2, 1, 3), v.permute(0, 2, 1, 3)
    start = torch.tensor([0, 37], dtype=torch.int32, device="cuda")
    c1, c2 = ctx.alloc_cache(B, H, T), ctx.alloc_cache(B, H, T)
    c1.zero_()
    c2.zero_()
    ctx.quantize_kv(kv_view.contiguous(), vv_view.contiguous(), start, c1, T)
    ctx.quantize_kv_strided(kv_view, vv_view, start, c2, T)
    assert ctx.device_status() == tq.TQ_OK
    assert torch.equal(c1, c2)


def test_paged_strided_equals_contiguous():
    d, B, H, N, max_blocks = 128, 2, 2, 300, 3
    ctx = tq.Context(d, 3, seed=4)
    k, v = _token_major(B, N, H, d, 2)
    kv_view, vv_view = k.permute(0, 2, 1, 3), v.permute(0, 2, 1, 3)
    start = torch.tensor([10, 0], dtype=torch.int32, device="cuda")
    n_blocks = B * max_blocks + 1
    table_np = np.random.default_rng(5).permutation(n_blocks)[:B * max_blocks].reshape(B, max_blocks)
    table = torch.from_numpy(table_np.astype(np.int32)).cuda()
    cache = ctx.alloc_cache(B, H, 128 * max_blocks)
    pool = ctx.alloc_pool(H, n_blocks)
    cache.zero_()
    pool.zero_()
    ctx.quantize_kv(kv_view.contiguous(), vv_view.contiguous(), start, cache, 128 * max_blocks)
    ctx.quantize_kv_paged_strided(kv_view, vv_view, start, pool, n_blocks, table)
    assert ctx.device_status() == tq.TQ_OK
    pb = tq.lib().tq_page_bytes(ctx._ctx)
    got = pagefmt.gather_paged(pool.cpu().numpy(), table_np, B, H, pb, max_blocks)
    assert np.array_equal(got, cache.cpu().numpy())


def test_bad_strides_are_rejected():
    ctx = tq.Context(128, 3)
    B, H, N, T = 1, 1, 16, 128
    k = torch.zeros(B, H, N, 128, dtype=torch.bfloat16, device="cuda")
    cache = ctx.alloc_cache(B, H, T)
    start = torch.zeros(B, dtype=torch.int32, device="cuda")
    lib = tq.lib()
    import ctypes
    for bad in ((N * 128, N * 128, 100, N * 128, N * 128, 128), (0, 0, -128, 0, 0, 128)):
        st = (ctypes.c_int64 * 6)(*bad)
        rc = lib.tq_quantize_kv_strided(ctx._ctx, k.data_ptr(), k.data_ptr(), st, B, H, N, start.data_ptr(),
                                        cache.data_ptr(), T, None)
        assert rc == tq.TQ_EINVAL
    rc = lib.tq_quantize_kv_strided(ctx._ctx, k.data_ptr(), k.data_ptr(), None, B, H, N, start.data_ptr(),
                                    cache.data_ptr(), T, None)
    assert rc == tq.TQ_EINVAL
